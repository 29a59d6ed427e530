// Fused FP8 quantization kernels (sm_103a): amax -> fp64 scale -> fp32 multiply -> clamp ->
// RNE saturating cast, one HBM read per element.
//
// Recipe: "FP8 Training: Quantization, Autograd, Torchao", section 2 "The quantization math".
// Fusion and layout design: "FP8 training on AMD GPUs with TorchTitan and TorchAO", "Triton
// Kernel Optimization": Level 1 (one kernel per quantization, no intermediates in HBM; the
// dual row/column-major output), Level 2 (column-wise scales with the output tile transposed
// on chip so the column-major writes are coalesced; single pass over the data), Level 3
// (relaxed atomics for the commutative amax reduction).
#include "common.cuh"
#include "internal.h"

namespace fp8lin {

template <int FMT>
struct FmtMax;
template <>
struct FmtMax<FP8_DT_E4M3> {
  static constexpr float v = kE4M3Max;
};
template <>
struct FmtMax<FP8_DT_E5M2> {
  static constexpr float v = kE5M2Max;
};

__host__ __device__ constexpr int64_t ceil_div64(int64_t a, int64_t b) { return (a + b - 1) / b; }
__host__ __device__ constexpr int64_t round_up64(int64_t a, int64_t b) { return ceil_div64(a, b) * b; }

// ==========================================================================================
// Rowwise: one scale per row. A team of TPR threads holds one row in registers (up to 8
// 16-byte vectors per thread), reduces |x| with packed-bf16 integer max, derives the scale in
// one thread, then casts from registers. Several teams share a CTA of at least 256 threads.
constexpr int kRowVPT = 8;

template <int FMT, int TPR>
__global__ void __launch_bounds__(TPR > 256 ? TPR : 256)
    quant_rows_kernel(const uint4* __restrict__ x, int64_t R, int nvec, uint2* __restrict__ q,
                      float* __restrict__ inv, const __grid_constant__ ScaleTab tab) {
  constexpr int CTA = TPR > 256 ? TPR : 256;
  constexpr int TEAMS = CTA / TPR;
  constexpr int WPT = TPR / 32;
  constexpr float FMAX = FmtMax<FMT>::v;
  __shared__ uint32_t red[CTA / 32];
  __shared__ float sc[TEAMS];
  const int team = threadIdx.x / TPR;
  const int t = threadIdx.x % TPR;
  const int warp = threadIdx.x / 32, lane = threadIdx.x % 32;

  for (int64_t base = (int64_t)blockIdx.x * TEAMS; base < R; base += (int64_t)gridDim.x * TEAMS) {
    const int64_t r = base + team;
    const bool active = r < R;
    const uint4* xr = x + r * nvec;
    uint4 v[kRowVPT];
    uint32_t acc = 0;
#pragma unroll
    for (int i = 0; i < kRowVPT; ++i) {
      const int c = t + i * TPR;
      if (active && c < nvec) {
        v[i] = ld_nc_v4(xr + c);
        acc = absmax_vec8(acc, v[i]);
      } else {
        v[i] = make_uint4(0, 0, 0, 0);
      }
    }
    const uint32_t m = __reduce_max_sync(0xffffffffu, absmax_fold(acc));
    if (lane == 0) red[warp] = m;
    __syncthreads();
    if (t == 0) {
      uint32_t mm = 0;
      for (int w = 0; w < WPT; ++w) mm = max(mm, red[team * WPT + w]);
      const Scale s = tab_scale(tab, mm);
      sc[team] = s.s32;
      if (active) inv[r] = s.inv32;
    }
    __syncthreads();
    const float s32 = sc[team];
    uint2* qr = q + r * nvec;
#pragma unroll
    for (int i = 0; i < kRowVPT; ++i) {
      const int c = t + i * TPR;
      if (active && c < nvec) qr[c] = quant_vec8<FMT>(v[i], s32, FMAX);
    }
  }
}

template <int FMT, int TPR>
static int run_rows(const void* x, int64_t R, int nvec, void* q, float* inv, const Ctx& c) {
  constexpr int CTA = TPR > 256 ? TPR : 256;
  constexpr int TEAMS = CTA / TPR;
  const int64_t need = ceil_div64(R, TEAMS);
  const int64_t cap = (int64_t)c.sm_count * (2048 / CTA);
  const int grid = (int)(need < cap ? need : cap);
  quant_rows_kernel<FMT, TPR><<<grid, CTA, 0, c.stream>>>(static_cast<const uint4*>(x), R, nvec,
                                                           static_cast<uint2*>(q), inv, scale_tab(FMT));
  return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

template <int FMT>
static int rows_dispatch(const void* x, int64_t R, int nvec, void* q, float* inv, const Ctx& c) {
  const int per = (nvec + kRowVPT - 1) / kRowVPT;  // threads needed at 8 vectors each
  if (per <= 32) return run_rows<FMT, 32>(x, R, nvec, q, inv, c);
  if (per <= 64) return run_rows<FMT, 64>(x, R, nvec, q, inv, c);
  if (per <= 128) return run_rows<FMT, 128>(x, R, nvec, q, inv, c);
  if (per <= 256) return run_rows<FMT, 256>(x, R, nvec, q, inv, c);
  if (per <= 512) return run_rows<FMT, 512>(x, R, nvec, q, inv, c);
  if (per <= 1024) return run_rows<FMT, 1024>(x, R, nvec, q, inv, c);
  return FP8_ERR_UNSUPPORTED;
}

int launch_quant_rows(const void* x, int64_t R, int64_t C, int fmt, void* q, float* inv, const Ctx& c) {
  if (R == 0) return FP8_OK;
  const int nvec = (int)(C / 8);
  return fmt == FP8_DT_E4M3 ? rows_dispatch<FP8_DT_E4M3>(x, R, nvec, q, inv, c)
                            : rows_dispatch<FP8_DT_E5M2>(x, R, nvec, q, inv, c);
}

// ==========================================================================================
// Tensorwise, phase 1: amax over the whole tensor. Grid-stride 16-byte loads, four in flight
// per thread, warp max by redux, one relaxed atomic max per CTA on the bf16 bit pattern.
__global__ void __launch_bounds__(256) amax_kernel(const uint4* __restrict__ x, int64_t nvec,
                                                   uint32_t* __restrict__ amax_ws) {
  __shared__ uint32_t red[8];
  uint32_t acc = 0;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < nvec; i += 4 * stride) {
    const uint4 a = ld_nc_v4(x + i), b = ld_nc_v4(x + i + stride);
    const uint4 d = ld_nc_v4(x + i + 2 * stride), e = ld_nc_v4(x + i + 3 * stride);
    acc = absmax_vec8(acc, a);
    acc = absmax_vec8(acc, b);
    acc = absmax_vec8(acc, d);
    acc = absmax_vec8(acc, e);
  }
  for (; i < nvec; i += stride) acc = absmax_vec8(acc, ld_nc_v4(x + i));
  const uint32_t m = __reduce_max_sync(0xffffffffu, absmax_fold(acc));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t mm = 0;
    for (int w = 0; w < 8; ++w) mm = max(mm, red[w]);
    red_max_relaxed(amax_ws, mm);
  }
}

// Tensorwise, phase 2: cast with the one scale; row-major output from registers and/or the
// column-major output through a transposed 64 x 128 tile in shared memory (dual output from
// one read). Tile: 128 rows x 64 columns.
constexpr int kTcRows = 128, kTcCols = 64, kTcPitch = 132;  // pitch: 33 words, conflict-light

template <int FMT>
__global__ void __launch_bounds__(256) quant_tensor_cast_kernel(const uint16_t* __restrict__ x, int64_t R,
                                                                int64_t C, const uint32_t* __restrict__ amax_ws,
                                                                uint8_t* __restrict__ q, uint8_t* __restrict__ qt,
                                                                float* __restrict__ inv,
                                                                const __grid_constant__ ScaleTab tab) {
  constexpr float FMAX = FmtMax<FMT>::v;
  __shared__ float s_sc;
  __shared__ __align__(16) uint8_t T[kTcCols * kTcPitch];
  if (threadIdx.x == 0) {
    const Scale s = tab_scale(tab, *amax_ws);
    s_sc = s.s32;
    if (blockIdx.x == 0 && blockIdx.y == 0) *inv = s.inv32;
  }
  __syncthreads();
  const float s32 = s_sc;
  const int64_t r0 = (int64_t)blockIdx.y * kTcRows, c0 = (int64_t)blockIdx.x * kTcCols;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int v = threadIdx.x + 256 * i;  // 128 rows x 8 vectors
    const int rr = v >> 3, cv = v & 7;
    const int64_t r = r0 + rr, col = c0 + cv * 8;
    uint2 o = make_uint2(0, 0);
    if (r < R && col < C) {
      o = quant_vec8<FMT>(ld_nc_v4(x + r * C + col), s32, FMAX);
      if (q) *reinterpret_cast<uint2*>(q + r * C + col) = o;
    }
    if (qt) {
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t w = j < 4 ? o.x : o.y;
        T[(cv * 8 + j) * kTcPitch + rr] = (uint8_t)(w >> (8 * (j & 3)));
      }
    }
  }
  if (!qt) return;
  __syncthreads();
  for (int i = threadIdx.x; i < kTcCols * (kTcRows / 16); i += 256) {
    const int cl = i >> 3, k = i & 7;
    const int64_t col = c0 + cl, r = r0 + 16 * k;
    if (col < C && r < R) {  // R % 16 == 0: the 16-byte chunk is all in range
      const uint32_t* src = reinterpret_cast<const uint32_t*>(T + cl * kTcPitch + 16 * k);
      *reinterpret_cast<uint4*>(qt + col * R + r) = make_uint4(src[0], src[1], src[2], src[3]);
    }
  }
}

int launch_quant_tensor(const void* x, int64_t R, int64_t C, int fmt, void* q, void* qt, float* inv,
                        uint32_t* amax_ws, const Ctx& c) {
  if (cudaMemsetAsync(amax_ws, 0, sizeof(uint32_t), c.stream) != cudaSuccess) return FP8_ERR_CUDA;
  const int64_t nvec = R * C / 8;
  if (nvec > 0) {
    const int64_t need = ceil_div64(nvec, 256 * 4);
    const int64_t cap = (int64_t)c.sm_count * 8;
    amax_kernel<<<(int)(need < cap ? need : cap), 256, 0, c.stream>>>(static_cast<const uint4*>(x), nvec, amax_ws);
    if (cudaGetLastError() != cudaSuccess) return FP8_ERR_CUDA;
  }
  dim3 grid((unsigned)ceil_div64(C, kTcCols), (unsigned)ceil_div64(R, kTcRows));
  if (grid.x == 0 || grid.y == 0) grid = dim3(1, 1);
  if (fmt == FP8_DT_E4M3)
    quant_tensor_cast_kernel<FP8_DT_E4M3><<<grid, 256, 0, c.stream>>>(
        static_cast<const uint16_t*>(x), R, C, amax_ws, static_cast<uint8_t*>(q), static_cast<uint8_t*>(qt), inv,
        scale_tab(fmt));
  else
    quant_tensor_cast_kernel<FP8_DT_E5M2><<<grid, 256, 0, c.stream>>>(
        static_cast<const uint16_t*>(x), R, C, amax_ws, static_cast<uint8_t*>(q), static_cast<uint8_t*>(qt), inv,
        scale_tab(fmt));
  return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

// ==========================================================================================
// Columnwise with column-major output: three stream-ordered kernels over (row group, 64-column
// strip, row tile) work units, which never straddle a group (segment) boundary.
//   1. colmax:   coalesced 16-byte loads (a warp reads four whole 128-byte row segments per
//                instruction); per-column |x| maxima folded in registers, shuffles and shared
//                memory; one relaxed atomic max per column per tile into a per-column scratch
//                word (the bf16 bit pattern of the maximum).
//   2. colscale: one thread per (group, column): the scale step; the fp32 scale replaces the
//                amax word in the scratch and the inverse scale goes to the output.
//   3. colcast:  the same loads, the fp32 multiply and the cast in registers; each 4-row column
//                pack becomes one 32-bit word of FP8 codes, written into a transposed tile in
//                shared memory (64 columns x 128 rows per box, TMA 128-byte swizzle; a thread's 8
//                columns are rotated by its chunk index so the stores are conflict-free); TMA
//                bulk-tensor stores write whole column-major boxes.
// The cast pass re-reads the input. Work units walk the strips of a row tile first, so the
// re-read mostly hits the 129 MB L2 when the tensor fits in it; larger tensors read it twice.
constexpr int kColThreads = 256;
constexpr int kColNB = 4;                  // 128-row blocks per work unit (512 rows)
constexpr int kColTile = 128 * kColNB;

struct ColParams {
  const uint16_t* x;
  int64_t rows_total;
  int64_t C;
  int64_t n_groups;
  int64_t group_rows;  // dense modes
  const int32_t* ends; // segment mode
  uint32_t* scratch;   // [n_groups, C]: amax bits, then fp32 scales
  float* inv;
  int32_t* status;
  int64_t n_strips;
  int mode;            // 0: 2-D [C, R] output; 1: batched [B, C, R]; 2: segments [C, P]
};

struct ColUnit {
  int64_t g, g0, n, pstart, write_end, rt;  // group, first row, rows, padded start, rows written, tile start
  int64_t c0;                                // first column of the strip
};

// Units: dense modes have n_groups * tiles * strips; segments a prefix over the segments.
// upre[e] = first unit of segment e; ppre[e] = padded start of segment e.
FP8_DEVI ColUnit col_unit(const ColParams& p, int64_t unit, const int32_t* upre, const int32_t* ppre) {
  ColUnit u;
  int64_t local;
  if (p.mode == 2) {
    int lo = 0, hi = (int)p.n_groups - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (upre[mid] <= unit) lo = mid;
      else hi = mid - 1;
    }
    u.g = lo;
    local = unit - upre[lo];
    u.g0 = lo ? p.ends[lo - 1] : 0;
    u.n = p.ends[lo] - u.g0;
    u.pstart = ppre[lo];
    u.write_end = round_up64(u.n, 128);
  } else {
    const int64_t tiles = ceil_div64(p.group_rows, kColTile);
    u.g = unit / (tiles * p.n_strips);
    local = unit % (tiles * p.n_strips);
    u.g0 = u.g * p.group_rows;
    u.n = p.group_rows;
    u.pstart = 0;
    u.write_end = u.n;
  }
  u.rt = (local / p.n_strips) * kColTile;
  u.c0 = (local % p.n_strips) * 64;
  return u;
}

// Validates the offsets (segment mode) and builds the unit / padded-start prefixes in shared
// memory; returns the number of units, or -1 after reporting bad offsets.
FP8_DEVI int64_t col_setup(const ColParams& p, int32_t* upre, int32_t* ppre) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (p.mode != 2) return p.n_groups * ceil_div64(p.group_rows, kColTile) * p.n_strips;
  int bad = 0;
  for (int64_t e = tid; e < p.n_groups; e += kColThreads) {
    const int64_t cur = p.ends[e], prev = e ? p.ends[e - 1] : 0;
    if (cur < prev || (e == p.n_groups - 1 && cur != p.rows_total)) bad = 1;
  }
  bad = __syncthreads_or(bad);
  if (bad) {
    if (blockIdx.x == 0 && tid == 0) set_status(p.status, FP8_DEV_BAD_OFFSETS);
    return -1;
  }
  if (warp == 0) {
    int cu = 0, cp = 0;
    for (int64_t base = 0; base < p.n_groups; base += 32) {
      const int64_t i = base + lane;
      int vu = 0, vp = 0;
      if (i < p.n_groups) {
        const int64_t n = p.ends[i] - (i ? p.ends[i - 1] : 0);
        vu = (int)(ceil_div64(n, kColTile) * p.n_strips);
        vp = (int)round_up64(n, 128);
      }
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int yu = __shfl_up_sync(0xffffffffu, vu, o);
        const int yp = __shfl_up_sync(0xffffffffu, vp, o);
        if (lane >= o) {
          vu += yu;
          vp += yp;
        }
      }
      if (i < p.n_groups) {
        upre[i + 1] = vu + cu;
        ppre[i + 1] = vp + cp;
      }
      cu += __shfl_sync(0xffffffffu, vu, 31);
      cp += __shfl_sync(0xffffffffu, vp, 31);
    }
    if (lane == 0) {
      upre[0] = 0;
      ppre[0] = 0;
    }
  }
  __syncthreads();
  return upre[p.n_groups];
}

// This thread's 4 rows x 8 columns of every 128-row block of the unit (zeros outside the
// group and the matrix): rows 128 b + 16 warp + 4 rq + jj, columns c0 + 8 ch .. + 7.
FP8_DEVI void col_load(const ColParams& p, const ColUnit& u, int warp, int ch, int rq, uint4 (&v)[kColNB][4]) {
  int64_t valid = u.n - u.rt;
  valid = valid < 0 ? 0 : (valid < kColTile ? valid : kColTile);
  const bool ch_ok = u.c0 + ch * 8 < p.C;
  const uint16_t* base = p.x + (u.g0 + u.rt) * p.C + u.c0 + ch * 8;
#pragma unroll
  for (int b = 0; b < kColNB; ++b)
#pragma unroll
    for (int jj = 0; jj < 4; ++jj) {
      const int row = 128 * b + 16 * warp + 4 * rq + jj;
      v[b][jj] = (ch_ok && row < valid) ? ld_nc_v4(base + (int64_t)row * p.C) : make_uint4(0, 0, 0, 0);
    }
}

__global__ void __launch_bounds__(kColThreads) colmax_kernel(const ColParams p) {
  __shared__ uint32_t red[8][8][4];
  extern __shared__ int32_t pre[];
  int32_t* upre = pre;
  int32_t* ppre = pre + (p.n_groups + 1);
  const int64_t total = col_setup(p, upre, ppre);
  if (total < 0) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ch = lane & 7, rq = lane >> 3;
  for (int64_t unit = blockIdx.x; unit < total; unit += gridDim.x) {
    const ColUnit u = col_unit(p, unit, upre, ppre);
    uint4 v[kColNB][4];
    col_load(p, u, warp, ch, rq, v);
    uint32_t m4[4] = {0, 0, 0, 0};
#pragma unroll
    for (int b = 0; b < kColNB; ++b)
#pragma unroll
      for (int jj = 0; jj < 4; ++jj) {
        m4[0] = absmax2(m4[0], v[b][jj].x);
        m4[1] = absmax2(m4[1], v[b][jj].y);
        m4[2] = absmax2(m4[2], v[b][jj].z);
        m4[3] = absmax2(m4[3], v[b][jj].w);
      }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      m4[i] = __vmaxu2(m4[i], __shfl_xor_sync(0xffffffffu, m4[i], 8));
      m4[i] = __vmaxu2(m4[i], __shfl_xor_sync(0xffffffffu, m4[i], 16));
    }
    if (rq == 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i) red[warp][ch][i] = m4[i];
    }
    __syncthreads();
    if (tid < 32) {  // pair t = columns 2t, 2t+1 = chunk t/4, word t%4
      uint32_t m = 0;
      for (int w = 0; w < 8; ++w) m = __vmaxu2(m, red[w][tid >> 2][tid & 3]);
      const int64_t col = u.c0 + 2 * tid;
      uint32_t* sc = p.scratch + u.g * p.C + col;
      if (col < p.C && (m & 0xFFFFu)) red_max_relaxed(sc, m & 0xFFFFu);
      if (col + 1 < p.C && (m >> 16)) red_max_relaxed(sc + 1, m >> 16);
    }
    __syncthreads();
  }
}

template <int FMT>
__global__ void __launch_bounds__(256) colscale_kernel(uint32_t* __restrict__ scratch, float* __restrict__ inv,
                                                       int64_t n, const __grid_constant__ ScaleTab tab) {
  const int64_t i = (int64_t)blockIdx.x * 256 + threadIdx.x;
  if (i >= n) return;
  const Scale s = tab_scale(tab, scratch[i]);
  reinterpret_cast<float*>(scratch)[i] = s.s32;
  inv[i] = s.inv32;
}

// Column j (0..7) of a 16-byte vector of 8 bf16, as fp32.
FP8_DEVI float col_of(const uint4& v, int j) {
  const uint32_t w = j < 2 ? v.x : (j < 4 ? v.y : (j < 6 ? v.z : v.w));
  return (j & 1) ? __uint_as_float(w & 0xFFFF0000u) : __uint_as_float(w << 16);
}

template <int FMT>
__global__ void __launch_bounds__(kColThreads) colcast_kernel(const __grid_constant__ CUtensorMap tm_out,
                                                              const ColParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* T = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  int32_t* upre = reinterpret_cast<int32_t*>(T + kColNB * 8192);
  int32_t* ppre = upre + (p.n_groups + 1);
  const int64_t total = col_setup(p, upre, ppre);
  if (total < 0) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ch = lane & 7, rq = lane >> 3;
  if (tid == 0) tma_prefetch_desc(&tm_out);
  const float* scales = reinterpret_cast<const float*>(p.scratch);
  for (int64_t unit = blockIdx.x; unit < total; unit += gridDim.x) {
    const ColUnit u = col_unit(p, unit, upre, ppre);
    uint4 v[kColNB][4];
    col_load(p, u, warp, ch, rq, v);
    float sc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) {
      const int64_t col = u.c0 + ch * 8 + j;
      sc[j] = col < p.C ? scales[u.g * p.C + col] : 0.0f;
    }
    int64_t wrows = u.write_end - u.rt;
    wrows = wrows < 0 ? 0 : (wrows < kColTile ? wrows : kColTile);
    const int nbox = (int)ceil_div64(wrows, 128);
    if (tid == 0) bulk_wait_read_all();  // the previous unit's stores have read the tile
    __syncthreads();
#pragma unroll
    for (int b = 0; b < kColNB; ++b) {
      if (b < nbox) {
        uint32_t o[8];
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const float s = sc[j];
          o[j] = cvt_fp8x2<FMT>(__fmul_rn(col_of(v[b][0], j), s), __fmul_rn(col_of(v[b][1], j), s)) |
                 (cvt_fp8x2<FMT>(__fmul_rn(col_of(v[b][2], j), s), __fmul_rn(col_of(v[b][3], j), s)) << 16);
        }
        // rotate by ch so that the lanes of a warp write 8 different column residues at once
#pragma unroll
        for (int sh = 1; sh < 8; sh <<= 1) {
          const bool rot = (ch & sh) != 0;
          uint32_t t[8];
#pragma unroll
          for (int j = 0; j < 8; ++j) t[j] = rot ? o[(j + sh) & 7] : o[j];
#pragma unroll
          for (int j = 0; j < 8; ++j) o[j] = t[j];
        }
        uint8_t* box = T + b * 8192;
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const int cl = ch * 8 + ((j + ch) & 7);
          *reinterpret_cast<uint32_t*>(box + cl * 128 + (((warp ^ cl) & 7) << 4) + rq * 4) = o[j];
        }
      }
    }
    fence_proxy_async_smem();
    __syncthreads();
    if (tid == 0) {
      for (int b = 0; b < nbox; ++b) {
        const int32_t xo = (int32_t)(u.pstart + u.rt + 128 * b);
        if (p.mode == 1)
          tma_store_3d(&tm_out, T + b * 8192, xo, (int32_t)u.c0, (int32_t)u.g);
        else
          tma_store_2d(&tm_out, T + b * 8192, xo, (int32_t)u.c0);
      }
      bulk_commit();
    }
  }
  if (tid == 0) bulk_wait_all();
}

int launch_quant_cols(const void* x, int64_t rows_total, int64_t C, int64_t n_groups, int64_t group_rows,
                      const int32_t* ends, int fmt, void* out_t, int64_t ld_out, float* inv, uint32_t* scratch,
                      const Ctx& c) {
  if (n_groups == 0 || C == 0) return FP8_OK;
  if (ends && n_groups > 6000) return FP8_ERR_UNSUPPORTED;  // prefix arrays live in shared memory
  ColParams p = {};
  p.x = static_cast<const uint16_t*>(x);
  p.rows_total = rows_total;
  p.C = C;
  p.n_groups = n_groups;
  p.group_rows = group_rows;
  p.ends = ends;
  p.scratch = scratch;
  p.inv = inv;
  p.status = c.status;
  p.n_strips = ceil_div64(C, 64);
  p.mode = ends ? 2 : (n_groups > 1 ? 1 : 0);

  CUtensorMap tout;
  int rc;
  if (p.mode == 1) {
    const uint64_t dims[3] = {(uint64_t)group_rows, (uint64_t)C, (uint64_t)n_groups};
    const uint64_t strides[2] = {(uint64_t)group_rows, (uint64_t)(C * group_rows)};
    const uint32_t box[3] = {128, 64, 1};
    rc = make_tmap(&tout, out_t, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  } else {
    const uint64_t inner = p.mode == 2 ? (uint64_t)ld_out : (uint64_t)group_rows;
    const uint64_t dims[2] = {inner, (uint64_t)C};
    const uint64_t strides[1] = {(uint64_t)ld_out};
    const uint32_t box[2] = {128, 64};
    rc = make_tmap(&tout, out_t, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  }
  if (rc != FP8_OK) return rc;

  const int64_t n_scales = n_groups * C;
  if (cudaMemsetAsync(scratch, 0, (size_t)n_scales * 4, c.stream) != cudaSuccess) return FP8_ERR_CUDA;
  // units: exact for dense modes; for segments an upper bound (each segment adds at most one
  // partial tile) -- the kernels compute the exact count from the offsets
  const int64_t units = p.mode == 2 ? (ceil_div64(rows_total, kColTile) + n_groups) * p.n_strips
                                    : n_groups * ceil_div64(group_rows, kColTile) * p.n_strips;
  const size_t pre_bytes = p.mode == 2 ? 8 * (size_t)(n_groups + 1) : 0;
  if (units > 0) {
    const int64_t cap_a = (int64_t)c.sm_count * 3;
    colmax_kernel<<<(unsigned)(units < cap_a ? units : cap_a), kColThreads, pre_bytes, c.stream>>>(p);
    if (cudaGetLastError() != cudaSuccess) return FP8_ERR_CUDA;
  }
  const unsigned gs = (unsigned)ceil_div64(n_scales, 256);
  if (fmt == FP8_DT_E4M3)
    colscale_kernel<FP8_DT_E4M3><<<gs, 256, 0, c.stream>>>(scratch, inv, n_scales, scale_tab(FP8_DT_E4M3));
  else
    colscale_kernel<FP8_DT_E5M2><<<gs, 256, 0, c.stream>>>(scratch, inv, n_scales, scale_tab(FP8_DT_E5M2));
  if (cudaGetLastError() != cudaSuccess) return FP8_ERR_CUDA;
  if (units > 0) {
    auto kern = fmt == FP8_DT_E4M3 ? colcast_kernel<FP8_DT_E4M3> : colcast_kernel<FP8_DT_E5M2>;
    const size_t smem = 1024 + kColNB * 8192 + pre_bytes;
    if (smem > 48 * 1024 && cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return FP8_ERR_CUDA;
    const int64_t cap_b = (int64_t)c.sm_count * 3;
    kern<<<(unsigned)(units < cap_b ? units : cap_b), kColThreads, smem, c.stream>>>(tout, p);
    if (cudaGetLastError() != cudaSuccess) return FP8_ERR_CUDA;
  }
  return FP8_OK;
}

}  // namespace fp8lin

namespace fp8lin {

int launch_quant_tensor_cast(const void* x, int64_t R, int64_t C, int fmt, void* q, void* qt, float* inv,
                             const uint32_t* amax_word, const Ctx& c) {
  dim3 grid((unsigned)ceil_div64(C, kTcCols), (unsigned)ceil_div64(R, kTcRows));
  if (grid.x == 0 || grid.y == 0) grid = dim3(1, 1);
  if (fmt == FP8_DT_E4M3)
    quant_tensor_cast_kernel<FP8_DT_E4M3><<<grid, 256, 0, c.stream>>>(
        static_cast<const uint16_t*>(x), R, C, amax_word, static_cast<uint8_t*>(q), static_cast<uint8_t*>(qt), inv,
        scale_tab(fmt));
  else
    quant_tensor_cast_kernel<FP8_DT_E5M2><<<grid, 256, 0, c.stream>>>(
        static_cast<const uint16_t*>(x), R, C, amax_word, static_cast<uint8_t*>(q), static_cast<uint8_t*>(qt), inv,
        scale_tab(fmt));
  return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

}  // namespace fp8lin
