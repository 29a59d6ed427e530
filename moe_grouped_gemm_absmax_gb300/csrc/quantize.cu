// Fused FP8 quantization kernels (sm_103a): amax -> fp64 scale -> fp32 multiply -> clamp ->
// RNE saturating cast, with no intermediate tensor in HBM.
//
// Recipe: "FP8 Training: Quantization, Autograd, Torchao", section 2 "The quantization math".
// Fusion and layout design: "FP8 training on AMD GPUs with TorchTitan and TorchAO", "Triton
// Kernel Optimization": Level 1 (one kernel per quantization, no intermediates in HBM; the
// dual row/column-major output), Level 2 (column-wise scales with the output tile transposed
// on chip so the column-major writes are coalesced), Level 3 (relaxed atomics for the
// commutative amax reduction).
//
// Reads of the bf16 input: the row-wise kernel reads each element once (a row's amax and its
// cast come from the same registers). Tensor and column granularity need the amax of a whole
// tensor or column before the first element can be cast, so they run an amax pass and a cast
// pass; the cast pass re-reads the input (from L2 where it still holds it).
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

// Rowwise for rows of up to 16384 elements: a team of WPR warps (1, 2 or 4) per row. A team issues
// all of its row's 16-byte loads at once (up to 16 per lane), folds |x|, combines its warps'
// maxima through shared memory behind a barrier of the team alone (none for one warp), takes the
// scale from the table (one row per team: every lane looks up the same entry), casts from
// registers and stores 8 codes per lane and vector. Persistent teams walk the rows with a grid
// stride, so at any time some teams load while others cast and store.
constexpr int kRowWarpVPL = 16;
template <int FMT, int WPR>
__global__ void __launch_bounds__(256) quant_rows_warp_kernel(const uint4* __restrict__ x, int64_t R, int nvec,
                                                              uint2* __restrict__ q, float* __restrict__ inv,
                                                              const __grid_constant__ ScaleTab tab) {
  constexpr int TPR = 32 * WPR;
  __shared__ uint32_t red[2][8];
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
  const int team = warp / WPR, t = threadIdx.x % TPR;
  const int64_t team0 = (int64_t)blockIdx.x * (8 / WPR) + team;
  const int64_t nteams = (int64_t)gridDim.x * (8 / WPR);
  int par = 0;
  for (int64_t r = team0; r < R; r += nteams) {
    const uint4* xr = x + r * nvec;
    uint4 v[kRowWarpVPL];
    uint32_t acc = 0;
#pragma unroll
    for (int i = 0; i < kRowWarpVPL; ++i) {
      const int c = t + TPR * i;
      v[i] = c < nvec ? ld_nc_v4(xr + c) : make_uint4(0, 0, 0, 0);
    }
#pragma unroll
    for (int i = 0; i < kRowWarpVPL; ++i) acc = absmax_vec8(acc, v[i]);
    uint32_t m = __reduce_max_sync(0xffffffffu, absmax_fold(acc));
    if (WPR > 1) {
      if (lane == 0) red[par][warp] = m;
      named_bar_sync(1 + team, TPR);
#pragma unroll
      for (int w = 0; w < WPR; ++w) m = max(m, red[par][team * WPR + w]);
      par ^= 1;
    }
    const Scale sc = tab_scale(tab, m);
    if (t == 0) inv[r] = sc.inv32;
    uint2* qr = q + r * nvec;
    const float2 s2 = make_float2(sc.s32, sc.s32);
#pragma unroll
    for (int i = 0; i < kRowWarpVPL; ++i) {
      const int c = t + TPR * i;
      if (c < nvec) {
        const uint4 d = v[i];
        float2 a = fmul2_rn(make_float2(__uint_as_float(d.x << 16), __uint_as_float(d.x & 0xFFFF0000u)), s2);
        float2 b = fmul2_rn(make_float2(__uint_as_float(d.y << 16), __uint_as_float(d.y & 0xFFFF0000u)), s2);
        uint2 o;
        o.x = cvt_fp8x2<FMT>(a.x, a.y) | (cvt_fp8x2<FMT>(b.x, b.y) << 16);
        a = fmul2_rn(make_float2(__uint_as_float(d.z << 16), __uint_as_float(d.z & 0xFFFF0000u)), s2);
        b = fmul2_rn(make_float2(__uint_as_float(d.w << 16), __uint_as_float(d.w & 0xFFFF0000u)), s2);
        o.y = cvt_fp8x2<FMT>(a.x, a.y) | (cvt_fp8x2<FMT>(b.x, b.y) << 16);
        qr[c] = o;
      }
    }
  }
}

template <int FMT, int WPR>
static int run_rows_warp(const void* x, int64_t R, int nvec, void* q, float* inv, const Ctx& c) {
  auto kern = quant_rows_warp_kernel<FMT, WPR>;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, 256, 0) != cudaSuccess || per_sm < 1) per_sm = 1;
  // as many teams as fit at once, but no more than the rows, with the rows spread evenly
  const int64_t slots = (int64_t)c.sm_count * per_sm * (8 / WPR);
  const int64_t waves = ceil_div64(R, slots);
  const int64_t teams = ceil_div64(R, waves);
  kern<<<(unsigned)ceil_div64(teams, 8 / WPR), 256, 0, c.stream>>>(static_cast<const uint4*>(x), R, nvec,
                                                                    static_cast<uint2*>(q), inv, scale_tab(FMT));
  return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

template <int FMT>
static int rows_warp_dispatch(const void* x, int64_t R, int nvec, void* q, float* inv, const Ctx& c) {
  if (nvec <= 32 * kRowWarpVPL) return run_rows_warp<FMT, 1>(x, R, nvec, q, inv, c);
  if (nvec <= 64 * kRowWarpVPL) return run_rows_warp<FMT, 2>(x, R, nvec, q, inv, c);
  return run_rows_warp<FMT, 4>(x, R, nvec, q, inv, c);
}

int launch_quant_rows(const void* x, int64_t R, int64_t C, int fmt, void* q, float* inv, const Ctx& c) {
  if (R == 0) return FP8_OK;
  const int nvec = (int)(C / 8);
  if (nvec >= 64 && nvec <= 128 * kRowWarpVPL)
    return fmt == FP8_DT_E4M3 ? rows_warp_dispatch<FP8_DT_E4M3>(x, R, nvec, q, inv, c)
                              : rows_warp_dispatch<FP8_DT_E5M2>(x, R, nvec, q, inv, c);
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
  const uint64_t keep = l2_evict_last();  // the cast pass reads the tensor again
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  for (; i + 3 * stride < nvec; i += 4 * stride) {
    const uint4 a = ld_nc_v4_hint(x + i, keep), b = ld_nc_v4_hint(x + i + stride, keep);
    const uint4 d = ld_nc_v4_hint(x + i + 2 * stride, keep), e = ld_nc_v4_hint(x + i + 3 * stride, keep);
    acc = absmax_vec8(acc, a);
    acc = absmax_vec8(acc, b);
    acc = absmax_vec8(acc, d);
    acc = absmax_vec8(acc, e);
  }
  for (; i < nvec; i += stride) acc = absmax_vec8(acc, ld_nc_v4_hint(x + i, keep));
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
                                                                int amax_shift, uint8_t* __restrict__ q,
                                                                uint8_t* __restrict__ qt, float* __restrict__ inv,
                                                                const __grid_constant__ ScaleTab tab) {
  constexpr float FMAX = FmtMax<FMT>::v;
  __shared__ float s_sc;
  __shared__ __align__(16) uint8_t T[kTcCols * kTcPitch];
  if (threadIdx.x == 0) {
    const Scale s = tab_scale(tab, *amax_ws >> amax_shift);  // bf16 pattern, or an fp32 word holding one
    s_sc = s.s32;
    if (blockIdx.x == 0 && blockIdx.y == 0) *inv = s.inv32;
  }
  __syncthreads();
  const float s32 = s_sc;
  // the input's last use and output nothing re-reads soon: neither should push out of L2 the
  // input lines other tiles still have to read
  const uint64_t last = l2_evict_first();
  const int64_t r0 = (int64_t)blockIdx.y * kTcRows, c0 = (int64_t)blockIdx.x * kTcCols;
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int v = threadIdx.x + 256 * i;  // 128 rows x 8 vectors
    const int rr = v >> 3, cv = v & 7;
    const int64_t r = r0 + rr, col = c0 + cv * 8;
    uint2 o = make_uint2(0, 0);
    if (r < R && col < C) {
      o = quant_vec8<FMT>(ld_nc_v4_hint(x + r * C + col, last), s32, FMAX);
      if (q) st_v2_hint(q + r * C + col, o, last);
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
      st_v4_hint(qt + col * R + r, make_uint4(src[0], src[1], src[2], src[3]), last);
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
        static_cast<const uint16_t*>(x), R, C, amax_ws, 0, static_cast<uint8_t*>(q), static_cast<uint8_t*>(qt), inv,
        scale_tab(fmt));
  else
    quant_tensor_cast_kernel<FP8_DT_E5M2><<<grid, 256, 0, c.stream>>>(
        static_cast<const uint16_t*>(x), R, C, amax_ws, 0, static_cast<uint8_t*>(q), static_cast<uint8_t*>(qt), inv,
        scale_tab(fmt));
  return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

// ==========================================================================================
// Columnwise with column-major output: two streaming passes of one warp-specialized kernel
// (one CTA per SM) over work units, a unit being a 256-row x 64-column tile of one row group
// (segment); units never straddle a group boundary and are ordered group, row tile, strip, and
// dealt to the CTAs round-robin, so that at any time the CTAs read neighbouring strips of the
// same rows (long row segments: DRAM pages and L2 lines are shared). In every CTA:
//   producer warp: streams its units' tiles into a shared-memory ring with TMA (128-byte
//              swizzle), 6 stages in pass 1 and 5 in pass 2: 160-192 KB of loads in flight per SM;
//   8 consumer warps read each tile from the ring (conflict-free through the swizzle).
//   pass 1 (max): a tile's per-column |x| maxima are folded by shuffles and shared memory into
//              one relaxed atomic max per column on a per-(group, column) scratch word (the bf16
//              bit pattern of the maximum).
//   pass 2 (cast): an amax warp beside the producer copies each tile's 64 column maxima from the
//              scratch words into the stage asynchronously (the copies themselves arrive on the
//              stage's barrier); one warp doing the scale step for the consumers ran at ~1 us per
//              tile, twice the time of the loads.
//              Each consumer warp then owns 32 rows of the tile: a lane takes a column pair, takes
//              their scales from the table in shared memory (the strip's first tile also writes
//              the inverse scales), multiplies in fp32 and casts in registers, writes its two
//              32-code rows of the transposed box (64 columns x 32 rows) in the warp's own
//              staging buffer, and the warp's elected lane stores the box by TMA (two alternating
//              buffers per warp), so the warps never wait on one another. Pass 2 walks the unit order backwards, so
//              its first reads are the tiles pass 1 read last, still in L2.
// The passes are stream-ordered launches: no CTA waits on another.
constexpr int kColThreads = 256;
constexpr int kColNB = 2;                  // 128-row blocks per work unit (256 rows)
constexpr int kColTile = 128 * kColNB;
constexpr int kColStagesMax = 6;  // ring stages: 6 in pass 1, 5 in pass 2 (its staging boxes take the rest)
template <bool CAST>
constexpr int col_stages() { return CAST ? 5 : 6; }
constexpr int kColStageBytes = kColTile * 128;         // 256 rows x 64 bf16
constexpr int kColOutBytes = (kColTile / 128) * 8192;  // 64 columns x 256 rows of codes
constexpr int kColWarpBox = 64 * 32;                   // pass 2: one warp's 64 columns x 32 rows of codes
constexpr int kColConsumerWarps = kColThreads / 32;    // 8
static_assert(2 * kColOutBytes == kColConsumerWarps * 2 * kColWarpBox, "pass-2 staging: two boxes per warp");
constexpr uint64_t kColDrainNs = 2000000000ull;        // fixed bound: loads in flight before exit

struct ColParams {
  const uint16_t* x;
  int64_t rows_total;
  int64_t C;
  int64_t n_groups;
  int64_t group_rows;  // dense modes
  const int32_t* ends; // segment mode
  uint32_t* scratch;   // [n_groups, C]: amax bits
  int amax_shift;      // pass 2 reads scratch >> amax_shift: 0 for bf16 patterns, 16 for fp32 words
  float* inv;
  int32_t* status;
  int64_t n_strips;
  uint64_t wait_ns;
  int mode;            // 0: 2-D [C, R] output; 1: batched [B, C, R]; 2: segments [C, P]
};

struct ColUnit {
  int64_t g, g0, n, pstart, write_end, rt;  // group, first row, rows, padded start, rows written, tile start
  int64_t strip, c0;                         // strip and its first column
};

// Unit i: group, row tile, strip. Segment mode: upre[e] = first unit of segment e, ppre[e] = its
// padded start, ppre[n_groups + 1 + e] = its first row (shared memory only: no global load on the
// producer's path).
// Unit indices fit 32 bits (the host checks), so the divisions are 32-bit.
FP8_DEVI ColUnit col_unit(const ColParams& p, int64_t i, const int32_t* upre, const int32_t* ppre) {
  ColUnit u;
  uint32_t local;
  if (p.mode == 2) {
    int lo = 0, hi = (int)p.n_groups - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (upre[mid] <= i) lo = mid;
      else hi = mid - 1;
    }
    u.g = lo;
    local = (uint32_t)(i - upre[lo]);
    const int32_t* rpre = ppre + (p.n_groups + 1);
    u.g0 = rpre[lo];
    u.n = rpre[lo + 1] - u.g0;
    u.pstart = ppre[lo];
    u.write_end = round_up64(u.n, 128);
  } else {
    const uint32_t per = (uint32_t)(p.n_strips * ceil_div64(p.group_rows, kColTile));
    const uint32_t g = (uint32_t)i / per;
    u.g = g;
    local = (uint32_t)i - g * per;
    u.g0 = u.g * p.group_rows;
    u.n = p.group_rows;
    u.pstart = 0;
    u.write_end = u.n;
  }
  const uint32_t ns = (uint32_t)p.n_strips;
  const uint32_t rt = local / ns;
  u.strip = local - rt * ns;
  u.rt = (int64_t)rt * kColTile;
  u.c0 = u.strip * 64;
  return u;
}

// Validates the offsets (segment mode) and builds the unit / padded-start / first-row prefixes in
// shared memory; returns the number of units, or -1 after reporting bad offsets.
FP8_DEVI int64_t col_setup(const ColParams& p, int32_t* upre, int32_t* ppre) {
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  if (p.mode != 2) return p.n_groups * p.n_strips * ceil_div64(p.group_rows, kColTile);
  int bad = 0;
  for (int64_t e = tid; e < p.n_groups; e += blockDim.x) {
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
        ppre[p.n_groups + 1 + i + 1] = p.ends[i];
      }
      cu += __shfl_sync(0xffffffffu, vu, 31);
      cp += __shfl_sync(0xffffffffu, vp, 31);
    }
    if (lane == 0) {
      upre[0] = 0;
      ppre[0] = 0;
      ppre[p.n_groups + 1] = 0;
    }
  }
  __syncthreads();
  return upre[p.n_groups];
}

// Column j (0..7) of a 16-byte vector of 8 bf16, as fp32.
FP8_DEVI float col_of(const uint4& v, int j) {
  const uint32_t w = j < 2 ? v.x : (j < 4 ? v.y : (j < 6 ? v.z : v.w));
  return (j & 1) ? __uint_as_float(w & 0xFFFF0000u) : __uint_as_float(w << 16);
}

// What the producer publishes with each stage: the unit's coordinates the consumers need.
struct ColInfo {
  int32_t g, c0, rt, valid, wrows, pstart;  // group, first column, tile start, rows of the group, rows written
};
struct ColShared {
  uint64_t full[kColStagesMax];   // the tile landed (TMA bytes) and the info was written
  uint64_t scl[kColStagesMax];    // pass 2: the stage's 64 amax words landed (32 async arrivals)
  uint64_t empty[kColStagesMax];  // the consumer warps are done with the stage
  ColInfo info[kColStagesMax];
  uint32_t am[kColStagesMax][64];  // pass 2: the amax words of the stage's 64 columns
  uint32_t red[kColConsumerWarps][8][4];
  int abort;
};
template <bool CAST>
struct ColSmem {
  static constexpr int bytes =
      1024 + col_stages<CAST>() * kColStageBytes + (CAST ? 2 * kColOutBytes : 0) + (int)sizeof(ColShared);
};

template <int FMT, bool CAST>
__global__ void __launch_bounds__(kColThreads + 64, 1) colstream_kernel(const __grid_constant__ CUtensorMap tm_in,
                                                                        const __grid_constant__ CUtensorMap tm_out,
                                                                        const ColParams p,
                                                                        const __grid_constant__ ScaleTab tab) {
  extern __shared__ uint8_t smem_raw[];
  constexpr int kColStages = col_stages<CAST>();
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* Tout = ring + kColStages * kColStageBytes;
  ColShared& S = *reinterpret_cast<ColShared*>(Tout + (CAST ? 2 * kColOutBytes : 0));
  int32_t* upre = reinterpret_cast<int32_t*>(&S + 1);
  int32_t* ppre = upre + (p.n_groups + 1);
  const int64_t M = col_setup(p, upre, ppre);
  if (M < 0) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the scale table in shared memory: the lanes of a warp look up different entries at once
  __shared__ ScaleTab stab;
  if (CAST) {
    static_assert(sizeof(ScaleTab) % 4 == 0, "table words");
    for (int i = tid; i < (int)(sizeof(ScaleTab) / 4); i += blockDim.x)
      reinterpret_cast<uint32_t*>(&stab)[i] = reinterpret_cast<const uint32_t*>(&tab)[i];
  }
  if (tid == 0) {
    for (int s = 0; s < kColStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.scl[s], 32);
      mbar_init(&S.empty[s], kColConsumerWarps);
    }
    S.abort = 0;
    fence_mbar_init();
    tma_prefetch_desc(&tm_in);
    if (CAST) tma_prefetch_desc(&tm_out);
  }
  // Groups without rows have no units: their inverse scales (amax 0) are written here.
  if (CAST && blockIdx.x == 0) {
    const Scale s0 = tab_scale(tab, 0u);
    for (int64_t g = 0; g < p.n_groups; ++g) {
      const int64_t n = p.mode == 2 ? p.ends[g] - (g ? p.ends[g - 1] : 0) : p.group_rows;
      if (n > 0) continue;
      for (int64_t c = tid; c < p.C; c += blockDim.x) p.inv[g * p.C + c] = s0.inv32;
    }
  }
  __syncthreads();
  // units are dealt round-robin, so the CTAs read neighbouring strips of the same rows at the same
  // time (DRAM pages stay open); pass 2 walks the order backwards, its first reads being the
  // units pass 1 read last, still in L2
  const int64_t cnt = (int64_t)blockIdx.x < M ? (M - 1 - blockIdx.x) / gridDim.x + 1 : 0;
  auto unit_at = [&](int64_t k) {
    const int64_t i = blockIdx.x + k * gridDim.x;
    return CAST ? M - 1 - i : i;
  };
  volatile int* cta_abort = &S.abort;

  if (warp == 0) {
    // ==================== producer warp: one lane issues the tiles by TMA ====================
    if (lane == 0) {
      // pass 1 keeps what it reads in L2 for pass 2; pass 2's reads are the last use
      const uint64_t pol = CAST ? l2_evict_first() : l2_evict_last();
      int s = 0;
      uint32_t ph = 0;
      int64_t k = 0;
      ColUnit un = {};
      if (cnt > 0) un = col_unit(p, unit_at(0), upre, ppre);
      for (; k < cnt; ++k) {
        if (!mbar_wait(&S.empty[s], ph ^ 1, cta_abort, p.wait_ns)) {
          if (!*cta_abort) {
            *cta_abort = 1;
            set_status(p.status, FP8_DEV_TIMEOUT);
          }
          break;
        }
        const ColUnit u = un;
        int64_t valid = u.n - u.rt, wr = u.write_end - u.rt;
        valid = valid < 0 ? 0 : (valid < kColTile ? valid : kColTile);
        wr = wr < 0 ? 0 : (wr < kColTile ? wr : kColTile);
        S.info[s] = ColInfo{(int32_t)u.g, (int32_t)u.c0, (int32_t)u.rt, (int32_t)valid, (int32_t)wr,
                            (int32_t)u.pstart};
        mbar_arrive_expect_tx(&S.full[s], kColStageBytes);
        tma_load_2d_hint(ring + s * kColStageBytes, &tm_in, &S.full[s], (int32_t)u.c0, (int32_t)(u.g0 + u.rt), pol);
        if (k + 1 < cnt) un = col_unit(p, unit_at(k + 1), upre, ppre);
        if (++s == kColStages) {
          s = 0;
          ph ^= 1;
        }
      }
      // the loads in flight land before the CTA may leave (all consumed unless aborted)
      const int64_t first = k > kColStages ? k - kColStages : 0;
      for (int64_t j = first; j < k; ++j)
        mbar_wait(&S.full[j % kColStages], (uint32_t)((j / kColStages) & 1), nullptr, kColDrainNs);
    }
  } else if (warp == kColConsumerWarps + 1) {
    // ======== pass 2 amax warp: each tile's 64 column maxima, beside the TMA producer ========
    // Once a stage is free, the words of its unit's columns lane and lane + 32 are copied
    // asynchronously into the stage's slot, and each lane's copies complete an arrival on the
    // stage's scl barrier when they land: nothing on this warp's path waits for memory.
    if (CAST) {
      int s = 0;
      uint32_t ph = 0;
      ColUnit un = {};
      if (cnt > 0) un = col_unit(p, unit_at(0), upre, ppre);
      for (int64_t k = 0; k < cnt; ++k) {
        const bool got = lane == 0 ? mbar_wait(&S.empty[s], ph ^ 1, cta_abort, p.wait_ns) : true;
        if (!__shfl_sync(0xffffffffu, got, 0)) {
          if (lane == 0 && !*cta_abort) {
            *cta_abort = 1;
            set_status(p.status, FP8_DEV_TIMEOUT);
          }
          break;
        }
#pragma unroll
        for (int h = 0; h < 2; ++h) {
          const int64_t col = un.c0 + lane + 32 * h;
          cp_async4(&S.am[s][lane + 32 * h], p.scratch + un.g * p.C + (col < p.C ? col : 0), col < p.C);
        }
        cp_async_arrive_noinc(&S.scl[s]);
        if (k + 1 < cnt) un = col_unit(p, unit_at(k + 1), upre, ppre);
        if (++s == kColStages) {
          s = 0;
          ph ^= 1;
        }
      }
      cp_async_wait<0>();  // no copy lands after the CTA has left
    }
  } else if (!CAST) {
    // ============ pass 1 consumers: thread = 4 rows x 8 columns of each 128-row block ============
    const int ct = tid - 32, cw = ct >> 5;
    const int ch = lane & 7, rq = lane >> 3;
    int s = 0;
    uint32_t ph = 0;
    for (int64_t k = 0; k < cnt; ++k) {
      const bool got = mbar_wait(&S.full[s], ph, cta_abort, p.wait_ns);
      if (!named_bar_and(2, kColThreads, got)) {  // uniform decision across the consumer warps
        if (!got && !*cta_abort) {
          *cta_abort = 1;
          set_status(p.status, FP8_DEV_TIMEOUT);
        }
        break;
      }
      const ColInfo info = S.info[s];
      const uint8_t* st = ring + s * kColStageBytes;
      uint4 v[kColNB][4];
      if (info.valid == kColTile) {
#pragma unroll
        for (int b = 0; b < kColNB; ++b)
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int r = 128 * b + 16 * cw + 4 * rq + jj;
            v[b][jj] = *reinterpret_cast<const uint4*>(st + r * 128 + ((ch ^ (r & 7)) << 4));
          }
      } else {
#pragma unroll
        for (int b = 0; b < kColNB; ++b)
#pragma unroll
          for (int jj = 0; jj < 4; ++jj) {
            const int r = 128 * b + 16 * cw + 4 * rq + jj;  // rows past the group read as zeros
            v[b][jj] = r < info.valid ? *reinterpret_cast<const uint4*>(st + r * 128 + ((ch ^ (r & 7)) << 4))
                                      : make_uint4(0, 0, 0, 0);
          }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[s]);  // this warp is done with the stage
      if (++s == kColStages) {
        s = 0;
        ph ^= 1;
      }
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
      for (int q = 0; q < 4; ++q) {
        m4[q] = __vmaxu2(m4[q], __shfl_xor_sync(0xffffffffu, m4[q], 8));
        m4[q] = __vmaxu2(m4[q], __shfl_xor_sync(0xffffffffu, m4[q], 16));
      }
      if (rq == 0) {
#pragma unroll
        for (int q = 0; q < 4; ++q) S.red[cw][ch][q] = m4[q];
      }
      named_bar_sync(1, kColThreads);
      if (ct < 32) {  // pair t = columns 2t, 2t+1 = chunk t/4, word t%4
        uint32_t m = 0;
#pragma unroll
        for (int w = 0; w < kColConsumerWarps; ++w) m = __vmaxu2(m, S.red[w][ct >> 2][ct & 3]);
        const int64_t col = info.c0 + 2 * ct;
        uint32_t* scw = p.scratch + (int64_t)info.g * p.C + col;
        if (col < p.C && (m & 0xFFFFu)) red_max_relaxed(scw, m & 0xFFFFu);
        if (col + 1 < p.C && (m >> 16)) red_max_relaxed(scw + 1, m >> 16);
      }
      named_bar_sync(1, kColThreads);
    }
  } else {
    // ====== pass 2 consumers: each warp casts 32 rows x 64 columns and stores them itself ======
    // Lane l owns the column pair (2 l, 2 l + 1); a 32-bit shared load holds the pair's values of
    // one row (the 128-byte swizzle permutes 16-byte chunks inside a row, so the 32 lanes still
    // read one row's 128 bytes). Its 2 x 32 codes go to the warp's staging box [64 columns][32
    // rows] and the warp's elected lane stores the box by TMA: no barrier across warps.
    const int cw = warp - 1;
    const int r0 = 32 * cw;  // the warp's rows within the unit
    const uint64_t out_pol = l2_evict_first();  // the codes are not re-read by this pass
    const uint32_t woff = ((uint32_t)(lane & 3) << 2);
    uint8_t* wbuf = Tout + cw * 2 * kColWarpBox;
    int s = 0, nb = 0;
    uint32_t ph = 0;
    for (int64_t k = 0; k < cnt; ++k) {
      bool got = mbar_wait(&S.full[s], ph, cta_abort, p.wait_ns);
      if (got) got = mbar_wait(&S.scl[s], ph, cta_abort, p.wait_ns);
      if (!__all_sync(0xffffffffu, got)) {
        if (lane == 0 && !*cta_abort) {
          *cta_abort = 1;
          set_status(p.status, FP8_DEV_TIMEOUT);
        }
        break;
      }
      const ColInfo info = S.info[s];
      // the scale step for the lane's two columns (the table in shared memory); the first row
      // tile of a strip also writes their inverse scales
      const uint2 am2 = *reinterpret_cast<const uint2*>(&S.am[s][2 * lane]);
      const Scale sv_lo = tab_scale(stab, am2.x >> p.amax_shift), sv_hi = tab_scale(stab, am2.y >> p.amax_shift);
      const float2 sc = make_float2(sv_lo.s32, sv_hi.s32);
      if (info.rt == 0 && cw == 0) {
        const int64_t col = info.c0 + 2 * lane;
        if (col < p.C) p.inv[(int64_t)info.g * p.C + col] = sv_lo.inv32;
        if (col + 1 < p.C) p.inv[(int64_t)info.g * p.C + col + 1] = sv_hi.inv32;
      }
      const uint8_t* st = ring + s * kColStageBytes + r0 * 128 + woff;
      uint32_t w[32];
      if (info.valid >= r0 + 32) {
#pragma unroll
        for (int r = 0; r < 32; ++r)
          w[r] = *reinterpret_cast<const uint32_t*>(st + r * 128 + ((((uint32_t)lane >> 2) ^ (uint32_t)(r & 7)) << 4));
      } else {
#pragma unroll
        for (int r = 0; r < 32; ++r)  // rows past the group read as zeros
          w[r] = r0 + r < info.valid
                     ? *reinterpret_cast<const uint32_t*>(st + r * 128 + ((((uint32_t)lane >> 2) ^ (uint32_t)(r & 7)) << 4))
                     : 0u;
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(&S.empty[s]);  // this warp is done with the stage
      if (++s == kColStages) {
        s = 0;
        ph ^= 1;
      }
      if (r0 >= info.wrows) continue;  // nothing of this warp's rows is written
      uint32_t olo[8], ohi[8];
      const float2 slo = make_float2(sc.x, sc.x), shi = make_float2(sc.y, sc.y);
#pragma unroll
      for (int r = 0; r < 32; r += 4) {
        // column 2 l: the low halves of rows r .. r + 3; column 2 l + 1: the high halves
        const float2 l01 = fmul2_rn(make_float2(__uint_as_float(w[r] << 16), __uint_as_float(w[r + 1] << 16)), slo);
        const float2 l23 = fmul2_rn(make_float2(__uint_as_float(w[r + 2] << 16), __uint_as_float(w[r + 3] << 16)), slo);
        const float2 h01 = fmul2_rn(make_float2(__uint_as_float(w[r] & 0xFFFF0000u), __uint_as_float(w[r + 1] & 0xFFFF0000u)), shi);
        const float2 h23 = fmul2_rn(make_float2(__uint_as_float(w[r + 2] & 0xFFFF0000u), __uint_as_float(w[r + 3] & 0xFFFF0000u)), shi);
        olo[r / 4] = cvt_fp8x2<FMT>(l01.x, l01.y) | (cvt_fp8x2<FMT>(l23.x, l23.y) << 16);
        ohi[r / 4] = cvt_fp8x2<FMT>(h01.x, h01.y) | (cvt_fp8x2<FMT>(h23.x, h23.y) << 16);
      }
      uint8_t* box = wbuf + nb * kColWarpBox;
      nb ^= 1;
      if (lane == 0) bulk_wait_read_1();  // the store that last read this box has done so
      __syncwarp();
      uint8_t* dst = box + lane * 64;  // rows 2 l and 2 l + 1 of the box: 32 codes each
      *reinterpret_cast<uint4*>(dst) = make_uint4(olo[0], olo[1], olo[2], olo[3]);
      *reinterpret_cast<uint4*>(dst + 16) = make_uint4(olo[4], olo[5], olo[6], olo[7]);
      *reinterpret_cast<uint4*>(dst + 32) = make_uint4(ohi[0], ohi[1], ohi[2], ohi[3]);
      *reinterpret_cast<uint4*>(dst + 48) = make_uint4(ohi[4], ohi[5], ohi[6], ohi[7]);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        const int32_t xo = info.pstart + info.rt + r0;
        if (p.mode == 1)
          tma_store_3d_hint(&tm_out, box, xo, info.c0, info.g, out_pol);
        else
          tma_store_2d_hint(&tm_out, box, xo, info.c0, out_pol);
        bulk_commit();
      }
    }
    if (lane == 0) bulk_wait_all();
  }
  __syncthreads();
}

// Workspace words of a column quantize: the amax per (group, column), rounded to 16 bytes.
int64_t col_ws_words(int64_t groups, int64_t C) { return round_up64(groups * C, 4); }

int launch_quant_cols(const void* x, int64_t rows_total, int64_t C, int64_t n_groups, int64_t group_rows,
                      const int32_t* ends, int fmt, void* out_t, int64_t ld_out, float* inv, uint32_t* scratch,
                      const Ctx& c, const uint32_t* amax_given) {
  if (n_groups == 0 || C == 0) return FP8_OK;
  if (ends && n_groups > 2048) return FP8_ERR_UNSUPPORTED;  // prefix arrays live in shared memory
  ColParams p = {};
  p.x = static_cast<const uint16_t*>(x);
  p.rows_total = rows_total;
  p.C = C;
  p.n_groups = n_groups;
  p.group_rows = group_rows;
  p.ends = ends;
  p.n_strips = ceil_div64(C, 64);
  p.scratch = scratch;
  p.inv = inv;
  p.status = c.status;
  p.wait_ns = c.wait_ns;
  p.mode = ends ? 2 : (n_groups > 1 ? 1 : 0);

  CUtensorMap tout, tin;
  int rc;
  if (p.mode == 1) {
    const uint64_t dims[3] = {(uint64_t)group_rows, (uint64_t)C, (uint64_t)n_groups};
    const uint64_t strides[2] = {(uint64_t)group_rows, (uint64_t)(C * group_rows)};
    const uint32_t box[3] = {32, 64, 1};  // one warp's box: 32 rows (bytes) x 64 columns
    rc = make_tmap(&tout, out_t, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
  } else {
    const uint64_t inner = p.mode == 2 ? (uint64_t)ld_out : (uint64_t)group_rows;
    const uint64_t dims[2] = {inner, (uint64_t)C};
    const uint64_t strides[1] = {(uint64_t)ld_out};
    const uint32_t box[2] = {32, 64};  // one warp's box: 32 rows (bytes) x 64 columns
    rc = make_tmap(&tout, out_t, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_NONE);
  }
  if (rc != FP8_OK) return rc;
  {
    const uint64_t dims[2] = {(uint64_t)C, (uint64_t)(rows_total > 0 ? rows_total : 1)};
    const uint64_t strides[1] = {(uint64_t)C * 2};
    const uint32_t box[2] = {64, kColTile};
    rc = make_tmap(&tin, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
    if (rc != FP8_OK) return rc;
  }

  if (amax_given) {
    p.scratch = const_cast<uint32_t*>(amax_given);  // read only (pass 2)
    p.amax_shift = 16;
  } else if (cudaMemsetAsync(scratch, 0, (size_t)col_ws_words(n_groups, C) * 4, c.stream) != cudaSuccess) {
    return FP8_ERR_CUDA;
  }
  // units: exact for dense modes; for segments an upper bound (each segment adds at most one
  // partial tile) -- the kernels compute the exact count from the offsets
  const int64_t units = p.mode == 2 ? (ceil_div64(rows_total, kColTile) + n_groups) * p.n_strips
                                    : n_groups * ceil_div64(group_rows, kColTile) * p.n_strips;
  if (units > INT32_MAX) return FP8_ERR_UNSUPPORTED;  // the kernels decode units in 32 bits
  const size_t pre = p.mode == 2 ? 12 * (size_t)(n_groups + 1) : 0;
  const int64_t grid = units > 0 ? (units < c.sm_count ? units : c.sm_count) : 1;
  const ScaleTab& tab = scale_tab(fmt);
  // pass 1: column maxima (skipped when the caller supplies them)
  if (units > 0 && !amax_given) {
    auto k1 = fmt == FP8_DT_E4M3 ? colstream_kernel<FP8_DT_E4M3, false> : colstream_kernel<FP8_DT_E5M2, false>;
    const size_t smem = ColSmem<false>::bytes + pre;
    if (cudaFuncSetAttribute(k1, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
      return FP8_ERR_CUDA;
    k1<<<(unsigned)grid, kColThreads + 64, smem, c.stream>>>(tin, tout, p, tab);
    if (cudaGetLastError() != cudaSuccess) return FP8_ERR_CUDA;
  }
  // pass 2: scales and cast (also writes the scales of groups without rows)
  auto k2 = fmt == FP8_DT_E4M3 ? colstream_kernel<FP8_DT_E4M3, true> : colstream_kernel<FP8_DT_E5M2, true>;
  const size_t smem2 = ColSmem<true>::bytes + pre;
  if (cudaFuncSetAttribute(k2, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem2) != cudaSuccess)
    return FP8_ERR_CUDA;
  k2<<<(unsigned)grid, kColThreads + 64, smem2, c.stream>>>(tin, tout, p, tab);
  return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

}  // namespace fp8lin

namespace fp8lin {

int launch_quant_tensor_cast(const void* x, int64_t R, int64_t C, int fmt, void* q, void* qt, float* inv,
                             const uint32_t* amax_word, const Ctx& c, int amax_shift) {
  dim3 grid((unsigned)ceil_div64(C, kTcCols), (unsigned)ceil_div64(R, kTcRows));
  if (grid.x == 0 || grid.y == 0) grid = dim3(1, 1);
  if (fmt == FP8_DT_E4M3)
    quant_tensor_cast_kernel<FP8_DT_E4M3><<<grid, 256, 0, c.stream>>>(
        static_cast<const uint16_t*>(x), R, C, amax_word, amax_shift, static_cast<uint8_t*>(q), static_cast<uint8_t*>(qt),
        inv,
        scale_tab(fmt));
  else
    quant_tensor_cast_kernel<FP8_DT_E5M2><<<grid, 256, 0, c.stream>>>(
        static_cast<const uint16_t*>(x), R, C, amax_word, amax_shift, static_cast<uint8_t*>(q), static_cast<uint8_t*>(qt),
        inv,
        scale_tab(fmt));
  return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

}  // namespace fp8lin

namespace fp8lin {

// Test hook: the cast of every quantize kernel (cvt.rn.satfinite, two values per instruction),
// applied to the fp32 values whose bit patterns are first, first + 1, ..., first + n - 1. The
// row-wise and column-wise kernels cast the scaled products without an explicit clamp (the
// saturating cvt gives the same code as clamping to +-fp8_max first), so this covers their cast
// step as it runs.
template <int FMT>
__global__ void __launch_bounds__(256) cast_bits_kernel(uint32_t first, int64_t n, uint8_t* __restrict__ out) {
  const int64_t stride = 2 * (int64_t)gridDim.x * blockDim.x;
  for (int64_t i = 2 * ((int64_t)blockIdx.x * blockDim.x + threadIdx.x); i < n; i += stride) {
    const float a = __uint_as_float(first + (uint32_t)i);
    const float b = __uint_as_float(first + (uint32_t)(i + 1));
    const uint32_t c = cvt_fp8x2<FMT>(a, b);
    out[i] = (uint8_t)c;
    if (i + 1 < n) out[i + 1] = (uint8_t)(c >> 8);
  }
}

int launch_cast_bits(uint32_t first, int64_t n, int fmt, void* out, const Ctx& c) {
  if (n <= 0) return FP8_OK;
  const int64_t need = ceil_div64(n, 2 * 256);
  const int64_t cap = (int64_t)c.sm_count * 8;
  const unsigned grid = (unsigned)(need < cap ? need : cap);
  if (fmt == FP8_DT_E4M3)
    cast_bits_kernel<FP8_DT_E4M3><<<grid, 256, 0, c.stream>>>(first, n, static_cast<uint8_t*>(out));
  else
    cast_bits_kernel<FP8_DT_E5M2><<<grid, 256, 0, c.stream>>>(first, n, static_cast<uint8_t*>(out));
  return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

}  // namespace fp8lin
