// Fused FP8 quantization kernels (sm_103a): amax -> fp64 scale -> fp32 multiply -> clamp ->
// RNE saturating cast, one HBM read per element.
//
// Recipe: "FP8 Training: Quantization, Autograd, Torchao", section 2 "The quantization math".
// Fusion and layout design: "FP8 training on AMD GPUs with TorchTitan and TorchAO", "Triton
// Kernel Optimization": Level 1 (one kernel per quantization, no intermediates in HBM; the
// dual row/column-major output), Level 2 (column-wise scales with the output tile transposed
// on chip so the column-major writes are coalesced; single pass over the data), Level 3
// (relaxed atomics for the commutative amax reduction).
#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"

namespace cg = cooperative_groups;

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
                      float* __restrict__ inv) {
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
      const Scale s = make_scale(bf16_bits_to_float(mm), FMAX);
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
                                                           static_cast<uint2*>(q), inv);
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
                                                                float* __restrict__ inv) {
  constexpr float FMAX = FmtMax<FMT>::v;
  __shared__ float s_sc;
  __shared__ __align__(16) uint8_t T[kTcCols * kTcPitch];
  if (threadIdx.x == 0) {
    const Scale s = make_scale(bf16_bits_to_float(*amax_ws), FMAX);
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
        static_cast<const uint16_t*>(x), R, C, amax_ws, static_cast<uint8_t*>(q), static_cast<uint8_t*>(qt), inv);
  else
    quant_tensor_cast_kernel<FP8_DT_E5M2><<<grid, 256, 0, c.stream>>>(
        static_cast<const uint16_t*>(x), R, C, amax_ws, static_cast<uint8_t*>(q), static_cast<uint8_t*>(qt), inv);
  return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

// ==========================================================================================
// Columnwise with column-major output, single pass. Work unit = (row group g, strip of 64
// columns). A cluster of kColCS CTAs shares the unit: each CTA pulls its share of the group's
// rows (up to kColCap rows) into shared memory with TMA (128-byte swizzled rows of 64 bf16),
// computes the per-column partial amax, the cluster exchanges the partials through distributed
// shared memory, every CTA derives the 64 scales, casts its rows into a transposed FP8 tile and
// writes whole 16-byte runs of the column-major output. A group larger than kColCS * kColCap
// rows falls back to two passes over the group (amax, then re-read and cast).
constexpr int kColCS = 8;
constexpr int kColCap = 1024;
constexpr int kColBox = 32;  // rows per TMA box
constexpr int kColThreads = 256;

struct ColSmem {
  uint8_t in[kColCap * 128];   // TMA destination: row r at r * 128, 16-byte chunks XOR (r % 8)
  uint8_t T[64 * kColCap];     // transposed codes: column c at c * kColCap, chunks XOR (c % 8)
  uint32_t red[8][32];
  uint32_t part[32];           // packed |bf16| maxima of column pairs (low half = even column)
  float s32[64];
  int64_t psum[8];
  uint64_t bar;
};

struct ColParams {
  int64_t rows_total;
  int64_t C;
  int64_t n_groups;
  int64_t group_rows;
  const int32_t* ends;
  uint8_t* out_t;
  int64_t ld_out;
  float* inv;
  int32_t* status;
  uint64_t wait_ns;
  int64_t n_strips;
};

template <int FMT>
FP8_DEVI uint32_t cast4(const float* f, float s, float fmax) {
  float y[4];
#pragma unroll
  for (int j = 0; j < 4; ++j) {
    float t = __fmul_rn(f[j], s);
    y[j] = t > fmax ? fmax : (t < -fmax ? -fmax : t);
  }
  return cvt_fp8x2<FMT>(y[0], y[1]) | (cvt_fp8x2<FMT>(y[2], y[3]) << 16);
}

template <int FMT>
__global__ void __launch_bounds__(kColThreads, 1)
    quant_cols_kernel(const __grid_constant__ CUtensorMap tmap, const ColParams p) {
  constexpr float FMAX = FmtMax<FMT>::v;
  cg::cluster_group cluster = cg::this_cluster();
  const unsigned rank = cluster.block_rank();
  extern __shared__ uint8_t smem_raw[];
  ColSmem& S = *reinterpret_cast<ColSmem*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t unit = blockIdx.x / kColCS;
  const int64_t g = unit / p.n_strips;
  const int64_t c0 = (unit % p.n_strips) * 64;

  // ---- the group's rows (and, for segments, its padded start) ----
  int64_t g0, g1, pstart = 0;
  if (p.ends) {
    int bad = 0;
    int64_t ps = 0;
    for (int64_t e = tid; e < p.n_groups; e += kColThreads) {
      const int64_t cur = p.ends[e], prev = e ? p.ends[e - 1] : 0;
      if (cur < prev || (e == p.n_groups - 1 && cur != p.rows_total)) bad = 1;
      if (e < g && cur >= prev) ps += round_up64(cur - prev, 128);
    }
    bad = __syncthreads_or(bad);
    if (bad) {
      if (blockIdx.x == 0 && tid == 0) set_status(p.status, FP8_DEV_BAD_OFFSETS);
      return;  // every CTA of every cluster takes this branch: no cluster barrier is pending
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) ps += __shfl_xor_sync(0xffffffffu, ps, o);
    if (lane == 0) S.psum[warp] = ps;
    __syncthreads();
    for (int w = 0; w < 8; ++w) pstart += S.psum[w];
    g0 = g ? p.ends[g - 1] : 0;
    g1 = p.ends[g];
  } else {
    g0 = g * p.group_rows;
    g1 = g0 + p.group_rows;
  }
  const int64_t n = g1 - g0;
  const int64_t write_end = p.ends ? round_up64(n, 128) : n;
  int64_t chunk;
  int rounds;
  if (n <= (int64_t)kColCS * kColCap) {
    chunk = round_up64(ceil_div64(n, kColCS), 16);
    rounds = n > 0 ? 1 : 0;
  } else {
    chunk = kColCap;
    rounds = (int)ceil_div64(n, (int64_t)kColCS * kColCap);
  }

  if (tid == 0) {
    mbar_init(&S.bar, 1);
    fence_mbar_init();
    tma_prefetch_desc(&tmap);
  }
  __syncthreads();

  uint32_t phase = 0;
  int ok = 1, pending = 0;
  auto load = [&](int64_t rel0, int64_t rows) {
    if (tid == 0) {
      const int nbox = (int)ceil_div64(rows, kColBox);
      mbar_arrive_expect_tx(&S.bar, (uint32_t)(nbox * kColBox * 128));
      for (int b = 0; b < nbox; ++b)
        tma_load_2d(S.in + b * kColBox * 128, &tmap, &S.bar, (int32_t)c0, (int32_t)(g0 + rel0 + b * kColBox));
    }
    pending = 1;
  };
  auto wait = [&]() {
    const bool w = mbar_wait(&S.bar, phase, nullptr, p.wait_ns);
    const int all = __syncthreads_and(w ? 1 : 0);
    if (all) {
      phase ^= 1;
      pending = 0;
    } else {
      ok = 0;
      if (tid == 0) set_status(p.status, FP8_DEV_TIMEOUT);
    }
  };

  // ---- pass 1: partial column amax over this CTA's rows ----
  uint32_t acc = 0;
  for (int j = 0; j < rounds && ok; ++j) {
    const int64_t rel0 = ((int64_t)j * kColCS + rank) * chunk;
    const int64_t valid = n - rel0 < chunk ? n - rel0 : chunk;
    if (valid <= 0) continue;
    if (j > 0) {
      fence_proxy_async_smem();
      __syncthreads();
    }
    load(rel0, valid);
    wait();
    if (!ok) break;
    for (int r = warp; r < valid; r += 8)
      acc = absmax2(acc, *reinterpret_cast<const uint32_t*>(S.in + r * 128 + (((lane >> 2) ^ (r & 7)) << 4) +
                                                            ((lane & 3) << 2)));
  }
  S.red[warp][lane] = acc;
  __syncthreads();
  if (warp == 0) {
    uint32_t m = 0;
    for (int w = 0; w < 8; ++w) m = __vmaxu2(m, S.red[w][lane]);
    S.part[lane] = m;
  }
  cluster.sync();
  if (warp == 0) {
    uint32_t m = 0;
    for (unsigned rr = 0; rr < (unsigned)kColCS; ++rr) m = __vmaxu2(m, cluster.map_shared_rank(S.part, rr)[lane]);
    const Scale s0 = make_scale(bf16_bits_to_float(m & 0xFFFFu), FMAX);
    const Scale s1 = make_scale(bf16_bits_to_float(m >> 16), FMAX);
    S.s32[2 * lane] = s0.s32;
    S.s32[2 * lane + 1] = s1.s32;
    if (rank == 0) {
      const int64_t col = c0 + 2 * lane;
      if (col < p.C) p.inv[g * p.C + col] = s0.inv32;
      if (col + 1 < p.C) p.inv[g * p.C + col + 1] = s1.inv32;
    }
  }
  __syncthreads();

  // ---- pass 2: cast into the transposed tile, write column-major runs ----
  for (int j = 0; j < rounds && ok; ++j) {
    const int64_t rel0 = ((int64_t)j * kColCS + rank) * chunk;
    const int64_t valid = n - rel0 < chunk ? (n - rel0 > 0 ? n - rel0 : 0) : chunk;
    const int64_t wrows = write_end - rel0 < chunk ? write_end - rel0 : chunk;
    if (wrows <= 0) continue;
    if (rounds > 1 && valid > 0) {
      fence_proxy_async_smem();
      __syncthreads();
      load(rel0, valid);
      wait();
      if (!ok) break;
    }
    // lane -> column (cc * 8 + lane % 8), rows r0 .. r0 + 3 with r0 = 16 b + 4 (lane / 8)
    for (int64_t b = warp; b * 16 < wrows; b += 8) {
      const int r0 = (int)(b * 16) + 4 * (lane >> 3);
#pragma unroll
      for (int cc = 0; cc < 8; ++cc) {
        const int cl = cc * 8 + (lane & 7);
        float f[4];
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int r = r0 + jj;
          const uint16_t h =
              *reinterpret_cast<const uint16_t*>(S.in + r * 128 + ((cc ^ (r & 7)) << 4) + ((lane & 7) << 1));
          f[jj] = r < valid ? bf16_bits_to_float(h) : 0.0f;
        }
        *reinterpret_cast<uint32_t*>(S.T + cl * kColCap + (((r0 >> 4) ^ (cl & 7)) << 4) + (r0 & 15)) =
            cast4<FMT>(f, S.s32[cl], FMAX);
      }
    }
    __syncthreads();
    const int nch = (int)(wrows / 16);
    for (int i = tid; i < 64 * nch; i += kColThreads) {
      const int cl = i / nch, k = i % nch;
      const int64_t col = c0 + cl;
      if (col < p.C) {
        const uint4 v = *reinterpret_cast<const uint4*>(S.T + cl * kColCap + ((k ^ (cl & 7)) << 4));
        const int64_t row0 = p.ends ? col * p.ld_out + pstart : (g * p.C + col) * p.ld_out;
        *reinterpret_cast<uint4*>(p.out_t + row0 + rel0 + 16 * k) = v;
      }
    }
    __syncthreads();
  }
  // Drain a load still in flight after a timeout, then keep this CTA's shared memory alive
  // until every peer has read its partial maxima.
  if (pending && tid == 0) mbar_wait(&S.bar, phase, nullptr, p.wait_ns);
  cluster.sync();
}

int launch_quant_cols(const void* x, int64_t rows_total, int64_t C, int64_t n_groups, int64_t group_rows,
                      const int32_t* ends, int fmt, void* out_t, int64_t ld_out, float* inv, const Ctx& c) {
  if (n_groups == 0 || C == 0) return FP8_OK;
  CUtensorMap tmap;
  const uint64_t dims[2] = {(uint64_t)C, (uint64_t)(rows_total > 0 ? rows_total : 1)};
  const uint64_t strides[1] = {(uint64_t)C * 2};
  const uint32_t box[2] = {64, kColBox};
  int rc = make_tmap(&tmap, x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B);
  if (rc != FP8_OK) return rc;
  ColParams p;
  p.rows_total = rows_total;
  p.C = C;
  p.n_groups = n_groups;
  p.group_rows = group_rows;
  p.ends = ends;
  p.out_t = static_cast<uint8_t*>(out_t);
  p.ld_out = ld_out;
  p.inv = inv;
  p.status = c.status;
  p.wait_ns = c.wait_ns;
  p.n_strips = ceil_div64(C, 64);
  const int64_t units = n_groups * p.n_strips;
  const size_t smem = sizeof(ColSmem) + 1024;
  auto kern = fmt == FP8_DT_E4M3 ? quant_cols_kernel<FP8_DT_E4M3> : quant_cols_kernel<FP8_DT_E5M2>;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return FP8_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(units * kColCS));
  cfg.blockDim = dim3(kColThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kColCS;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, tmap, p) != cudaSuccess) return FP8_ERR_CUDA;
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
        static_cast<const uint16_t*>(x), R, C, amax_word, static_cast<uint8_t*>(q), static_cast<uint8_t*>(qt), inv);
  else
    quant_tensor_cast_kernel<FP8_DT_E5M2><<<grid, 256, 0, c.stream>>>(
        static_cast<const uint16_t*>(x), R, C, amax_word, static_cast<uint8_t*>(q), static_cast<uint8_t*>(qt), inv);
  return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

}  // namespace fp8lin
