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
// Columnwise with column-major output, single pass, register-resident.
//
// Work unit = (row group g, strips of 64 columns). A group of n rows needs k CTAs (k = the
// power of two >= n / (128 NB), at most the cluster size cs); a cluster of cs CTAs then
// processes cs / k strips of the group at once, one sub-team of k CTAs per strip, each member
// holding up to 128 NB rows of its strip in registers:
//   - loads: a thread reads 4 consecutive rows x 8 columns (four 16-byte loads; a warp reads 4
//     whole 128-byte rows per instruction), keeps them in registers and folds |x| into packed
//     per-column maxima;
//   - the CTA's column maxima go to shared memory; one cluster barrier; each CTA folds its
//     sub-team peers' maxima through distributed shared memory and derives the 64 scales;
//   - cast from registers: each 4-row column pack becomes one 32-bit word of FP8 codes; the
//     words are written into a transposed tile (64 columns x 128 rows per box, TMA 128-byte
//     swizzle; the order of a thread's 8 columns is rotated by its chunk index so the shared
//     stores are conflict-free), then TMA bulk-tensor stores write the column-major output.
// Clusters are persistent and walk the units. Groups of more than cs * 128 NB rows take two
// passes (amax over all rows, then re-read and cast).
constexpr int kColThreads = 256;
constexpr int kColCtrlBytes = 4096;

struct ColCtrl {
  uint32_t part[2][32];    // this CTA's packed |bf16| column-pair maxima, by unit parity
  uint32_t red[8][8][4];   // per warp, per 8-column chunk, 4 packed pairs
  float s32[64];
  int32_t total_units;
  int32_t bad;
};
static_assert(sizeof(ColCtrl) <= kColCtrlBytes, "column kernel control block");

struct ColParams {
  const uint16_t* x;
  int64_t rows_total;
  int64_t C;
  int64_t n_groups;
  int64_t group_rows;  // dense modes
  const int32_t* ends; // segment mode
  float* inv;
  int32_t* status;
  int64_t n_strips;
  int cs;              // CTAs per cluster
  int mode;            // 0: 2-D [C, R] output; 1: batched [B, C, R]; 2: segments [C, P]
  int dense_k;         // dense modes: CTAs per strip
};

struct ColUnit {
  int64_t g, g0, n, pstart, write_end, chunk;
  int64_t strip;       // this CTA's strip (may be >= n_strips: idle member)
  int k, member, sub, rounds;
};

FP8_DEVI int ceil_pow2_int(int64_t v) {
  int k = 1;
  while (k < v) k <<= 1;
  return k;
}

// Sub-team size of a group of n rows: k CTAs of cap rows each, a power of two <= cs.
FP8_DEVI int team_size(int64_t n, int cap, int cs) {
  const int64_t need = ceil_div64(n, cap);
  const int k = ceil_pow2_int(need < 1 ? 1 : need);
  return k > cs ? cs : k;
}

template <int NB>
FP8_DEVI ColUnit col_unit(const ColParams& p, int64_t unit, const int32_t* upre, const int32_t* ppre, int rank) {
  constexpr int CAP = 128 * NB;
  ColUnit u;
  int64_t local;
  if (p.mode == 2) {
    int lo = 0, hi = (int)p.n_groups - 1;  // the segment whose unit range holds `unit`
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
    u.k = team_size(u.n, CAP, p.cs);
  } else {
    u.k = p.dense_k;
    const int64_t upg = ceil_div64(p.n_strips, p.cs / u.k);
    u.g = unit / upg;
    local = unit % upg;
    u.g0 = u.g * p.group_rows;
    u.n = p.group_rows;
    u.pstart = 0;
    u.write_end = u.n;
  }
  u.sub = rank / u.k;
  u.member = rank % u.k;
  u.strip = local * (p.cs / u.k) + u.sub;
  if (u.n <= (int64_t)u.k * CAP) {
    u.chunk = round_up64(ceil_div64(u.n, u.k), 128);
    u.rounds = u.n > 0 ? 1 : 0;
  } else {
    u.chunk = CAP;
    u.rounds = (int)ceil_div64(u.n, (int64_t)u.k * CAP);
  }
  return u;
}



// Column j (0..7) of a 16-byte vector of 8 bf16, as fp32.
FP8_DEVI float col_of(const uint4& v, int j) {
  const uint32_t w = j < 2 ? v.x : (j < 4 ? v.y : (j < 6 ? v.z : v.w));
  return (j & 1) ? __uint_as_float(w & 0xFFFF0000u) : __uint_as_float(w << 16);
}

template <int FMT, int NB>
__global__ void __launch_bounds__(kColThreads, NB <= 4 ? 2 : 1)
    quant_cols_kernel(const __grid_constant__ CUtensorMap tm_out, const ColParams p) {
  constexpr int CAP = 128 * NB;
  cg::cluster_group cluster = cg::this_cluster();
  const int rank = (int)cluster.block_rank();
  const int cs = p.cs;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* T = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  ColCtrl& S = *reinterpret_cast<ColCtrl*>(T + CAP * 64);
  int32_t* upre = reinterpret_cast<int32_t*>(reinterpret_cast<uint8_t*>(&S) + kColCtrlBytes);  // [E + 1]
  int32_t* ppre = upre + (p.n_groups + 1);                                                    // [E + 1]
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int ch = lane & 7, rq = lane >> 3;  // 8-column chunk, row quad within the warp's 16 rows
  const int64_t cluster_id = blockIdx.x / cs, n_clusters = gridDim.x / cs;

  // ---- units: dense modes have a fixed count; segments need the offsets ----
  int64_t total_units;
  if (p.mode == 2) {
    int bad = 0;
    for (int64_t e = tid; e < p.n_groups; e += kColThreads) {
      const int64_t cur = p.ends[e], prev = e ? p.ends[e - 1] : 0;
      if (cur < prev || (e == p.n_groups - 1 && cur != p.rows_total)) bad = 1;
    }
    bad = __syncthreads_or(bad);
    if (bad) {
      if (blockIdx.x == 0 && tid == 0) set_status(p.status, FP8_DEV_BAD_OFFSETS);
      return;  // every CTA takes this branch before any cluster barrier
    }
    if (warp == 0) {  // prefix of units per segment and of padded segment lengths
      int cu = 0, cp = 0;
      for (int64_t base = 0; base < p.n_groups; base += 32) {
        const int64_t i = base + lane;
        int vu = 0, vp = 0;
        if (i < p.n_groups) {
          const int64_t n = p.ends[i] - (i ? p.ends[i - 1] : 0);
          const int k = team_size(n, CAP, cs);
          vu = (int)ceil_div64(p.n_strips, cs / k);
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
    total_units = upre[p.n_groups];
  } else {
    total_units = p.n_groups * ceil_div64(p.n_strips, cs / p.dense_k);
  }
  if (tid == 0) tma_prefetch_desc(&tm_out);

  int parity = 0;
  for (int64_t unit = cluster_id; unit < total_units; unit += n_clusters, parity ^= 1) {
    const ColUnit u = col_unit<NB>(p, unit, upre, ppre, rank);
    const bool on = u.strip < p.n_strips;
    const int64_t c0 = u.strip * 64;
    const bool ch_ok = on && c0 + ch * 8 < p.C;
    // this thread's rows within a member's chunk: block b, rows 128 b + 16 warp + 4 rq + jj
    uint4 v[NB][4];
    auto load_round = [&](int r, int64_t* rel0_out, int64_t* valid_out) {
      const int64_t rel0 = ((int64_t)r * u.k + u.member) * u.chunk;
      int64_t valid = u.n - rel0;
      valid = valid < 0 ? 0 : (valid < u.chunk ? valid : u.chunk);
      const uint16_t* base = p.x + (u.g0 + rel0) * p.C + c0 + ch * 8;
#pragma unroll
      for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          const int row = 128 * b + 16 * warp + 4 * rq + jj;
          v[b][jj] = (ch_ok && row < valid) ? ld_nc_v4(base + (int64_t)row * p.C) : make_uint4(0, 0, 0, 0);
        }
      *rel0_out = rel0;
      *valid_out = valid;
    };

    // ---- pass 1: packed per-column maxima (x: cols 0-1, y: 2-3, z: 4-5, w: 6-7 of the chunk) ----
    uint32_t m4[4] = {0, 0, 0, 0};
    for (int r = 0; r < u.rounds; ++r) {
      int64_t rel0, valid;
      load_round(r, &rel0, &valid);
#pragma unroll
      for (int b = 0; b < NB; ++b)
#pragma unroll
        for (int jj = 0; jj < 4; ++jj) {
          m4[0] = absmax2(m4[0], v[b][jj].x);
          m4[1] = absmax2(m4[1], v[b][jj].y);
          m4[2] = absmax2(m4[2], v[b][jj].z);
          m4[3] = absmax2(m4[3], v[b][jj].w);
        }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      m4[i] = __vmaxu2(m4[i], __shfl_xor_sync(0xffffffffu, m4[i], 8));
      m4[i] = __vmaxu2(m4[i], __shfl_xor_sync(0xffffffffu, m4[i], 16));
    }
    if (rq == 0) {
#pragma unroll
      for (int i = 0; i < 4; ++i) S.red[warp][ch][i] = m4[i];
    }
    __syncthreads();
    if (tid < 32) {  // pair t = columns 2t, 2t+1 = chunk t/4, word t%4
      uint32_t m = 0;
      for (int w = 0; w < 8; ++w) m = __vmaxu2(m, S.red[w][tid >> 2][tid & 3]);
      S.part[parity][tid] = m;
    }
    cluster.sync();
    if (tid < 32) {
      uint32_t m = 0;
      for (int i = 0; i < u.k; ++i)
        m = __vmaxu2(m, cluster.map_shared_rank(&S.part[parity][0], u.sub * u.k + i)[tid]);
      constexpr float FMAX = FmtMax<FMT>::v;
      const Scale s0 = make_scale(bf16_bits_to_float(m & 0xFFFFu), FMAX);
      const Scale s1 = make_scale(bf16_bits_to_float(m >> 16), FMAX);
      S.s32[2 * tid] = s0.s32;
      S.s32[2 * tid + 1] = s1.s32;
      if (on && u.member == 0) {  // an empty segment gets the scales of an all-zero group
        const int64_t col = c0 + 2 * tid;
        if (col < p.C) p.inv[u.g * p.C + col] = s0.inv32;
        if (col + 1 < p.C) p.inv[u.g * p.C + col + 1] = s1.inv32;
      }
    }
    if (tid == 0) bulk_wait_read_all();  // the previous unit's stores have read the tile
    __syncthreads();
    float sc[8];
#pragma unroll
    for (int j = 0; j < 8; ++j) sc[j] = S.s32[ch * 8 + j];

    // ---- pass 2: cast from registers into the transposed tile, store column-major ----
    for (int r = 0; r < u.rounds; ++r) {
      int64_t rel0, valid;
      if (u.rounds > 1) {
        load_round(r, &rel0, &valid);
      } else {
        rel0 = (int64_t)u.member * u.chunk;
      }
      int64_t wrows = u.write_end - rel0;
      wrows = wrows < 0 ? 0 : (wrows < u.chunk ? wrows : u.chunk);
      const int nbox = (int)ceil_div64(wrows, 128);
      if (on && nbox > 0) {
#pragma unroll
        for (int b = 0; b < NB; ++b) {
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
      }
      fence_proxy_async_smem();
      __syncthreads();
      if (tid == 0 && on && nbox > 0) {
        for (int b = 0; b < nbox; ++b) {
          const int32_t xo = (int32_t)(u.pstart + rel0 + 128 * b);
          if (p.mode == 1)
            tma_store_3d(&tm_out, T + b * 8192, xo, (int32_t)c0, (int32_t)u.g);
          else
            tma_store_2d(&tm_out, T + b * 8192, xo, (int32_t)c0);
        }
        bulk_commit();
      }
      if (u.rounds > 1) {
        if (tid == 0) bulk_wait_read_all();
        __syncthreads();
      }
    }
  }
  if (tid == 0) bulk_wait_all();
  cluster.sync();  // peers may still read this CTA's partial maxima
}

template <int FMT, int NB>
static int run_cols(const ColParams& p0, const CUtensorMap& tout, const Ctx& c) {
  auto kern = quant_cols_kernel<FMT, NB>;
  ColParams p = p0;
  const size_t ctrl = kColCtrlBytes + (p.mode == 2 ? 8 * (size_t)(p.n_groups + 1) : 0);
  const size_t smem = 1024 + (size_t)128 * NB * 64 + ctrl;
  static bool attr_done = false;
  if (!attr_done) {
    if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 1024 + 128 * 8 * 64 + 65536) !=
            cudaSuccess ||
        cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1) != cudaSuccess)
      return FP8_ERR_CUDA;
    attr_done = true;
  }
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.blockDim = dim3(kColThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int slots = 0;
  for (int cs : {16, 8}) {
    attr[0].val.clusterDim.x = cs;
    cfg.gridDim = dim3(cs);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, kern, &cfg) == cudaSuccess && n > 0) {
      p.cs = cs;
      slots = n;
      break;
    }
    cudaGetLastError();
  }
  if (slots == 0) return FP8_ERR_CUDA;
  int64_t units;
  if (p.mode == 2) {
    units = p.n_groups * p.n_strips;  // upper bound; the kernel computes the exact count
  } else {
    int k = 1;
    while (k * 128 * NB < p.group_rows && k < p.cs) k <<= 1;
    p.dense_k = k;
    units = p.n_groups * ((p.n_strips + p.cs / k - 1) / (p.cs / k));
  }
  const int64_t clusters = units < slots ? units : slots;
  attr[0].val.clusterDim.x = p.cs;
  cfg.gridDim = dim3((unsigned)(clusters * p.cs));
  if (cudaLaunchKernelEx(&cfg, kern, tout, p) != cudaSuccess) return FP8_ERR_CUDA;
  return FP8_OK;
}

int launch_quant_cols(const void* x, int64_t rows_total, int64_t C, int64_t n_groups, int64_t group_rows,
                      const int32_t* ends, int fmt, void* out_t, int64_t ld_out, float* inv, const Ctx& c) {
  if (n_groups == 0 || C == 0) return FP8_OK;
  if (ends && n_groups > 6000) return FP8_ERR_UNSUPPORTED;  // prefix arrays live in shared memory
  ColParams p = {};
  p.x = static_cast<const uint16_t*>(x);
  p.rows_total = rows_total;
  p.C = C;
  p.n_groups = n_groups;
  p.group_rows = group_rows;
  p.ends = ends;
  p.inv = inv;
  p.status = c.status;
  p.n_strips = ceil_div64(C, 64);
  p.mode = ends ? 2 : (n_groups > 1 ? 1 : 0);
  p.cs = 16;
  p.dense_k = 1;

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
  // 4 blocks of 128 rows per CTA (two CTAs per SM) unless a dense group needs more than
  // 16 x 512 rows, then 8 blocks (one CTA per SM).
  const bool big = p.mode != 2 && group_rows > 16 * 512;
  if (fmt == FP8_DT_E4M3)
    return big ? run_cols<FP8_DT_E4M3, 8>(p, tout, c) : run_cols<FP8_DT_E4M3, 4>(p, tout, c);
  return big ? run_cols<FP8_DT_E5M2, 8>(p, tout, c) : run_cols<FP8_DT_E5M2, 4>(p, tout, c);
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
