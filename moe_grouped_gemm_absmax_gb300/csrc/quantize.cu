// Tensorwise and column-wise FP8 quantization (sm_103a): amax -> fp64 scale (by table) -> fp32
// multiply -> clamp -> RNE saturating cast, with no intermediate tensor in HBM. (Row-wise: rows.cu.)
//
// Recipe: "FP8 Training: Quantization, Autograd, Torchao", section 2 "The quantization math".
// Fusion and layout design: "FP8 training on AMD GPUs with TorchTitan and TorchAO", "Triton
// Kernel Optimization": Level 1 (one kernel per quantization, no intermediates in HBM; the
// dual row/column-major output), Level 2 (column-wise scales with the output tile transposed
// on chip so the column-major writes are coalesced), Level 3 (relaxed atomics for the
// commutative amax reduction).
//
// Tensor and column granularity need the amax of a whole tensor or column before the first element
// can be cast, so the input is read twice: an amax pass whose loads keep the lines in L2, then the
// cast pass, which reads them again mostly from L2.
#include "common.cuh"
#include "internal.h"

namespace fp8lin {


// ==========================================================================================
// Tensorwise cast with a given amax (fp8_quantize_from_amax, the allocation-free variant): one scale; row-major output from registers and/or the
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

// ==========================================================================================
// Tensorwise in one launch. Every CTA is resident at once (cooperative launch), so the CTAs can
// meet at a grid barrier between the two steps the recipe needs:
//   amax   a grid-stride read of the whole tensor (8 independent 16-byte loads in flight per thread;
//          the loads keep their lines in L2 for the cast), |x| folded as packed bf16 maxima, one
//          relaxed atomic max per CTA on the workspace's amax word;
//   barrier each CTA counts itself on the workspace's barrier word with a release increment (its
//          atomic max is ordered before it) and waits, bounded, until all have (acquire loads);
//   cast   the scale from the table, then the cast of the tensor read again, mostly from L2:
//          row-major only by a grid-stride walk in the amax pass's order, 8-byte stores; with the
//          column-major copy by 128 x 64 tiles transposed through shared memory (dual output).
// A wait that runs out sets FP8_DEV_TIMEOUT and the CTA leaves without casting (the failure-detection
// test hook fp8_set_test_stall makes it wait for one arrival that never comes).
constexpr int kTfThreads = 256;
constexpr int kTfUnroll = 8;

template <int FMT>
__global__ void __launch_bounds__(kTfThreads) quant_tensor_fused_kernel(
    const uint16_t* __restrict__ x, int64_t R, int64_t C, uint32_t* __restrict__ ws, uint8_t* __restrict__ q,
    uint8_t* __restrict__ qt, float* __restrict__ inv, int32_t* status, uint64_t wait_ns, int test_stall,
    const __grid_constant__ ScaleTab tab) {
  constexpr float FMAX = FmtMax<FMT>::v;
  __shared__ uint32_t red[kTfThreads / 32];
  __shared__ float s_sc;
  __shared__ int s_ok;
  __shared__ __align__(16) uint8_t T[kTcCols * kTcPitch];
  const int tid = threadIdx.x;
  const uint4* xv = reinterpret_cast<const uint4*>(x);
  const int64_t nvec = R * C / 8;
  const int64_t stride = (int64_t)gridDim.x * kTfThreads;
  const int64_t first = (int64_t)blockIdx.x * kTfThreads + tid;

  // ---- amax ----
  {
    const uint64_t keep = l2_evict_last();
    uint32_t acc = 0;
    int64_t i = first;
    for (; i + (kTfUnroll - 1) * stride < nvec; i += kTfUnroll * stride) {
      uint4 v[kTfUnroll];
#pragma unroll
      for (int u = 0; u < kTfUnroll; ++u) v[u] = ld_nc_v4_hint(xv + i + u * stride, keep);
#pragma unroll
      for (int u = 0; u < kTfUnroll; ++u) acc = absmax_vec8(acc, v[u]);
    }
    for (; i < nvec; i += stride) acc = absmax_vec8(acc, ld_nc_v4_hint(xv + i, keep));
    const uint32_t m = __reduce_max_sync(0xffffffffu, absmax_fold(acc));
    if ((tid & 31) == 0) red[tid >> 5] = m;
  }
  __syncthreads();
  // ---- grid barrier, then the scale ----
  if (tid == 0) {
    uint32_t mm = 0;
    for (int w = 0; w < kTfThreads / 32; ++w) mm = max(mm, red[w]);
    if (mm) red_max_relaxed(ws, mm);
    red_add_release_gpu(ws + 1, 1u);
    // the failure-detection test hook waits for one arrival more than there are CTAs
    const bool ok = wait_count_geq(ws + 1, gridDim.x + (test_stall ? 1u : 0u), wait_ns);
    if (!ok) set_status(status, FP8_DEV_TIMEOUT);
    const Scale sc = tab_scale(tab, ld_relaxed_gpu(ws));
    s_sc = sc.s32;
    s_ok = ok;
    if (blockIdx.x == 0 && ok) *inv = sc.inv32;
  }
  __syncthreads();
  if (!s_ok) return;
  const float s32 = s_sc;
  const uint64_t last = l2_evict_first();  // the input's last use; output nothing re-reads soon

  // ---- cast: row-major only ----
  if (!qt) {
    uint2* qv = reinterpret_cast<uint2*>(q);
    int64_t i = first;
    for (; i + (kTfUnroll - 1) * stride < nvec; i += kTfUnroll * stride) {
      uint4 v[kTfUnroll];
#pragma unroll
      for (int u = 0; u < kTfUnroll; ++u) v[u] = ld_nc_v4_hint(xv + i + u * stride, last);
#pragma unroll
      for (int u = 0; u < kTfUnroll; ++u) st_v2_hint(qv + i + u * stride, quant_vec8<FMT>(v[u], s32, FMAX), last);
    }
    for (; i < nvec; i += stride) st_v2_hint(qv + i, quant_vec8<FMT>(ld_nc_v4_hint(xv + i, last), s32, FMAX), last);
    return;
  }
  // ---- cast: tiles of 128 rows x 64 columns, the column-major copy through shared memory; the
  // next tile's loads are in flight while the current one is cast, transposed and stored ----
  const int64_t ncb = ceil_div64(C, kTcCols), ntiles = ceil_div64(R, kTcRows) * ncb;
  auto load_tile = [&](int64_t t, uint4* v) {
    const int64_t r0 = (t / ncb) * kTcRows, c0 = (t % ncb) * kTcCols;
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int vi = tid + kTfThreads * k;  // 128 rows x 8 vectors
      const int64_t r = r0 + (vi >> 3), col = c0 + (vi & 7) * 8;
      v[k] = (r < R && col < C) ? ld_nc_v4_hint(x + r * C + col, last) : make_uint4(0, 0, 0, 0);
    }
  };
  uint4 nx[4];
  if ((int64_t)blockIdx.x < ntiles) load_tile(blockIdx.x, nx);
  for (int64_t t = blockIdx.x; t < ntiles; t += gridDim.x) {
    const int64_t r0 = (t / ncb) * kTcRows, c0 = (t % ncb) * kTcCols;
    uint4 v[4];
#pragma unroll
    for (int k = 0; k < 4; ++k) v[k] = nx[k];
    if (t + gridDim.x < ntiles) load_tile(t + gridDim.x, nx);
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      const int vi = tid + kTfThreads * k;
      const int rr = vi >> 3, cv = vi & 7;
      const int64_t r = r0 + rr, col = c0 + cv * 8;
      const uint2 o = quant_vec8<FMT>(v[k], s32, FMAX);
      if (q && r < R && col < C) st_v2_hint(q + r * C + col, o, last);
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        const uint32_t w = j < 4 ? o.x : o.y;
        T[(cv * 8 + j) * kTcPitch + rr] = (uint8_t)(w >> (8 * (j & 3)));
      }
    }
    __syncthreads();
    for (int i = tid; i < kTcCols * (kTcRows / 16); i += kTfThreads) {
      const int cl = i >> 3, k = i & 7;
      const int64_t col = c0 + cl, r = r0 + 16 * k;
      if (col < C && r < R) {  // R % 16 == 0: the 16-byte chunk is all in range
        const uint32_t* src = reinterpret_cast<const uint32_t*>(T + cl * kTcPitch + 16 * k);
        st_v4_hint(qt + col * R + r, make_uint4(src[0], src[1], src[2], src[3]), last);
      }
    }
    __syncthreads();  // T is rewritten by the next tile
  }
}

int launch_quant_tensor(const void* x, int64_t R, int64_t C, int fmt, void* q, void* qt, float* inv,
                        uint32_t* ws, const Ctx& c) {
  // ws[0]: the amax word, ws[1]: the barrier count; both start at zero
  if (cudaMemsetAsync(ws, 0, 2 * sizeof(uint32_t), c.stream) != cudaSuccess) return FP8_ERR_CUDA;
  auto kern = fmt == FP8_DT_E4M3 ? quant_tensor_fused_kernel<FP8_DT_E4M3> : quant_tensor_fused_kernel<FP8_DT_E5M2>;
  int per_sm = 0;
  if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kTfThreads, 0) != cudaSuccess || per_sm < 1)
    return FP8_ERR_CUDA;
  const int64_t nvec = R * C / 8;
  const int64_t work = qt ? ceil_div64(R, kTcRows) * ceil_div64(C, kTcCols) : ceil_div64(nvec, kTfThreads * kTfUnroll);
  const int64_t cap = (int64_t)c.sm_count * per_sm;
  const unsigned grid = (unsigned)(work < 1 ? 1 : (work < cap ? work : cap));
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs resident: they meet at the grid barrier
  attr[0].val.cooperative = 1;
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kTfThreads);
  cfg.dynamicSmemBytes = 0;
  cfg.stream = c.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, static_cast<const uint16_t*>(x), R, C, ws, static_cast<uint8_t*>(q),
                         static_cast<uint8_t*>(qt), inv, c.status, c.wait_ns, c.test_stall, scale_tab(fmt)) != cudaSuccess)
    return FP8_ERR_CUDA;
  return FP8_OK;
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
//              its first reads are the tiles pass 1 read last.
// Both passes run in one launch: every CTA is resident (cooperative launch), and between the passes
// each CTA counts itself on the workspace's barrier word (release) and waits, bounded, until all
// have, so every column maximum is complete before pass 2 reads it. Pass 1's loads keep their lines
// in L2 and pass 2 re-reads them right after the barrier, mostly from L2. With the maxima given
// (fp8_quantize_from_amax) the launch runs pass 2 alone.
constexpr int kColThreads = 256;
constexpr int kColNB = 2;                  // 128-row blocks per work unit (256 rows)
constexpr int kColTile = 128 * kColNB;
constexpr int kColStages = 5;  // ring stages (pass 2's staging boxes take the rest of shared memory)
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
  int first_pass;      // 0: both passes; 1: pass 2 alone (maxima given)
  uint32_t* barrier;   // grid-barrier count between the passes (zeroed by the launcher)
  int test_stall;      // failure-detection test hook: the barrier waits for one arrival more
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
  uint64_t full[kColStages];   // the tile landed (TMA bytes) and the info was written
  uint64_t scl[kColStages];    // pass 2: the stage's 64 amax words landed (32 async arrivals)
  uint64_t empty[kColStages];  // the consumer warps are done with the stage
  ColInfo info[kColStages];
  uint32_t am[kColStages][64];  // pass 2: the amax words of the stage's 64 columns
  uint32_t red[kColConsumerWarps][8][4];
  int abort;
};
constexpr int kColSmemBytes = 1024 + kColStages * kColStageBytes + 2 * kColOutBytes + (int)sizeof(ColShared);

template <int FMT>
__global__ void __launch_bounds__(kColThreads + 64, 1) colstream_kernel(const __grid_constant__ CUtensorMap tm_in,
                                                                        const __grid_constant__ CUtensorMap tm_out,
                                                                        const ColParams p,
                                                                        const __grid_constant__ ScaleTab tab) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* ring = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* Tout = ring + kColStages * kColStageBytes;
  ColShared& S = *reinterpret_cast<ColShared*>(Tout + 2 * kColOutBytes);
  int32_t* upre = reinterpret_cast<int32_t*>(&S + 1);
  int32_t* ppre = upre + (p.n_groups + 1);
  const int64_t M = col_setup(p, upre, ppre);
  if (M < 0) return;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  // the scale table in shared memory: the lanes of a warp look up different entries at once
  __shared__ ScaleTab stab;
  static_assert(sizeof(ScaleTab) % 4 == 0, "table words");
  for (int i = tid; i < (int)(sizeof(ScaleTab) / 4); i += blockDim.x)
    reinterpret_cast<uint32_t*>(&stab)[i] = reinterpret_cast<const uint32_t*>(&tab)[i];
  auto init_barriers = [&]() {
    for (int s = 0; s < kColStages; ++s) {
      mbar_init(&S.full[s], 1);
      mbar_init(&S.scl[s], 32);
      mbar_init(&S.empty[s], kColConsumerWarps);
    }
    fence_mbar_init();
  };
  if (tid == 0) {
    init_barriers();
    S.abort = 0;
    tma_prefetch_desc(&tm_in);
    tma_prefetch_desc(&tm_out);
  }
  // Groups without rows have no units: their inverse scales (amax 0) are written here.
  if (blockIdx.x == 0) {
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
  volatile int* cta_abort = &S.abort;

  for (int pass = p.first_pass; pass < 2; ++pass) {
  const bool CAST = pass == 1;
  if (CAST && p.first_pass == 0) {
    // between the passes: every CTA's column maxima are complete before any CTA reads one
    __syncthreads();
    if (tid == 0) {
      if (!*cta_abort) {
        __threadfence();
        red_add_release_gpu(p.barrier, 1u);
        if (!wait_count_geq(p.barrier, gridDim.x + (p.test_stall ? 1u : 0u), p.wait_ns)) {
          *cta_abort = 1;
          set_status(p.status, FP8_DEV_TIMEOUT);
        }
      }
      if (!*cta_abort) {  // every load of pass 1 was consumed: fresh barriers for pass 2
        for (int s = 0; s < kColStages; ++s) {
          mbar_inval(&S.full[s]);
          mbar_inval(&S.scl[s]);
          mbar_inval(&S.empty[s]);
        }
        init_barriers();
      }
    }
    __syncthreads();
    if (*cta_abort) break;
  }
  auto unit_at = [&](int64_t k) {
    const int64_t i = blockIdx.x + k * gridDim.x;
    return CAST ? M - 1 - i : i;
  };

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
  }  // passes
  __syncthreads();
}

// Workspace words of a column quantize: the amax per (group, column), rounded to 16 bytes.
int64_t col_ws_words(int64_t groups, int64_t C) { return round_up64(groups * C, 4) + 4; }  // + the barrier count

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
  p.test_stall = c.test_stall;

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
    p.first_pass = 1;
  } else {
    if (cudaMemsetAsync(scratch, 0, (size_t)col_ws_words(n_groups, C) * 4, c.stream) != cudaSuccess) return FP8_ERR_CUDA;
    p.first_pass = 0;
    p.barrier = scratch + round_up64(n_groups * C, 4);
  }
  // units: exact for dense modes; for segments an upper bound (each segment adds at most one
  // partial tile) -- the kernels compute the exact count from the offsets
  const int64_t units = p.mode == 2 ? (ceil_div64(rows_total, kColTile) + n_groups) * p.n_strips
                                    : n_groups * ceil_div64(group_rows, kColTile) * p.n_strips;
  if (units > INT32_MAX) return FP8_ERR_UNSUPPORTED;  // the kernels decode units in 32 bits
  const size_t pre = p.mode == 2 ? 12 * (size_t)(n_groups + 1) : 0;
  const int64_t grid = units > 0 ? (units < c.sm_count ? units : c.sm_count) : 1;
  const ScaleTab& tab = scale_tab(fmt);
  auto kern = fmt == FP8_DT_E4M3 ? colstream_kernel<FP8_DT_E4M3> : colstream_kernel<FP8_DT_E5M2>;
  const size_t smem = kColSmemBytes + pre;
  if (cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)smem) != cudaSuccess)
    return FP8_ERR_CUDA;
  cudaLaunchConfig_t cfg = {};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;  // all CTAs resident: they meet between the passes
  attr[0].val.cooperative = 1;
  cfg.gridDim = dim3((unsigned)grid);
  cfg.blockDim = dim3(kColThreads + 64);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = c.stream;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (cudaLaunchKernelEx(&cfg, kern, tin, tout, p, tab) != cudaSuccess) return FP8_ERR_CUDA;
  return FP8_OK;
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
