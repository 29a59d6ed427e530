// Tensorwise FP8 quantization (sm_103a): amax -> fp64 scale (by table) -> fp32 multiply -> clamp ->
// RNE saturating cast, with no intermediate tensor in HBM. (Row-wise: rows.cu; column-wise: cols.cu.)
//
// Recipe: "FP8 Training: Quantization, Autograd, Torchao", section 2 "The quantization math".
// Fusion and layout design: "FP8 training on AMD GPUs with TorchTitan and TorchAO", "Triton
// Kernel Optimization": Level 1 (one kernel per quantization, no intermediates in HBM; the
// dual row/column-major output), Level 2 (column-wise scales with the output tile transposed
// on chip so the column-major writes are coalesced), Level 3 (relaxed atomics for the
// commutative amax reduction).
//
// Tensor granularity needs the amax of the whole tensor before the first element can be cast, so
// the input is read twice: an amax pass whose loads keep the lines in L2, then the cast pass,
// which reads them again mostly from L2.
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
//          column-major copy by 128 x 64 tiles transposed through shared memory (only where the
//          stash kernel of tensor.cu cannot store the row-major codes by TMA: C % 16 != 0).
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
  // with a column-major output: tensor.cu, part of the tensor kept on chip between the reads
  // (row-major alone is as fast by the grid-stride walk below: 34 / 95 us for 8192 x 4096 /
  // 8192 x 14336 against 34 / 105 us)
  if (qt && tensor_stash_ok(R, C, q != nullptr, true))
    return launch_quant_tensor_stash(x, R, C, fmt, q, qt, inv, ws, c);
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
