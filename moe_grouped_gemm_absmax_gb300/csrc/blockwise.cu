// Blockwise quantization on sm_103a: one scale per fixed-size tile ("FP8 training on AMD GPUs
// with TorchTitan and TorchAO", section "AMD FP8 format in TorchAO"). The tile shapes are not
// given there; this library takes 1 x 128 tiles for activations and gradients (a scale per row and
// 128 consecutive elements of the contraction) and 128 x 128 tiles for weights, each tile
// quantized by the recipe of "FP8 Training: Quantization, Autograd, Torchao" section 2 (amax,
// fp64 scale with eps from the host-built table, fp32 multiply, clamp, cast, fp64 reciprocal).
//
// A CTA owns a 128 x 128 bf16 tile (256 threads, eight 16-byte loads each):
//   1 x 128:   the 16 lanes holding a row reduce its maximum with four shuffles, take the scale
//              from the table and cast from registers (8-byte coalesced stores);
//   128 x 128: the tile's maximum by warp shuffles and shared memory, one scale for all; the
//              row-major codes straight from registers, the column-major codes (the transposed
//              operand of the grad-input GEMM; a square tile keeps its scale under transposition)
//              through shared memory as 128-byte rows.
#include "common.cuh"
#include "internal.h"

namespace fp8lin {

namespace {

constexpr int kBT = 128;               // tile rows and columns
constexpr int kBThreads = 256;
constexpr int kBInPitch = kBT + 8;     // bf16 per staged input row
constexpr int kBOutPitch = kBT + 16;   // bytes per staged output row
constexpr int kBSmem = kBT * kBInPitch * 2 + kBT * kBOutPitch;

template <int FMT>
struct BlkMax;
template <>
struct BlkMax<FP8_DT_E4M3> {
  static constexpr float v = 448.0f;
};
template <>
struct BlkMax<FP8_DT_E5M2> {
  static constexpr float v = 57344.0f;
};

struct BlkArgs {
  const uint16_t* x;
  int64_t R, C;
  uint8_t* q;      // row-major codes [R, C], or null
  uint8_t* qt;     // column-major codes [C, R] (128 x 128 tiles only), or null
  float* inv;      // 1 x 128: [R, C / 128]; 128 x 128: [ceil(R / 128), C / 128] (may be null with qt)
  float* inv_t;    // 128 x 128 with qt: [C / 128, R / 128] (the same values, transposed), or null
};

template <int FMT, bool TILE, bool ROWS, bool COLS>
__global__ void __launch_bounds__(kBThreads) blk_quant_kernel(const BlkArgs a, const __grid_constant__ ScaleTab tab) {
  extern __shared__ __align__(16) uint8_t blk_smem[];
  __shared__ uint32_t wmax[kBThreads / 32];
  __shared__ Scale tile_scale;
  constexpr float FMAX = BlkMax<FMT>::v;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int64_t c0 = (int64_t)blockIdx.x * kBT, r0 = (int64_t)blockIdx.y * kBT;
  const int valid = (int)(a.R - r0 < kBT ? a.R - r0 : kBT);
  const int cc = (lane & 15) * 8;
  uint4 v[8];
#pragma unroll
  for (int it = 0; it < 8; ++it) {
    const int rr = it * 16 + warp * 2 + (lane >> 4);
    v[it] = rr < valid ? ld_nc_v4(a.x + (r0 + rr) * a.C + c0 + cc) : make_uint4(0, 0, 0, 0);
  }
  if (!TILE) {
    // 1 x 128: one scale per row of the tile
    const int64_t ncb = a.C / kBT;
#pragma unroll
    for (int it = 0; it < 8; ++it) {
      const int rr = it * 16 + warp * 2 + (lane >> 4);
      uint32_t m = absmax_fold(absmax_vec8(0u, v[it]));
#pragma unroll
      for (int o = 1; o < 16; o <<= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
      const Scale sc = tab_scale(tab, m);
      const uint2 o8 = quant_vec8<FMT>(v[it], sc.s32, FMAX);
      if (rr < valid) {
        *reinterpret_cast<uint2*>(a.q + (r0 + rr) * a.C + c0 + cc) = o8;
        if ((lane & 15) == 0) a.inv[(r0 + rr) * ncb + (c0 >> 7)] = sc.inv32;
      }
    }
    return;
  }
  // 128 x 128: the tile's maximum, one scale
  uint32_t m = 0;
#pragma unroll
  for (int it = 0; it < 8; ++it) m = absmax_vec8(m, v[it]);
  m = absmax_fold(m);
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) m = max(m, __shfl_xor_sync(0xffffffffu, m, o));
  if (lane == 0) wmax[warp] = m;
  __syncthreads();
  if (tid == 0) {
    uint32_t t = 0;
#pragma unroll
    for (int w = 0; w < kBThreads / 32; ++w) t = max(t, wmax[w]);
    const Scale sc = tab_scale(tab, t);
    tile_scale = sc;
    const int64_t ncb = a.C / kBT;
    if (a.inv) a.inv[blockIdx.y * ncb + blockIdx.x] = sc.inv32;
    if (COLS && a.inv_t) a.inv_t[blockIdx.x * (a.R / kBT) + blockIdx.y] = sc.inv32;
  }
  __syncthreads();
  const float s32 = tile_scale.s32;
  if (ROWS) {
#pragma unroll
    for (int it = 0; it < 8; ++it) {
      const int rr = it * 16 + warp * 2 + (lane >> 4);
      if (rr < valid) *reinterpret_cast<uint2*>(a.q + (r0 + rr) * a.C + c0 + cc) = quant_vec8<FMT>(v[it], s32, FMAX);
    }
  }
  if (COLS) {
    uint16_t* sx = reinterpret_cast<uint16_t*>(blk_smem);
    uint8_t* so = blk_smem + kBT * kBInPitch * 2;
#pragma unroll
    for (int it = 0; it < 8; ++it) {
      const int rr = it * 16 + warp * 2 + (lane >> 4);
      *reinterpret_cast<uint4*>(sx + rr * kBInPitch + cc) = v[it];
    }
    __syncthreads();
    // thread: columns (2 cp, 2 cp + 1), rows 32 qb .. 32 qb + 31, from packed 32-bit loads
    const int cp = tid & 63, qb = tid >> 6;
    const int rb = 32 * qb;
    uint32_t lo[8], hi[8];
#pragma unroll
    for (int r = 0; r < 32; r += 4) {
      uint32_t w4[4];
#pragma unroll
      for (int i = 0; i < 4; ++i) w4[i] = *reinterpret_cast<const uint32_t*>(sx + (rb + r + i) * kBInPitch + 2 * cp);
      const uint32_t l01 = (w4[0] & 0xFFFFu) | (w4[1] << 16), l23 = (w4[2] & 0xFFFFu) | (w4[3] << 16);
      const uint32_t h01 = (w4[0] >> 16) | (w4[1] & 0xFFFF0000u), h23 = (w4[2] >> 16) | (w4[3] & 0xFFFF0000u);
      lo[r / 4] = quant_bf16x2<FMT>(l01, s32, FMAX) | (quant_bf16x2<FMT>(l23, s32, FMAX) << 16);
      hi[r / 4] = quant_bf16x2<FMT>(h01, s32, FMAX) | (quant_bf16x2<FMT>(h23, s32, FMAX) << 16);
    }
    uint8_t* dlo = so + (2 * cp) * kBOutPitch + rb;
    uint8_t* dhi = dlo + kBOutPitch;
    *reinterpret_cast<uint4*>(dlo) = make_uint4(lo[0], lo[1], lo[2], lo[3]);
    *reinterpret_cast<uint4*>(dlo + 16) = make_uint4(lo[4], lo[5], lo[6], lo[7]);
    *reinterpret_cast<uint4*>(dhi) = make_uint4(hi[0], hi[1], hi[2], hi[3]);
    *reinterpret_cast<uint4*>(dhi + 16) = make_uint4(hi[4], hi[5], hi[6], hi[7]);
    __syncthreads();
#pragma unroll
    for (int i = 0; i < kBT / 32; ++i) {
      const int cr = i * 32 + warp * 4 + (lane >> 3);
      const int ch = (lane & 7) * 16;
      *reinterpret_cast<uint4*>(a.qt + (c0 + cr) * a.R + r0 + ch) = *reinterpret_cast<const uint4*>(so + cr * kBOutPitch + ch);
    }
  }
}

template <int FMT, bool TILE, bool ROWS, bool COLS>
int run_blk(const BlkArgs& a, const Ctx& c) {
  auto kern = blk_quant_kernel<FMT, TILE, ROWS, COLS>;
  const int smem = COLS ? kBSmem : 0;
  if (COLS && cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, smem) != cudaSuccess)
    return FP8_ERR_CUDA;
  const dim3 grid((unsigned)(a.C / kBT), (unsigned)((a.R + kBT - 1) / kBT));
  kern<<<grid, kBThreads, smem, c.stream>>>(a, scale_tab(FMT));
  return cudaGetLastError() == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

template <int FMT>
int dispatch_blk(const BlkArgs& a, bool tile, const Ctx& c) {
  if (!tile) return run_blk<FMT, false, true, false>(a, c);
  if (a.q && a.qt) return run_blk<FMT, true, true, true>(a, c);
  if (a.q) return run_blk<FMT, true, true, false>(a, c);
  return run_blk<FMT, true, false, true>(a, c);
}

}  // namespace

int launch_blk_quant(const void* x, int64_t R, int64_t C, int fmt, bool tile128, void* q, void* qt, float* inv,
                     float* inv_t, const Ctx& c) {
  if (C % kBT || (!q && !qt) || (!tile128 && qt) || (qt && R % kBT)) return FP8_ERR_UNSUPPORTED;
  if ((R + kBT - 1) / kBT > 65535) return FP8_ERR_UNSUPPORTED;
  if (R == 0 || C == 0) return FP8_OK;
  if (!tile128) {  // 1 x 128 tiles: the row kernel's teams where the row length suits them
    const int rc = launch_quant_rows_blk128(x, R, C, fmt, q, inv, c);
    if (rc != FP8_ERR_UNSUPPORTED) return rc;
  }
  BlkArgs a;
  a.x = static_cast<const uint16_t*>(x);
  a.R = R;
  a.C = C;
  a.q = static_cast<uint8_t*>(q);
  a.qt = static_cast<uint8_t*>(qt);
  a.inv = inv;
  a.inv_t = inv_t;
  return fmt == FP8_DT_E4M3 ? dispatch_blk<FP8_DT_E4M3>(a, tile128, c) : dispatch_blk<FP8_DT_E5M2>(a, tile128, c);
}

}  // namespace fp8lin
