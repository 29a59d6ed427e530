// Row-wise FP8 quantization (sm_103a): one scale per row, each element read once. A row's amax
// and its cast come from the same registers: amax -> fp64 scale (by table) -> fp32 multiply ->
// RNE saturating cast -> row-major codes, with no intermediate tensor in HBM.
//
// Recipe: "FP8 Training: Quantization, Autograd, Torchao", section 2 "The quantization math" (per
// row of A and per output column of B, i.e. along the contraction dimension). Fusion: "FP8 training
// on AMD GPUs with TorchTitan and TorchAO", "Triton Kernel Optimization", Level 1 (one kernel per
// quantization, no intermediates in HBM).
#include "common.cuh"
#include "internal.h"

namespace fp8lin {

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
//
// B128: blockwise 1 x 128 tiles instead of whole rows ("FP8 training on AMD GPUs with TorchTitan and
// TorchAO", "AMD FP8 format in TorchAO": a scale per tile). A tile is 16 consecutive 16-byte vectors,
// i.e. the vectors one load step gives 16 consecutive lanes of a warp; those lanes reduce its amax by
// shuffles, take its scale from the table, and the first of them writes the tile's inverse scale
// (inv [R, C / 128]).
constexpr int kRowWarpVPL = 16;
template <int FMT, int WPR, bool B128 = false>
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
    if (B128) {
      uint2* qr = q + r * nvec;
#pragma unroll
      for (int i = 0; i < kRowWarpVPL; ++i) {
        const int c = t + TPR * i;
        uint32_t a = absmax_fold(absmax_vec8(0u, v[i]));
#pragma unroll
        for (int o = 1; o < 16; o <<= 1) a = max(a, __shfl_xor_sync(0xffffffffu, a, o));  // the 16-lane tile
        if (c >= nvec) continue;  // uniform across the tile's 16 lanes (nvec % 16 == 0)
        const Scale sc = tab_scale(tab, a);
        if ((t & 15) == 0) inv[r * (nvec / 16) + c / 16] = sc.inv32;
        const float2 s2 = make_float2(sc.s32, sc.s32);
        const uint4 d = v[i];
        float2 e = fmul2_rn(make_float2(__uint_as_float(d.x << 16), __uint_as_float(d.x & 0xFFFF0000u)), s2);
        float2 f = fmul2_rn(make_float2(__uint_as_float(d.y << 16), __uint_as_float(d.y & 0xFFFF0000u)), s2);
        uint2 o;
        o.x = cvt_fp8x2<FMT>(e.x, e.y) | (cvt_fp8x2<FMT>(f.x, f.y) << 16);
        e = fmul2_rn(make_float2(__uint_as_float(d.z << 16), __uint_as_float(d.z & 0xFFFF0000u)), s2);
        f = fmul2_rn(make_float2(__uint_as_float(d.w << 16), __uint_as_float(d.w & 0xFFFF0000u)), s2);
        o.y = cvt_fp8x2<FMT>(e.x, e.y) | (cvt_fp8x2<FMT>(f.x, f.y) << 16);
        qr[c] = o;
      }
      continue;
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

template <int FMT, int WPR, bool B128 = false>
static int run_rows_warp(const void* x, int64_t R, int nvec, void* q, float* inv, const Ctx& c) {
  auto kern = quant_rows_warp_kernel<FMT, WPR, B128>;
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

// Blockwise 1 x 128 tiles of rows of 512-16384 elements (C % 128 == 0): the row kernel's teams with
// a scale per 16-lane tile. Returns FP8_ERR_UNSUPPORTED outside that range.
int launch_quant_rows_blk128(const void* x, int64_t R, int64_t C, int fmt, void* q, float* inv, const Ctx& c) {
  const int nvec = (int)(C / 8);
  if (C % 128 || nvec < 64 || nvec > 128 * kRowWarpVPL) return FP8_ERR_UNSUPPORTED;
  if (R == 0) return FP8_OK;
  const bool e4 = fmt == FP8_DT_E4M3;
  if (nvec <= 32 * kRowWarpVPL)
    return e4 ? run_rows_warp<FP8_DT_E4M3, 1, true>(x, R, nvec, q, inv, c) : run_rows_warp<FP8_DT_E5M2, 1, true>(x, R, nvec, q, inv, c);
  if (nvec <= 64 * kRowWarpVPL)
    return e4 ? run_rows_warp<FP8_DT_E4M3, 2, true>(x, R, nvec, q, inv, c) : run_rows_warp<FP8_DT_E5M2, 2, true>(x, R, nvec, q, inv, c);
  return e4 ? run_rows_warp<FP8_DT_E4M3, 4, true>(x, R, nvec, q, inv, c) : run_rows_warp<FP8_DT_E5M2, 4, true>(x, R, nvec, q, inv, c);
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

}  // namespace fp8lin
