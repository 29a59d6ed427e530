// Allocation-free variant of the tensorwise quantize, for callers that cannot allocate device
// memory (see fp8_quantize_tensor_noalloc in include/fp8lin.h).
//
// The ordinary entry point reduces the tensor's amax through a caller-provided workspace word.
// Here the reduction's scratch is this file's static device array instead: the first kernel
// writes one partial maximum per CTA into it, a second kernel folds those partials into the
// array's last slot, and the existing cast kernel reads that slot. Every slot a call reads is
// written earlier in the same call, so nothing has to be cleared between calls.
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace fp8lin {
namespace {

constexpr int kSlots = FP8_NOALLOC_MAX_PARTIALS;  // partial maxima, one per CTA of phase 1
constexpr int kVecPerCta = 4096;                  // 16-byte vectors (8 bf16) per phase-1 CTA

// Shared by every call on this device; lives until the process exits.
static __device__ __align__(256) uint32_t g_scratch[kSlots + 1];

__global__ void __launch_bounds__(256) amax_partials_kernel(const uint4* __restrict__ x, int64_t nvec,
                                                            uint32_t* __restrict__ partials) {
  __shared__ uint32_t red[8];
  const int64_t base = (int64_t)blockIdx.x * kVecPerCta;
  uint32_t acc = 0;
#pragma unroll 4
  for (int i = threadIdx.x; i < kVecPerCta; i += 256) {
    const int64_t v = base + i;
    if (v < nvec) acc = absmax_vec8(acc, ld_nc_v4(x + v));
  }
  const uint32_t m = __reduce_max_sync(0xffffffffu, absmax_fold(acc));
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x == 0) {
    uint32_t mm = 0;
    for (int w = 0; w < 8; ++w) mm = max(mm, red[w]);
    partials[blockIdx.x] = mm;
  }
}

__global__ void __launch_bounds__(1024) amax_finalize_kernel(uint32_t* __restrict__ scratch, int n_partials) {
  __shared__ uint32_t red[32];
  uint32_t acc = 0;
  for (int i = threadIdx.x; i < n_partials; i += 1024) acc = max(acc, scratch[i]);
  const uint32_t m = __reduce_max_sync(0xffffffffu, acc);
  if ((threadIdx.x & 31) == 0) red[threadIdx.x >> 5] = m;
  __syncthreads();
  if (threadIdx.x < 32) {
    const uint32_t mm = __reduce_max_sync(0xffffffffu, red[threadIdx.x]);
    if (threadIdx.x == 0) scratch[kSlots] = mm;  // the final amax word
  }
}

// Device address of g_scratch, looked up once per device with that device current.
constexpr int kMaxDevices = 64;
uint32_t* scratch_address(int device, int* rc) {
  static std::mutex mu;
  static uint32_t* addr[kMaxDevices];
  if (device < 0 || device >= kMaxDevices) {
    *rc = FP8_ERR_DEVICE;
    return nullptr;
  }
  std::lock_guard<std::mutex> lock(mu);
  if (!addr[device]) {
    void* p = nullptr;
    if (cudaGetSymbolAddress(&p, g_scratch) != cudaSuccess || p == nullptr) {
      *rc = FP8_ERR_CUDA;
      return nullptr;
    }
    addr[device] = static_cast<uint32_t*>(p);
  }
  *rc = FP8_OK;
  return addr[device];
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace
}  // namespace fp8lin

using namespace fp8lin;

extern "C" int fp8_quantize_tensor_noalloc(const fp8_tensor* x, int out_dtype, int layout, fp8_tensor* out,
                                           fp8_tensor* out_t, fp8_tensor* inv_scale, void* stream) {
  // Host-side checks first: they need no device.
  if (!x || x->dtype != FP8_DT_BF16 || x->ndim != 2 || x->shape[0] < 0 || x->shape[1] < 0) return FP8_ERR_INVALID_ARG;
  if (out_dtype != FP8_DT_E4M3 && out_dtype != FP8_DT_E5M2) return FP8_ERR_INVALID_ARG;
  if (layout < 1 || layout > 3) return FP8_ERR_INVALID_ARG;
  if (!inv_scale || !inv_scale->ptr || inv_scale->dtype != FP8_DT_F32 || inv_scale->ndim < 1 || inv_scale->ndim > 3)
    return FP8_ERR_INVALID_ARG;
  int64_t inv_n = 1;
  for (int i = 0; i < inv_scale->ndim; ++i) {
    if (inv_scale->shape[i] != 1) return FP8_ERR_INVALID_ARG;  // exactly one scale
    inv_n *= inv_scale->shape[i];
  }
  if (inv_n != 1) return FP8_ERR_INVALID_ARG;
  const int64_t R = x->shape[0], C = x->shape[1];
  if (C % 8 != 0) return FP8_ERR_ALIGNMENT;
  // each extent within the limit before the product (no overflow), then the element count:
  // more elements than the array's partial maxima cover is rejected
  if (R >= ((int64_t)1 << 31) || C > FP8_NOALLOC_MAX_ELEMENTS) return FP8_ERR_UNSUPPORTED;
  if (R * C > FP8_NOALLOC_MAX_ELEMENTS) return FP8_ERR_UNSUPPORTED;
  const bool want_row = layout & FP8_LAYOUT_ROW_MAJOR, want_col = layout & FP8_LAYOUT_COL_MAJOR;
  if (want_row) {
    if (!out || out->dtype != out_dtype || out->ndim != 2 || out->shape[0] != R || out->shape[1] != C)
      return FP8_ERR_INVALID_ARG;
    if ((R * C > 0 && !out->ptr) || !aligned16(out->ptr)) return FP8_ERR_ALIGNMENT;
  }
  if (want_col) {
    if (!out_t || out_t->dtype != out_dtype || out_t->ndim != 2 || out_t->shape[0] != C || out_t->shape[1] != R)
      return FP8_ERR_INVALID_ARG;
    if (R % 16 != 0 || (R * C > 0 && !out_t->ptr) || !aligned16(out_t->ptr)) return FP8_ERR_ALIGNMENT;
  }
  if ((R * C > 0 && !x->ptr) || !aligned16(x->ptr)) return FP8_ERR_ALIGNMENT;

  Ctx c;
  int rc = make_ctx(&c, stream, nullptr);
  if (rc != FP8_OK) return rc;
  uint32_t* scratch = scratch_address(c.device, &rc);
  if (rc != FP8_OK) return rc;

  const int64_t nvec = R * C / 8;
  const int n_partials = (int)((nvec + kVecPerCta - 1) / kVecPerCta);
  if (n_partials > 0) {
    amax_partials_kernel<<<n_partials, 256, 0, c.stream>>>(static_cast<const uint4*>(x->ptr), nvec, scratch);
    if (cudaGetLastError() != cudaSuccess) return FP8_ERR_CUDA;
  }
  amax_finalize_kernel<<<1, 1024, 0, c.stream>>>(scratch, n_partials);  // 0 partials -> amax 0
  if (cudaGetLastError() != cudaSuccess) return FP8_ERR_CUDA;
  return launch_quant_tensor_cast(x->ptr, R, C, out_dtype, want_row ? out->ptr : nullptr,
                                  want_col ? out_t->ptr : nullptr, static_cast<float*>(inv_scale->ptr),
                                  scratch + kSlots, c);
}
