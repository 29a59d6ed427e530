// Device helpers shared by the fp8lin kernels (sm_103a): inline PTX for mbarriers, TMA,
// tcgen05 / tensor memory, FP8 conversion, bounded waits and the status word.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fp8lin.h"

#define FP8_DEVI __device__ __forceinline__

namespace fp8lin {

// ------------------------------------------------------------------------------------------
// Formats: largest finite magnitude (e4m3fn 1.75 * 2^8, e5m2 1.75 * 2^15).
constexpr float kE4M3Max = 448.0f;
constexpr float kE5M2Max = 57344.0f;
// Lower clamp of amax in the scale step.
constexpr double kEps = 1e-12;

FP8_DEVI uint32_t smem_u32(const void* p) { return static_cast<uint32_t>(__cvta_generic_to_shared(p)); }

FP8_DEVI uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// Status word: conditions found on the device are OR-ed in with a relaxed atomic.
FP8_DEVI void set_status(int32_t* st, int32_t bits) {
  if (st) atomicOr(st, bits);
}

// ------------------------------------------------------------------------------------------
// Scale step: scale64 = fp8_max / max(amax, eps) with an IEEE fp64 division; the fp32 multiply
// uses scale64 rounded to fp32; the inverse handed to the GEMM is the correctly rounded fp64
// reciprocal of scale64, rounded to fp32.
//
// The kernels take this step by table, with no fp64 arithmetic on the device (GB300's fp64 rate
// is a small fraction of its fp32 rate, and the row-wise kernel would take the step once per
// row). amax is a bf16 value m * 2^E with m one of 128 mantissas in [1, 2). Scaling by a power
// of two commutes with round-to-nearest while the results stay normal, so
//   RN64(fp8_max / amax)   = RN64(fp8_max / m) * 2^-E
//   RN64(1 / scale64)      = RN64(1 / RN64(fp8_max / m)) * 2^E
// and the same holds after rounding each to fp32. ScaleTab keeps, per m, the two fp32 factors,
// computed on the host in IEEE fp64; the kernel applies 2^-E / 2^E exactly on the fp32 exponent
// field. For every amax >= eps (and <= the largest bf16) both fp32 results are normal
// (e5m2: scale <= 57344 / 1e-12 ~ 5.7e16; e4m3: scale >= 448 / 3.4e38 ~ 1.3e-36), so the table
// reproduces the fp64 step bit for bit. amax below eps takes the eps entry; amax = +Inf gives
// scale 0 and inverse +Inf, a NaN amax NaN for both, as the fp64 step would.
struct Scale {
  float s32;
  float inv32;
};
struct ScaleTab {
  float s[128];     // RN32(RN64(fp8_max / m)), m = 1 + i / 128
  float inv[128];   // RN32(RN64(1 / RN64(fp8_max / m)))
  uint32_t eps_below;  // bf16 patterns below this one encode values < eps
  float eps_s, eps_inv;
};
FP8_DEVI Scale tab_scale(const ScaleTab& t, uint32_t amax_bits) {
  Scale r;
  if (amax_bits < t.eps_below) {
    r.s32 = t.eps_s;
    r.inv32 = t.eps_inv;
  } else if (amax_bits < 0x7F80u) {
    const int e = (int)(amax_bits >> 7) - 127;
    const uint32_t m7 = amax_bits & 0x7Fu;
    r.s32 = __int_as_float(__float_as_int(t.s[m7]) - (e << 23));
    r.inv32 = __int_as_float(__float_as_int(t.inv[m7]) + (e << 23));
  } else if (amax_bits == 0x7F80u) {
    r.s32 = 0.0f;
    r.inv32 = __int_as_float(0x7F800000);
  } else {
    r.s32 = __int_as_float(0x7FC00000);
    r.inv32 = r.s32;
  }
  return r;
}

// Largest finite magnitude of a format, at compile time.
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

// Two IEEE fp32 products in one instruction (mul.rn.f32x2): bit-identical to two __fmul_rn.
FP8_DEVI float2 fmul2_rn(float2 a, float2 b) {
  uint64_t ra, rb, rd;
  asm("mov.b64 %0, {%1, %2};" : "=l"(ra) : "f"(a.x), "f"(a.y));
  asm("mov.b64 %0, {%1, %2};" : "=l"(rb) : "f"(b.x), "f"(b.y));
  asm("mul.rn.f32x2 %0, %1, %2;" : "=l"(rd) : "l"(ra), "l"(rb));
  float2 d;
  asm("mov.b64 {%0, %1}, %2;" : "=f"(d.x), "=f"(d.y) : "l"(rd));
  return d;
}

// Round-to-nearest-even, saturating casts of two fp32 values into two packed FP8 codes;
// `lo` lands in the low byte (the lower address).
template <int FMT>
FP8_DEVI uint32_t cvt_fp8x2(float lo, float hi) {
  uint16_t r;
  if (FMT == FP8_DT_E4M3)
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  else
    asm("cvt.rn.satfinite.e5m2x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
  return r;
}

// x * scale in fp32, clamp to +-fp8_max (NaN passes through), cast. Two bf16 in, two codes out.
template <int FMT>
FP8_DEVI uint32_t quant_bf16x2(uint32_t two_bf16, float s32, float fmax) {
  float a = __fmul_rn(__uint_as_float(two_bf16 << 16), s32);
  float b = __fmul_rn(__uint_as_float(two_bf16 & 0xFFFF0000u), s32);
  a = a > fmax ? fmax : (a < -fmax ? -fmax : a);
  b = b > fmax ? fmax : (b < -fmax ? -fmax : b);
  return cvt_fp8x2<FMT>(a, b);
}

// 8 bf16 (one 16-byte vector) -> 8 codes (8 bytes).
template <int FMT>
FP8_DEVI uint2 quant_vec8(uint4 v, float s32, float fmax) {
  uint2 o;
  o.x = quant_bf16x2<FMT>(v.x, s32, fmax) | (quant_bf16x2<FMT>(v.y, s32, fmax) << 16);
  o.y = quant_bf16x2<FMT>(v.z, s32, fmax) | (quant_bf16x2<FMT>(v.w, s32, fmax) << 16);
  return o;
}

// MX block scale (OCP MX v1.0): X = 2^(floor(log2(amax)) - emax_elem), exponent clamped below at -127.
// E8M0 code of a block from the bf16 pattern of its amax (sign cleared). For a normal amax,
// floor(log2 amax) = exponent field - 127, so the code (exponent + 127) is field - emax_elem,
// clamped at 0; a zero or subnormal amax lies below the clamp. Inf / NaN give the NaN code.
template <int FMT>
FP8_DEVI uint32_t mx_code(uint32_t amax_bits) {
  constexpr int kEmax = FMT == FP8_DT_E4M3 ? 8 : 15;
  const int ef = (int)(amax_bits >> 7);
  if (ef == 255) return 0xFFu;
  return ef > kEmax ? (uint32_t)(ef - kEmax) : 0u;
}

// 1 / X = 2^(127 - code) as an fp32 (a normal number for every code the rule produces).
FP8_DEVI float mx_inv(uint32_t code) {
  return code == 0xFFu ? __uint_as_float(0x7FC00000u) : __uint_as_float((254u - code) << 23);
}

// Two bf16 (one packed word) times a power of two, cast: the product is exact, so the only
// rounding is the cast's (nearest even, saturating at the format's largest finite value).
template <int FMT>
FP8_DEVI uint32_t mx_cast2(uint32_t two_bf16, float inv) {
  const float2 p = fmul2_rn(make_float2(__uint_as_float(two_bf16 << 16), __uint_as_float(two_bf16 & 0xFFFF0000u)),
                            make_float2(inv, inv));
  return cvt_fp8x2<FMT>(p.x, p.y);
}

// Elementwise unsigned max of the |bf16| patterns in two packed pairs. For non-negative
// bf16 values the bit pattern orders like the value, so amax needs no float compare.
FP8_DEVI uint32_t absmax2(uint32_t acc, uint32_t v) { return __vmaxu2(acc, v & 0x7FFF7FFFu); }
FP8_DEVI uint32_t absmax_vec8(uint32_t acc, uint4 v) {
  acc = absmax2(acc, v.x);
  acc = absmax2(acc, v.y);
  acc = absmax2(acc, v.z);
  return absmax2(acc, v.w);
}
// Larger of the two halves of a packed pair, as a bf16 pattern in the low 16 bits.
FP8_DEVI uint32_t absmax_fold(uint32_t acc) {
  uint32_t lo = acc & 0xFFFFu, hi = acc >> 16;
  return lo > hi ? lo : hi;
}

// Relaxed (no fences) atomic max, for the commutative amax reduction.
FP8_DEVI void red_max_relaxed(uint32_t* addr, uint32_t v) {
  asm volatile("red.relaxed.gpu.global.max.u32 [%0], %1;" ::"l"(addr), "r"(v) : "memory");
}

// ------------------------------------------------------------------------------------------
// Streaming global loads / stores.
FP8_DEVI uint4 ld_nc_v4(const void* p) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p));
  return r;
}

// L2 cache policies (createpolicy) for loads and stores that carry a cache hint. evict_last: lines
// that a later pass reads again (the amax pass of a two-pass quantize keeps its input in L2 for
// the cast pass); evict_first: a line's last use, or output that nothing reads soon, so that it
// does not push out lines still to be re-read.
FP8_DEVI uint64_t l2_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
FP8_DEVI uint64_t l2_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
FP8_DEVI uint4 ld_nc_v4_hint(const void* p, uint64_t pol) {
  uint4 r;
  asm volatile("ld.global.nc.L1::no_allocate.L2::cache_hint.v4.u32 {%0,%1,%2,%3}, [%4], %5;"
               : "=r"(r.x), "=r"(r.y), "=r"(r.z), "=r"(r.w)
               : "l"(p), "l"(pol));
  return r;
}
FP8_DEVI void st_v2_hint(void* p, uint2 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v2.u32 [%0], {%1, %2}, %3;" ::"l"(p), "r"(v.x), "r"(v.y), "l"(pol) : "memory");
}
FP8_DEVI void st_v4_hint(void* p, uint4 v, uint64_t pol) {
  asm volatile("st.global.L2::cache_hint.v4.u32 [%0], {%1, %2, %3, %4}, %5;" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
               "r"(v.w), "l"(pol)
               : "memory");
}

// Grid barrier words (global memory, gpu scope): a release increment orders this thread's earlier
// memory operations (e.g. a relaxed atomic max) before the count; the acquire load of the waiter
// then sees them.
FP8_DEVI void red_add_release_gpu(uint32_t* p, uint32_t v) {
  asm volatile("red.release.gpu.global.add.u32 [%0], %1;" ::"l"(p), "r"(v) : "memory");
}
FP8_DEVI uint32_t ld_acquire_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.acquire.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
FP8_DEVI uint32_t ld_relaxed_gpu(const uint32_t* p) {
  uint32_t v;
  asm volatile("ld.relaxed.gpu.global.u32 %0, [%1];" : "=r"(v) : "l"(p) : "memory");
  return v;
}
// Bounded wait until *p >= target (polling with a short back-off). False when limit_ns elapsed.
FP8_DEVI bool wait_count_geq(const uint32_t* p, uint32_t target, uint64_t limit_ns) {
  if (ld_acquire_gpu(p) >= target) return true;
  const uint64_t t0 = globaltimer();
  uint32_t ns = 32;
  for (;;) {
    __nanosleep(ns);
    if (ns < 128) ns <<= 1;
    if (ld_acquire_gpu(p) >= target) return true;
    if (globaltimer() - t0 > limit_ns) return false;
  }
}

// ------------------------------------------------------------------------------------------
// mbarrier
FP8_DEVI void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
FP8_DEVI void mbar_inval(uint64_t* bar) {
  asm volatile("mbarrier.inval.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
FP8_DEVI void fence_mbar_init() { asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory"); }
FP8_DEVI void fence_proxy_async_smem() { asm volatile("fence.proxy.async.shared::cta;" ::: "memory"); }
FP8_DEVI void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(smem_u32(bar)), "r"(bytes)
               : "memory");
}
FP8_DEVI void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
FP8_DEVI bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(smem_u32(bar)), "r"(parity)
      : "memory");
  return ok != 0;
}

// Bounded wait for the phase of `parity` to complete. Returns false when `limit_ns` elapsed or
// when another role raised `*abort` (abort may be null).
FP8_DEVI bool mbar_wait(uint64_t* bar, uint32_t parity, const volatile int* abort, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 15u) == 0) {
      if (abort && *abort) return false;
      if (globaltimer() - t0 > limit_ns) return false;
    }
  }
}

// ------------------------------------------------------------------------------------------
// TMA (cp.async.bulk.tensor): global -> shared, completion counted on an mbarrier in bytes.
FP8_DEVI void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}
FP8_DEVI void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y)
      : "memory");
}
FP8_DEVI void tma_load_3d(void* dst, const CUtensorMap* m, uint64_t* bar, int32_t x, int32_t y, int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z)
      : "memory");
}
FP8_DEVI void tma_load_4d(void* dst, const CUtensorMap* m, uint64_t* bar, int32_t x, int32_t y, int32_t z,
                          int32_t w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}

// The same loads with an L2 cache policy (see l2_evict_last / l2_evict_first).
FP8_DEVI void tma_load_2d_hint(void* dst, const CUtensorMap* m, uint64_t* bar, int32_t x, int32_t y, uint64_t pol) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(pol)
      : "memory");
}

// TMA bulk-tensor stores shared -> global, tracked per thread in bulk async-groups.
FP8_DEVI void tma_store_2d(const CUtensorMap* m, const void* src, int32_t x, int32_t y) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group [%0, {%2, %3}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(smem_u32(src)), "r"(x), "r"(y)
               : "memory");
}
FP8_DEVI void tma_store_3d(const CUtensorMap* m, const void* src, int32_t x, int32_t y, int32_t z) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group [%0, {%2, %3, %4}], [%1];" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z)
               : "memory");
}
FP8_DEVI void tma_store_2d_hint(const CUtensorMap* m, const void* src, int32_t x, int32_t y, uint64_t pol) {
  asm volatile("cp.async.bulk.tensor.2d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3}], [%1], %4;" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(smem_u32(src)), "r"(x), "r"(y), "l"(pol)
               : "memory");
}
FP8_DEVI void tma_store_3d_hint(const CUtensorMap* m, const void* src, int32_t x, int32_t y, int32_t z, uint64_t pol) {
  asm volatile("cp.async.bulk.tensor.3d.global.shared::cta.bulk_group.L2::cache_hint [%0, {%2, %3, %4}], [%1], %5;" ::"l"(
                   reinterpret_cast<uint64_t>(m)),
               "r"(smem_u32(src)), "r"(x), "r"(y), "r"(z), "l"(pol)
               : "memory");
}
FP8_DEVI void bulk_commit() { asm volatile("cp.async.bulk.commit_group;" ::: "memory"); }
FP8_DEVI void bulk_wait_read_all() { asm volatile("cp.async.bulk.wait_group.read 0;" ::: "memory"); }
FP8_DEVI void bulk_wait_all() { asm volatile("cp.async.bulk.wait_group 0;" ::: "memory"); }
FP8_DEVI void bulk_wait_read_1() { asm volatile("cp.async.bulk.wait_group.read 1;" ::: "memory"); }

// Asynchronous 4-byte copy global -> shared (zero-filled when `valid` is false), tracked per thread
// in commit groups: a move of a register that a plain load is still filling waits for the load,
// an asynchronous copy into shared memory does not.
FP8_DEVI void cp_async4(void* smem_dst, const void* gsrc, bool valid) {
  asm volatile("cp.async.ca.shared.global [%0], [%1], 4, %2;" ::"r"(smem_u32(smem_dst)), "l"(gsrc),
               "r"(valid ? 4 : 0)
               : "memory");
}
FP8_DEVI void cp_async_commit() { asm volatile("cp.async.commit_group;" ::: "memory"); }
// The mbarrier receives one arrival from this thread once all of its earlier cp.async copies have
// landed (the barrier's expected count includes that arrival).
FP8_DEVI void cp_async_arrive_noinc(uint64_t* bar) {
  asm volatile("cp.async.mbarrier.arrive.noinc.shared::cta.b64 [%0];" ::"r"(smem_u32(bar)) : "memory");
}
template <int N>
FP8_DEVI void cp_async_wait() { asm volatile("cp.async.wait_group %0;" ::"n"(N) : "memory"); }

// ------------------------------------------------------------------------------------------
// tcgen05: tensor memory allocation, MMA issue, commit, loads, fences.
FP8_DEVI void tmem_alloc(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
FP8_DEVI void tmem_relinquish() { asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory"); }
FP8_DEVI void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
FP8_DEVI void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
FP8_DEVI void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// D(tmem) (+)= A(smem desc) * B(smem desc); kind::f8f6f4 (FP8 operands, K = 32 per issue).
FP8_DEVI void umma_f8f6f4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// kind::f16 (BF16 operands, K = 16 per issue).
FP8_DEVI void umma_f16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when every tcgen05 operation this thread issued so far has completed.
FP8_DEVI void umma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(smem_u32(bar))
               : "memory");
}

// ---- CTA pairs (cta_group::2): the two CTAs of a 2-CTA cluster share one MMA ----
FP8_DEVI uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
FP8_DEVI uint32_t mapa_shared(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}
FP8_DEVI void cluster_barrier() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}
// Arrive on an mbarrier given by its shared::cluster address (possibly in the peer CTA).
FP8_DEVI void mbar_arrive_cluster(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
// Relaxed arrivals (no release ordering), for barriers that only say "this warp's tensor-memory
// loads of an accumulator have completed" (tcgen05.wait::ld returned, the values are in registers,
// and tcgen05.fence::before_thread_sync precedes the arrival): no memory write of the arriving warp
// has to become visible to the waiting thread. A release arrival would first wait for the warp's
// outstanding memory operations; at cluster scope that took about 1 us per tile in the jagged-K
// GEMM, whose epilogue had just issued its output stores.
FP8_DEVI void mbar_arrive_cluster_relaxed(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.relaxed.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}
FP8_DEVI void mbar_arrive_relaxed(uint64_t* bar) {
  asm volatile("mbarrier.arrive.relaxed.cta.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
FP8_DEVI void tmem_alloc_pair(uint32_t* dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(dst_smem)),
               "r"(ncols)
               : "memory");
}
FP8_DEVI void tmem_relinquish_pair() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
}
FP8_DEVI void tmem_dealloc_pair(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
FP8_DEVI void umma_f8f6f4_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
FP8_DEVI void umma_f16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, p;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive once on the mbarrier at this offset in every CTA of `cta_mask` when the pair's MMAs
// issued so far have completed.
FP8_DEVI void umma_commit_pair(uint64_t* bar, uint16_t cta_mask) {
  asm volatile(
      "tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;" ::"r"(
          smem_u32(bar)),
      "h"(cta_mask)
      : "memory");
}
// TMA loads whose completion is counted on an mbarrier that may live in the peer CTA.
FP8_DEVI void tma_load_2d_pair(void* dst, const CUtensorMap* m, uint32_t bar_cluster_addr, int32_t x, int32_t y) {
  asm volatile(
      "cp.async.bulk.tensor.2d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster_addr), "r"(x), "r"(y)
      : "memory");
}
FP8_DEVI void tma_load_3d_pair(void* dst, const CUtensorMap* m, uint32_t bar_cluster_addr, int32_t x, int32_t y,
                               int32_t z) {
  asm volatile(
      "cp.async.bulk.tensor.3d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster_addr), "r"(x), "r"(y), "r"(z)
      : "memory");
}

FP8_DEVI void tma_load_4d_pair(void* dst, const CUtensorMap* m, uint32_t bar_cluster_addr, int32_t x, int32_t y,
                               int32_t z, int32_t w) {
  asm volatile(
      "cp.async.bulk.tensor.4d.cta_group::2.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4, %5, %6}], [%2];" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster_addr), "r"(x), "r"(y), "r"(z), "r"(w)
      : "memory");
}

// ---- MX block scaling: E8M0 scale factors in tensor memory ----
// tcgen05.mma.kind::mxf8f6f4.block_scale.scale_vec::1X: one E8M0 scale per row per 32 K
// elements (one MMA of K = 32). Scale factors live in tensor memory; a column of 32-bit words
// holds four consecutive K-block scales per lane and the instruction descriptor picks the byte
// (scale-factor id = K block % 4). Rows of A (and of B) map to tensor memory as row % 32 -> lane
// (in each of the four lane quarters), row / 32 -> column. tcgen05.cp .32x128b.warpx4 copies a
// 512-byte shared-memory block [32 lanes][4 columns][4 bytes] into that layout, repeated in the
// four lane quarters.
FP8_DEVI void umma_mx(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa_tmem,
                      uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
FP8_DEVI void umma_mx_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc, uint32_t sfa_tmem,
                           uint32_t sfb_tmem, uint32_t accumulate) {
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "setp.ne.b32 p, %6, 0;\n\t"
      "tcgen05.mma.cta_group::2.kind::mxf8f6f4.block_scale.scale_vec::1X [%0], %1, %2, %3, [%4], [%5], p;\n\t}" ::"r"(
          d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate)
      : "memory");
}
// shared memory -> tensor memory, 32 rows x 128 bits, repeated in the four lane quarters.
// Issued by the MMA thread; tcgen05.mma issued after it by the same thread sees the copy.
FP8_DEVI void tmem_cp_sf(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}
// CTA pairs: each CTA's shared memory into its own tensor memory, issued by the even CTA.
FP8_DEVI void tmem_cp_sf_pair(uint32_t taddr, uint64_t sdesc) {
  asm volatile("tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;" ::"r"(taddr), "l"(sdesc) : "memory");
}

// 32 lanes x 32 bit, 32 consecutive columns.
FP8_DEVI void tmem_ld32(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr));
}
// Waits for this thread's tensor-memory loads (tcgen05.wait::ld), naming the 32 registers of the
// load it completes as in/out operands: the compiler may not read, move or reuse them between the
// asynchronous load and this wait.
FP8_DEVI void tmem_ld_wait_regs(uint32_t* r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15]),
                 "+r"(r[16]), "+r"(r[17]), "+r"(r[18]), "+r"(r[19]), "+r"(r[20]), "+r"(r[21]), "+r"(r[22]), "+r"(r[23]),
                 "+r"(r[24]), "+r"(r[25]), "+r"(r[26]), "+r"(r[27]), "+r"(r[28]), "+r"(r[29]), "+r"(r[30]), "+r"(r[31])
               :
               : "memory");
}
// 32 lanes x 32 bit, 16 consecutive columns, and its wait (as above).
FP8_DEVI void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
                 "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
               : "r"(taddr));
}
FP8_DEVI void tmem_ld_wait_regs16(uint32_t* r) {
  asm volatile("tcgen05.wait::ld.sync.aligned;"
               : "+r"(r[0]), "+r"(r[1]), "+r"(r[2]), "+r"(r[3]), "+r"(r[4]), "+r"(r[5]), "+r"(r[6]), "+r"(r[7]),
                 "+r"(r[8]), "+r"(r[9]), "+r"(r[10]), "+r"(r[11]), "+r"(r[12]), "+r"(r[13]), "+r"(r[14]), "+r"(r[15])
               :
               : "memory");
}

// Named barriers (ids > 0) for a subset of warps; bar_and also reduces a predicate (all true).
FP8_DEVI void named_bar_sync(uint32_t id, uint32_t nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}
FP8_DEVI bool named_bar_and(uint32_t id, uint32_t nthreads, bool v) {
  uint32_t r;
  asm volatile(
      "{\n\t.reg .pred p, q;\n\t"
      "setp.ne.u32 p, %1, 0;\n\t"
      "bar.red.and.pred q, %2, %3, p;\n\t"
      "selp.u32 %0, 1, 0, q;\n\t}"
      : "=r"(r)
      : "r"((uint32_t)v), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// Shared-memory matrix descriptor (tcgen05 format): start address, leading- and
// stride-dimension byte offsets (in 16-byte units), version 1, swizzle mode in bits 61..63
// (2 = 128-byte swizzle).
FP8_DEVI uint64_t smem_desc(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Shared-memory descriptor without swizzle for the scale-factor copies: 8-row x 16-byte core
// matrices, rows 16 bytes apart, core matrices `sbo_bytes` apart along the rows.
FP8_DEVI uint64_t smem_desc_plain(uint32_t saddr, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;
}

// Instruction descriptor for kind::mxf8f6f4 with block scaling: operand formats, K-major A and
// B, N >> 3 at bit 17, E8M0 scales (bit 23), M >> 4 at bit 24. The scale-factor ids (which byte
// of the scale column an MMA uses) go in bits 4-5 (B) and 29-30 (A), added per MMA.
__host__ __device__ constexpr uint32_t make_idesc_mx(uint32_t a_fmt, uint32_t b_fmt, uint32_t M, uint32_t N) {
  return (a_fmt << 7) | (b_fmt << 10) | ((N >> 3) << 17) | (1u << 23) | ((M >> 4) << 24);
}
FP8_DEVI uint32_t idesc_sf_ids(uint32_t idesc, uint32_t a_id, uint32_t b_id) {
  return idesc | (b_id << 4) | (a_id << 29);
}

// Instruction descriptor for kind::f16 / kind::f8f6f4: fp32 accumulator, operand formats,
// operand majors (0 = K-major, 1 = MN-major), N >> 3 at bit 17, M >> 4 at bit 24.
__host__ __device__ constexpr uint32_t make_idesc(uint32_t a_fmt, uint32_t b_fmt, uint32_t a_mn, uint32_t b_mn,
                                                  uint32_t M, uint32_t N) {
  return (1u << 4) | (a_fmt << 7) | (b_fmt << 10) | (a_mn << 15) | (b_mn << 16) | ((N >> 3) << 17) |
         ((M >> 4) << 24);
}
// Operand format codes: kind::f8f6f4 e4m3 = 0, e5m2 = 1; kind::f16 bf16 = 1.
constexpr uint32_t kFmtE4M3 = 0, kFmtE5M2 = 1, kFmtBF16 = 1;

}  // namespace fp8lin
