// C ABI of fp8lin: argument checking, launch context, TMA descriptor encoding, and the
// composition of the Linear forward / backward passes from the quantize and GEMM launchers.
#include <cudaTypedefs.h>

#include <string.h>

#include <atomic>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace fp8lin {

static std::atomic<uint64_t> g_wait_ns{4000000000ull};

// Table of the scale step (see ScaleTab): for the 128 bf16 mantissas m in [1, 2), the fp64
// quotient fp8_max / m and its fp64 reciprocal, each rounded to fp32; the eps entry for amax
// below eps; eps_below = the smallest bf16 pattern whose value is >= eps.
static ScaleTab build_tab(double fp8_max) {
  ScaleTab t;
  for (int m7 = 0; m7 < 128; ++m7) {
    const double m = 1.0 + m7 / 128.0;
    const double s = fp8_max / m;
    t.s[m7] = (float)s;
    t.inv[m7] = (float)(1.0 / s);
  }
  const double se = fp8_max / kEps;
  t.eps_s = (float)se;
  t.eps_inv = (float)(1.0 / se);
  uint32_t b = 0;
  while (b < 0x7F80u) {
    uint32_t u = b << 16;
    float f;
    memcpy(&f, &u, 4);
    if ((double)f >= kEps) break;
    ++b;
  }
  t.eps_below = b;
  return t;
}

const ScaleTab& scale_tab(int fmt) {
  static const ScaleTab e4 = build_tab(kE4M3Max), e5 = build_tab(kE5M2Max);
  return fmt == FP8_DT_E4M3 ? e4 : e5;
}
static std::atomic<int> g_test_stall{0};

int make_ctx(Ctx* ctx, void* stream, int32_t* status) {
  static std::mutex mu;
  static int sms[64];
  static int ok[64];
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return FP8_ERR_DEVICE;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (ok[dev] == 0) {
      int major = 0, minor = 0, n = 0;
      if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess)
        return FP8_ERR_DEVICE;
      ok[dev] = (major == 10 && minor == 3) ? 1 : -1;  // the kernels are built for sm_103a only
      sms[dev] = n;
    }
    if (ok[dev] < 0) return FP8_ERR_DEVICE;
    ctx->sm_count = sms[dev];
  }
  ctx->device = dev;
  ctx->stream = static_cast<cudaStream_t>(stream);
  ctx->status = status;
  ctx->wait_ns = g_wait_ns.load();
  ctx->test_stall = g_test_stall.load();
  return FP8_OK;
}

static PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* p = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(p);
  });
  return fn;
}

int make_tmap(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int rank, const uint64_t* dims,
              const uint64_t* strides_bytes, const uint32_t* box, CUtensorMapSwizzle swz) {
  auto fn = encode_fn();
  if (!fn) return FP8_ERR_CUDA;
  cuuint64_t d[5];
  cuuint64_t s[4];
  cuuint32_t b[5], e[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    b[i] = box[i];
    e[i] = 1;
    if (i + 1 < rank) s[i] = strides_bytes[i];
  }
  CUresult r = fn(map, dt, (cuuint32_t)rank, const_cast<void*>(base), d, s, b, e, CU_TENSOR_MAP_INTERLEAVE_NONE, swz,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS ? FP8_OK : FP8_ERR_CUDA;
}

}  // namespace fp8lin

using namespace fp8lin;

// ------------------------------------------------------------------------------------------
// argument helpers

static bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
static bool is_fp8(int dt) { return dt == FP8_DT_E4M3 || dt == FP8_DT_E5M2; }
static bool is_out(int dt) { return dt == FP8_DT_BF16 || dt == FP8_DT_F32; }
static int64_t numel(const fp8_tensor* t) {
  int64_t n = 1;
  for (int i = 0; i < t->ndim; ++i) n *= t->shape[i];
  return n;
}
static bool valid_desc(const fp8_tensor* t) {
  if (!t || t->ndim < 1 || t->ndim > 3) return false;
  for (int i = 0; i < t->ndim; ++i)
    if (t->shape[i] < 0) return false;
  return t->ptr != nullptr || numel(t) == 0;
}
static bool shape_is(const fp8_tensor* t, int nd, int64_t a, int64_t b = -1, int64_t c = -1) {
  if (t->ndim != nd) return false;
  const int64_t s[3] = {a, b, c};
  for (int i = 0; i < nd; ++i)
    if (t->shape[i] != s[i]) return false;
  return true;
}
static int64_t round_up(int64_t a, int64_t b) { return (a + b - 1) / b * b; }

#define FP8_CHECK(cond, code) \
  do {                        \
    if (!(cond)) return (code); \
  } while (0)
#define FP8_TRY(expr)        \
  do {                       \
    int rc_ = (expr);        \
    if (rc_ != FP8_OK) return rc_; \
  } while (0)

// ------------------------------------------------------------------------------------------

extern "C" int64_t fp8_mx_scale_bytes(int64_t rows, int64_t k) { return mx_scale_bytes(rows, k); }

extern "C" int64_t fp8_jagged_padded_rows(int64_t rows, int64_t n_segments) {
  if (rows < 0 || n_segments < 0) return -1;
  return round_up(rows + 127 * n_segments, 128);
}

extern "C" uint64_t fp8_set_wait_limit_ns(uint64_t ns) { return g_wait_ns.exchange(ns ? ns : 1); }

extern "C" int fp8_set_test_stall(int enable) { return g_test_stall.exchange(enable ? 1 : 0); }

extern "C" int fp8_test_cast_bits(uint32_t first_bits, int64_t n, int out_dtype, void* out, void* stream) {
  if (!is_fp8(out_dtype) || n < 0 || n > ((int64_t)1 << 32) - (int64_t)first_bits) return FP8_ERR_INVALID_ARG;
  if (n > 0 && !out) return FP8_ERR_INVALID_ARG;
  Ctx c;
  const int rc = make_ctx(&c, stream, nullptr);
  if (rc != FP8_OK) return rc;
  return launch_cast_bits(first_bits, n, out_dtype, out, c);
}

extern "C" const char* fp8_status_string(int code) {
  switch (code) {
    case FP8_OK: return "ok";
    case FP8_ERR_INVALID_ARG: return "invalid argument (null pointer, dtype, rank or shape)";
    case FP8_ERR_UNSUPPORTED: return "unsupported combination of arguments";
    case FP8_ERR_ALIGNMENT: return "pointer or contiguous row not 16-byte aligned";
    case FP8_ERR_WORKSPACE: return "workspace missing or too small";
    case FP8_ERR_CUDA: return "CUDA runtime or launch failure";
    case FP8_ERR_DEVICE: return "no sm_103 device current";
    case FP8_DEV_BAD_OFFSETS: return "device: offsets not non-decreasing or last != total rows";
    case FP8_DEV_TIMEOUT: return "device: a bounded wait ran out";
    case FP8_DEV_BAD_OFFSETS | FP8_DEV_TIMEOUT: return "device: bad offsets and a wait ran out";
    default: return "unknown status";
  }
}

// ------------------------------------------------------------------------------------------
// fp8_quantize

static int quantize_impl(const fp8_tensor* x, int gran, int out_dtype, int layout, fp8_tensor* out,
                         fp8_tensor* out_t, fp8_tensor* inv, const fp8_tensor* offsets, void* ws, size_t ws_bytes,
                         const Ctx& c) {
  FP8_CHECK(valid_desc(x) && x->dtype == FP8_DT_BF16 && (x->ndim == 2 || x->ndim == 3), FP8_ERR_INVALID_ARG);
  FP8_CHECK(is_fp8(out_dtype), FP8_ERR_INVALID_ARG);
  FP8_CHECK(layout >= 1 && layout <= 3, FP8_ERR_INVALID_ARG);
  FP8_CHECK(valid_desc(inv) && inv->dtype == (gran == FP8_GRAN_MX ? FP8_DT_E8M0 : FP8_DT_F32), FP8_ERR_INVALID_ARG);
  const int nd = x->ndim;
  const int64_t B = nd == 3 ? x->shape[0] : 1, R = x->shape[nd - 2], C = x->shape[nd - 1];
  FP8_CHECK(C % 8 == 0 && aligned16(x->ptr), FP8_ERR_ALIGNMENT);
  FP8_CHECK(B * R < (int64_t(1) << 31), FP8_ERR_UNSUPPORTED);
  const bool want_row = layout & FP8_LAYOUT_ROW_MAJOR, want_col = layout & FP8_LAYOUT_COL_MAJOR;
  if (want_row) {
    FP8_CHECK(valid_desc(out) && out->dtype == out_dtype && out->ndim == nd, FP8_ERR_INVALID_ARG);
    for (int i = 0; i < nd; ++i) FP8_CHECK(out->shape[i] == x->shape[i], FP8_ERR_INVALID_ARG);
    FP8_CHECK(aligned16(out->ptr), FP8_ERR_ALIGNMENT);
  }
  if (want_col) {
    FP8_CHECK(valid_desc(out_t) && out_t->dtype == out_dtype, FP8_ERR_INVALID_ARG);
    FP8_CHECK(aligned16(out_t->ptr), FP8_ERR_ALIGNMENT);
  }
  switch (gran) {
    case FP8_GRAN_TENSOR: {
      FP8_CHECK(offsets == nullptr, FP8_ERR_UNSUPPORTED);
      FP8_CHECK(numel(inv) == 1, FP8_ERR_INVALID_ARG);
      if (want_col) {
        FP8_CHECK(nd == 2, FP8_ERR_UNSUPPORTED);
        FP8_CHECK(shape_is(out_t, 2, C, R), FP8_ERR_INVALID_ARG);
        FP8_CHECK(R % 16 == 0, FP8_ERR_ALIGNMENT);
      }
      FP8_CHECK(ws && ws_bytes >= 8 && (reinterpret_cast<uintptr_t>(ws) & 7u) == 0, FP8_ERR_WORKSPACE);
      return launch_quant_tensor(x->ptr, B * R, C, out_dtype, want_row ? out->ptr : nullptr,
                                 want_col ? out_t->ptr : nullptr, static_cast<float*>(inv->ptr),
                                 static_cast<uint32_t*>(ws), c);
    }
    case FP8_GRAN_ROW: {
      FP8_CHECK(offsets == nullptr, FP8_ERR_UNSUPPORTED);
      FP8_CHECK(layout == FP8_LAYOUT_ROW_MAJOR, FP8_ERR_UNSUPPORTED);
      FP8_CHECK(numel(inv) == B * R, FP8_ERR_INVALID_ARG);
      FP8_CHECK(C <= 65536, FP8_ERR_UNSUPPORTED);
      return launch_quant_rows(x->ptr, B * R, C, out_dtype, out->ptr, static_cast<float*>(inv->ptr), c);
    }
    case FP8_GRAN_COL: {
      FP8_CHECK(layout == FP8_LAYOUT_COL_MAJOR, FP8_ERR_UNSUPPORTED);
      const int64_t groups = offsets ? (valid_desc(offsets) && offsets->ndim == 1 ? offsets->shape[0] : 0) : B;
      FP8_CHECK(ws && (reinterpret_cast<uintptr_t>(ws) & 15u) == 0 &&
                    ws_bytes >= (size_t)col_ws_words(groups > 0 ? groups : 1, C, B * R) * 4,
                FP8_ERR_WORKSPACE);
      uint32_t* scratch = static_cast<uint32_t*>(ws);
      if (offsets) {
        FP8_CHECK(nd == 2, FP8_ERR_UNSUPPORTED);
        FP8_CHECK(valid_desc(offsets) && offsets->dtype == FP8_DT_I32 && offsets->ndim == 1 && offsets->shape[0] >= 1,
                  FP8_ERR_INVALID_ARG);
        const int64_t E = offsets->shape[0];
        FP8_CHECK(out_t->ndim == 2 && out_t->shape[0] == C, FP8_ERR_INVALID_ARG);
        const int64_t P = out_t->shape[1];
        FP8_CHECK(P >= R + 127 * E, FP8_ERR_INVALID_ARG);
        FP8_CHECK(P % 16 == 0, FP8_ERR_ALIGNMENT);
        FP8_CHECK(numel(inv) == E * C, FP8_ERR_INVALID_ARG);
        return launch_quant_cols(x->ptr, R, C, E, 0, static_cast<const int32_t*>(offsets->ptr), out_dtype,
                                 out_t->ptr, P, static_cast<float*>(inv->ptr), scratch, c);
      }
      FP8_CHECK(R % 16 == 0, FP8_ERR_ALIGNMENT);
      if (nd == 2)
        FP8_CHECK(shape_is(out_t, 2, C, R), FP8_ERR_INVALID_ARG);
      else
        FP8_CHECK(shape_is(out_t, 3, B, C, R), FP8_ERR_INVALID_ARG);
      FP8_CHECK(numel(inv) == B * C, FP8_ERR_INVALID_ARG);
      return launch_quant_cols(x->ptr, B * R, C, B, R, nullptr, out_dtype, out_t->ptr, R,
                               static_cast<float*>(inv->ptr), scratch, c);
    }
    case FP8_GRAN_MX: {
      FP8_CHECK(C % 128 == 0, FP8_ERR_UNSUPPORTED);
      uint8_t* sf = static_cast<uint8_t*>(inv->ptr);
      if (offsets) {
        FP8_CHECK(nd == 2, FP8_ERR_UNSUPPORTED);
        FP8_CHECK(valid_desc(offsets) && offsets->dtype == FP8_DT_I32 && offsets->ndim == 1 && offsets->shape[0] >= 1,
                  FP8_ERR_INVALID_ARG);
        const int64_t E = offsets->shape[0];
        // the padded row count: from out_t, else from the size of the row-major scales
        if (C == 0) return FP8_OK;  // no columns: no codes and no scales to write
        const int64_t P = want_col ? (out_t->ndim == 2 ? out_t->shape[1] : -1) : numel(inv) * 32 / C;
        FP8_CHECK(P >= R + 127 * E && P % 128 == 0, FP8_ERR_INVALID_ARG);
        if (want_col) FP8_CHECK(shape_is(out_t, 2, C, P), FP8_ERR_INVALID_ARG);
        const int64_t row_bytes = want_row ? mx_scale_bytes(P, C) : 0, col_bytes = want_col ? mx_scale_bytes(C, P) : 0;
        FP8_CHECK(numel(inv) == row_bytes + col_bytes, FP8_ERR_INVALID_ARG);
        FP8_CHECK(ws && (reinterpret_cast<uintptr_t>(ws) & 15u) == 0 && ws_bytes >= (size_t)round_up(4 * (E + 1), 16),
                  FP8_ERR_WORKSPACE);
        return launch_mx_quant(x->ptr, 1, R, C, out_dtype, want_row ? out->ptr : nullptr, sf,
                               want_col ? out_t->ptr : nullptr, P, sf + row_bytes,
                               static_cast<const int32_t*>(offsets->ptr), E, static_cast<int32_t*>(ws), c);
      }
      if (want_col) {
        FP8_CHECK(R % 128 == 0, FP8_ERR_UNSUPPORTED);
        if (nd == 2)
          FP8_CHECK(shape_is(out_t, 2, C, R), FP8_ERR_INVALID_ARG);
        else
          FP8_CHECK(shape_is(out_t, 3, B, C, R), FP8_ERR_INVALID_ARG);
      }
      const int64_t row_bytes = want_row ? B * mx_scale_bytes(R, C) : 0;
      const int64_t col_bytes = want_col ? B * mx_scale_bytes(C, R) : 0;
      FP8_CHECK(numel(inv) == row_bytes + col_bytes, FP8_ERR_INVALID_ARG);
      return launch_mx_quant(x->ptr, B, R, C, out_dtype, want_row ? out->ptr : nullptr, sf,
                             want_col ? out_t->ptr : nullptr, R, sf + row_bytes, nullptr, 0, nullptr, c);
    }
    case FP8_GRAN_BLOCK_1x128: {
      FP8_CHECK(offsets == nullptr && nd == 2 && layout == FP8_LAYOUT_ROW_MAJOR, FP8_ERR_UNSUPPORTED);
      FP8_CHECK(C % 128 == 0, FP8_ERR_UNSUPPORTED);
      FP8_CHECK(numel(inv) == R * (C / 128), FP8_ERR_INVALID_ARG);
      return launch_blk_quant(x->ptr, R, C, out_dtype, false, out->ptr, nullptr, static_cast<float*>(inv->ptr),
                              nullptr, c);
    }
    case FP8_GRAN_BLOCK_128x128: {
      FP8_CHECK(offsets == nullptr && nd == 2, FP8_ERR_UNSUPPORTED);
      FP8_CHECK(C % 128 == 0 && (!want_col || R % 128 == 0), FP8_ERR_UNSUPPORTED);
      if (want_col) FP8_CHECK(shape_is(out_t, 2, C, R), FP8_ERR_INVALID_ARG);
      const int64_t nrow = want_row ? ((R + 127) / 128) * (C / 128) : 0, ncol = want_col ? (C / 128) * (R / 128) : 0;
      FP8_CHECK(numel(inv) == nrow + ncol, FP8_ERR_INVALID_ARG);
      float* iv = static_cast<float*>(inv->ptr);
      return launch_blk_quant(x->ptr, R, C, out_dtype, true, want_row ? out->ptr : nullptr,
                              want_col ? out_t->ptr : nullptr, want_row ? iv : nullptr, want_col ? iv + nrow : nullptr,
                              c);
    }
    default:
      return FP8_ERR_INVALID_ARG;
  }
}

extern "C" int fp8_quantize(const fp8_tensor* x, int granularity, int out_dtype, int layout, fp8_tensor* out,
                            fp8_tensor* out_t, fp8_tensor* inv_scales, const fp8_tensor* offsets, void* workspace,
                            size_t workspace_bytes, int32_t* d_status, void* stream) {
  Ctx c;
  FP8_TRY(make_ctx(&c, stream, d_status));
  return quantize_impl(x, granularity, out_dtype, layout, out, out_t, inv_scales, offsets, workspace,
                       workspace_bytes, c);
}

// ------------------------------------------------------------------------------------------
// fp8_scaled_mm

static int dense_gemm(const void* A, int a_dt, int a_mn, const void* B, int b_dt, int b_mn, const float* sA,
                      int64_t sA_len, const float* sB, int64_t sB_len, void* out, int out_dt, int64_t M, int64_t N,
                      int64_t K, const Ctx& c, uint32_t* row_amax = nullptr, uint32_t* col_amax = nullptr,
                      int amax_whole = 0) {
  GemmArgs g = {};
  g.row_amax = row_amax;
  g.col_amax = col_amax;
  g.amax_whole = amax_whole;
  g.A = A;
  g.B = B;
  g.a_dtype = a_dt;
  g.b_dtype = b_dt;
  g.a_mn = a_mn;
  g.b_mn = b_mn;
  g.sA = sA;
  g.sB = sB;
  g.sA_len = sA_len;
  g.sB_len = sB_len;
  g.out = out;
  g.out_dtype = out_dt;
  g.M = M;
  g.N = N;
  g.K = K;
  g.mode = -1;
  return launch_gemm(g, c);
}

// An empty contraction (K == 0): every output element is an empty sum, stored as +0.
static int zero_out(const fp8_tensor* out, int64_t M, int64_t N, const Ctx& c) {
  const size_t bytes = (size_t)M * (size_t)N * (out->dtype == FP8_DT_F32 ? 4u : 2u);
  return cudaMemsetAsync(out->ptr, 0, bytes, c.stream) == cudaSuccess ? FP8_OK : FP8_ERR_CUDA;
}

static int scaled_mm_impl(const fp8_tensor* A, const fp8_tensor* B, const fp8_tensor* sA, const fp8_tensor* sB,
                          fp8_tensor* out, int flags, const Ctx& c, uint32_t* row_amax = nullptr,
                          uint32_t* col_amax = nullptr, int amax_whole = 0) {
  FP8_CHECK(valid_desc(A) && valid_desc(B) && valid_desc(out) && A->ndim == 2 && B->ndim == 2 && out->ndim == 2,
            FP8_ERR_INVALID_ARG);
  FP8_CHECK(is_out(out->dtype), FP8_ERR_INVALID_ARG);
  FP8_CHECK(aligned16(A->ptr) && aligned16(B->ptr) && aligned16(out->ptr), FP8_ERR_ALIGNMENT);
  const bool fp8 = is_fp8(A->dtype);
  if (fp8) {
    FP8_CHECK(is_fp8(B->dtype), FP8_ERR_INVALID_ARG);
    FP8_CHECK(!(A->dtype == FP8_DT_E5M2 && B->dtype == FP8_DT_E5M2), FP8_ERR_UNSUPPORTED);
    FP8_CHECK((flags & (FP8_MM_A_MN_MAJOR | FP8_MM_B_MN_MAJOR)) == 0, FP8_ERR_UNSUPPORTED);
    const int64_t M = A->shape[0], K = A->shape[1], N = B->shape[0];
    FP8_CHECK(B->shape[1] == K && shape_is(out, 2, M, N), FP8_ERR_INVALID_ARG);
    FP8_CHECK(K % 16 == 0, FP8_ERR_ALIGNMENT);
    FP8_CHECK(valid_desc(sA) && valid_desc(sB), FP8_ERR_INVALID_ARG);
    if (sA->dtype == FP8_DT_E8M0 || sB->dtype == FP8_DT_E8M0) {  // MX block scales
      FP8_CHECK(sA->dtype == FP8_DT_E8M0 && sB->dtype == FP8_DT_E8M0, FP8_ERR_INVALID_ARG);
      FP8_CHECK(K % 128 == 0, FP8_ERR_UNSUPPORTED);
      FP8_CHECK(numel(sA) == mx_scale_bytes(M, K) && numel(sB) == mx_scale_bytes(N, K), FP8_ERR_INVALID_ARG);
      FP8_CHECK(aligned16(sA->ptr) && aligned16(sB->ptr), FP8_ERR_ALIGNMENT);
      FP8_CHECK(M < (int64_t(1) << 31) && N < (int64_t(1) << 31) && K < (int64_t(1) << 31), FP8_ERR_UNSUPPORTED);
      if (M == 0 || N == 0) return FP8_OK;
      if (K == 0) return zero_out(out, M, N, c);
      GemmArgs g = {};
      g.A = A->ptr;
      g.B = B->ptr;
      g.a_dtype = A->dtype;
      g.b_dtype = B->dtype;
      g.out = out->ptr;
      g.out_dtype = out->dtype;
      g.M = M;
      g.N = N;
      g.K = K;
      g.mode = -1;
      g.mx = 1;
      g.sfa = sA->ptr;
      g.sfb = sB->ptr;
      g.sfa_rows = M;
      return launch_gemm(g, c);
    }
    FP8_CHECK(sA->dtype == FP8_DT_F32 && sB->dtype == FP8_DT_F32, FP8_ERR_INVALID_ARG);
    if (flags & FP8_MM_BLOCKWISE) {  // [B]: sA [M, K/128], sB [ceil(N/128), K/128]
      FP8_CHECK(K % 128 == 0 && !row_amax && !col_amax, FP8_ERR_UNSUPPORTED);
      FP8_CHECK(numel(sA) == M * (K / 128) && numel(sB) == ((N + 127) / 128) * (K / 128), FP8_ERR_INVALID_ARG);
      FP8_CHECK(M < (int64_t(1) << 31) && N < (int64_t(1) << 31) && K < (int64_t(1) << 31), FP8_ERR_UNSUPPORTED);
      if (M == 0 || N == 0) return FP8_OK;
      if (K == 0) return zero_out(out, M, N, c);
      GemmArgs g = {};
      g.A = A->ptr;
      g.B = B->ptr;
      g.a_dtype = A->dtype;
      g.b_dtype = B->dtype;
      g.sA = static_cast<const float*>(sA->ptr);
      g.sB = static_cast<const float*>(sB->ptr);
      g.out = out->ptr;
      g.out_dtype = out->dtype;
      g.M = M;
      g.N = N;
      g.K = K;
      g.mode = -1;
      g.blockwise = 1;
      return launch_gemm(g, c);
    }
    const int64_t la = numel(sA), lb = numel(sB);
    FP8_CHECK((la == 1 || la == M) && (lb == 1 || lb == N), FP8_ERR_INVALID_ARG);
    FP8_CHECK(M < (int64_t(1) << 31) && N < (int64_t(1) << 31) && K < (int64_t(1) << 31), FP8_ERR_UNSUPPORTED);
    if (M == 0 || N == 0) return FP8_OK;
    if (K == 0) return zero_out(out, M, N, c);
    return dense_gemm(A->ptr, A->dtype, 0, B->ptr, B->dtype, 0, static_cast<const float*>(sA->ptr), la,
                      static_cast<const float*>(sB->ptr), lb, out->ptr, out->dtype, M, N, K, c, row_amax, col_amax,
                      amax_whole);
  }
  FP8_CHECK(A->dtype == FP8_DT_BF16 && B->dtype == FP8_DT_BF16, FP8_ERR_INVALID_ARG);
  FP8_CHECK(sA == nullptr && sB == nullptr, FP8_ERR_INVALID_ARG);
  const int a_mn = (flags & FP8_MM_A_MN_MAJOR) ? 1 : 0, b_mn = (flags & FP8_MM_B_MN_MAJOR) ? 1 : 0;
  const int64_t M = a_mn ? A->shape[1] : A->shape[0], K = a_mn ? A->shape[0] : A->shape[1];
  const int64_t N = b_mn ? B->shape[1] : B->shape[0], K2 = b_mn ? B->shape[0] : B->shape[1];
  FP8_CHECK(K == K2 && shape_is(out, 2, M, N), FP8_ERR_INVALID_ARG);
  FP8_CHECK(A->shape[1] % 8 == 0 && B->shape[1] % 8 == 0, FP8_ERR_ALIGNMENT);
  if (M == 0 || N == 0) return FP8_OK;
  if (K == 0) return zero_out(out, M, N, c);
  return dense_gemm(A->ptr, FP8_DT_BF16, a_mn, B->ptr, FP8_DT_BF16, b_mn, nullptr, 0, nullptr, 0, out->ptr,
                    out->dtype, M, N, K, c, row_amax, col_amax, amax_whole);
}

extern "C" int fp8_scaled_mm(const fp8_tensor* A, const fp8_tensor* B, const fp8_tensor* sA, const fp8_tensor* sB,
                             fp8_tensor* out, int flags, int32_t* d_status, void* stream) {
  Ctx c;
  FP8_TRY(make_ctx(&c, stream, d_status));
  return scaled_mm_impl(A, B, sA, sB, out, flags, c);
}

extern "C" int fp8_scaled_mm_amax(const fp8_tensor* A, const fp8_tensor* B, const fp8_tensor* sA,
                                  const fp8_tensor* sB, fp8_tensor* out, int flags, fp8_tensor* row_amax,
                                  fp8_tensor* col_amax, int32_t* d_status, void* stream) {
  Ctx c;
  FP8_TRY(make_ctx(&c, stream, d_status));
  FP8_CHECK(valid_desc(out) && out->ndim == 2 && out->dtype == FP8_DT_BF16, FP8_ERR_UNSUPPORTED);
  FP8_CHECK(!(sA && sA->dtype == FP8_DT_E8M0), FP8_ERR_UNSUPPORTED);  // MX outputs: no side outputs
  const int64_t M = out->shape[0], N = out->shape[1];
  uint32_t* ra = nullptr;
  uint32_t* ca = nullptr;
  if (row_amax) {
    FP8_CHECK(valid_desc(row_amax) && row_amax->dtype == FP8_DT_F32 && numel(row_amax) == M, FP8_ERR_INVALID_ARG);
    ra = static_cast<uint32_t*>(row_amax->ptr);
  }
  int whole = 0;
  if (col_amax) {
    FP8_CHECK(valid_desc(col_amax) && col_amax->dtype == FP8_DT_F32 && (numel(col_amax) == N || numel(col_amax) == 1),
              FP8_ERR_INVALID_ARG);
    ca = static_cast<uint32_t*>(col_amax->ptr);
    whole = numel(col_amax) == 1 && N != 1;
  }
  // the maxima are folded in with atomic max from zero
  if (ra && M > 0 && cudaMemsetAsync(ra, 0, (size_t)M * 4, c.stream) != cudaSuccess) return FP8_ERR_CUDA;
  if (ca && cudaMemsetAsync(ca, 0, (size_t)numel(col_amax) * 4, c.stream) != cudaSuccess) return FP8_ERR_CUDA;
  return scaled_mm_impl(A, B, sA, sB, out, flags, c, ra, ca, whole);
}

extern "C" int fp8_scaled_mm_quant(const fp8_tensor* A, const fp8_tensor* B, const fp8_tensor* sA,
                                   const fp8_tensor* sB, int flags, int out_granularity, fp8_tensor* out_q,
                                   fp8_tensor* out_scales, int32_t* d_status, void* stream) {
  Ctx c;
  FP8_TRY(make_ctx(&c, stream, d_status));
  FP8_CHECK(valid_desc(A) && valid_desc(B) && valid_desc(sA) && valid_desc(sB) && valid_desc(out_q) &&
                valid_desc(out_scales) && A->ndim == 2 && B->ndim == 2 && out_q->ndim == 2,
            FP8_ERR_INVALID_ARG);
  FP8_CHECK(is_fp8(A->dtype) && is_fp8(B->dtype) && is_fp8(out_q->dtype), FP8_ERR_INVALID_ARG);
  FP8_CHECK(!(A->dtype == FP8_DT_E5M2 && B->dtype == FP8_DT_E5M2), FP8_ERR_UNSUPPORTED);
  FP8_CHECK((flags & (FP8_MM_A_MN_MAJOR | FP8_MM_B_MN_MAJOR | FP8_MM_BLOCKWISE)) == 0, FP8_ERR_UNSUPPORTED);
  FP8_CHECK(sA->dtype == FP8_DT_F32 && sB->dtype == FP8_DT_F32, FP8_ERR_INVALID_ARG);
  const int64_t M = A->shape[0], K = A->shape[1], N = B->shape[0];
  FP8_CHECK(B->shape[1] == K && shape_is(out_q, 2, M, N), FP8_ERR_INVALID_ARG);
  const int64_t la = numel(sA), lb = numel(sB);
  FP8_CHECK((la == 1 || la == M) && (lb == 1 || lb == N), FP8_ERR_INVALID_ARG);
  FP8_CHECK(K % 16 == 0 && aligned16(A->ptr) && aligned16(B->ptr) && aligned16(out_q->ptr), FP8_ERR_ALIGNMENT);
  FP8_CHECK(N % 128 == 0, FP8_ERR_UNSUPPORTED);  // whole 128-column row segments per epilogue lane
  FP8_CHECK(K > 0, FP8_ERR_UNSUPPORTED);          // an empty contraction: not implemented here
  FP8_CHECK(M < (int64_t(1) << 31) && N < (int64_t(1) << 31) && K < (int64_t(1) << 31), FP8_ERR_UNSUPPORTED);
  int mx = 0;
  if (out_granularity == FP8_GRAN_BLOCK_1x128) {
    FP8_CHECK(out_scales->dtype == FP8_DT_F32 && numel(out_scales) == M * (N / 128), FP8_ERR_INVALID_ARG);
  } else if (out_granularity == FP8_GRAN_MX) {
    FP8_CHECK(out_scales->dtype == FP8_DT_E8M0 && numel(out_scales) == mx_scale_bytes(M, N), FP8_ERR_INVALID_ARG);
    FP8_CHECK(aligned16(out_scales->ptr), FP8_ERR_ALIGNMENT);
    mx = 1;
  } else {
    return FP8_ERR_UNSUPPORTED;
  }
  if (M == 0 || N == 0) return FP8_OK;
  GemmArgs g = {};
  g.A = A->ptr;
  g.B = B->ptr;
  g.a_dtype = A->dtype;
  g.b_dtype = B->dtype;
  g.sA = static_cast<const float*>(sA->ptr);
  g.sB = static_cast<const float*>(sB->ptr);
  g.sA_len = la;
  g.sB_len = lb;
  g.out = nullptr;
  g.out_dtype = FP8_DT_BF16;
  g.M = M;
  g.N = N;
  g.K = K;
  g.mode = -1;
  g.q_out = out_q->ptr;
  g.q_scales = out_scales->ptr;
  g.q_mx = mx;
  g.q_fmt = out_q->dtype;
  return launch_gemm(g, c);
}

extern "C" int fp8_quantize_from_amax(const fp8_tensor* x, int granularity, int out_dtype, int layout,
                                      fp8_tensor* out, fp8_tensor* out_t, fp8_tensor* inv_scales,
                                      const fp8_tensor* amax, int32_t* d_status, void* stream) {
  Ctx c;
  FP8_TRY(make_ctx(&c, stream, d_status));
  FP8_CHECK(valid_desc(x) && x->dtype == FP8_DT_BF16 && x->ndim == 2, FP8_ERR_INVALID_ARG);
  FP8_CHECK(is_fp8(out_dtype) && layout >= 1 && layout <= 3, FP8_ERR_INVALID_ARG);
  FP8_CHECK(valid_desc(inv_scales) && inv_scales->dtype == FP8_DT_F32, FP8_ERR_INVALID_ARG);
  FP8_CHECK(valid_desc(amax) && amax->dtype == FP8_DT_F32, FP8_ERR_INVALID_ARG);
  const int64_t R = x->shape[0], C = x->shape[1];
  FP8_CHECK(C % 8 == 0 && aligned16(x->ptr), FP8_ERR_ALIGNMENT);
  const bool want_row = layout & FP8_LAYOUT_ROW_MAJOR, want_col = layout & FP8_LAYOUT_COL_MAJOR;
  if (want_row) {
    FP8_CHECK(valid_desc(out) && out->dtype == out_dtype && shape_is(out, 2, R, C), FP8_ERR_INVALID_ARG);
    FP8_CHECK(aligned16(out->ptr), FP8_ERR_ALIGNMENT);
  }
  if (want_col) {
    FP8_CHECK(valid_desc(out_t) && out_t->dtype == out_dtype && shape_is(out_t, 2, C, R), FP8_ERR_INVALID_ARG);
    FP8_CHECK(aligned16(out_t->ptr) && R % 16 == 0, FP8_ERR_ALIGNMENT);
  }
  const uint32_t* am = static_cast<const uint32_t*>(amax->ptr);
  if (granularity == FP8_GRAN_TENSOR) {
    FP8_CHECK(numel(amax) == 1 && numel(inv_scales) == 1, FP8_ERR_INVALID_ARG);
    return launch_quant_tensor_cast(x->ptr, R, C, out_dtype, want_row ? out->ptr : nullptr,
                                    want_col ? out_t->ptr : nullptr, static_cast<float*>(inv_scales->ptr), am, c, 16);
  }
  if (granularity == FP8_GRAN_COL) {
    FP8_CHECK(layout == FP8_LAYOUT_COL_MAJOR, FP8_ERR_UNSUPPORTED);
    FP8_CHECK(numel(amax) == C && numel(inv_scales) == C, FP8_ERR_INVALID_ARG);
    FP8_CHECK(R < (int64_t(1) << 31), FP8_ERR_UNSUPPORTED);
    return launch_quant_cols(x->ptr, R, C, 1, R, nullptr, out_dtype, out_t->ptr, R,
                             static_cast<float*>(inv_scales->ptr), nullptr, c, am);
  }
  return FP8_ERR_UNSUPPORTED;  // row granularity reads x once already
}

// ------------------------------------------------------------------------------------------
// fp8_grouped_mm

extern "C" int fp8_grouped_mm(const fp8_tensor* A, const fp8_tensor* B, const fp8_tensor* offsets,
                              const fp8_tensor* sA, const fp8_tensor* sB, fp8_tensor* out, int mode, int flags,
                              int32_t* d_status, void* stream) {
  (void)flags;
  Ctx c;
  FP8_TRY(make_ctx(&c, stream, d_status));
  FP8_CHECK(valid_desc(A) && valid_desc(B) && valid_desc(out) && valid_desc(offsets) && valid_desc(sA) &&
                valid_desc(sB),
            FP8_ERR_INVALID_ARG);
  FP8_CHECK(is_fp8(A->dtype) && is_fp8(B->dtype) && is_out(out->dtype), FP8_ERR_INVALID_ARG);
  FP8_CHECK(!(A->dtype == FP8_DT_E5M2 && B->dtype == FP8_DT_E5M2), FP8_ERR_UNSUPPORTED);
  FP8_CHECK(offsets->dtype == FP8_DT_I32 && offsets->ndim == 1 && offsets->shape[0] >= 1, FP8_ERR_INVALID_ARG);
  const bool mx = sA->dtype == FP8_DT_E8M0;
  FP8_CHECK(mx ? sB->dtype == FP8_DT_E8M0 : (sA->dtype == FP8_DT_F32 && sB->dtype == FP8_DT_F32), FP8_ERR_INVALID_ARG);
  FP8_CHECK(aligned16(A->ptr) && aligned16(B->ptr) && aligned16(out->ptr), FP8_ERR_ALIGNMENT);
  if (mx) FP8_CHECK(aligned16(sA->ptr) && aligned16(sB->ptr), FP8_ERR_ALIGNMENT);
  const int64_t E = offsets->shape[0];
  GemmArgs g = {};
  g.A = A->ptr;
  g.B = B->ptr;
  g.a_dtype = A->dtype;
  g.b_dtype = B->dtype;
  g.sA = static_cast<const float*>(sA->ptr);
  g.sB = static_cast<const float*>(sB->ptr);
  g.out = out->ptr;
  g.out_dtype = out->dtype;
  g.mode = mode;
  g.ends = static_cast<const int32_t*>(offsets->ptr);
  g.E = E;
  if (mx) {
    g.mx = 1;
    g.sfa = sA->ptr;
    g.sfb = sB->ptr;
    g.sA = nullptr;
    g.sB = nullptr;
  }
  if (mode == FP8_GROUPED_JAGGED_M) {
    FP8_CHECK(A->ndim == 2 && B->ndim == 3 && B->shape[0] == E, FP8_ERR_INVALID_ARG);
    const int64_t M = A->shape[0], K = A->shape[1], N = B->shape[1];
    FP8_CHECK(B->shape[2] == K && shape_is(out, 2, M, N), FP8_ERR_INVALID_ARG);
    FP8_CHECK(K > 0, FP8_ERR_UNSUPPORTED);  // an empty contraction: not implemented here
    if (mx) {
      FP8_CHECK(K % 128 == 0, FP8_ERR_UNSUPPORTED);
      const int64_t P = numel(sA) * 32 / K;  // the segment-padded rows of A's scales
      FP8_CHECK(numel(sA) == mx_scale_bytes(P, K) && P % 128 == 0 && P >= M + 127 * E, FP8_ERR_INVALID_ARG);
      FP8_CHECK(numel(sB) == E * mx_scale_bytes(N, K), FP8_ERR_INVALID_ARG);
      FP8_CHECK(M < (int64_t(1) << 31) && E * N < (int64_t(1) << 31), FP8_ERR_UNSUPPORTED);
      g.M = M;
      g.N = N;
      g.K = K;
      g.sfa_rows = P;
      if (M == 0 || N == 0) return FP8_OK;
      return launch_gemm(g, c);
    }
    FP8_CHECK(numel(sA) == M && numel(sB) == E * N, FP8_ERR_INVALID_ARG);
    FP8_CHECK(K % 16 == 0, FP8_ERR_ALIGNMENT);
    FP8_CHECK(M < (int64_t(1) << 31) && E * N < (int64_t(1) << 31), FP8_ERR_UNSUPPORTED);
    g.M = M;
    g.N = N;
    g.K = K;
    g.sA_len = M;
    g.sB_len = E * N;
    if (M == 0 || N == 0) return FP8_OK;
    return launch_gemm(g, c);
  }
  if (mode == FP8_GROUPED_JAGGED_K) {
    FP8_CHECK(A->ndim == 2 && B->ndim == 2 && A->shape[1] == B->shape[1], FP8_ERR_INVALID_ARG);
    const int64_t N = A->shape[0], Kd = B->shape[0], P = A->shape[1];
    FP8_CHECK(shape_is(out, 3, E, N, Kd), FP8_ERR_INVALID_ARG);
    FP8_CHECK(P > 0, FP8_ERR_UNSUPPORTED);  // no padded token columns at all: not implemented here
    if (mx) {
      FP8_CHECK(P % 128 == 0, FP8_ERR_UNSUPPORTED);
      FP8_CHECK(numel(sA) == mx_scale_bytes(N, P) && numel(sB) == mx_scale_bytes(Kd, P), FP8_ERR_INVALID_ARG);
      g.M = N;
      g.N = Kd;
      g.K = P;
      g.k_dim = Kd;
      g.sfa_rows = N;
      if (N == 0 || Kd == 0) return FP8_OK;
      return launch_gemm(g, c);
    }
    FP8_CHECK(numel(sA) == E * N && numel(sB) == E * Kd, FP8_ERR_INVALID_ARG);
    FP8_CHECK(P % 16 == 0, FP8_ERR_ALIGNMENT);
    g.M = N;
    g.N = Kd;
    g.K = P;
    g.k_dim = Kd;
    g.sA_len = E * N;
    g.sB_len = E * Kd;
    if (N == 0 || Kd == 0) return FP8_OK;
    return launch_gemm(g, c);
  }
  return FP8_ERR_INVALID_ARG;
}

// ------------------------------------------------------------------------------------------
// Linear forward / backward

static fp8_tensor T2(void* p, int dt, int64_t a, int64_t b) {
  fp8_tensor t = {};
  t.ptr = p;
  t.dtype = dt;
  t.ndim = 2;
  t.shape[0] = a;
  t.shape[1] = b;
  return t;
}
static fp8_tensor T1(void* p, int dt, int64_t a) {
  fp8_tensor t = {};
  t.ptr = p;
  t.dtype = dt;
  t.ndim = 1;
  t.shape[0] = a;
  return t;
}

// Workspace layout of the backward pass (each piece 256-byte aligned).
struct BwdLayout {
  size_t amax, dy_q, dy_inv, dyt_q, dyt_inv, wt_q, wt_inv, xt_q, xt_inv, col_scratch, col_scratch_bytes, total;
};
static BwdLayout bwd_layout(int64_t M, int64_t K, int64_t N, int gran, int wgrad) {
  BwdLayout L = {};
  size_t off = 0;
  auto take = [&](size_t bytes) {
    size_t o = off;
    off += (size_t)round_up((int64_t)bytes, 256);
    return o;
  };
  const bool rows = gran == FP8_GRAN_ROW, fp8w = wgrad == FP8_WGRAD_FP8;
  if (gran == FP8_GRAN_BLOCK_1x128) {  // dY in 1 x 128 tiles
    L.dy_q = take((size_t)(M * N));
    L.dy_inv = take((size_t)(M * ((N + 127) / 128)) * 4);
    L.total = off;
    return L;
  }
  if (gran == FP8_GRAN_MX) {  // dY in both layouts; its row-major then column-major MX scales
    L.dy_q = take((size_t)(M * N));
    L.dyt_q = fp8w ? take((size_t)(N * M)) : 0;
    L.dy_inv = take((size_t)(mx_scale_bytes(M, N) + (fp8w ? mx_scale_bytes(N, M) : 0)));
    L.total = off;
    return L;
  }
  L.amax = take(8);
  L.dy_q = take((size_t)(M * N));
  L.dy_inv = take((size_t)(rows ? M : 1) * 4);
  L.dyt_q = fp8w ? take((size_t)(N * M)) : 0;
  L.dyt_inv = (fp8w && rows) ? take((size_t)N * 4) : 0;
  L.wt_q = rows ? take((size_t)(K * N)) : 0;
  L.wt_inv = rows ? take((size_t)K * 4) : 0;
  L.xt_q = (fp8w && rows) ? take((size_t)(K * M)) : 0;
  L.xt_inv = (fp8w && rows) ? take((size_t)K * 4) : 0;
  // per-column scratch of the column-wise quantizations (used one after the other)
  // the column quantizes of W [N, K], dY [M, N] and x [M, K] share one scratch
  int64_t cw = col_ws_words(1, K, N);
  if (col_ws_words(1, N, M) > cw) cw = col_ws_words(1, N, M);
  if (col_ws_words(1, K, M) > cw) cw = col_ws_words(1, K, M);
  L.col_scratch = rows ? take((size_t)cw * 4) : 0;
  L.col_scratch_bytes = rows ? (size_t)cw * 4 : 0;
  L.total = off;
  return L;
}

// MX quantize of a bf16 [R, C] matrix: row-major codes q [R, C] with scales q_sf and, when qt is
// given, the column-major copy qt [C, R] with scales qt_sf, from one read of x.
static int mx_both(const fp8_tensor* x, int fmt, const fp8_tensor* q, const fp8_tensor* q_sf, const fp8_tensor* qt,
                   const fp8_tensor* qt_sf, const Ctx& c) {
  FP8_CHECK(valid_desc(x) && x->ndim == 2 && x->dtype == FP8_DT_BF16, FP8_ERR_INVALID_ARG);
  const int64_t R = x->shape[0], C = x->shape[1];
  FP8_CHECK(C % 128 == 0 && (!qt || R % 128 == 0), FP8_ERR_UNSUPPORTED);
  FP8_CHECK(valid_desc(q) && q->dtype == fmt && shape_is(q, 2, R, C), FP8_ERR_INVALID_ARG);
  FP8_CHECK(valid_desc(q_sf) && q_sf->dtype == FP8_DT_E8M0 && numel(q_sf) == mx_scale_bytes(R, C),
            FP8_ERR_INVALID_ARG);
  FP8_CHECK(aligned16(x->ptr) && aligned16(q->ptr) && aligned16(q_sf->ptr), FP8_ERR_ALIGNMENT);
  if (qt) {
    FP8_CHECK(valid_desc(qt) && qt->dtype == fmt && shape_is(qt, 2, C, R), FP8_ERR_INVALID_ARG);
    FP8_CHECK(valid_desc(qt_sf) && qt_sf->dtype == FP8_DT_E8M0 && numel(qt_sf) == mx_scale_bytes(C, R),
              FP8_ERR_INVALID_ARG);
    FP8_CHECK(aligned16(qt->ptr) && aligned16(qt_sf->ptr), FP8_ERR_ALIGNMENT);
  }
  return launch_mx_quant(x->ptr, 1, R, C, fmt, q->ptr, q_sf->ptr, qt ? qt->ptr : nullptr, R,
                         qt ? qt_sf->ptr : nullptr, nullptr, 0, nullptr, c);
}

extern "C" size_t fp8_workspace_size(int op, int64_t d0, int64_t d1, int64_t d2, int granularity, int wgrad_mode) {
  switch (op) {
    case FP8_OP_QUANTIZE:  // (d0, d1) = (groups, columns) for FP8_GRAN_COL; (segments, -) for MX
      if (granularity == FP8_GRAN_TENSOR) return 8;  // amax word, grid-barrier count
      if (granularity == FP8_GRAN_MX) return d0 > 0 ? (size_t)round_up(4 * (d0 + 1), 16) : 0;
      // (d0, d1, d2) = (groups, columns, rows of x over all groups) for FP8_GRAN_COL
      if (granularity == FP8_GRAN_COL)
        return (size_t)col_ws_words(d0 > 0 ? d0 : 1, d1 > 0 ? d1 : 0, d2 > 0 ? d2 : 0) * 4;
      return 0;
    case FP8_OP_LINEAR_FWD:
      return granularity == FP8_GRAN_TENSOR ? 256 : 0;
    case FP8_OP_LINEAR_BWD:
      return bwd_layout(d0, d1, d2, granularity, wgrad_mode).total;
    default:
      return 0;
  }
}

extern "C" int fp8_linear_fwd(const fp8_tensor* x, const fp8_tensor* w, int granularity, int flags, fp8_tensor* y,
                              fp8_linear_saved* saved, void* workspace, size_t workspace_bytes, int32_t* d_status,
                              void* stream) {
  Ctx c;
  FP8_TRY(make_ctx(&c, stream, d_status));
  FP8_CHECK(valid_desc(x) && valid_desc(w) && valid_desc(y) && saved, FP8_ERR_INVALID_ARG);
  FP8_CHECK(x->ndim == 2 && w->ndim == 2 && x->dtype == FP8_DT_BF16 && w->dtype == FP8_DT_BF16, FP8_ERR_INVALID_ARG);
  const int64_t M = x->shape[0], K = x->shape[1], N = w->shape[0];
  FP8_CHECK(w->shape[1] == K, FP8_ERR_INVALID_ARG);
  if (granularity == FP8_GRAN_TENSOR) {
    FP8_CHECK(workspace && workspace_bytes >= 8, FP8_ERR_WORKSPACE);
    const int xl = saved->xt_q.ptr ? FP8_LAYOUT_BOTH : FP8_LAYOUT_ROW_MAJOR;
    FP8_TRY(quantize_impl(x, FP8_GRAN_TENSOR, FP8_DT_E4M3, xl, &saved->x_q, &saved->xt_q, &saved->x_inv, nullptr,
                          workspace, workspace_bytes, c));
    FP8_TRY(quantize_impl(w, FP8_GRAN_TENSOR, FP8_DT_E4M3, FP8_LAYOUT_BOTH, &saved->w_q, &saved->wt_q, &saved->w_inv,
                          nullptr, workspace, workspace_bytes, c));
  } else if (granularity == FP8_GRAN_MX) {
    // x and W in both layouts, each from one read (the column-major copies feed the backward
    // GEMMs); x's column-major copy only when the caller keeps one (FP8 weight gradient)
    FP8_CHECK(M % 128 == 0 && K % 128 == 0 && N % 128 == 0, FP8_ERR_UNSUPPORTED);
    FP8_TRY(mx_both(x, FP8_DT_E4M3, &saved->x_q, &saved->x_inv, saved->xt_q.ptr ? &saved->xt_q : nullptr,
                    &saved->xt_inv, c));
    FP8_TRY(mx_both(w, FP8_DT_E4M3, &saved->w_q, &saved->w_inv, &saved->wt_q, &saved->wt_inv, c));
  } else if (granularity == FP8_GRAN_BLOCK_1x128) {
    // [B]: x in 1 x 128 tiles; W in 128 x 128 tiles, both layouts from one read (the scales of
    // the transposed copy are the same tiles, transposed)
    FP8_CHECK(K % 128 == 0 && N % 128 == 0, FP8_ERR_UNSUPPORTED);
    FP8_CHECK(valid_desc(&saved->x_inv) && saved->x_inv.dtype == FP8_DT_F32 && numel(&saved->x_inv) == M * (K / 128),
              FP8_ERR_INVALID_ARG);
    FP8_CHECK(valid_desc(&saved->w_inv) && valid_desc(&saved->wt_inv) && numel(&saved->w_inv) == (N / 128) * (K / 128) &&
                  numel(&saved->wt_inv) == (N / 128) * (K / 128) && saved->w_inv.dtype == FP8_DT_F32 &&
                  saved->wt_inv.dtype == FP8_DT_F32,
              FP8_ERR_INVALID_ARG);
    FP8_CHECK(shape_is(&saved->x_q, 2, M, K) && shape_is(&saved->w_q, 2, N, K) && shape_is(&saved->wt_q, 2, K, N),
              FP8_ERR_INVALID_ARG);
    FP8_TRY(quantize_impl(x, FP8_GRAN_BLOCK_1x128, FP8_DT_E4M3, FP8_LAYOUT_ROW_MAJOR, &saved->x_q, nullptr,
                          &saved->x_inv, nullptr, nullptr, 0, c));
    FP8_TRY(launch_blk_quant(w->ptr, N, K, FP8_DT_E4M3, true, saved->w_q.ptr, saved->wt_q.ptr,
                             static_cast<float*>(saved->w_inv.ptr), static_cast<float*>(saved->wt_inv.ptr), c));
    return scaled_mm_impl(&saved->x_q, &saved->w_q, &saved->x_inv, &saved->w_inv, y,
                          (flags & FP8_MM_FAST_ACCUM) | FP8_MM_BLOCKWISE, c);
  } else if (granularity == FP8_GRAN_ROW) {
    FP8_TRY(quantize_impl(x, FP8_GRAN_ROW, FP8_DT_E4M3, FP8_LAYOUT_ROW_MAJOR, &saved->x_q, nullptr, &saved->x_inv,
                          nullptr, nullptr, 0, c));
    FP8_TRY(quantize_impl(w, FP8_GRAN_ROW, FP8_DT_E4M3, FP8_LAYOUT_ROW_MAJOR, &saved->w_q, nullptr, &saved->w_inv,
                          nullptr, nullptr, 0, c));
  } else {
    return FP8_ERR_INVALID_ARG;
  }
  (void)M;
  (void)N;
  return scaled_mm_impl(&saved->x_q, &saved->w_q, &saved->x_inv, &saved->w_inv, y, flags & FP8_MM_FAST_ACCUM, c);
}

extern "C" int fp8_linear_bwd(const fp8_tensor* dy, const fp8_linear_saved* saved, const fp8_tensor* x,
                              const fp8_tensor* w, int granularity, int wgrad_mode, fp8_tensor* dx, fp8_tensor* dw,
                              void* workspace, size_t workspace_bytes, int32_t* d_status, void* stream) {
  Ctx c;
  FP8_TRY(make_ctx(&c, stream, d_status));
  FP8_CHECK(valid_desc(dy) && saved && dy->ndim == 2 && dy->dtype == FP8_DT_BF16, FP8_ERR_INVALID_ARG);
  FP8_CHECK(granularity == FP8_GRAN_TENSOR || granularity == FP8_GRAN_ROW || granularity == FP8_GRAN_MX ||
                granularity == FP8_GRAN_BLOCK_1x128,
            FP8_ERR_INVALID_ARG);
  FP8_CHECK(wgrad_mode == FP8_WGRAD_FP8 || wgrad_mode == FP8_WGRAD_BF16, FP8_ERR_INVALID_ARG);
  const int64_t M = dy->shape[0], N = dy->shape[1];
  FP8_CHECK(saved->x_q.ndim == 2 && saved->x_q.shape[0] == M, FP8_ERR_INVALID_ARG);
  const int64_t K = saved->x_q.shape[1];
  const bool rows = granularity == FP8_GRAN_ROW, fp8w = wgrad_mode == FP8_WGRAD_FP8;
  const bool need_dw = dw && dw->ptr;
  const BwdLayout L = bwd_layout(M, K, N, granularity, wgrad_mode);
  FP8_CHECK(workspace && workspace_bytes >= L.total, FP8_ERR_WORKSPACE);
  FP8_CHECK(aligned16(workspace), FP8_ERR_ALIGNMENT);
  uint8_t* ws = static_cast<uint8_t*>(workspace);
  fp8_tensor dy_q = T2(ws + L.dy_q, FP8_DT_E5M2, M, N);
  if (granularity == FP8_GRAN_BLOCK_1x128) {
    // [B]: dY in 1 x 128 tiles (along N) for dX = dY W with W's 128 x 128 tiles transposed;
    // the weight gradient in bf16
    FP8_CHECK(!(fp8w && need_dw), FP8_ERR_UNSUPPORTED);
    FP8_CHECK(N % 128 == 0 && K % 128 == 0, FP8_ERR_UNSUPPORTED);
    fp8_tensor dy_inv = T1(ws + L.dy_inv, FP8_DT_F32, M * (N / 128));
    if (dx && dx->ptr) {
      FP8_TRY(quantize_impl(dy, FP8_GRAN_BLOCK_1x128, FP8_DT_E5M2, FP8_LAYOUT_ROW_MAJOR, &dy_q, nullptr, &dy_inv,
                            nullptr, nullptr, 0, c));
      FP8_TRY(scaled_mm_impl(&dy_q, &saved->wt_q, &dy_inv, &saved->wt_inv, dx, FP8_MM_BLOCKWISE, c));
    }
    if (need_dw) {
      FP8_CHECK(valid_desc(x) && x->dtype == FP8_DT_BF16 && shape_is(x, 2, M, K), FP8_ERR_INVALID_ARG);
      FP8_TRY(scaled_mm_impl(dy, x, nullptr, nullptr, dw, FP8_MM_A_MN_MAJOR | FP8_MM_B_MN_MAJOR, c));
    }
    return FP8_OK;
  }
  if (granularity == FP8_GRAN_MX) {
    // dY in both layouts from one read: rows (blocks along N) for dX = dY W, columns (blocks
    // along M) for dW = dY^T x
    FP8_CHECK(M % 128 == 0 && N % 128 == 0 && K % 128 == 0, FP8_ERR_UNSUPPORTED);
    const bool want_dyt = fp8w && need_dw;
    fp8_tensor dy_sf = T1(ws + L.dy_inv, FP8_DT_E8M0, mx_scale_bytes(M, N));
    fp8_tensor dyt_q = T2(fp8w ? ws + L.dyt_q : nullptr, FP8_DT_E5M2, N, M);
    fp8_tensor dyt_sf = T1(ws + L.dy_inv + mx_scale_bytes(M, N), FP8_DT_E8M0, mx_scale_bytes(N, M));
    FP8_TRY(mx_both(dy, FP8_DT_E5M2, &dy_q, &dy_sf, want_dyt ? &dyt_q : nullptr, &dyt_sf, c));
    if (dx && dx->ptr) FP8_TRY(scaled_mm_impl(&dy_q, &saved->wt_q, &dy_sf, &saved->wt_inv, dx, 0, c));
    if (need_dw) {
      if (fp8w) {
        FP8_CHECK(saved->xt_q.ptr, FP8_ERR_INVALID_ARG);
        FP8_TRY(scaled_mm_impl(&dyt_q, &saved->xt_q, &dyt_sf, &saved->xt_inv, dw, 0, c));
      } else {
        FP8_CHECK(valid_desc(x) && x->dtype == FP8_DT_BF16 && shape_is(x, 2, M, K), FP8_ERR_INVALID_ARG);
        FP8_TRY(scaled_mm_impl(dy, x, nullptr, nullptr, dw, FP8_MM_A_MN_MAJOR | FP8_MM_B_MN_MAJOR, c));
      }
    }
    return FP8_OK;
  }
  fp8_tensor dy_inv = T1(ws + L.dy_inv, FP8_DT_F32, rows ? M : 1);
  fp8_tensor dyt_q = T2(fp8w ? ws + L.dyt_q : nullptr, FP8_DT_E5M2, N, M);
  if (!rows) {
    const int layout = (fp8w && need_dw) ? FP8_LAYOUT_BOTH : FP8_LAYOUT_ROW_MAJOR;
    FP8_TRY(quantize_impl(dy, FP8_GRAN_TENSOR, FP8_DT_E5M2, layout, &dy_q, &dyt_q, &dy_inv, nullptr, ws + L.amax, 8,
                          c));
    if (dx && dx->ptr)
      FP8_TRY(scaled_mm_impl(&dy_q, &saved->wt_q, &dy_inv, &saved->w_inv, dx, 0, c));
    if (need_dw) {
      if (fp8w) {
        FP8_CHECK(saved->xt_q.ptr, FP8_ERR_INVALID_ARG);
        FP8_TRY(scaled_mm_impl(&dyt_q, &saved->xt_q, &dy_inv, &saved->x_inv, dw, 0, c));
      } else {
        FP8_CHECK(valid_desc(x) && x->dtype == FP8_DT_BF16, FP8_ERR_INVALID_ARG);
        FP8_TRY(scaled_mm_impl(dy, x, nullptr, nullptr, dw, FP8_MM_A_MN_MAJOR | FP8_MM_B_MN_MAJOR, c));
      }
    }
    return FP8_OK;
  }
  // row granularity
  FP8_TRY(quantize_impl(dy, FP8_GRAN_ROW, FP8_DT_E5M2, FP8_LAYOUT_ROW_MAJOR, &dy_q, nullptr, &dy_inv, nullptr,
                        nullptr, 0, c));
  if (dx && dx->ptr) {
    FP8_CHECK(valid_desc(w) && w->dtype == FP8_DT_BF16 && shape_is(w, 2, N, K), FP8_ERR_INVALID_ARG);
    fp8_tensor wt_q = T2(ws + L.wt_q, FP8_DT_E4M3, K, N);
    fp8_tensor wt_inv = T1(ws + L.wt_inv, FP8_DT_F32, K);
    FP8_TRY(quantize_impl(w, FP8_GRAN_COL, FP8_DT_E4M3, FP8_LAYOUT_COL_MAJOR, nullptr, &wt_q, &wt_inv, nullptr,
                          ws + L.col_scratch, L.col_scratch_bytes, c));
    FP8_TRY(scaled_mm_impl(&dy_q, &wt_q, &dy_inv, &wt_inv, dx, 0, c));
  }
  if (need_dw) {
    FP8_CHECK(valid_desc(x) && x->dtype == FP8_DT_BF16 && shape_is(x, 2, M, K), FP8_ERR_INVALID_ARG);
    if (fp8w) {
      fp8_tensor dyt_inv = T1(ws + L.dyt_inv, FP8_DT_F32, N);
      fp8_tensor xt_q = T2(ws + L.xt_q, FP8_DT_E4M3, K, M);
      fp8_tensor xt_inv = T1(ws + L.xt_inv, FP8_DT_F32, K);
      FP8_TRY(quantize_impl(dy, FP8_GRAN_COL, FP8_DT_E5M2, FP8_LAYOUT_COL_MAJOR, nullptr, &dyt_q, &dyt_inv, nullptr,
                            ws + L.col_scratch, L.col_scratch_bytes, c));
      FP8_TRY(quantize_impl(x, FP8_GRAN_COL, FP8_DT_E4M3, FP8_LAYOUT_COL_MAJOR, nullptr, &xt_q, &xt_inv, nullptr,
                            ws + L.col_scratch, L.col_scratch_bytes, c));
      FP8_TRY(scaled_mm_impl(&dyt_q, &xt_q, &dyt_inv, &xt_inv, dw, 0, c));
    } else {
      FP8_TRY(scaled_mm_impl(dy, x, nullptr, nullptr, dw, FP8_MM_A_MN_MAJOR | FP8_MM_B_MN_MAJOR, c));
    }
  }
  return FP8_OK;
}
