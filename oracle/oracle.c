/*
 * Oracle for the FP8 dynamic-scaling linear (plain C, fp64 where the pages do not fix the
 * precision). TEST INFRASTRUCTURE ONLY: see oracle.h for who may use it and for the sources.
 *
 * Build: gcc -O2 -fopenmp -ffp-contract=off -fno-fast-math -fPIC -shared (no FMA contraction,
 * no reassociation: each line below rounds exactly as written).
 */
#include "oracle.h"

#include <math.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* The clamp floor applied to amax before the division ("EPS" in the recipe of [P3] section 2;
 * the pages name it without a value; 1e-12 is the reading taken here). */
static const double ORC_EPS = 1e-12;

/* ---------------------------------------------------------------------------------------- */
/* Formats ([P3] section 3): e4m3 = 1 sign, 4 exponent (bias 7), 3 mantissa bits, no Inf,
 * S.1111.111 is NaN, largest finite 1.75 * 2^8 = 448. e5m2 = 1 sign, 5 exponent (bias 15),
 * 2 mantissa bits, IEEE-style Inf/NaN at exponent 31, largest finite 1.75 * 2^15 = 57344.   */

typedef struct {
  int man_bits;   /* stored mantissa bits */
  int bias;       /* exponent bias */
  int emin;       /* exponent of the smallest normal */
  int max_efield; /* largest exponent field of a finite value */
  int max_mfield; /* largest mantissa field at max_efield */
} orc_fmt;

static orc_fmt fmt_of(int fmt) {
  orc_fmt f;
  if (fmt == ORC_E4M3) {
    f.man_bits = 3; f.bias = 7; f.emin = -6; f.max_efield = 15; f.max_mfield = 6;
  } else {
    f.man_bits = 2; f.bias = 15; f.emin = -14; f.max_efield = 30; f.max_mfield = 3;
  }
  return f;
}

double orc_fp8_max(int fmt) {
  orc_fmt f = fmt_of(fmt);
  return ldexp(1.0 + (double)f.max_mfield / (double)(1 << f.man_bits), f.max_efield - f.bias);
}

double orc_fp8_decode(uint8_t code, int fmt) {
  orc_fmt f = fmt_of(fmt);
  int s = code >> 7;
  int ebits = (fmt == ORC_E4M3) ? 4 : 5;
  int e = (code >> f.man_bits) & ((1 << ebits) - 1);
  int m = code & ((1 << f.man_bits) - 1);
  double v;
  if (fmt == ORC_E4M3 && e == 15 && m == 7) return NAN;
  if (fmt == ORC_E5M2 && e == 31) {
    if (m != 0) return NAN;
    return s ? -INFINITY : INFINITY;
  }
  if (e == 0)
    v = ldexp((double)m, f.emin - f.man_bits); /* subnormal: m * 2^(emin - p) */
  else
    v = ldexp(1.0 + (double)m / (double)(1 << f.man_bits), e - f.bias);
  return s ? -v : v;
}

static uint8_t max_code(orc_fmt f) {
  return (uint8_t)((f.max_efield << f.man_bits) | f.max_mfield);
}

uint8_t orc_fp8_encode(float v, int fmt) {
  orc_fmt f = fmt_of(fmt);
  uint32_t bits;
  memcpy(&bits, &v, 4);
  uint8_t sign = (uint8_t)((bits >> 31) << 7);
  uint32_t efield = (bits >> 23) & 0xFF;
  uint32_t frac = bits & 0x7FFFFF;
  if (efield == 0xFF) {
    if (frac != 0) return (uint8_t)(sign | 0x7F); /* NaN stays NaN */
    return (uint8_t)(sign | max_code(f));         /* Inf saturates to the largest finite */
  }
  if (efield == 0 && frac == 0) return sign; /* signed zero */

  /* |v| = sig * 2^x exactly, with lg = floor(log2 |v|). */
  uint32_t sig;
  int x, lg;
  if (efield == 0) {
    sig = frac;
    x = -149;
    int hb = 31;
    while (!((sig >> hb) & 1u)) --hb;
    lg = hb - 149;
  } else {
    sig = frac | 0x800000u;
    x = (int)efield - 150;
    lg = (int)efield - 127;
  }
  /* Target binade: the value's own exponent, floored at the smallest normal (below that the
   * quantum is the subnormal step). Quantum q = 2^(E8 - p); n = round(|v| / q), ties even. */
  int E8 = lg > f.emin ? lg : f.emin;
  int qe = E8 - f.man_bits;
  int shift = qe - x; /* > 0: fp32 always carries more bits than the target */
  uint32_t n;
  if (shift > 25) {
    n = 0; /* |v| < q / 2 */
  } else {
    n = sig >> shift;
    uint32_t rem = sig & ((1u << shift) - 1u);
    uint32_t half = 1u << (shift - 1);
    if (rem > half || (rem == half && (n & 1u))) n += 1;
  }
  if (n == 0) return sign;
  /* Rounding can carry into the next binade. */
  if (n == (1u << (f.man_bits + 1))) {
    n >>= 1;
    E8 += 1;
  }
  uint32_t efield8, mfield8;
  if (n < (1u << f.man_bits)) { /* subnormal result (only when E8 == emin) */
    efield8 = 0;
    mfield8 = n;
  } else {
    efield8 = (uint32_t)(E8 + f.bias);
    mfield8 = n - (1u << f.man_bits);
  }
  if ((int)efield8 > f.max_efield || ((int)efield8 == f.max_efield && (int)mfield8 > f.max_mfield))
    return (uint8_t)(sign | max_code(f)); /* saturate */
  return (uint8_t)(sign | (efield8 << f.man_bits) | mfield8);
}

void orc_fp8_encode_array(const float* v, int64_t n, int fmt, uint8_t* out) {
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) out[i] = orc_fp8_encode(v[i], fmt);
}

void orc_fp8_decode_array(const uint8_t* c, int64_t n, int fmt, double* out) {
  for (int64_t i = 0; i < n; ++i) out[i] = orc_fp8_decode(c[i], fmt);
}

/* ---------------------------------------------------------------------------------------- */
/* The quantization recipe of [P3] section 2, one group at a time.                          */

static float bf16_to_float(uint16_t b) {
  uint32_t u = (uint32_t)b << 16;
  float f;
  memcpy(&f, &u, 4);
  return f;
}

void orc_scale(float amax, int fmt, double* scale64, float* scale32, float* inv32) {
  double fp8_max = orc_fp8_max(fmt);
  /* amax promoted to fp64, clamped from below by eps, then fp8_max divided by it in fp64. */
  double a = (double)amax;
  if (a < ORC_EPS) a = ORC_EPS;
  double s = fp8_max / a;
  if (scale64) *scale64 = s;
  /* The multiply of an fp32 tensor by this 0-dim fp64 scale runs in fp32, so the scale the
   * multiply sees is the fp64 value rounded to fp32. */
  if (scale32) *scale32 = (float)s;
  /* The inverse is the fp64 reciprocal of the fp64 scale; the GEMM takes it as fp32. */
  if (inv32) *inv32 = (float)(1.0 / s);
}

/* x * scale in fp32, clamp to +-fp8_max, cast (RNE, saturating). */
static uint8_t scale_clamp_cast(float xf, float scale32, float fp8_max, int fmt) {
  float y = xf * scale32;
  if (y > fp8_max) y = fp8_max;
  if (y < -fp8_max) y = -fp8_max;
  return orc_fp8_encode(y, fmt);
}

void orc_quantize_tensor(const uint16_t* x, int64_t n, int fmt, uint8_t* q, float* inv) {
  /* step 1: amax of |x| (fp32; max involves no rounding) */
  float amax = 0.0f;
  for (int64_t i = 0; i < n; ++i) {
    float a = fabsf(bf16_to_float(x[i]));
    if (a > amax) amax = a;
  }
  /* step 2: scale */
  float scale32, inv32;
  orc_scale(amax, fmt, NULL, &scale32, &inv32);
  /* step 3: scale, clamp, cast */
  float fmax8 = (float)orc_fp8_max(fmt);
#pragma omp parallel for schedule(static)
  for (int64_t i = 0; i < n; ++i) q[i] = scale_clamp_cast(bf16_to_float(x[i]), scale32, fmax8, fmt);
  *inv = inv32;
}

void orc_quantize_rows(const uint16_t* x, int64_t R, int64_t C, int fmt, uint8_t* q, float* inv) {
  float fmax8 = (float)orc_fp8_max(fmt);
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < R; ++r) {
    const uint16_t* xr = x + r * C;
    float amax = 0.0f;
    for (int64_t c = 0; c < C; ++c) {
      float a = fabsf(bf16_to_float(xr[c]));
      if (a > amax) amax = a;
    }
    float scale32, inv32;
    orc_scale(amax, fmt, NULL, &scale32, &inv32);
    for (int64_t c = 0; c < C; ++c) q[r * C + c] = scale_clamp_cast(bf16_to_float(xr[c]), scale32, fmax8, fmt);
    inv[r] = inv32;
  }
}

/* Columns of the row range [r0, r1) of x [*, C] (row-major), one scale per column. */
static void quantize_col_range(const uint16_t* x, int64_t r0, int64_t r1, int64_t C, int fmt,
                               uint8_t* q, float* inv) {
  float fmax8 = (float)orc_fp8_max(fmt);
#pragma omp parallel for schedule(static)
  for (int64_t c = 0; c < C; ++c) {
    float amax = 0.0f;
    for (int64_t r = r0; r < r1; ++r) {
      float a = fabsf(bf16_to_float(x[r * C + c]));
      if (a > amax) amax = a;
    }
    float scale32, inv32;
    orc_scale(amax, fmt, NULL, &scale32, &inv32);
    for (int64_t r = r0; r < r1; ++r) q[r * C + c] = scale_clamp_cast(bf16_to_float(x[r * C + c]), scale32, fmax8, fmt);
    inv[c] = inv32;
  }
}

void orc_quantize_cols(const uint16_t* x, int64_t B, int64_t R, int64_t C, int fmt, uint8_t* q,
                       float* inv) {
  for (int64_t b = 0; b < B; ++b)
    quantize_col_range(x + b * R * C, 0, R, C, fmt, q + b * R * C, inv + b * C);
}

static int check_ends(const int32_t* ends, int64_t E, int64_t total) {
  int64_t prev = 0;
  for (int64_t e = 0; e < E; ++e) {
    if (ends[e] < prev) return -1;
    prev = ends[e];
  }
  return (E > 0 && prev == total) ? 0 : -1;
}

int orc_quantize_jagged_cols(const uint16_t* x, int64_t R, int64_t C, const int32_t* ends,
                             int64_t E, int fmt, uint8_t* q, float* inv) {
  if (check_ends(ends, E, R)) return -1;
  for (int64_t e = 0; e < E; ++e) {
    int64_t r0 = e ? ends[e - 1] : 0, r1 = ends[e];
    /* an empty segment still gets the scales of an all-zero group (amax 0 -> eps) */
    quantize_col_range(x, r0, r1, C, fmt, q, inv + e * C);
  }
  return 0;
}

/* ---------------------------------------------------------------------------------------- */
/* GEMMs: the dequant contract of [P3] section 2 (the GEMM multiplies its result by
 * scale_a * scale_b, the inverse scales), the layouts of [P3] section 4, the grouped contract
 * of [P1] "Scaling FP8 to MoE Architectures". Products of decoded FP8 values are exact in fp64;
 * the fp64 sum runs in k order.                                                              */

static void decode_table(int fmt, double* t) {
  for (int c = 0; c < 256; ++c) t[c] = orc_fp8_decode((uint8_t)c, fmt);
}

void orc_gemm_fp8(const uint8_t* A, int fmtA, int64_t a_sm, int64_t a_sk, const uint8_t* B,
                  int fmtB, int64_t b_sn, int64_t b_sk, const float* sA, int64_t sA_len,
                  const float* sB, int64_t sB_len, int64_t M, int64_t N, int64_t K,
                  const int64_t* rows, int64_t n_rows, double* out, double* absacc) {
  double ta[256], tb[256];
  decode_table(fmtA, ta);
  decode_table(fmtB, tb);
  int64_t cnt = rows ? n_rows : M;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < cnt; ++i) {
    int64_t m = rows ? rows[i] : i;
    double sa = (double)(sA_len == 1 ? sA[0] : sA[m]);
    for (int64_t n = 0; n < N; ++n) {
      double sb = (double)(sB_len == 1 ? sB[0] : sB[n]);
      double acc = 0.0, aacc = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        double p = ta[A[m * a_sm + k * a_sk]] * tb[B[n * b_sn + k * b_sk]];
        acc += p;
        aacc += fabs(p);
      }
      out[i * N + n] = sa * sb * acc;
      if (absacc) absacc[i * N + n] = fabs(sa * sb) * aacc;
    }
  }
}

void orc_gemm_bf16(const uint16_t* A, int64_t a_sm, int64_t a_sk, const uint16_t* B, int64_t b_sn,
                   int64_t b_sk, int64_t M, int64_t N, int64_t K, const int64_t* rows,
                   int64_t n_rows, double* out, double* absacc) {
  int64_t cnt = rows ? n_rows : M;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < cnt; ++i) {
    int64_t m = rows ? rows[i] : i;
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0, aacc = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        double p = (double)bf16_to_float(A[m * a_sm + k * a_sk]) * (double)bf16_to_float(B[n * b_sn + k * b_sk]);
        acc += p;
        aacc += fabs(p);
      }
      out[i * N + n] = acc;
      if (absacc) absacc[i * N + n] = aacc;
    }
  }
}

int orc_grouped_gemm_m(const uint8_t* A, int fmtA, const uint8_t* W, int fmtW, const float* sA,
                       const float* sB, const int32_t* ends, int64_t E, int64_t M, int64_t N,
                       int64_t K, const int64_t* rows, int64_t n_rows, double* out,
                       double* absacc) {
  if (check_ends(ends, E, M)) return -1;
  double ta[256], tb[256];
  decode_table(fmtA, ta);
  decode_table(fmtW, tb);
  int64_t cnt = rows ? n_rows : M;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < cnt; ++i) {
    int64_t r = rows ? rows[i] : i;
    int64_t e = 0;
    while (ends[e] <= r) ++e; /* the segment holding row r */
    const uint8_t* We = W + e * N * K;
    double sa = (double)sA[r];
    for (int64_t n = 0; n < N; ++n) {
      double sb = (double)sB[e * N + n];
      double acc = 0.0, aacc = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        double p = ta[A[r * K + k]] * tb[We[n * K + k]];
        acc += p;
        aacc += fabs(p);
      }
      out[i * N + n] = sa * sb * acc;
      if (absacc) absacc[i * N + n] = fabs(sa * sb) * aacc;
    }
  }
  return 0;
}

int orc_grouped_gemm_k(const uint8_t* G, int fmtG, const uint8_t* X, int fmtX, const float* sG,
                       const float* sX, const int32_t* ends, int64_t E, int64_t M, int64_t N,
                       int64_t K, const int64_t* nsel, int64_t n_sel, double* out,
                       double* absacc) {
  if (check_ends(ends, E, M)) return -1;
  double tg[256], tx[256];
  decode_table(fmtG, tg);
  decode_table(fmtX, tx);
  int64_t cnt = nsel ? n_sel : N;
  for (int64_t e = 0; e < E; ++e) {
    int64_t r0 = e ? ends[e - 1] : 0, r1 = ends[e];
#pragma omp parallel for schedule(dynamic, 1)
    for (int64_t i = 0; i < cnt; ++i) {
      int64_t n = nsel ? nsel[i] : i;
      double sg = (double)sG[e * N + n];
      for (int64_t k = 0; k < K; ++k) {
        double sx = (double)sX[e * K + k];
        double acc = 0.0, aacc = 0.0;
        for (int64_t r = r0; r < r1; ++r) {
          double p = tg[G[r * N + n]] * tx[X[r * K + k]];
          acc += p;
          aacc += fabs(p);
        }
        out[(e * cnt + i) * K + k] = sg * sx * acc;
        if (absacc) absacc[(e * cnt + i) * K + k] = fabs(sg * sx) * aacc;
      }
    }
  }
  return 0;
}

/* ---------------------------------------------------------------------------------------- */
/* Blockwise scaling. [P1] "AMD FP8 format in TorchAO" names a scale per fixed-size tile as the
 * third granularity; the tile shapes are not given there. Reading: 1 x 128 tiles for activations
 * and gradients (a scale per row and 128 consecutive elements of the contraction) and 128 x 128
 * tiles for weights, each tile quantized by the recipe of [P3] section 2 (amax over the tile,
 * fp64 scale with eps, fp32 multiply, clamp, cast, fp64 reciprocal). Edge tiles are smaller. */

void orc_quantize_blocks(const uint16_t* x, int64_t R, int64_t C, int64_t br, int64_t bc, int fmt,
                         uint8_t* q, float* inv) {
  float fmax8 = (float)orc_fp8_max(fmt);
  int64_t nbr = (R + br - 1) / br, nbc = (C + bc - 1) / bc;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t b = 0; b < nbr * nbc; ++b) {
    int64_t r0 = (b / nbc) * br, c0 = (b % nbc) * bc;
    int64_t r1 = r0 + br < R ? r0 + br : R, c1 = c0 + bc < C ? c0 + bc : C;
    float amax = 0.0f;
    for (int64_t r = r0; r < r1; ++r)
      for (int64_t c = c0; c < c1; ++c) {
        float a = fabsf(bf16_to_float(x[r * C + c]));
        if (a > amax) amax = a;
      }
    float scale32, inv32;
    orc_scale(amax, fmt, NULL, &scale32, &inv32);
    for (int64_t r = r0; r < r1; ++r)
      for (int64_t c = c0; c < c1; ++c) q[r * C + c] = scale_clamp_cast(bf16_to_float(x[r * C + c]), scale32, fmax8, fmt);
    inv[b] = inv32;
  }
}

/* Blockwise GEMM: out[i, n] = sum_k sA[m, k / 128] * sB[n / 128, k / 128] * dec(A[m, k]) * dec(B[n, k]),
 * m = rows[i] (or i); A [M, K] and B [N, K] row-major codes; sA [M, ceil(K / 128)] (1 x 128
 * tiles of A), sB [ceil(N / 128), ceil(K / 128)] (128 x 128 tiles of B). Each term is the fp64
 * product of the two inverse scales and the two decoded values; the sum runs in k order. */
void orc_gemm_blockwise(const uint8_t* A, int fmtA, const uint8_t* B, int fmtB, const float* sA,
                        const float* sB, int64_t M, int64_t N, int64_t K, const int64_t* rows,
                        int64_t n_rows, double* out, double* absacc) {
  double ta[256], tb[256];
  decode_table(fmtA, ta);
  decode_table(fmtB, tb);
  int64_t kb = (K + 127) / 128;
  int64_t cnt = rows ? n_rows : M;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < cnt; ++i) {
    int64_t m = rows ? rows[i] : i;
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0, aacc = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        double s = (double)sA[m * kb + k / 128] * (double)sB[(n / 128) * kb + k / 128];
        double p = s * (ta[A[m * K + k]] * tb[B[n * K + k]]);
        acc += p;
        aacc += fabs(p);
      }
      out[i * N + n] = acc;
      if (absacc) absacc[i * N + n] = aacc;
    }
  }
}

/* ---------------------------------------------------------------------------------------- */
/* MXFP8. The pages name it as the fourth scaling granularity, a scale per group stored with the
 * data ([P1] section "AMD FP8 format in TorchAO"), and as the next step for quantization and the
 * grouped GEMM ([P1] "Summary and Next Steps"); they fix nothing more. The block, the shared
 * scale and its rule are taken from the published OCP Microscaling Formats (MX) specification
 * v1.0 (sections 5.1-5.2 and 6.3):
 *   - a block is 32 consecutive elements along the contraction dimension;
 *   - its shared scale is X = 2^(floor(log2(amax)) - emax_elem), emax_elem being the exponent
 *     of the element format's largest normal (8 for e4m3: 448 = 1.75 * 2^8; 15 for e5m2);
 *   - X is stored as E8M0: an unsigned biased exponent, bias 127, codes 0..254 for
 *     2^-127..2^127 and 255 for NaN;
 *   - each element is x / X cast to the element format, rounding to nearest even and
 *     saturating at the largest finite value.
 * An exponent below -127 (an all-zero block, log2(0) = -inf, or amax < 2^-119) is clamped to
 * -127. A NaN or infinite amax gives the NaN scale. */

static int mx_emax_elem(int fmt) { return fmt == ORC_E4M3 ? 8 : 15; }

uint8_t orc_mx_scale(float amax, int fmt) {
  if (isnan(amax) || isinf(amax)) return 0xFF;
  int e = -127;
  if (amax > 0.0f) {
    int ex;
    frexp((double)amax, &ex); /* amax = f * 2^ex, f in [0.5, 1): floor(log2(amax)) = ex - 1 */
    e = (ex - 1) - mx_emax_elem(fmt);
    if (e < -127) e = -127;
    if (e > 127) e = 127;
  }
  return (uint8_t)(e + 127);
}

double orc_e8m0_decode(uint8_t code) { return code == 0xFF ? NAN : ldexp(1.0, (int)code - 127); }

int orc_mx_quantize_rows(const uint16_t* x, int64_t R, int64_t C, int fmt, uint8_t* q, uint8_t* sc) {
  if (C % 32) return -1;
  const int64_t nb = C / 32;
  const double fmax8 = orc_fp8_max(fmt);
#pragma omp parallel for schedule(static)
  for (int64_t r = 0; r < R; ++r) {
    for (int64_t b = 0; b < nb; ++b) {
      const uint16_t* xb = x + r * C + b * 32;
      float amax = 0.0f;
      for (int i = 0; i < 32; ++i) {
        float a = fabsf(bf16_to_float(xb[i]));
        if (a > amax || isnan(a)) amax = a;
      }
      uint8_t code = orc_mx_scale(amax, fmt);
      double X = orc_e8m0_decode(code);
      for (int i = 0; i < 32; ++i) {
        /* x / X is exact in fp64 (X is a power of two). Its fp32 copy is exact too, except for
         * magnitudes below 2^-126, far under half the smallest FP8 subnormal, which encode to a
         * signed zero either way. */
        double v = (double)bf16_to_float(xb[i]) / X;
        if (v > fmax8) v = fmax8;
        if (v < -fmax8) v = -fmax8;
        q[r * C + b * 32 + i] = orc_fp8_encode((float)v, fmt);
      }
      sc[r * nb + b] = code;
    }
  }
  return 0;
}

/* MX GEMM: out[i, n] = sum_k X_A[m, k / 32] * X_B[n, k / 32] * dec(A[m, k]) * dec(B[n, k]),
 * m = rows[i] (or i); A [M, K] and B [N, K] row-major codes, sA [M, K / 32] and sB [N, K / 32]
 * E8M0 codes. Every term is exact in fp64 (a product of two FP8 values and two powers of two);
 * the sum runs in k order. */
int orc_gemm_mx(const uint8_t* A, int fmtA, const uint8_t* B, int fmtB, const uint8_t* sA,
                const uint8_t* sB, int64_t M, int64_t N, int64_t K, const int64_t* rows,
                int64_t n_rows, double* out, double* absacc) {
  if (K % 32) return -1;
  const int64_t nb = K / 32;
  double ta[256], tb[256], ts[256];
  decode_table(fmtA, ta);
  decode_table(fmtB, tb);
  for (int c = 0; c < 256; ++c) ts[c] = orc_e8m0_decode((uint8_t)c);
  int64_t cnt = rows ? n_rows : M;
#pragma omp parallel for schedule(dynamic, 1)
  for (int64_t i = 0; i < cnt; ++i) {
    int64_t m = rows ? rows[i] : i;
    for (int64_t n = 0; n < N; ++n) {
      double acc = 0.0, aacc = 0.0;
      for (int64_t k = 0; k < K; ++k) {
        double p = ts[sA[m * nb + k / 32]] * ts[sB[n * nb + k / 32]] * (ta[A[m * K + k]] * tb[B[n * K + k]]);
        acc += p;
        aacc += fabs(p);
      }
      out[i * N + n] = acc;
      if (absacc) absacc[i * N + n] = aacc;
    }
  }
  return 0;
}

int orc_num_threads(void) {
#ifdef _OPENMP
  return omp_get_max_threads();
#else
  return 1;
#endif
}

/* The thread count of the parallel loops that follow (timing only: results do not depend on it). */
void orc_set_num_threads(int n) {
#ifdef _OPENMP
  if (n > 0) omp_set_num_threads(n);
#else
  (void)n;
#endif
}
