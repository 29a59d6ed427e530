/*
 * Oracle for the FP8 dynamic-scaling linear: a plain, slow CPU restatement of what the
 * hot path computes.
 *
 * TEST INFRASTRUCTURE ONLY. Nothing on the product path may include, link or call this.
 * Only tests/, __graft_entry__.smoke() and bench.py's cpu_baseline / reference leg use it.
 * It shares no code, header, table or constant with the CUDA library.
 *
 * Sources (web pages, cited by title and section):
 *  [P3]  "FP8 Training: Quantization, Autograd, Torchao", section 2 "The quantization math"
 *        (the amax -> fp64 scale -> multiply -> clamp -> cast recipe and the inverse scale),
 *        section 3 "Format choice: e4m3 vs e5m2" (the two formats and their maxima),
 *        section 4 "_scaled_mm layout requirements" (the three GEMMs of a Linear) and
 *        section 5 "use_fast_accum".
 *  [P1]  "FP8 training on AMD GPUs with TorchTitan and TorchAO", section "Scaling FP8 to MoE
 *        Architectures" and Figure 3 (grouped GEMM: per-row activation scales,
 *        per-expert-column weight scales, an offsets tensor routing rows to experts); section
 *        "AMD FP8 format in TorchAO" (the four granularities, MXFP8 among them) and "Summary
 *        and Next Steps" (MXFP8 quantization and grouped GEMM as the next step).
 *  [OCP] OCP Microscaling Formats (MX) Specification v1.0, a published standard outside the
 *        pages: the MX block of 32, the E8M0 scale and the rule that derives it from amax.
 *
 * Every floating-point step is written out in the order the recipe states. Inputs in bf16
 * are passed as raw uint16 bit patterns; FP8 values as raw uint8 codes.
 */
#ifndef FP8_ORACLE_H
#define FP8_ORACLE_H

#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORC_E4M3 = 0, ORC_E5M2 = 1 };

/* Largest finite magnitude of the format: 448 (e4m3) or 57344 (e5m2). */
double orc_fp8_max(int fmt);
/* Value of one FP8 code, from its sign / exponent / mantissa fields. NaN codes give NaN. */
double orc_fp8_decode(uint8_t code, int fmt);
/* Round-to-nearest-even, saturating (finite) conversion of an fp32 value to an FP8 code. */
uint8_t orc_fp8_encode(float v, int fmt);
void orc_fp8_encode_array(const float* v, int64_t n, int fmt, uint8_t* out);
void orc_fp8_decode_array(const uint8_t* c, int64_t n, int fmt, double* out);

/* The scale step for one group's amax: scale64 = fp8_max / max(amax, eps) in fp64,
 * scale32 = that value rounded to fp32 (what the fp32 multiply sees), inv32 = the fp64
 * reciprocal of scale64 rounded to fp32 (the dequant scale handed to the GEMM). */
void orc_scale(float amax, int fmt, double* scale64, float* scale32, float* inv32);

/* Quantize with one scale for the whole tensor. q: codes in x's order. inv: one float. */
void orc_quantize_tensor(const uint16_t* x, int64_t n, int fmt, uint8_t* q, float* inv);
/* One scale per row of x [R, C] (amax over the row). q [R, C], inv [R]. */
void orc_quantize_rows(const uint16_t* x, int64_t R, int64_t C, int fmt, uint8_t* q, float* inv);
/* One scale per (batch b, column c) of x [B, R, C] (amax over the R rows of the column).
 * q [B, R, C] in x's own (row-major) order, inv [B, C]. */
void orc_quantize_cols(const uint16_t* x, int64_t B, int64_t R, int64_t C, int fmt, uint8_t* q,
                       float* inv);
/* One scale per (segment e, column c) of x [R, C], where segment e holds rows
 * [ends[e-1], ends[e]) (ends[-1] = 0). q [R, C] row-major, inv [E, C]. An empty segment's
 * scales are those of an all-zero group. Returns 0, or -1 when ends is not non-decreasing or
 * its last entry is not R. */
int orc_quantize_jagged_cols(const uint16_t* x, int64_t R, int64_t C, const int32_t* ends,
                             int64_t E, int fmt, uint8_t* q, float* inv);

/* Scaled FP8 GEMM, fp64 accumulation of decoded values:
 *   out[i, n] = sA[m] * sB[n] * sum_k dec(A[m, k]) * dec(B[n, k]),  m = rows[i] (or i)
 * A(m, k) is read at A[m * a_sm + k * a_sk]; B(n, k) at B[n * b_sn + k * b_sk].
 * sA has M entries (or 1 when sA_len == 1); sB has N entries (or 1).
 * absacc (optional) receives |sA * sB| * sum_k |dec(a) * dec(b)|, the tolerance reference.
 * rows == NULL computes all M rows. */
void orc_gemm_fp8(const uint8_t* A, int fmtA, int64_t a_sm, int64_t a_sk, const uint8_t* B,
                  int fmtB, int64_t b_sn, int64_t b_sk, const float* sA, int64_t sA_len,
                  const float* sB, int64_t sB_len, int64_t M, int64_t N, int64_t K,
                  const int64_t* rows, int64_t n_rows, double* out, double* absacc);

/* Plain bf16 GEMM with fp64 accumulation (the high-precision weight-gradient GEMM):
 *   out[i, n] = sum_k A(m, k) * B(n, k), strides as for orc_gemm_fp8. */
void orc_gemm_bf16(const uint16_t* A, int64_t a_sm, int64_t a_sk, const uint16_t* B, int64_t b_sn,
                   int64_t b_sk, int64_t M, int64_t N, int64_t K, const int64_t* rows,
                   int64_t n_rows, double* out, double* absacc);

/* MoE grouped GEMM, rows jagged by expert:
 *   out[i, n] = sA[r] * sB[e, n] * sum_k dec(A[r, k]) * dec(W[e, n, k]),  r = rows[i] (or i),
 * e the expert whose segment holds row r. A [M, K], W [E, N, K], sA [M], sB [E, N].
 * Returns 0, or -1 for bad ends. */
int orc_grouped_gemm_m(const uint8_t* A, int fmtA, const uint8_t* W, int fmtW, const float* sA,
                       const float* sB, const int32_t* ends, int64_t E, int64_t M, int64_t N,
                       int64_t K, const int64_t* rows, int64_t n_rows, double* out,
                       double* absacc);

/* MoE grouped GEMM, contraction jagged by expert (per-expert weight gradient):
 *   out[e, i, k] = sG[e, n] * sX[e, k] * sum_{r in segment e} dec(G[r, n]) * dec(X[r, k]),
 * n = nsel[i] (or i). G [M, N] and X [M, K] row-major codes; sG [E, N], sX [E, K].
 * An empty segment gives zeros. out is [E, n_sel, K]. Returns 0, or -1 for bad ends. */
int orc_grouped_gemm_k(const uint8_t* G, int fmtG, const uint8_t* X, int fmtX, const float* sG,
                       const float* sX, const int32_t* ends, int64_t E, int64_t M, int64_t N,
                       int64_t K, const int64_t* nsel, int64_t n_sel, double* out,
                       double* absacc);

/* Blockwise scaling (tiles of br x bc; the reading takes 1 x 128 for activations and gradients,
 * 128 x 128 for weights): each tile quantized by the recipe. q [R, C] codes, inv
 * [ceil(R/br), ceil(C/bc)] inverse scales. */
void orc_quantize_blocks(const uint16_t* x, int64_t R, int64_t C, int64_t br, int64_t bc, int fmt,
                         uint8_t* q, float* inv);
/* Blockwise GEMM: out[i, n] = sum_k sA[m, k/128] sB[n/128, k/128] dec(A[m, k]) dec(B[n, k]),
 * m = rows[i] (or i). A [M, K], B [N, K] row-major; sA [M, ceil(K/128)], sB [ceil(N/128),
 * ceil(K/128)]. absacc gets the sum of the terms' magnitudes. */
void orc_gemm_blockwise(const uint8_t* A, int fmtA, const uint8_t* B, int fmtB, const float* sA,
                        const float* sB, int64_t M, int64_t N, int64_t K, const int64_t* rows,
                        int64_t n_rows, double* out, double* absacc);

/* MXFP8 (OCP Microscaling Formats v1.0; the pages name the format only): the E8M0 scale code
 * of a 32-element block with this amax, 2^(floor(log2 amax) - emax_elem) clamped below at
 * 2^-127 (255 = NaN for a NaN or infinite amax); the value of an E8M0 code. */
uint8_t orc_mx_scale(float amax, int fmt);
double orc_e8m0_decode(uint8_t code);
/* Blocks of 32 consecutive elements along each row of x [R, C] (C a multiple of 32): q [R, C]
 * codes, sc [R, C / 32] E8M0 scale codes. Returns 0, or -1 when C % 32 != 0. */
int orc_mx_quantize_rows(const uint16_t* x, int64_t R, int64_t C, int fmt, uint8_t* q, uint8_t* sc);
/* MX GEMM: out[i, n] = sum_k X_A[m, k/32] X_B[n, k/32] dec(A[m, k]) dec(B[n, k]), m = rows[i]
 * (or i). A [M, K], B [N, K] row-major; sA [M, K/32], sB [N, K/32] E8M0 codes. absacc gets the
 * sum of the terms' magnitudes. Returns 0, or -1 when K % 32 != 0. */
int orc_gemm_mx(const uint8_t* A, int fmtA, const uint8_t* B, int fmtB, const uint8_t* sA,
                const uint8_t* sB, int64_t M, int64_t N, int64_t K, const int64_t* rows,
                int64_t n_rows, double* out, double* absacc);

/* Number of OpenMP threads the oracle runs on. */
int orc_num_threads(void);
void orc_set_num_threads(int n);

#ifdef __cplusplus
}
#endif
#endif
