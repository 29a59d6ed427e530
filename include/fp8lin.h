/*
 * fp8lin — FP8 dynamic-scaling linear for NVIDIA GB300 (sm_103a): C ABI.
 *
 * What it computes (sources are web pages, cited by title and section):
 *  [Q]  "FP8 Training: Quantization, Autograd, Torchao", section 2 "The quantization math":
 *       per group (tensor, row or column) amax = max|x| in fp32; scale = fp8_max / max(amax, eps)
 *       in fp64; q = cast(clamp(x * scale, -fp8_max, fp8_max)); the GEMM receives the inverse
 *       scale (the fp64 reciprocal of scale) and multiplies its result by scale_a * scale_b.
 *  [F]  same page, section 3 "Format choice: e4m3 vs e5m2": e4m3 (max 448) for activations and
 *       weights, e5m2 (max 57344) for gradients.
 *  [L]  same page, section 4 "_scaled_mm layout requirements": the three GEMMs of a Linear
 *       (forward out = x W^T, grad-input dX = dY W, grad-weight dW = dY^T x) with A row-major
 *       and B column-major, i.e. both operands contiguous along the contraction dimension
 *       ("K-major"); section 5 "use_fast_accum" (forward True, backward False).
 *  [G]  "FP8 training on AMD GPUs with TorchTitan and TorchAO", section "Scaling FP8 to MoE
 *       Architectures" and Figure 3: a grouped GEMM over experts routed by an offsets tensor,
 *       with per-row activation scales and per-expert per-column weight scales.
 *  [W]  same page, Figure 1 caption: the high-precision weight-gradient recipe (forward and
 *       grad-input GEMMs in FP8, the weight-gradient GEMM in BF16).
 *  [T]  same page, "Level 1" and "Level 2" of "Triton Kernel Optimization": one fused kernel per
 *       quantization (no intermediate tensors in HBM), the column-wise variant that writes a
 *       column-major output through on-chip staging (no separate transpose copy), and the
 *       dual output (row- and column-major from one read).
 *  [B]  same page, section "AMD FP8 format in TorchAO": blockwise scaling, one scale per
 *       fixed-size tile. The tile shapes are not given; this library takes 1 x 128 tiles for
 *       activations and gradients (a scale per row and 128 consecutive contraction elements) and
 *       128 x 128 tiles for weights, each tile quantized by the recipe [Q]. The GEMM computes
 *       sum_k sA[m, k/128] sB[n/128, k/128] A[m, k] B[n, k]: the tensor cores accumulate each
 *       128-deep K block separately in fp32 and the epilogue warps add the block products scaled
 *       by sA * sB into fp32 registers.
 *  [MX] same page, section "AMD FP8 format in TorchAO" (MXFP8: a scale per group stored with the
 *       data) and "Summary and Next Steps" (MXFP8 quantization and grouped GEMM next). The pages
 *       give no more; block, scale and rule are those of the OCP Microscaling Formats (MX)
 *       specification v1.0: blocks of 32 consecutive elements along the contraction dimension,
 *       one E8M0 scale X = 2^(floor(log2(amax)) - emax_elem) per block (emax_elem 8 for e4m3,
 *       15 for e5m2; exponent clamped below at -127), elements x / X cast round-to-nearest-even
 *       with saturation. The GEMM computes sum_k X_A[m, k/32] X_B[n, k/32] A[m, k] B[n, k].
 *
 * Conventions for every entry point:
 *  - Tensors are described by fp8_tensor: a DEVICE pointer (global memory, 16-byte aligned),
 *    a dtype, and a logical shape, always dense and row-major (last index contiguous). A
 *    "column-major [R, C]" operand is passed as the row-major tensor of shape [C, R].
 *  - Ownership: the caller allocates and frees every buffer, including the workspace. The
 *    library never allocates device memory, never synchronizes the host, and never reads a
 *    device buffer (offsets included) on the host.
 *  - Streams: every call is asynchronous on `stream` (a cudaStream_t; NULL = legacy default
 *    stream). Outputs are defined once the stream reaches the call, and only if both the
 *    return value and the device status word are 0.
 *  - Return value: synchronous argument checking. FP8_OK, or an FP8_ERR_* code; on error
 *    nothing was launched.
 *  - d_status (optional, device int32): conditions found on the device are OR-ed into it
 *    (FP8_DEV_*). The caller zeroes it and reads it after its own synchronization. When a
 *    call's kernels find such a condition they stop early and leave outputs undefined.
 *  - Scales, in and out, are always fp32 INVERSE (dequantization) scales ([Q]).
 *  - Not re-entrant on one workspace: calls that share a workspace must be stream-ordered.
 */
#ifndef FP8LIN_H
#define FP8LIN_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* element types */
enum {
  FP8_DT_BF16 = 1,
  FP8_DT_F32 = 2,
  FP8_DT_E4M3 = 3, /* OCP float8 e4m3fn: bias 7, no Inf, max 448 */
  FP8_DT_E5M2 = 4, /* OCP float8 e5m2: bias 15, max 57344 */
  FP8_DT_I32 = 5,
  FP8_DT_E8M0 = 6  /* OCP E8M0 scale codes (MX): 2^(code - 127), 0xFF = NaN; one byte each */
};

/* scale granularity */
enum {
  FP8_GRAN_TENSOR = 0,
  FP8_GRAN_ROW = 1,
  FP8_GRAN_COL = 2,
  FP8_GRAN_MX = 3,
  FP8_GRAN_BLOCK_1x128 = 4,   /* blockwise [B]: one scale per row and 128 consecutive columns */
  FP8_GRAN_BLOCK_128x128 = 5  /* blockwise [B]: one scale per 128 x 128 tile */
};

/*
 * MX scale layout (FP8_GRAN_MX; [MX]). An MX operand with R rows (its non-contraction index) and
 * contraction length K (K % 128 == 0) carries E8M0 codes for blocks of 32 along K, stored in
 * 512-byte blocks [ceil(R / 128)][K / 128][512]; inside a block the code of row r, K block j
 * (elements 32 j .. 32 j + 31) is at byte (r % 32) * 16 + ((r / 32) % 4) * 4 + (j % 4). This is
 * the order in which the tensor cores' block-scaled MMA reads scales from tensor memory, so the
 * GEMM copies each block unchanged. Rows past R in the last 128-row block are never read for
 * results. Bytes: fp8_mx_scale_bytes(R, K). Batched operands ([B, R, K]) repeat the layout per
 * batch entry. With segment offsets, rows are placed in the segment-padded row space (segment e
 * at padded rows pstart_e = sum_{j<e} roundup(count_j, 128)), P rows in all.
 */

/* output layouts of fp8_quantize (bit mask) */
enum { FP8_LAYOUT_ROW_MAJOR = 1, FP8_LAYOUT_COL_MAJOR = 2, FP8_LAYOUT_BOTH = 3 };

/* GEMM flags (bit mask) */
enum {
  FP8_MM_FAST_ACCUM = 1, /* accepted for parity with the pages' forward GEMM; the tcgen05
                            accumulator is fp32 in tensor memory either way */
  FP8_MM_A_MN_MAJOR = 2, /* BF16 only: A is given as [K, M] (M contiguous) */
  FP8_MM_B_MN_MAJOR = 4, /* BF16 only: B is given as [K, N] (N contiguous) */
  FP8_MM_BLOCKWISE = 8   /* FP8 only: sA [M, K/128] (1 x 128 tiles of A) and sB [ceil(N/128), K/128]
                            (128 x 128 tiles of B) inverse scales, K % 128 == 0 ([B]) */
};

/* grouped GEMM modes */
enum { FP8_GROUPED_JAGGED_M = 0, FP8_GROUPED_JAGGED_K = 1 };

/* weight-gradient recipe of fp8_linear_bwd */
enum { FP8_WGRAD_FP8 = 0, FP8_WGRAD_BF16 = 1 };

/* operations for fp8_workspace_size */
enum { FP8_OP_QUANTIZE = 0, FP8_OP_LINEAR_FWD = 1, FP8_OP_LINEAR_BWD = 2 };

/* synchronous return codes */
enum {
  FP8_OK = 0,
  FP8_ERR_INVALID_ARG = 1, /* null pointer, wrong dtype, rank or shape mismatch */
  FP8_ERR_UNSUPPORTED = 2, /* a valid request this library does not implement */
  FP8_ERR_ALIGNMENT = 3,   /* pointer not 16-byte aligned, or a contiguous dimension whose
                              byte length is not a multiple of 16 (e.g. K % 16 for FP8) */
  FP8_ERR_WORKSPACE = 4,   /* workspace missing or smaller than fp8_workspace_size() */
  FP8_ERR_CUDA = 5,        /* a CUDA runtime call or kernel launch failed */
  FP8_ERR_DEVICE = 6       /* no usable sm_103 device current */
};

/* device status bits (OR-ed into *d_status) */
enum {
  FP8_DEV_BAD_OFFSETS = 1 << 8, /* offsets not non-decreasing, or last entry != total rows */
  FP8_DEV_TIMEOUT = 1 << 9      /* a bounded on-device wait ran out; the kernel drained and
                                   returned */
};

typedef struct fp8_tensor {
  void* ptr;        /* device pointer, 16-byte aligned */
  int32_t dtype;    /* FP8_DT_* */
  int32_t ndim;     /* 1, 2 or 3 */
  int64_t shape[3]; /* logical shape, dense row-major */
} fp8_tensor;

/*
 * fp8_quantize — the quantization chain of [Q] in one fused pass per output ([T]).
 *
 *  x           bf16 [R, C], or [B, R, C] for a batch of matrices (e.g. MoE expert weights).
 *              C % 8 == 0 (16-byte rows).
 *  granularity FP8_GRAN_TENSOR: one scale for all of x.
 *              FP8_GRAN_BLOCK_1x128 ([B]): one scale per row and 128 columns; ROW_MAJOR only;
 *                               2-D x, C % 128 == 0; inv_scales fp32 [R, C / 128].
 *              FP8_GRAN_BLOCK_128x128 ([B]): one scale per 128 x 128 tile; 2-D x, C % 128 == 0
 *                               (and R % 128 == 0 for COL_MAJOR); inv_scales fp32: ROW_MAJOR
 *                               [ceil(R/128), C/128]; COL_MAJOR [C/128, R/128] (the scales of the
 *                               transposed operand); BOTH the first followed by the second.
 *              FP8_GRAN_MX:     MXFP8 ([MX]): one E8M0 scale per 32 elements; C % 128 == 0.
 *                               ROW_MAJOR: blocks along rows, `out` in x's shape, scales over
 *                               (rows R, contraction C). COL_MAJOR: blocks down columns (R % 128
 *                               == 0 without offsets), `out_t` [C, R] ([B, C, R]), scales over
 *                               (rows C, contraction R). BOTH: both from one read.
 *                               With `offsets` (2-D x): segments padded to 128 rows; `out_t` is
 *                               [C, P] as for COL granularity and the row-major scales use the
 *                               padded row space, P % 128 == 0, P >= R + 127 E.
 *              FP8_GRAN_ROW:    one scale per row (amax over the C entries of the row);
 *                               a 3-D x is treated as [B*R, C].
 *              FP8_GRAN_COL:    one scale per column (amax over the R rows of the column), per
 *                               batch entry for 3-D x; with `offsets`, one scale per
 *                               (segment, column) where segment e holds rows
 *                               [offsets[e-1], offsets[e]) (offsets[-1] = 0) of a 2-D x.
 *  out_dtype   FP8_DT_E4M3 or FP8_DT_E5M2 ([F]).
 *  layout      FP8_LAYOUT_ROW_MAJOR: `out` = codes in x's shape.
 *              FP8_LAYOUT_COL_MAJOR: `out_t` = codes transposed: [C, R] (2-D), [B, C, R]
 *                (3-D), or, with offsets, [C, P] in the segment-padded layout: segment e
 *                starts at column pstart_e = sum_{j<e} roundup(count_j, 128) and is followed
 *                by zero codes up to the next multiple of 128. P >= R + 127 E and
 *                P % 16 == 0; fp8_jagged_padded_rows(R, E) gives the recommended P.
 *                For 2-D/3-D, R % 16 == 0.
 *              FP8_LAYOUT_BOTH: both (tensor granularity only: one read, two outputs).
 *              ROW granularity supports ROW_MAJOR; COL granularity supports COL_MAJOR.
 *  inv_scales  fp32: [1] (tensor), [R] or [B*R] (row), [C], [B, C] or [E, C] (col).
 *              MX: E8M0 bytes in the MX scale layout: ROW_MAJOR B * fp8_mx_scale_bytes(R, C)
 *              (with offsets fp8_mx_scale_bytes(P, C)); COL_MAJOR B * fp8_mx_scale_bytes(C, R)
 *              (with offsets fp8_mx_scale_bytes(C, P)); BOTH the row-major scales followed by
 *              the column-major ones.
 *  offsets     NULL, or int32 [E] cumulative segment ends (COL granularity, 2-D x only);
 *              E <= 2048.
 *              Checked on the device: a bad vector sets FP8_DEV_BAD_OFFSETS.
 *  workspace   device memory, 16-byte aligned, of fp8_workspace_size(FP8_OP_QUANTIZE, groups,
 *              C, rows, granularity) bytes: 8 bytes for tensor granularity (the amax word and a
 *              grid-barrier count); for column granularity 128 bytes (the 64 column maxima of a
 *              256-row x 64-column tile) per tile, (ceil(rows / 256) + groups) * ceil(C / 64)
 *              tiles, rows = all rows of x (B * R for 3-D x)
 *              (groups = B for 3-D x, E with offsets, else 1); 0 for row
 *              granularity (workspace may then be NULL). MX: 4 * (E + 1) bytes rounded up to
 *              16 with offsets (the padded segment starts), else 0. Calls sharing a workspace must be
 *              stream-ordered: the quantize clears and uses it.
 * Bit-exactness: codes and inverse scales equal the recipe evaluated with an fp64 division,
 * an fp32 multiply and a round-to-nearest-even saturating cast (eps = 1e-12).
 */
int fp8_quantize(const fp8_tensor* x, int granularity, int out_dtype, int layout, fp8_tensor* out,
                 fp8_tensor* out_t, fp8_tensor* inv_scales, const fp8_tensor* offsets,
                 void* workspace, size_t workspace_bytes, int32_t* d_status, void* stream);

/*
 * fp8_scaled_mm — out[m, n] = sA[m] * sB[n] * sum_k A[m, k] * B[n, k]   ([Q], [L]).
 *
 *  A    FP8 (e4m3 or e5m2) [M, K], K-major. Or BF16 [M, K] (or [K, M] with FP8_MM_A_MN_MAJOR).
 *  B    FP8 [N, K], K-major (the pages' column-major B). Or BF16 [N, K] (or [K, N] with
 *       FP8_MM_B_MN_MAJOR). FP8 operand pairs: e4m3 x e4m3, e5m2 x e4m3, e4m3 x e5m2.
 *  sA   fp32 [1] (tensorwise) or [M] (rowwise) inverse scales; NULL for BF16 operands.
 *  sB   fp32 [1] or [N]; NULL for BF16 operands.
 *  out  bf16 or fp32 [M, N]. Accumulation is fp32 in tensor memory; the dequantization
 *       sA[m] * sB[n] is applied once in the epilogue, followed by one rounding to out's type.
 *  K * element size must be a multiple of 16 bytes; M and N are arbitrary (>= 1). K == 0 (an
 *  empty contraction) writes out = 0 (every element an empty sum) with one cudaMemsetAsync.
 *  MX ([MX]): sA and sB of dtype FP8_DT_E8M0 select the block-scaled GEMM,
 *       out[m, n] = sum_k X_A[m, k/32] X_B[n, k/32] A[m, k] B[n, k], with A, B FP8 K-major,
 *       sA fp8_mx_scale_bytes(M, K) bytes and sB fp8_mx_scale_bytes(N, K) bytes in the MX scale
 *       layout, K % 128 == 0. The block scales are applied inside the tensor-core MMA
 *       (tcgen05.mma block_scale); the epilogue only rounds.
 */
int fp8_scaled_mm(const fp8_tensor* A, const fp8_tensor* B, const fp8_tensor* sA,
                  const fp8_tensor* sB, fp8_tensor* out, int flags, int32_t* d_status,
                  void* stream);

/*
 * fp8_grouped_mm — the MoE grouped GEMM of [G], one persistent launch; the offsets stay on the
 * device. offsets: int32 [E] cumulative segment ends (non-decreasing, last = total rows);
 * empty segments are allowed anywhere. The contraction must have at least one column: K >= 1
 * (JAGGED_M) and P >= 1 (JAGGED_K), else FP8_ERR_UNSUPPORTED.
 *
 * FP8_GROUPED_JAGGED_M (forward / grad-input):
 *   out[r, n] = sA[r] * sB[e, n] * sum_k A[r, k] * B[e, n, k]   for r in segment e.
 *   A FP8 [M, K]; B FP8 [E, N, K] (K-major per expert); sA fp32 [M]; sB fp32 [E, N];
 *   out bf16/fp32 [M, N]. Rows of empty experts do not exist; no other rows are touched.
 * FP8_GROUPED_JAGGED_K (per-expert weight gradient):
 *   out[e, n, k] = sA[e, n] * sB[e, k] * sum_{r in segment e} G[r, n] * X[r, k].
 *   A = G^T and B = X^T in the segment-padded column-major layout written by fp8_quantize
 *   (COL granularity with offsets): A FP8 [N, P], B FP8 [K, P]; sA fp32 [E, N]; sB fp32 [E, K];
 *   out bf16/fp32 [E, N, K]. An empty segment gives out[e] = 0.
 * MX ([MX]; sA, sB of dtype FP8_DT_E8M0, K % 128 == 0, scales in the MX scale layout):
 *   JAGGED_M: sA = the segment-padded row-major scales of A (fp8_quantize MX ROW_MAJOR with
 *   offsets; P = 32 * bytes / K rows, P % 128 == 0, P >= M + 127 E); sB = E * fp8_mx_scale_bytes(N,
 *   K) bytes. JAGGED_K: A = G^T [N, P] and B = X^T [K, P] from fp8_quantize MX COL_MAJOR with
 *   offsets; sA = fp8_mx_scale_bytes(N, P), sB = fp8_mx_scale_bytes(K, P) bytes.
 */
int fp8_grouped_mm(const fp8_tensor* A, const fp8_tensor* B, const fp8_tensor* offsets,
                   const fp8_tensor* sA, const fp8_tensor* sB, fp8_tensor* out, int mode,
                   int flags, int32_t* d_status, void* stream);

/*
 * fp8_scaled_mm_amax — fp8_scaled_mm with the amax reduction of the NEXT quantization as side
 * outputs of the epilogue ([T] Level 1: fewer kernels, no extra pass over HBM): row_amax[m] =
 * max_n |out[m, n]| and col_amax[n] = max_m |out[m, n]| of the result as stored (bf16), as fp32
 * values; col_amax may also be a single fp32 word, which then receives the maximum over the
 * whole output (the tensorwise amax). These are exactly the maxima fp8_quantize computes on
 * `out`, so fp8_quantize_from_amax then quantizes `out` from one read instead of two. out must
 * be bf16, M and N as fp8_scaled_mm (dense); FP8 (not MX) or BF16 operands. Either amax pointer
 * may be NULL. The call zeroes the amax buffers on its stream before the GEMM.
 */
int fp8_scaled_mm_amax(const fp8_tensor* A, const fp8_tensor* B, const fp8_tensor* sA,
                       const fp8_tensor* sB, fp8_tensor* out, int flags, fp8_tensor* row_amax,
                       fp8_tensor* col_amax, int32_t* d_status, void* stream);

/*
 * fp8_scaled_mm_quant — fp8_scaled_mm whose epilogue writes the NEXT quantization of its result
 * instead of the result itself ([T] Level 1: the quantize fused into the producing kernel, no bf16
 * round trip through HBM). The result out[m, n] = sA[m] sB[n] sum_k A[m, k] B[n, k] is rounded once
 * to bf16 (exactly what fp8_scaled_mm stores in a bf16 output), then quantized along its rows:
 *  out_granularity FP8_GRAN_BLOCK_1x128 ([B]): one scale per row and 128 columns by the recipe [Q];
 *                  out_scales fp32 [M, N / 128] inverse scales.
 *                  FP8_GRAN_MX ([MX]): blocks of 32 columns with E8M0 scales; out_scales E8M0
 *                  bytes fp8_mx_scale_bytes(M, N) in the MX scale layout (rows M, contraction N),
 *                  16-byte aligned.
 *  out_q           FP8 (E4M3 or E5M2) [M, N] row-major codes.
 *  A, B, sA, sB, flags as fp8_scaled_mm with FP8 operands and fp32 tensor / row scales
 *  (FP8_MM_FAST_ACCUM only). N % 128 == 0; K >= 1 (K == 0: FP8_ERR_UNSUPPORTED).
 * The codes and scales are bit-identical to fp8_scaled_mm with a bf16 output followed by
 * fp8_quantize (FP8_GRAN_BLOCK_1x128 or FP8_GRAN_MX, ROW_MAJOR) of that output. No workspace.
 */
int fp8_scaled_mm_quant(const fp8_tensor* A, const fp8_tensor* B, const fp8_tensor* sA,
                        const fp8_tensor* sB, int flags, int out_granularity, fp8_tensor* out_q,
                        fp8_tensor* out_scales, int32_t* d_status, void* stream);

/*
 * fp8_quantize_from_amax — the scale and cast steps of fp8_quantize ([Q] section 2) with the amax
 * step given: amax fp32 [1] (FP8_GRAN_TENSOR; ROW_MAJOR, COL_MAJOR or BOTH) or [C] (FP8_GRAN_COL,
 * COL_MAJOR), holding bf16 values (the maxima of a bf16 tensor always are). x bf16 [R, C]; the
 * outputs, inverse scales and their layouts as for fp8_quantize. When amax holds the true maxima
 * of x (e.g. from fp8_scaled_mm_amax) the results are bit-identical to fp8_quantize's, from one
 * read of x where fp8_quantize needs two. Row granularity: FP8_ERR_UNSUPPORTED (fp8_quantize
 * reads each row once already). No workspace.
 */
int fp8_quantize_from_amax(const fp8_tensor* x, int granularity, int out_dtype, int layout,
                           fp8_tensor* out, fp8_tensor* out_t, fp8_tensor* inv_scales,
                           const fp8_tensor* amax, int32_t* d_status, void* stream);

/* FP8 copies and inverse scales kept from the forward pass for the backward pass
 * ([Q] section 6: the autograd function saves the quantized tensors, not the bf16 inputs).
 * All buffers are caller-owned. */
typedef struct fp8_linear_saved {
  fp8_tensor x_q;    /* e4m3 [M, K] */
  fp8_tensor x_inv;  /* fp32 [1] (tensor) or [M] (row); MX: E8M0 fp8_mx_scale_bytes(M, K) */
  fp8_tensor w_q;    /* e4m3 [N, K] */
  fp8_tensor w_inv;  /* fp32 [1] or [N]; MX: E8M0 fp8_mx_scale_bytes(N, K) */
  fp8_tensor xt_q;   /* tensor and MX granularity: e4m3 [K, M], x column-major (FP8 weight
                        gradient); ptr may be NULL when the backward pass uses FP8_WGRAD_BF16 */
  fp8_tensor wt_q;   /* tensor and MX granularity: e4m3 [K, N], W column-major (grad-input) */
  fp8_tensor xt_inv; /* MX only: E8M0 fp8_mx_scale_bytes(K, M) (blocks of 32 along M) */
  fp8_tensor wt_inv; /* MX only: E8M0 fp8_mx_scale_bytes(K, N) (blocks of 32 along N) */
} fp8_linear_saved;

/*
 * fp8_linear_fwd — y = x W^T through FP8 ([Q], [L]): quantize x and W (e4m3; tensor, row, MX or
 * blockwise granularity), then one scaled GEMM. Blockwise (FP8_GRAN_BLOCK_1x128, [B]): x in 1 x 128
 * tiles (x_inv [M, K/128]), W in 128 x 128 tiles in both layouts (w_inv [N/128, K/128], wt_inv
 * [K/128, N/128]); K and N multiples of 128; the backward pass supports FP8_WGRAD_BF16 only. x bf16 [M, K], w bf16 [N, K], y bf16/fp32 [M, N].
 * Tensor and MX granularity write x and W in both layouts (dual output) so that the backward
 * pass needs no transpose copy. MX ([MX]) needs M, K and N multiples of 128.
 */
int fp8_linear_fwd(const fp8_tensor* x, const fp8_tensor* w, int granularity, int flags,
                   fp8_tensor* y, fp8_linear_saved* saved, void* workspace,
                   size_t workspace_bytes, int32_t* d_status, void* stream);

/*
 * fp8_linear_bwd — dX = dY W and dW = dY^T x ([L], [W]).
 *  dy      bf16 [M, N]; quantized to e5m2 ([F]).
 *  saved   from fp8_linear_fwd with the same granularity.
 *  x, w    the bf16 forward inputs. Row granularity needs w (W quantized per column over N for
 *          the grad-input GEMM). FP8_WGRAD_BF16 needs x; FP8_WGRAD_FP8 with row granularity
 *          needs x (quantized per column over M). MX uses the saved column-major copies and
 *          quantizes dY to MX e5m2 in both layouts from one read.
 *  dx      bf16/fp32 [M, K]; dw bf16/fp32 [N, K]. Either may be NULL to skip that GEMM.
 *  Both backward GEMMs run with full accumulation ([Q] section 5).
 */
int fp8_linear_bwd(const fp8_tensor* dy, const fp8_linear_saved* saved, const fp8_tensor* x,
                   const fp8_tensor* w, int granularity, int wgrad_mode, fp8_tensor* dx,
                   fp8_tensor* dw, void* workspace, size_t workspace_bytes, int32_t* d_status,
                   void* stream);

/* Test hook for failure detection: while enabled, every GEMM launch first waits on a barrier
 * that nothing signals, the grid barrier of the tensorwise quantize waits for one arrival more
 * than there are CTAs, the column-wise quantize sees no tile maxima as written, and the MX
 * quantize with a column-major output of a dense tensor loads no tile into its ring; the wait
 * runs out after the wait limit (fp8_set_wait_limit_ns), the kernel reports FP8_DEV_TIMEOUT,
 * drains and returns. Off by default. Returns the previous setting. */
int fp8_set_test_stall(int enable);

/* Test hook for the cast step ([Q] section 2: round to nearest even, saturating; [F] formats):
 * out[i] = the FP8 code (out_dtype E4M3 or E5M2) that the quantize kernels' cast gives the fp32
 * value whose bit pattern is first_bits + i, for 0 <= i < n (first_bits + n <= 2^32). out: n
 * bytes of device memory. Values beyond +-fp8_max saturate to it, as clamping first would give.
 * Asynchronous on `stream`. Returns FP8_OK, FP8_ERR_INVALID_ARG, FP8_ERR_DEVICE or FP8_ERR_CUDA. */
int fp8_test_cast_bits(uint32_t first_bits, int64_t n, int out_dtype, void* out, void* stream);

/*
 * fp8_quantize_tensor_noalloc — the tensorwise quantize of fp8_quantize (FP8_GRAN_TENSOR) for
 * callers that cannot allocate device memory. The pages have no counterpart: this entry point
 * exists for callers that hold no allocator and receive no workspace, such as plugin or callback
 * interfaces that hand the library only its input and output buffers, and runtimes that reserve
 * all device memory at start-up and forbid cudaMalloc afterwards (cudaMalloc may also
 * synchronize the device, which latency-bound callers avoid).
 *
 * Same arguments and results as fp8_quantize with FP8_GRAN_TENSOR, minus the workspace and the
 * status word: x bf16 [R, C] (2-D), out / out_t / inv_scale as there. The amax reduction uses a
 * fixed array in the library's own device memory instead of a workspace: one partial maximum per
 * 32768 input elements, FP8_NOALLOC_MAX_PARTIALS of them (about 64 KiB), allocated when the
 * library is loaded on a device and held by every device that loads it until the process exits.
 *  - x with more than FP8_NOALLOC_MAX_ELEMENTS elements is rejected with FP8_ERR_UNSUPPORTED
 *    before anything is launched.
 *  - The first call on each device looks up the array's device address (with that device
 *    current); make that first call before any stream capture.
 *  - Every call on a device shares the one array and leaves its last contents there; each call
 *    writes every slot it reads before reading it, so nothing needs clearing between calls. Calls
 *    that can run at the same time on the GPU (different streams without ordering between them)
 *    race on the array and give wrong scales: order them on one stream or with events.
 *  - Allocates nothing: no cudaMalloc / cudaFree and no allocating library routine.
 */
#define FP8_NOALLOC_MAX_PARTIALS 16384
#define FP8_NOALLOC_MAX_ELEMENTS (16384LL * 32768LL)
int fp8_quantize_tensor_noalloc(const fp8_tensor* x, int out_dtype, int layout, fp8_tensor* out,
                                fp8_tensor* out_t, fp8_tensor* inv_scale, void* stream);

/* Workspace bytes for an operation. FP8_OP_QUANTIZE: (d0, d1, d2) = (groups, columns, rows of x
 * over all groups) as described at fp8_quantize (d2 is used by column granularity only).
 * FP8_OP_LINEAR_FWD / FP8_OP_LINEAR_BWD: (d0, d1, d2) = (M, K, N). */
size_t fp8_workspace_size(int op, int64_t d0, int64_t d1, int64_t d2, int granularity,
                          int wgrad_mode);

/* Padded row count P for the segment-padded column-major layout (see fp8_quantize): the room
 * the segments need, rows + 127 * n_segments, rounded up to a multiple of 128 so that every row
 * of the [C, P] operand starts on a 128-byte line (the grouped GEMM's tile loads then read whole
 * L2 lines; a P that is only a multiple of 16 is accepted but makes each 128-byte row chunk
 * straddle two lines). Returns -1 for negative arguments. */
int64_t fp8_jagged_padded_rows(int64_t rows, int64_t n_segments);

/* Bytes of the MX scales of an operand with `rows` rows and contraction length k (see the MX
 * scale layout): ceil(rows / 128) * 128 * k / 32. Returns -1 unless rows >= 0 and k % 128 == 0. */
int64_t fp8_mx_scale_bytes(int64_t rows, int64_t k);

/* Text for an FP8_ERR_* return code or an FP8_DEV_* status word. */
const char* fp8_status_string(int code);

/* Upper bound, in nanoseconds, of every on-device wait (default 4e9). A wait that runs out
 * sets FP8_DEV_TIMEOUT and the kernel drains and returns. Tests lower it to exercise that
 * path without faulting the GPU. Returns the previous value. */
uint64_t fp8_set_wait_limit_ns(uint64_t ns);

#ifdef __cplusplus
}
#endif
#endif /* FP8LIN_H */
