// Host-side internals of fp8lin: launch context, tensor-map encoding and the kernel launchers
// that the C ABI (api.cu) composes.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/fp8lin.h"

namespace fp8lin {

struct Ctx {
  cudaStream_t stream;
  int32_t* status;   // device status word (may be null)
  uint64_t wait_ns;  // bound of every on-device wait
  int sm_count;
  int device;
  int test_stall;    // failure-detection test hook (see fp8_set_test_stall)
};

struct ScaleTab;
// The scale table of a format (FP8_DT_E4M3 / FP8_DT_E5M2), built once on the host in fp64.
const ScaleTab& scale_tab(int fmt);

// Fills ctx for the current device; returns FP8_OK or FP8_ERR_DEVICE.
int make_ctx(Ctx* ctx, void* stream, int32_t* status);

// 2-D / 3-D tiled tensor maps (row-major tensors; dims listed innermost first).
int make_tmap(CUtensorMap* map, const void* base, CUtensorMapDataType dt, int rank, const uint64_t* dims,
              const uint64_t* strides_bytes /* rank-1 entries */, const uint32_t* box, CUtensorMapSwizzle swz);

// --- quantize launchers (quantize.cu) ---
// Rowwise: x bf16 [R, C] -> q [R, C], inv [R].
int launch_quant_rows(const void* x, int64_t R, int64_t C, int fmt, void* q, float* inv, const Ctx& c);
// Blockwise 1 x 128 by the row kernel: x bf16 [R, C] -> q [R, C], inv [R, C / 128]; 512 <= C <= 16384,
// C % 128 == 0, else FP8_ERR_UNSUPPORTED (nothing launched).
int launch_quant_rows_blk128(const void* x, int64_t R, int64_t C, int fmt, void* q, float* inv, const Ctx& c);
// Tensorwise in one cooperative launch: amax of x [R, C] into ws[0], a grid barrier on ws[1] (both
// zeroed here), then the cast into q (row-major, may be null) and/or qt ([C, R], may be null); inv [1].
int launch_quant_tensor(const void* x, int64_t R, int64_t C, int fmt, void* q, void* qt, float* inv,
                        uint32_t* amax_ws, const Ctx& c);
// The same with up to 12 tiles of 128 x 64 per SM kept in shared memory between the two reads
// (tensor.cu); for shapes where tensor_stash_ok holds (the outputs can leave by TMA).
bool tensor_stash_ok(int64_t R, int64_t C, bool has_q, bool has_qt);
int launch_quant_tensor_stash(const void* x, int64_t R, int64_t C, int fmt, void* q, void* qt, float* inv,
                              uint32_t* amax_ws, const Ctx& c);
// Columnwise with column-major output. x viewed as [rows_total, C]. Groups of rows share one
// scale per column: either n_groups consecutive groups of group_rows rows (ends == null) or the
// segments given by ends[n_groups] (segment-padded output, padded row count ld_out).
// out_t row (g, c) starts at out_t + (g * C + c) * ld_out (dense) or out_t + c * ld_out + pstart_g
// (segments). inv [n_groups, C]. scratch: col_ws_words(n_groups, C, rows_total) words of device
// memory, 16-byte aligned (unused when the maxima are given).
// Workspace words (4 bytes each) a column quantize of `groups` x C scales over rows_total rows of
// input (all groups) needs.
int64_t col_ws_words(int64_t groups, int64_t C, int64_t rows_total);
// amax_given (optional): the column maxima as fp32 words [n_groups, C] (bf16 values); pass 1 is
// skipped and scratch is not used.
int launch_quant_cols(const void* x, int64_t rows_total, int64_t C, int64_t n_groups, int64_t group_rows,
                      const int32_t* ends, int fmt, void* out_t, int64_t ld_out, float* inv, uint32_t* scratch,
                      const Ctx& c, const uint32_t* amax_given = nullptr);

// --- MX quantize (mx.cu) ---
// Bytes of the E8M0 scales of an operand with `rows` rows and contraction length k (k % 128 == 0):
// [ceil(rows / 128)][k / 128][512]; -1 for bad arguments.
int64_t mx_scale_bytes(int64_t rows, int64_t k);
// x bf16 [batches, R, C] (C % 128 == 0). q: row-major codes (blocks along C) with scales sf; qt:
// column-major codes [batches, C, ld_t] (blocks along R; R % 128 == 0 unless segmented) with
// scales sft. Either output may be null. With ends (batches == 1): segments of rows, padded row
// space of ld_t rows (ld_t % 128 == 0) for sf's rows and qt's columns; pstart_ws: E + 1 words.
int launch_mx_quant(const void* x, int64_t batches, int64_t R, int64_t C, int fmt, void* q, void* sf, void* qt,
                    int64_t ld_t, void* sft, const int32_t* ends, int64_t E, int32_t* pstart_ws, const Ctx& c);

// --- blockwise quantize (blockwise.cu) ---
// x bf16 [R, C] (C % 128 == 0). tile128 false: 1 x 128 tiles, row-major codes q, inv [R, C/128].
// tile128 true: 128 x 128 tiles; q row-major and/or qt column-major [C, R] (R % 128 == 0);
// inv [ceil(R/128), C/128] (may be null when qt is given) and inv_t [C/128, R/128] (with qt).
int launch_blk_quant(const void* x, int64_t R, int64_t C, int fmt, bool tile128, void* q, void* qt, float* inv,
                     float* inv_t, const Ctx& c);

// --- GEMM launchers (gemm.cu) ---
struct GemmArgs {
  // operands
  const void* A;
  const void* B;
  int a_dtype, b_dtype;   // FP8_DT_*
  int a_mn, b_mn;         // BF16 only: operand stored MN-major
  const float* sA;        // [1] or [M] (dense), [M] (jagged M), [E, M-dim] (jagged K); null for BF16
  const float* sB;
  int64_t sA_len, sB_len; // dense: 1 or M / 1 or N
  void* out;
  int out_dtype;          // FP8_DT_BF16 / FP8_DT_F32
  int64_t M, N, K;        // dense problem; jagged M: M = total rows; jagged K: K = padded rows P
  // grouped
  int mode;               // -1 dense, FP8_GROUPED_JAGGED_M, FP8_GROUPED_JAGGED_K
  const int32_t* ends;
  int64_t E;
  int64_t k_dim;          // jagged K: the output's last dimension (X's columns)
  // MX (block-scaled) operands: E8M0 scales in [row blocks][K / 128][512 B] blocks
  int mx;
  const void* sfa;        // A's scales; rows: M, or the segment-padded row count (jagged M)
  const void* sfb;        // B's scales; rows: N (per expert for jagged M)
  int64_t sfa_rows;
  // side outputs (dense, bf16 out): max |out| per row / per column as fp32 words, or null
  uint32_t* row_amax;
  uint32_t* col_amax;
  int amax_whole;         // col_amax is one word: the maximum over the whole output
  int blockwise;          // FP8 operands with blockwise inverse scales: sA [M, K/128] (1 x 128 tiles),
                          // sB [ceil(N/128), K/128] (128 x 128 tiles); dense only
  // quantized output (dense FP8, N % 128 == 0): codes [M, N] in q_fmt and scales of the result's
  // bf16 rounding, 1 x 128 blocks (q_mx 0: fp32 inverse scales [M, N/128]) or MX blocks of 32
  // (q_mx 1: E8M0 bytes in the MX scale layout for rows M, contraction N); out is then unused
  void* q_out;
  void* q_scales;
  int q_mx;
  int q_fmt;
};
int launch_gemm(const GemmArgs& g, const Ctx& c);

}  // namespace fp8lin

namespace fp8lin {
// Cast phase of the tensorwise quantize alone: reads the bf16 pattern of amax at `amax_word`
// (already reduced) and writes q / qt / inv exactly as launch_quant_tensor does.
// amax_shift: 0 when amax_word holds a bf16 pattern, 16 when it holds the fp32 value.
// Test hook: out[i] = the kernels' cast (fmt) of the fp32 value with bit pattern first + i.
int launch_cast_bits(uint32_t first, int64_t n, int fmt, void* out, const Ctx& c);
int launch_quant_tensor_cast(const void* x, int64_t R, int64_t C, int fmt, void* q, void* qt, float* inv,
                             const uint32_t* amax_word, const Ctx& c, int amax_shift = 0);
}  // namespace fp8lin
