"""The amax step of a quantization fused into the GEMM that produces the tensor ("FP8 training on
AMD GPUs with TorchTitan and TorchAO", "Triton Kernel Optimization", Level 1: fewer kernels and no
intermediate pass over HBM; Level 2: the column-wise quantize from one read).

fp8_scaled_mm_amax writes max |out| per row / per column / over the whole output from its
epilogue; fp8_quantize_from_amax runs the scale and cast steps from given maxima. Checked:
  - the GEMM result against the oracle (as for fp8_scaled_mm);
  - the side outputs equal the maxima of the result as stored (a property of the output that
    holds at any size);
  - fp8_quantize_from_amax with maxima taken from the bf16 input by their plain definition
    (numpy max |x|) is bit-identical to the oracle's quantize;
  - the fused chain (GEMM with side output, then quantize from amax) against the oracle: on
    integer-valued operands with power-of-two scales the fp32 accumulation is exact, so the
    oracle's own GEMM rounded once to bf16 is the stored output, and the oracle's column-wise
    quantize of it fixes the chain's codes and scales; the chain also equals the unfused one
    (GEMM, then the two-pass fp8_quantize) bit for bit."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_util import bits, check_gemm, codes, f32_bits, upload_codes, upload_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp8():
    import moe_grouped_gemm_absmax_gb300 as m
    return m


def _absmax_rows_cols(t):
    a = t.float().abs()
    return a.amax(dim=1), a.amax(dim=0), a.amax()


@pytest.mark.parametrize("M,N,K", [(300, 520, 256), (4096, 2560, 512)])  # single CTAs; CTA pairs
def test_gemm_amax_side_outputs(fp8, M, N, K):
    x, w, _ = W.linear_inputs(M, K, N, seed=M, outliers=True)
    cx, ix = oracle.quantize_rows(bits(x), oracle.E4M3)
    cw, iw = oracle.quantize_rows(bits(w), oracle.E4M3)
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    ra = torch.full((M,), -1.0, device="cuda")
    ca = torch.full((N,), -1.0, device="cuda")
    whole = torch.full((1,), -1.0, device="cuda")
    A, B, sA, sB = upload_codes(cx, oracle.E4M3), upload_codes(cw, oracle.E4M3), upload_f32(ix), upload_f32(iw)
    fp8.fp8_scaled_mm_amax(A, B, sA, sB, out, row_amax=ra, col_amax=ca)
    out2 = torch.empty_like(out)
    fp8.fp8_scaled_mm_amax(A, B, sA, sB, out2, col_amax=whole)
    torch.cuda.synchronize()
    rows = np.unique(np.concatenate([np.random.default_rng(1).choice(M, min(M, 64), replace=False), [0, M - 1]]))
    ref, acc = oracle.gemm_fp8(cx, oracle.E4M3, cw, oracle.E4M3, ix, iw, rows=rows)
    check_gemm(out[torch.as_tensor(rows, device="cuda")], ref, acc, True)
    assert torch.equal(out, out2)
    r, c, t = _absmax_rows_cols(out)
    assert torch.equal(ra, r) and torch.equal(ca, c) and torch.equal(whole[0], t)


def test_gemm_amax_bf16_operands(fp8):
    """The bf16 weight-gradient GEMM (MN-major operands) with a column amax."""
    M, K, N = 512, 384, 640  # out [K, N] = a^T b, contraction over M
    a = W.normal_bf16((M, K), 1.0, 6).cuda()
    b = W.normal_bf16((M, N), 1e-3, 7).cuda()
    out = torch.empty((K, N), dtype=torch.bfloat16, device="cuda")
    ca = torch.empty((N,), device="cuda")
    fp8.fp8_scaled_mm_amax(a, b, None, None, out, fp8.MM_A_MN_MAJOR | fp8.MM_B_MN_MAJOR, col_amax=ca)
    torch.cuda.synchronize()
    ref, acc = oracle.gemm_bf16(bits(a.cpu()), bits(b.cpu()), a_trans=True, b_trans=True)
    check_gemm(out, ref, acc, True)
    assert torch.equal(ca, out.float().abs().amax(dim=0))


@pytest.mark.parametrize("R,C,fmt", [(512, 384, oracle.E5M2), (1024, 200, oracle.E4M3)])
def test_quantize_from_amax_matches_oracle(fp8, R, C, fmt):
    g = W.column_gain_bf16((R, C), 1e-3, -2, 2, seed=R)
    xb = bits(g)
    mag = np.abs((xb.astype(np.uint32) << 16).view(np.float32))  # |x| from the bf16 patterns
    col_amax = torch.from_numpy(mag.max(axis=0).astype(np.float32)).cuda()
    tens_amax = torch.from_numpy(np.array([mag.max()], np.float32)).cuda()
    dt = 3 if fmt == oracle.E4M3 else 4
    fdt = torch.float8_e4m3fn if fmt == oracle.E4M3 else torch.float8_e5m2
    x = g.cuda()
    qt = torch.empty((C, R), dtype=fdt, device="cuda")
    inv = torch.empty(C, device="cuda")
    fp8.fp8_quantize_from_amax(x, fp8.GRAN_COL, dt, fp8.LAYOUT_COL_MAJOR, None, qt, inv, col_amax)
    q2 = torch.empty((R, C), dtype=fdt, device="cuda")
    qt2 = torch.empty((C, R), dtype=fdt, device="cuda")
    inv2 = torch.empty(1, device="cuda")
    fp8.fp8_quantize_from_amax(x, fp8.GRAN_TENSOR, dt, fp8.LAYOUT_BOTH, q2, qt2, inv2, tens_amax)
    torch.cuda.synchronize()
    qo, io = oracle.quantize_cols(xb, fmt)
    assert np.array_equal(codes(qt), qo.T) and np.array_equal(f32_bits(inv), io.view(np.uint32))
    qo, io = oracle.quantize_tensor(xb, fmt)
    assert np.array_equal(codes(q2), qo) and np.array_equal(codes(qt2), qo.T)
    assert np.array_equal(f32_bits(inv2), io.view(np.uint32))


def _exact_operands(M, N, K, seed):
    """FP8 operands whose products and sums are exact in fp32: integer values in [-8, 8] (exact in
    e5m2 and e4m3), per-row / per-column inverse scales that are powers of two, K * 64 < 2^24."""
    rng = np.random.default_rng(seed)
    a = rng.integers(-8, 9, size=(M, K)).astype(np.float32)
    b = rng.integers(-8, 9, size=(N, K)).astype(np.float32)
    sa = (2.0 ** rng.integers(-6, 3, size=M)).astype(np.float32)
    sb = (2.0 ** rng.integers(-6, 3, size=N)).astype(np.float32)
    return oracle.encode(a, oracle.E5M2), oracle.encode(b, oracle.E4M3), sa, sb


def test_fused_chain_matches_oracle(fp8):
    """The grad-input GEMM dX = dY W (e5m2 x e4m3, rowwise scales) with its column amax, then dX
    quantized column-wise (e5m2, column-major) from those maxima: the stored dX, the maxima, the
    codes and the inverse scales against the oracle; the chain against the unfused one."""
    M, N, K = 1024, 768, 512  # dX [M, N], contraction K
    ca, cb, sa, sb = _exact_operands(M, N, K, 9)
    ref, _ = oracle.gemm_fp8(ca, oracle.E5M2, cb, oracle.E4M3, sa, sb)
    ref_bf16 = torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16)  # exact -> one RNE rounding
    rb = bits(ref_bf16)
    qo, io = oracle.quantize_cols(rb, oracle.E5M2)
    dx = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    col = torch.empty(N, device="cuda")
    fp8.fp8_scaled_mm_amax(upload_codes(ca, oracle.E5M2), upload_codes(cb, oracle.E4M3), upload_f32(sa),
                           upload_f32(sb), dx, 0, col_amax=col)
    qt = torch.empty((N, M), dtype=torch.float8_e5m2, device="cuda")
    inv = torch.empty(N, device="cuda")
    fp8.fp8_quantize_from_amax(dx, fp8.GRAN_COL, fp8.DT_E5M2, fp8.LAYOUT_COL_MAJOR, None, qt, inv, col)
    _, qt_ref, inv_ref = fp8.quantize_alloc(dx, fp8.GRAN_COL, fp8.DT_E5M2)
    torch.cuda.synchronize()
    assert np.array_equal(bits(dx.cpu()), rb)
    assert np.array_equal(col.cpu().numpy(), ref_bf16.float().abs().amax(dim=0).numpy())
    assert np.array_equal(codes(qt), qo.T) and np.array_equal(f32_bits(inv), io.view(np.uint32))
    assert torch.equal(qt.view(torch.uint8), qt_ref.view(torch.uint8)) and torch.equal(inv, inv_ref)


def test_rejects(fp8):
    a = torch.zeros((128, 128), dtype=torch.float8_e4m3fn, device="cuda")
    s = torch.ones(1, device="cuda")
    out32 = torch.empty((128, 128), device="cuda")
    with pytest.raises(fp8.Fp8Error):  # side outputs need a bf16 result
        fp8.fp8_scaled_mm_amax(a, a, s, s, out32, col_amax=torch.empty(128, device="cuda"))
    x = torch.zeros((128, 128), dtype=torch.bfloat16, device="cuda")
    with pytest.raises(fp8.Fp8Error):  # row granularity is one read already
        fp8.fp8_quantize_from_amax(x, fp8.GRAN_ROW, 3, fp8.LAYOUT_ROW_MAJOR,
                                   torch.empty((128, 128), dtype=torch.float8_e4m3fn, device="cuda"), None,
                                   torch.empty(128, device="cuda"), torch.empty(128, device="cuda"))
