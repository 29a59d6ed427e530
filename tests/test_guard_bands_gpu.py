"""Guard bands around outputs: every output buffer below sits between two 4 KiB sentinel regions
of one allocation, and after the call both regions must be unchanged (no write past either end
of an output), while the output itself matches the oracle as in the parity tests. Shapes are
ragged (rows and columns that are not multiples of the tiles), on single CTAs and CTA pairs.
Contracts: "FP8 Training: Quantization, Autograd, Torchao", sections 2 and 4; "FP8 training on AMD
GPUs with TorchTitan and TorchAO", "Scaling FP8 to MoE Architectures" and Figure 3."""
import math

import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_util import bits, check_gemm, codes, f32_bits, segpad_cols, upload_codes, upload_f32

pytestmark = pytest.mark.gpu
GUARD = 4096
SENTINEL = 0xA5


@pytest.fixture(scope="module")
def fp8():
    import moe_grouped_gemm_absmax_gb300 as m
    return m


class Guarded:
    """An output tensor of `shape` / `dtype` inside one byte buffer with GUARD sentinel bytes on
    each side."""

    def __init__(self, shape, dtype):
        self.nbytes = math.prod(shape) * torch.empty(0, dtype=dtype).element_size()
        self.buf = torch.full((GUARD + self.nbytes + GUARD,), SENTINEL, dtype=torch.uint8, device="cuda")
        self.t = self.buf[GUARD:GUARD + self.nbytes].view(dtype).view(shape)

    def intact(self):
        b = self.buf.cpu().numpy()
        return bool((b[:GUARD] == SENTINEL).all() and (b[GUARD + self.nbytes:] == SENTINEL).all())


def qrows(x, fmt):
    c, inv = oracle.quantize_rows(bits(x), fmt)
    return c, inv, upload_codes(c, fmt), upload_f32(inv)


@pytest.mark.parametrize("M,N,K,out_dtype", [(300, 520, 272, torch.float32), (300, 520, 272, torch.bfloat16),
                                             (1300, 4700, 160, torch.bfloat16), (1024, 4864, 256, torch.float32),
                                             (1, 1, 16, torch.bfloat16)])
def test_dense_gemm(fp8, M, N, K, out_dtype):
    x = W.normal_bf16((M, K), 1.0, M + 3)
    w = W.normal_bf16((N, K), 0.02, N + 5)
    ca, ia, qa, sa = qrows(x, oracle.E4M3)
    cb, ib, qb, sb = qrows(w, oracle.E4M3)
    out = Guarded((M, N), out_dtype)
    fp8.fp8_scaled_mm(qa, qb, sa, sb, out.t)
    torch.cuda.synchronize()
    assert out.intact()
    rows = np.unique(np.concatenate([[0, M - 1], np.random.default_rng(2).choice(M, min(M, 96), replace=False)]))
    ref, acc = oracle.gemm_fp8(ca, oracle.E4M3, cb, oracle.E4M3, ia, ib, rows=rows)
    check_gemm(out.t[torch.as_tensor(rows, device="cuda")], ref, acc, out_dtype == torch.bfloat16)


def test_bf16_gemm_mn_major(fp8):
    """The bf16 weight-gradient layout (both operands MN-major) on CTA pairs, ragged N."""
    M, N, K = 1032, 4856, 192
    a = W.normal_bf16((M, K), 1.0, 31)
    b = W.normal_bf16((N, K), 1.0, 32)
    out = Guarded((M, N), torch.bfloat16)
    fp8.fp8_scaled_mm(a.T.contiguous().cuda(), b.T.contiguous().cuda(), None, None, out.t,
                      fp8.MM_A_MN_MAJOR | fp8.MM_B_MN_MAJOR)
    torch.cuda.synchronize()
    assert out.intact()
    rows = np.unique(np.concatenate([[0, M - 1], np.random.default_rng(3).choice(M, 64, replace=False)]))
    ref, acc = oracle.gemm_bf16(bits(a), bits(b), rows=rows)
    check_gemm(out.t[torch.as_tensor(rows, device="cuda")], ref, acc, True)


@pytest.mark.parametrize("counts,N,K,out_dtype", [([100, 0, 37, 300, 1], 300, 256, torch.float32),
                                                  ([0, 2100, 3, 0, 33], 1040, 512, torch.bfloat16)])
def test_grouped_jagged_m(fp8, counts, N, K, out_dtype):
    E, M = len(counts), sum(counts)
    A = W.normal_bf16((M, K), 1.0, 41)
    Wt = W.normal_bf16((E, N, K), 0.02, 42)
    ca, ia = oracle.quantize_rows(bits(A), oracle.E4M3)
    cw, iw = oracle.quantize_rows(bits(Wt).reshape(E * N, K), oracle.E4M3)
    ends = W.ends_from_counts(counts)
    out = Guarded((M, N), out_dtype)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp8.fp8_grouped_mm(upload_codes(ca, oracle.E4M3), upload_codes(cw.reshape(E, N, K), oracle.E4M3),
                       torch.from_numpy(ends).cuda(), upload_f32(ia), upload_f32(iw.reshape(E, N)), out.t,
                       fp8.GROUPED_JAGGED_M, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and out.intact()
    ref, acc = oracle.grouped_gemm_m(ca, oracle.E4M3, cw.reshape(E, N, K), oracle.E4M3, ia, iw.reshape(E, N), ends)
    check_gemm(out.t, ref, acc, out_dtype == torch.bfloat16)


@pytest.mark.parametrize("counts,N,Kd,out_dtype", [([100, 0, 300, 37], 72, 200, torch.float32),
                                                   ([300, 0, 260, 90], 520, 2560, torch.bfloat16)])
def test_grouped_jagged_k(fp8, counts, N, Kd, out_dtype):
    E, M = len(counts), sum(counts)
    G = W.normal_bf16((M, N), 1e-3, 43)
    X = W.normal_bf16((M, Kd), 1.0, 44)
    ends = W.ends_from_counts(counts)
    cg, sg = oracle.quantize_jagged_cols(bits(G), ends, oracle.E5M2)
    cx, sx = oracle.quantize_jagged_cols(bits(X), ends, oracle.E4M3)
    P = fp8.fp8_jagged_padded_rows(M, E)
    out = Guarded((E, N, Kd), out_dtype)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp8.fp8_grouped_mm(upload_codes(segpad_cols(cg, ends, P), oracle.E5M2),
                       upload_codes(segpad_cols(cx, ends, P), oracle.E4M3), torch.from_numpy(ends).cuda(),
                       upload_f32(sg), upload_f32(sx), out.t, fp8.GROUPED_JAGGED_K, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and out.intact()
    ref, acc = oracle.grouped_gemm_k(cg, oracle.E5M2, cx, oracle.E4M3, sg, sx, ends)
    check_gemm(out.t, ref, acc, out_dtype == torch.bfloat16)


@pytest.mark.parametrize("R,C", [(300, 520), (17, 8), (5, 16392), (129, 4096)])
def test_quantize_rows(fp8, R, C):
    x = W.outlier_channels_bf16((R, C), 1.0, 0.01, 50.0, R + C)
    q = Guarded((R, C), torch.float8_e4m3fn)
    inv = Guarded((R,), torch.float32)
    fp8.fp8_quantize(x.cuda(), fp8.GRAN_ROW, fp8.DT_E4M3, fp8.LAYOUT_ROW_MAJOR, q.t, None, inv.t)
    torch.cuda.synchronize()
    assert q.intact() and inv.intact()
    qo, io = oracle.quantize_rows(bits(x), oracle.E4M3)
    assert np.array_equal(codes(q.t), qo) and np.array_equal(f32_bits(inv.t), io.view(np.uint32))


@pytest.mark.parametrize("R,C", [(272, 200), (16, 8), (1040, 4104)])
def test_quantize_tensor_dual(fp8, R, C):
    x = W.normal_bf16((R, C), 1.0, R * 3 + C)
    q = Guarded((R, C), torch.float8_e5m2)
    qt = Guarded((C, R), torch.float8_e5m2)
    inv = Guarded((1,), torch.float32)
    ws = torch.empty(4, dtype=torch.int32, device="cuda")
    fp8.fp8_quantize(x.cuda(), fp8.GRAN_TENSOR, fp8.DT_E5M2, fp8.LAYOUT_BOTH, q.t, qt.t, inv.t, None, ws)
    torch.cuda.synchronize()
    assert q.intact() and qt.intact() and inv.intact()
    qo, io = oracle.quantize_tensor(bits(x), oracle.E5M2)
    assert np.array_equal(codes(q.t), qo) and np.array_equal(codes(qt.t), qo.T)
    assert np.array_equal(f32_bits(inv.t), io.view(np.uint32))


@pytest.mark.parametrize("R,C", [(272, 200), (528, 4104)])
def test_quantize_cols(fp8, R, C):
    x = W.column_gain_bf16((R, C), 1e-3, -2, 2, seed=R + C)
    qt = Guarded((C, R), torch.float8_e4m3fn)
    inv = Guarded((C,), torch.float32)
    fp8.fp8_quantize(x.cuda(), fp8.GRAN_COL, fp8.DT_E4M3, fp8.LAYOUT_COL_MAJOR, None, qt.t, inv.t, None,
                     fp8.col_workspace(1, C, R, "cuda"))
    torch.cuda.synchronize()
    assert qt.intact() and inv.intact()
    qo, io = oracle.quantize_cols(bits(x), oracle.E4M3)
    assert np.array_equal(codes(qt.t), qo.T) and np.array_equal(f32_bits(inv.t), io.view(np.uint32))


def test_quantize_jagged_cols(fp8):
    counts = [100, 0, 300, 37, 129]
    E, M, C = len(counts), sum(counts), 200
    x = W.normal_bf16((M, C), 1e-3, 47)
    ends = W.ends_from_counts(counts)
    P = fp8.fp8_jagged_padded_rows(M, E)
    qt = Guarded((C, P), torch.float8_e5m2)
    inv = Guarded((E, C), torch.float32)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp8.fp8_quantize(x.cuda(), fp8.GRAN_COL, fp8.DT_E5M2, fp8.LAYOUT_COL_MAJOR, None, qt.t, inv.t,
                     torch.from_numpy(ends).cuda(), fp8.col_workspace(E, C, M, "cuda"), status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0 and qt.intact() and inv.intact()
    qo, io = oracle.quantize_jagged_cols(bits(x), ends, oracle.E5M2)
    got = codes(qt.t)
    want = segpad_cols(qo, ends, P)
    # the padding between segments is part of the layout (zero codes); columns past the last
    # segment's padded end are not written by the kernel
    used = sum(-(-c // 128) * 128 for c in counts)
    assert np.array_equal(got[:, :used], want[:, :used])
    assert np.array_equal(f32_bits(inv.t), io.view(np.uint32))
