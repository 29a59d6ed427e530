"""GPU parity of the MoE grouped FP8 GEMM (one persistent launch; offsets stay on the device)
against the fp64 oracle. Contract: "FP8 training on AMD GPUs with TorchTitan and TorchAO",
"Scaling FP8 to MoE Architectures" and Figure 3 (per-row activation scales, per-expert-column
weight scales, offsets routing rows to experts)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_util import bits, check_gemm, segpad_cols, upload_codes, upload_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp8():
    import moe_grouped_gemm_absmax_gb300 as m
    return m


def _jagged_m_case(fp8, counts, N, K, out_dtype=torch.float32, seed=0, fa=oracle.E4M3):
    counts = [int(c) for c in counts]
    E, M = len(counts), sum(counts)
    A = W.normal_bf16((M, K), 1.0, seed)
    Wt = W.normal_bf16((E, N, K), 0.02, seed + 1)
    ca, ia = oracle.quantize_rows(bits(A), fa)
    cw, iw = oracle.quantize_rows(bits(Wt).reshape(E * N, K), oracle.E4M3)
    cw, iw = cw.reshape(E, N, K), iw.reshape(E, N)
    ends = W.ends_from_counts(counts)
    out = torch.full((M, N), float("nan"), dtype=out_dtype, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp8.fp8_grouped_mm(upload_codes(ca, fa), upload_codes(cw, oracle.E4M3), torch.from_numpy(ends).cuda(),
                       upload_f32(ia), upload_f32(iw), out, fp8.GROUPED_JAGGED_M, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return out, (ca, fa, cw, ia, iw, ends)


@pytest.mark.parametrize("counts,N,K", [
    ([100, 0, 37, 300, 1], 300, 256),
    ([0, 0, 64], 256, 128),
    ([128, 128], 512, 384),
    ([0, 5, 0, 250, 0], 72, 64),
    ([1], 16, 16),
])
def test_jagged_m(fp8, counts, N, K):
    out, (ca, fa, cw, ia, iw, ends) = _jagged_m_case(fp8, counts, N, K)
    ref, absacc = oracle.grouped_gemm_m(ca, fa, cw, oracle.E4M3, ia, iw, ends)
    check_gemm(out, ref, absacc, False)


@pytest.mark.parametrize("counts,N,K,out_dtype,fa", [
    ([1, 15, 16, 17, 0, 255, 256, 257, 1200, 300], 300, 256, torch.float32, oracle.E4M3),
    ([0, 2100, 3, 0, 33], 1040, 512, torch.bfloat16, oracle.E5M2),
    ([513, 511, 1024, 0], 264, 128, torch.bfloat16, oracle.E4M3),
    ([64, 65, 100, 128, 129, 200, 240, 241, 31, 32, 48, 49, 1000], 520, 256, torch.bfloat16, oracle.E4M3),
    ([1000, 49, 48, 32, 31, 241, 240, 200, 129, 128, 100, 65, 64], 136, 384, torch.float32, oracle.E5M2),
])
def test_jagged_m_pairs(fp8, counts, N, K, out_dtype, fa):
    """At least 2048 rows: CTA pairs with 256-row tiles that start at each expert's first row:
    experts with 1, 15, 16, 17 tokens, 255-257, empty experts, N not a multiple of 256, e4m3 and
    e5m2 activations, fp32 and bf16 outputs. An expert's last tile with fewer than 256 rows runs
    transposed with row boxes of 32, 64 or 128 per CTA (tails up to 64, 128, 255 rows): the last
    two cases put tails on both sides of each boundary (64/65, 128/129), at 31/32, 48/49 and
    240/241."""
    out, (ca, fa_, cw, ia, iw, ends) = _jagged_m_case(fp8, counts, N, K, out_dtype, seed=9, fa=fa)
    ref, absacc = oracle.grouped_gemm_m(ca, fa_, cw, oracle.E4M3, ia, iw, ends)
    check_gemm(out, ref, absacc, out_dtype == torch.bfloat16)


def test_jagged_m_zipf_bf16(fp8):
    """DeepSeek-V3-style routing at reduced size: 64 experts, Zipf(1.1) counts with forced-empty
    experts (first and last included), bf16 output, e5m2 activations x e4m3 weights."""
    counts = W.zipf_counts(4096, 64, 1.1, 4, 3, empty_first=True, empty_last=True)
    out, (ca, fa, cw, ia, iw, ends) = _jagged_m_case(fp8, counts, 384, 512, torch.bfloat16, seed=5, fa=oracle.E5M2)
    rows = np.unique(np.concatenate([np.random.default_rng(1).choice(4096, 256, replace=False),
                                     ends[ends > 0] - 1, np.concatenate([[0], ends[:-1]])[np.diff(np.concatenate([[0], ends])) > 0]]))
    ref, absacc = oracle.grouped_gemm_m(ca, fa, cw, oracle.E4M3, ia, iw, ends, rows=rows)
    check_gemm(out[torch.from_numpy(rows).cuda()], ref, absacc, True)


def test_jagged_m_single_expert_equals_dense(fp8):
    M, N, K = 300, 260, 192
    out, (ca, fa, cw, ia, iw, ends) = _jagged_m_case(fp8, [M], N, K)
    dense = torch.empty((M, N), dtype=torch.float32, device="cuda")
    fp8.fp8_scaled_mm(upload_codes(ca, fa), upload_codes(cw[0], oracle.E4M3), upload_f32(ia), upload_f32(iw[0]), dense)
    torch.cuda.synchronize()
    ref, absacc = oracle.gemm_fp8(ca, fa, cw[0], oracle.E4M3, ia, iw[0])
    check_gemm(out, ref, absacc, False)
    check_gemm(dense, ref, absacc, False)


# the last case has enough 256 x 256 tiles per expert set to run on CTA pairs
@pytest.mark.parametrize("counts,N,Kd", [([100, 0, 300, 37], 72, 200), ([0, 0, 130], 256, 256), ([500], 128, 64),
                                         ([1, 127, 128, 129, 0], 40, 24), ([300, 0, 260, 90], 520, 2560)])
@pytest.mark.parametrize("pitch16", [False, True])
def test_jagged_k(fp8, counts, N, Kd, pitch16):
    """pitch16: the padded operands' row pitch is a multiple of 16 but not of 128 bytes."""
    counts = [int(c) for c in counts]
    E, M = len(counts), sum(counts)
    G = W.normal_bf16((M, N), 1e-3, 7)
    X = W.normal_bf16((M, Kd), 1.0, 8)
    ends = W.ends_from_counts(counts)
    cg, sg = oracle.quantize_jagged_cols(bits(G), ends, oracle.E5M2)
    cx, sx = oracle.quantize_jagged_cols(bits(X), ends, oracle.E4M3)
    P = fp8.fp8_jagged_padded_rows(M, E)
    if pitch16:
        P = W.ceil_div(M + 127 * E, 16) * 16
        P += 16 if P % 128 == 0 else 0
    out = torch.full((E, N, Kd), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp8.fp8_grouped_mm(upload_codes(segpad_cols(cg, ends, P), oracle.E5M2), upload_codes(segpad_cols(cx, ends, P), oracle.E4M3),
                       torch.from_numpy(ends).cuda(), upload_f32(sg), upload_f32(sx), out, fp8.GROUPED_JAGGED_K,
                       status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    ref, absacc = oracle.grouped_gemm_k(cg, oracle.E5M2, cx, oracle.E4M3, sg, sx, ends)
    check_gemm(out, ref, absacc, False)


def test_grouped_bad_offsets(fp8):
    A = torch.zeros((64, 32), dtype=torch.float8_e4m3fn, device="cuda")
    B = torch.zeros((2, 16, 32), dtype=torch.float8_e4m3fn, device="cuda")
    sA = torch.ones(64, device="cuda")
    sB = torch.ones((2, 16), device="cuda")
    out = torch.zeros((64, 16), device="cuda")
    for bad in ([40, 30], [10, 63]):
        st = torch.zeros(1, dtype=torch.int32, device="cuda")
        fp8.fp8_grouped_mm(A, B, torch.tensor(bad, dtype=torch.int32, device="cuda"), sA, sB, out,
                           fp8.GROUPED_JAGGED_M, status=st)
        torch.cuda.synchronize()
        assert int(st.item()) == fp8.DEV_BAD_OFFSETS
