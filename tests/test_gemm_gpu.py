"""GPU parity of the tcgen05 scaled GEMMs against the fp64 oracle.

Bar: |gpu - oracle| <= tol * sum_k |sA a_k sB b_k| per element, tol = 2e-3 (full accumulation)
or 1e-2 (fast_accum), plus, for a bf16 output, the output rounding itself (half an ulp of bf16,
<= 2^-8 |oracle|). Contract: "FP8 Training: Quantization, Autograd, Torchao", sections 2, 4, 5."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_util import bits, check_gemm, upload_codes, upload_f32

pytestmark = pytest.mark.gpu
TOL = 2e-3


@pytest.fixture(scope="module")
def fp8():
    import moe_grouped_gemm_absmax_gb300 as m
    return m


def check(got, ref, absacc, out_bf16, tol=TOL):
    check_gemm(got, ref, absacc, out_bf16, tol)


def qrows(x, fmt):
    """Oracle rowwise quantization; returns host codes/scales and their device copies."""
    c, inv = oracle.quantize_rows(bits(x), fmt)
    return c, inv, upload_codes(c, fmt), upload_f32(inv)


# (1024, 4864, 256) and (1300, 4700, 160) have enough 256 x 256 tiles to run on CTA pairs
@pytest.mark.parametrize("M,N,K", [(128, 256, 128), (300, 520, 272), (1, 1, 16), (129, 257, 4096), (1000, 2000, 512),
                                   (1024, 4864, 256), (1300, 4700, 160)])
@pytest.mark.parametrize("types", [("e4m3", "e4m3"), ("e5m2", "e4m3"), ("e4m3", "e5m2")])
@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
def test_dense_rowwise(fp8, M, N, K, types, out_dtype):
    fa = oracle.E4M3 if types[0] == "e4m3" else oracle.E5M2
    fb = oracle.E4M3 if types[1] == "e4m3" else oracle.E5M2
    x = W.normal_bf16((M, K), 1.0, M + K)
    w = W.normal_bf16((N, K), 0.02, N + K)
    ca, ia, qa, sa = qrows(x, fa)
    cb, ib, qb, sb = qrows(w, fb)
    out = torch.empty((M, N), dtype=out_dtype, device="cuda")
    fp8.fp8_scaled_mm(qa, qb, sa, sb, out)
    torch.cuda.synchronize()
    ref, absacc = oracle.gemm_fp8(ca, fa, cb, fb, ia, ib)
    check(out, ref, absacc, out_dtype == torch.bfloat16)


def test_dense_tensorwise_and_fast_accum(fp8):
    M, N, K = 256, 256, 512
    x = W.normal_bf16((M, K), 1.0, 1)
    w = W.normal_bf16((N, K), 0.02, 2)
    ca, ia = oracle.quantize_tensor(bits(x), oracle.E4M3)
    cb, ib = oracle.quantize_tensor(bits(w), oracle.E4M3)
    qa, sa, qb, sb = upload_codes(ca, 0), upload_f32(ia), upload_codes(cb, 0), upload_f32(ib)
    ref, absacc = oracle.gemm_fp8(ca, oracle.E4M3, cb, oracle.E4M3, ia, ib)
    for flags, tol in ((0, TOL), (fp8.MM_FAST_ACCUM, 1e-2)):
        out = torch.empty((M, N), dtype=torch.float32, device="cuda")
        fp8.fp8_scaled_mm(qa, qb, sa, sb, out, flags)
        torch.cuda.synchronize()
        check(out, ref, absacc, False, tol)


def test_dense_large_sampled_rows(fp8):
    """A multi-wave problem (more tiles than SMs): every row of four 128-row tiles and a sample."""
    M, N, K = 2048, 4096, 2048
    x = W.normal_bf16((M, K), 1.0, 11)
    w = W.normal_bf16((N, K), 0.02, 12)
    ca, ia, qa, sa = qrows(x, oracle.E4M3)
    cb, ib, qb, sb = qrows(w, oracle.E4M3)
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    fp8.fp8_scaled_mm(qa, qb, sa, sb, out)
    torch.cuda.synchronize()
    rows = np.concatenate([np.arange(0, 128), np.arange(1920, 2048), np.random.default_rng(0).choice(M, 64, replace=False)])
    ref, absacc = oracle.gemm_fp8(ca, oracle.E4M3, cb, oracle.E4M3, ia, ib, rows=rows)
    check(out[torch.from_numpy(rows).cuda()], ref, absacc, True)


@pytest.mark.parametrize("a_mn,b_mn", [(0, 0), (1, 0), (0, 1), (1, 1)])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (200, 296, 136), (512, 768, 1024), (1032, 4864, 192)])
def test_bf16(fp8, a_mn, b_mn, M, N, K):
    a = W.normal_bf16((M, K), 1.0, 21 + M)
    b = W.normal_bf16((N, K), 1.0, 22 + N)
    A = a.T.contiguous() if a_mn else a
    B = b.T.contiguous() if b_mn else b
    flags = (fp8.MM_A_MN_MAJOR if a_mn else 0) | (fp8.MM_B_MN_MAJOR if b_mn else 0)
    out = torch.empty((M, N), dtype=torch.float32, device="cuda")
    fp8.fp8_scaled_mm(A.cuda(), B.cuda(), None, None, out, flags)
    torch.cuda.synchronize()
    ref, absacc = oracle.gemm_bf16(bits(a), bits(b))
    check(out, ref, absacc, False)
