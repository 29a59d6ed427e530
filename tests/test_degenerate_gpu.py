"""Degenerate sizes at the C ABI.

- An empty contraction (K = 0) is an empty sum. The dense scaled GEMMs write it as +0 in every
  output element, as the oracle's GEMM gives it, and fold it into zero side-output maxima.
- The grouped GEMMs and the fused quantized output do not implement an empty contraction. They
  reject it with FP8_ERR_UNSUPPORTED, MX scales included; these checks come before any arithmetic
  on the sizes.
- An MX quantize of a tensor with no columns writes nothing.

Definition: "FP8 Training: Quantization, Autograd, Torchao", section 4 (the scaled GEMM,
out = sA sB sum_k a b)."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import check_gemm

pytestmark = pytest.mark.gpu
E4, E5 = torch.float8_e4m3fn, torch.float8_e5m2


@pytest.fixture(scope="module")
def fp8():
    import moe_grouped_gemm_absmax_gb300 as m
    return m


def _all_plus_zero(t):
    return int(t.contiguous().view(torch.uint8).count_nonzero()) == 0


@pytest.mark.parametrize("out_dtype", [torch.float32, torch.bfloat16])
@pytest.mark.parametrize("rowwise", [False, True])
def test_empty_contraction_fp8(fp8, out_dtype, rowwise):
    M, N = 300, 520
    A = torch.empty((M, 0), dtype=E4, device="cuda")
    B = torch.empty((N, 0), dtype=E5, device="cuda")
    sA = torch.full((M if rowwise else 1,), 0.5, device="cuda")
    sB = torch.full((N if rowwise else 1,), 3.0, device="cuda")
    out = torch.full((M, N), float("nan"), dtype=out_dtype, device="cuda")
    fp8.fp8_scaled_mm(A, B, sA, sB, out)
    torch.cuda.synchronize()
    ref, absacc = oracle.gemm_fp8(np.zeros((M, 0), np.uint8), oracle.E4M3, np.zeros((N, 0), np.uint8), oracle.E5M2,
                                  sA.cpu().numpy(), sB.cpu().numpy())
    assert not ref.any() and not absacc.any()
    check_gemm(out, ref, absacc, out_dtype == torch.bfloat16)
    assert _all_plus_zero(out)


@pytest.mark.parametrize("kind", ["blockwise", "mx"])
def test_empty_contraction_block_scaled(fp8, kind):
    M, N = 200, 300
    A = torch.empty((M, 0), dtype=E4, device="cuda")
    B = torch.empty((N, 0), dtype=E4, device="cuda")
    if kind == "blockwise":
        sA = torch.empty((M, 0), device="cuda")
        sB = torch.empty(((N + 127) // 128, 0), device="cuda")
        flags = fp8.MM_BLOCKWISE
    else:  # E8M0 scale bytes: fp8_mx_scale_bytes(M, 0) = 0
        sA = torch.empty(0, dtype=torch.uint8, device="cuda")
        sB = torch.empty(0, dtype=torch.uint8, device="cuda")
        flags = 0
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    fp8.fp8_scaled_mm(A, B, sA, sB, out, flags)
    torch.cuda.synchronize()
    assert _all_plus_zero(out)


def test_empty_contraction_bf16_with_side_maxima(fp8):
    M, N = 130, 264
    A = torch.empty((M, 0), dtype=torch.bfloat16, device="cuda")
    B = torch.empty((N, 0), dtype=torch.bfloat16, device="cuda")
    out = torch.full((M, N), float("nan"), dtype=torch.bfloat16, device="cuda")
    ra = torch.full((M,), 7.0, device="cuda")
    ca = torch.full((N,), 7.0, device="cuda")
    fp8.fp8_scaled_mm_amax(A, B, None, None, out, row_amax=ra, col_amax=ca)
    torch.cuda.synchronize()
    assert _all_plus_zero(out) and _all_plus_zero(ra) and _all_plus_zero(ca)


def test_grouped_empty_contraction_is_unsupported(fp8):
    E, M, N = 3, 64, 32
    ends = torch.tensor([10, 40, 64], dtype=torch.int32, device="cuda")
    A = torch.empty((M, 0), dtype=E4, device="cuda")
    B = torch.empty((E, N, 0), dtype=E4, device="cuda")
    out = torch.zeros((M, N), device="cuda")
    scales = ((torch.ones(M, device="cuda"), torch.ones((E, N), device="cuda")),
              (torch.empty(0, dtype=torch.uint8, device="cuda"), torch.empty(0, dtype=torch.uint8, device="cuda")))
    for sA, sB in scales:  # fp32 row / expert-column scales, then MX scales
        with pytest.raises(fp8.Fp8Error) as e:
            fp8.fp8_grouped_mm(A, B, ends, sA, sB, out, fp8.GROUPED_JAGGED_M)
        assert e.value.code == 2
    G = torch.empty((N, 0), dtype=E5, device="cuda")
    X = torch.empty((16, 0), dtype=E4, device="cuda")
    outk = torch.zeros((E, N, 16), device="cuda")
    with pytest.raises(fp8.Fp8Error) as e:
        fp8.fp8_grouped_mm(G, X, torch.zeros(E, dtype=torch.int32, device="cuda"), torch.ones((E, N), device="cuda"),
                           torch.ones((E, 16), device="cuda"), outk, fp8.GROUPED_JAGGED_K)
    assert e.value.code == 2
    torch.cuda.synchronize()


def test_fused_quant_empty_contraction_is_unsupported(fp8):
    M, N = 128, 256
    A = torch.empty((M, 0), dtype=E4, device="cuda")
    B = torch.empty((N, 0), dtype=E4, device="cuda")
    q = torch.empty((M, N), dtype=E4, device="cuda")
    sc = torch.empty((M, N // 128), device="cuda")
    with pytest.raises(fp8.Fp8Error) as e:
        fp8.fp8_scaled_mm_quant(A, B, torch.ones(1, device="cuda"), torch.ones(1, device="cuda"), q, sc,
                                fp8.GRAN_BLOCK_1x128)
    assert e.value.code == 2


def test_mx_quantize_without_columns(fp8):
    """Segments given, row-major only: nothing to write, and no size derived from the (empty)
    scales."""
    R = 100
    x = torch.empty((R, 0), dtype=torch.bfloat16, device="cuda")
    q = torch.empty((R, 0), dtype=E4, device="cuda")
    sf = torch.empty(0, dtype=torch.uint8, device="cuda")
    ends = torch.tensor([30, 30, 100], dtype=torch.int32, device="cuda")
    ws = torch.zeros(16, dtype=torch.int32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp8.fp8_quantize(x, fp8.GRAN_MX, fp8.DT_E4M3, fp8.LAYOUT_ROW_MAJOR, q, None, sf, ends, ws, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
