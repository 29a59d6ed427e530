"""The GEMM whose epilogue writes its result's next quantization (fp8_scaled_mm_quant): "FP8
training on AMD GPUs with TorchTitan and TorchAO", "Triton Kernel Optimization", Level 1 (the
quantize fused into the producing kernel), with 1 x 128 blocks ("AMD FP8 format in TorchAO",
blockwise scaling) or MX blocks of 32 (OCP MX v1.0) along the rows of the result.

Checked against the oracle:
  - bit for bit: on integer-valued operands with power-of-two scales the fp32 accumulation is
    exact, so the oracle's GEMM rounded once to bf16 is the value the epilogue quantizes, and the
    oracle's blockwise / MX quantize of it fixes the codes and scales;
  - general operands (the oracle's row-wise codes of seeded bf16 inputs): the dequantized codes
    within the GEMM tolerance of the oracle's fp64 GEMM plus the quantization's own error (half a
    code step at the block's scale);
  - guard bands around the codes and the scales."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_util import bits, mx_unblock_rows, upload_codes, upload_f32

pytestmark = pytest.mark.gpu
E4, E5 = oracle.E4M3, oracle.E5M2


@pytest.fixture(scope="module")
def fp8():
    import moe_grouped_gemm_absmax_gb300 as m
    return m


def _exact_operands(M, N, K, seed):
    rng = np.random.default_rng(seed)
    a = rng.integers(-8, 9, size=(M, K)).astype(np.float32)
    b = rng.integers(-8, 9, size=(N, K)).astype(np.float32)
    sa = (2.0 ** rng.integers(-6, 3, size=M)).astype(np.float32)
    sb = (2.0 ** rng.integers(-6, 3, size=N)).astype(np.float32)
    return oracle.encode(a, E4), oracle.encode(b, E4), sa, sb


def _run(fp8, ca, cb, sa, sb, gran, fmt, guard=0):
    """fp8_scaled_mm_quant on device copies; returns (codes, scales) as host arrays (the scale bytes
    of MX as stored); with guard > 0 the outputs sit between sentinel regions that are checked."""
    M, N = ca.shape[0], cb.shape[0]
    fdt = torch.float8_e4m3fn if fmt == E4 else torch.float8_e5m2
    nq = M * N
    ns = fp8.fp8_mx_scale_bytes(M, N) if gran == fp8.GRAN_MX else M * (N // 128) * 4
    qb = torch.full((2 * guard + nq,), 0xA5, dtype=torch.uint8, device="cuda")
    sbuf = torch.full((2 * guard + ns,), 0xA5, dtype=torch.uint8, device="cuda")
    q = qb[guard:guard + nq].view(fdt).view(M, N)
    sc = sbuf[guard:guard + ns] if gran == fp8.GRAN_MX else sbuf[guard:guard + ns].view(torch.float32).view(M, N // 128)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp8.fp8_scaled_mm_quant(upload_codes(ca, E4), upload_codes(cb, E4), upload_f32(sa), upload_f32(sb), q, sc, gran,
                            status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    if guard:
        for buf, n in ((qb, nq), (sbuf, ns)):
            h = buf.cpu().numpy()
            assert (h[:guard] == 0xA5).all() and (h[guard + n:] == 0xA5).all(), "write outside the output"
    return q.view(torch.uint8).cpu().numpy(), sc


@pytest.mark.parametrize("gran_name", ["GRAN_BLOCK_1x128", "GRAN_MX"])
@pytest.mark.parametrize("fmt", [E4, E5])
@pytest.mark.parametrize("M,N,K", [(300, 512, 256), (1300, 4608, 160)])  # single CTAs; CTA pairs
def test_matches_oracle_bit_for_bit(fp8, gran_name, fmt, M, N, K):
    gran = getattr(fp8, gran_name)
    ca, cb, sa, sb = _exact_operands(M, N, K, M + N)
    ref, _ = oracle.gemm_fp8(ca, E4, cb, E4, sa, sb)
    rb = bits(torch.from_numpy(ref.astype(np.float32)).to(torch.bfloat16))  # exact -> one RNE rounding
    q, sc = _run(fp8, ca, cb, sa, sb, gran, fmt, guard=4096)
    if gran == fp8.GRAN_MX:
        qo, so = oracle.mx_quantize_rows(rb, fmt)
        assert np.array_equal(q, qo)
        assert np.array_equal(mx_unblock_rows(sc, np.arange(M), N), so)
    else:
        qo, so = oracle.quantize_blocks(rb, fmt, 1, 128)
        assert np.array_equal(q, qo)
        assert np.array_equal(sc.cpu().numpy().view(np.uint32), so.view(np.uint32))


@pytest.mark.parametrize("gran_name", ["GRAN_BLOCK_1x128", "GRAN_MX"])
def test_general_operands_within_bound(fp8, gran_name):
    """x W^T of the oracle's row-wise codes of seeded bf16 inputs (outlier channels in x): the
    dequantized result within the GEMM bound plus half a code step at each block's scale."""
    gran = getattr(fp8, gran_name)
    M, K, N = 512, 768, 1024
    x, w, _ = W.linear_inputs(M, K, N, seed=21, outliers=True)
    ca, ia = oracle.quantize_rows(bits(x), E4)
    cb, ib = oracle.quantize_rows(bits(w), E4)
    ref, acc = oracle.gemm_fp8(ca, E4, cb, E4, ia, ib)
    q, sc = _run(fp8, ca, cb, ia, ib, gran, E4)
    dec = oracle.decode(q, E4)
    if gran == fp8.GRAN_MX:
        blk = oracle.e8m0_decode(mx_unblock_rows(sc, np.arange(M), N))  # X per block of 32
        scale = np.repeat(blk, 32, axis=1)
    else:
        scale = np.repeat(sc.cpu().numpy().astype(np.float64), 128, axis=1)  # inverse scale per 1 x 128 block
    deq = dec * scale
    gemm_err = 2e-3 * acc + 2.0 ** -8 * np.abs(ref)
    # e4m3: a code step is 2^-3 of the value's binade (half: 2^-4), subnormals 2^-9 (half: 2^-10);
    # MX puts a block's largest element in [256, 512) code units, so values above 448 X saturate
    mag = np.abs(ref) + gemm_err
    quant_err = 2.0 ** -4 * mag + 2.0 ** -10 * scale
    if gran == fp8.GRAN_MX:
        quant_err += np.maximum(0.0, mag - 448.0 * scale)
    bad = np.abs(deq - ref) > gemm_err + quant_err + 1e-30
    assert not bad.any(), f"{bad.sum()} elements outside the bound"


def test_rejects(fp8):
    a = torch.zeros((128, 128), dtype=torch.float8_e4m3fn, device="cuda")
    s = torch.ones(1, device="cuda")
    q = torch.empty((128, 64), dtype=torch.float8_e4m3fn, device="cuda")
    b = torch.zeros((64, 128), dtype=torch.float8_e4m3fn, device="cuda")
    with pytest.raises(fp8.Fp8Error):  # N % 128 != 0
        fp8.fp8_scaled_mm_quant(a, b, s, s, q, torch.empty((128, 1), device="cuda"), fp8.GRAN_BLOCK_1x128)
    q2 = torch.empty((128, 128), dtype=torch.float8_e4m3fn, device="cuda")
    with pytest.raises(fp8.Fp8Error):  # row granularity is not an output recipe here
        fp8.fp8_scaled_mm_quant(a, a, s, s, q2, torch.empty(128, device="cuda"), fp8.GRAN_ROW)
