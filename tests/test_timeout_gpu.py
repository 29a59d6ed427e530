"""Failure detection without a GPU fault: every on-device wait of the GEMM kernels, of the grid
barrier of the tensorwise quantize, of the column-wise quantize's partial maxima and of the MX
quantize's load ring is bounded. The test hook fp8_set_test_stall makes the GEMM's MMA issuer wait
on a barrier that nothing signals, the tensorwise quantize wait for one CTA more than it
launched, the column-wise gatherers read no partial as written and the MX producer load nothing;
with a short wait limit the wait runs out, and the kernel must report
FP8_DEV_TIMEOUT in the status word, stop its other warps, drain its in-flight TMA loads and MMAs,
free its tensor memory and return, leaving the context usable (a normal call afterwards is
correct)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_util import bits, check_gemm, upload_codes, upload_f32

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp8():
    import moe_grouped_gemm_absmax_gb300 as m
    return m


def _operands(M, N, K, seed):
    x = W.normal_bf16((M, K), 1.0, seed)
    w = W.normal_bf16((N, K), 0.02, seed + 1)
    ca, ia = oracle.quantize_rows(bits(x), oracle.E4M3)
    cb, ib = oracle.quantize_rows(bits(w), oracle.E4M3)
    return ca, ia, cb, ib


@pytest.mark.parametrize("M,N,K", [(256, 512, 2048), (2048, 4096, 1024)])  # single CTAs, CTA pairs
def test_wait_limit_expiry_reports_timeout_and_context_survives(fp8, M, N, K):
    ca, ia, cb, ib = _operands(M, N, K, 5)
    A, B, sA, sB = upload_codes(ca, 0), upload_codes(cb, 0), upload_f32(ia), upload_f32(ib)
    out = torch.zeros((M, N), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    old = fp8.fp8_set_wait_limit_ns(2_000_000)  # 2 ms
    fp8.fp8_set_test_stall(True)
    try:
        fp8.fp8_scaled_mm(A, B, sA, sB, out, status=st)
        torch.cuda.synchronize()
    finally:
        fp8.fp8_set_test_stall(False)
        fp8.fp8_set_wait_limit_ns(old)
    assert int(st.item()) & fp8.DEV_TIMEOUT
    # the same call with the normal bound succeeds and is correct
    st.zero_()
    fp8.fp8_scaled_mm(A, B, sA, sB, out, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rows = np.arange(0, M, max(1, M // 64))
    ref, absacc = oracle.gemm_fp8(ca, oracle.E4M3, cb, oracle.E4M3, ia, ib, rows=rows)
    check_gemm(out[torch.from_numpy(rows).cuda()], ref, absacc, True)


def test_tensorwise_barrier_expiry_reports_timeout_and_context_survives(fp8):
    x = W.normal_bf16((1024, 2048), 1.0, 17)
    xd = x.cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    old = fp8.fp8_set_wait_limit_ns(2_000_000)  # 2 ms
    fp8.fp8_set_test_stall(True)
    try:
        fp8.quantize_alloc(xd, fp8.GRAN_TENSOR, fp8.DT_E4M3, layout=fp8.LAYOUT_BOTH, status=st)
        torch.cuda.synchronize()
    finally:
        fp8.fp8_set_test_stall(False)
        fp8.fp8_set_wait_limit_ns(old)
    assert int(st.item()) & fp8.DEV_TIMEOUT
    st.zero_()
    q, qt, inv = fp8.quantize_alloc(xd, fp8.GRAN_TENSOR, fp8.DT_E4M3, layout=fp8.LAYOUT_BOTH, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    qo, io = oracle.quantize_tensor(bits(x), oracle.E4M3)
    assert np.array_equal(q.view(torch.uint8).cpu().numpy(), qo)
    assert np.array_equal(qt.view(torch.uint8).cpu().numpy(), qo.T)
    assert np.array_equal(inv.cpu().numpy().view(np.uint32), io.view(np.uint32))


@pytest.mark.parametrize("counts", [None, [300, 0, 700, 24]])  # dense, jagged segments
def test_colwise_barrier_expiry_reports_timeout_and_context_survives(fp8, counts):
    R, C = 1024, 512
    x = W.column_gain_bf16((R, C), 1e-3, -2, 2, seed=23)
    xd = x.cuda()
    offs = torch.tensor(W.ends_from_counts(counts), device="cuda") if counts else None
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    old = fp8.fp8_set_wait_limit_ns(2_000_000)  # 2 ms
    fp8.fp8_set_test_stall(True)
    try:
        fp8.quantize_alloc(xd, fp8.GRAN_COL, fp8.DT_E5M2, offsets=offs, status=st)
        torch.cuda.synchronize()
    finally:
        fp8.fp8_set_test_stall(False)
        fp8.fp8_set_wait_limit_ns(old)
    assert int(st.item()) & fp8.DEV_TIMEOUT
    st.zero_()
    _, qt, inv = fp8.quantize_alloc(xd, fp8.GRAN_COL, fp8.DT_E5M2, offsets=offs, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    if counts is None:
        qo, io = oracle.quantize_cols(bits(x), oracle.E5M2)
        assert np.array_equal(qt.view(torch.uint8).cpu().numpy(), qo.T)
    else:
        ends = W.ends_from_counts(counts)
        qo, io = oracle.quantize_jagged_cols(bits(x), ends, oracle.E5M2)
        from tests.gpu_util import segpad_cols
        used = sum(-(-c // 128) * 128 for c in counts)
        got = qt.view(torch.uint8).cpu().numpy()
        assert np.array_equal(got[:, :used], segpad_cols(qo, ends, qt.shape[1])[:, :used])
    assert np.array_equal(inv.cpu().numpy().view(np.uint32), io.view(np.uint32))


def test_mx_ring_expiry_reports_timeout_and_context_survives(fp8):
    """The pipelined MX quantize (column-major output of a dense tensor): with the hook on its
    producer loads nothing, the consumers' bounded wait runs out, the status says so, and the
    next call on the same context is bit-exact against the oracle."""
    x = W.normal_bf16((512, 384), 1.0, 23)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    old = fp8.fp8_set_wait_limit_ns(2_000_000)  # 2 ms
    fp8.fp8_set_test_stall(True)
    try:
        fp8.mx_quantize_alloc(x.cuda(), fp8.DT_E4M3, fp8.LAYOUT_BOTH, status=st)
        torch.cuda.synchronize()
    finally:
        fp8.fp8_set_test_stall(False)
        fp8.fp8_set_wait_limit_ns(old)
    assert int(st.item()) & fp8.DEV_TIMEOUT
    st.zero_()
    q, qt, sf, sft = fp8.mx_quantize_alloc(x.cuda(), fp8.DT_E4M3, fp8.LAYOUT_BOTH, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    qo, so = oracle.mx_quantize_cols(bits(x), oracle.E4M3)
    assert np.array_equal(qt.cpu().view(torch.uint8).numpy(), qo)
    qr, sr = oracle.mx_quantize_rows(bits(x), oracle.E4M3)
    assert np.array_equal(q.cpu().view(torch.uint8).numpy(), qr)
