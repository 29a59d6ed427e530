"""Parity at the full workload sizes, in the launch configuration the benchmark times: each test
builds the benchmark's own step (same tensors, same entry points, same flags), runs it once, and
checks sampled outputs against the oracle, which computes them one by one from the seeded bf16
inputs (quantize: whole sampled rows / columns, bit-exact; GEMMs: sampled output elements within
the tolerance of "FP8 Training: Quantization, Autograd, Torchao" section 2, 2e-3 * sum|a*b| with
full accumulation, 1e-2 with fast accumulation, plus half a bf16 ulp for bf16 outputs).

The oracle never sees a value the GPU produced: every reference code and scale below is the
oracle's own quantization of the input rows / columns it needs."""
import numpy as np
import pytest
import torch

import oracle
from tests.gpu_util import bits, check_gemm, codes, f32_bits, mx_unblock_rows

pytestmark = pytest.mark.gpu

E4, E5 = oracle.E4M3, oracle.E5M2


@pytest.fixture(scope="module")
def fp8():
    import moe_grouped_gemm_absmax_gb300 as m
    return m


@pytest.fixture(scope="module")
def bench():
    import bench as b
    return b


def _rows(t, idx):
    """bf16 bit patterns of rows `idx` of a device tensor (an input, never a GPU result)."""
    return bits(t[torch.as_tensor(idx, device=t.device)].cpu())


def _cols(t, idx):
    return bits(t[:, torch.as_tensor(idx, device=t.device)].cpu())


def _check_rows_q(x, q, inv, idx, fmt):
    qo, io = oracle.quantize_rows(_rows(x, idx), fmt)
    sel = torch.as_tensor(idx, device=q.device)
    assert np.array_equal(codes(q[sel]), qo)
    assert np.array_equal(f32_bits(inv[sel]), io.view(np.uint32))
    return qo, io


def test_llama3_mlp_up_linear(fp8, bench):
    """M=8192 tokens, K=4096, N=14336; rowwise recipe, bf16 weight gradient (the default bench)."""
    st = bench.make_step(fp8, "llama3-8b-mlp-up")
    st.run()
    torch.cuda.synchronize()
    rng = np.random.default_rng(11)
    M, K, N = st.M, st.K, st.N
    mi = np.sort(rng.choice(M, 8, replace=False))
    ni = np.sort(rng.choice(N, 48, replace=False))
    ki = np.sort(rng.choice(K, 48, replace=False))
    # quantize: sampled rows of x, W, dY; sampled columns of W (column-major copy)
    xq, ix = _check_rows_q(st.x, st.xq, st.xi, mi, E4)
    wq, iw = _check_rows_q(st.w, st.wq, st.wi, ni, E4)
    dyq, idy = _check_rows_q(st.dy, st.dyq, st.dyi, mi, E5)
    wcq, iwc = oracle.quantize_cols(_cols(st.w, ki), E4)  # [N, 48] in W's order, one scale per column
    ksel = torch.as_tensor(ki, device="cuda")
    assert np.array_equal(codes(st.wtq[ksel]), wcq.T)
    assert np.array_equal(f32_bits(st.wti[ksel]), iwc.view(np.uint32))
    # forward (fast accumulation) on the sampled (m, n)
    ref, acc = oracle.gemm_fp8(xq, E4, wq, E4, ix, iw)
    got = st.y[torch.as_tensor(mi, device="cuda")][:, torch.as_tensor(ni, device="cuda")]
    check_gemm(got, ref, acc, True, 1e-2)
    # grad-input on the sampled (m, k): dY rows x W columns quantized over N
    ref, acc = oracle.gemm_fp8(dyq, E5, wcq, E4, idy, iwc, b_trans=True)
    got = st.dx[torch.as_tensor(mi, device="cuda")][:, ksel]
    check_gemm(got, ref, acc, True)
    # bf16 weight gradient on the sampled (n, k): sum over all M tokens
    ref, acc = oracle.gemm_bf16(_cols(st.dy, ni), _cols(st.x, ki), a_trans=True, b_trans=True)
    got = st.dw[torch.as_tensor(ni, device="cuda")][:, ksel]
    check_gemm(got, ref, acc, True)


def test_colwise_gradient_and_rows(fp8, bench):
    """bf16 [8192, 14336] column-gain gradient -> e5m2 per-column scales, column-major codes;
    plus the rowwise e4m3 quantize of [8192, 4096]."""
    st = bench.make_step(fp8, "colwise-8192x14336")
    st.run()
    torch.cuda.synchronize()
    rng = np.random.default_rng(12)
    ci = np.sort(np.concatenate([rng.choice(st.C, 40, replace=False), [0, st.C - 1]]))
    qo, io = oracle.quantize_cols(_cols(st.g, ci), E5)
    sel = torch.as_tensor(ci, device="cuda")
    assert np.array_equal(codes(st.gt[sel]), qo.T)
    assert np.array_equal(f32_bits(st.gi[sel]), io.view(np.uint32))
    _check_rows_q(st.xx, st.xq, st.xi, np.sort(rng.choice(st.RX, 32, replace=False)), E4)


def _expert_of(ends, m):
    return int(np.searchsorted(ends, m, side="right"))


def test_dsv3_grouped_forward(fp8, bench):
    """256 experts, K=7168, N=2048, 131072 routed rows (Zipf counts with empty experts)."""
    st = bench.make_step(fp8, "dsv3-moe-fwd")
    st.run()
    torch.cuda.synchronize()
    ends = st.ends.cpu().numpy()
    assert (st.counts == 0).any()  # the workload has empty experts
    rng = np.random.default_rng(13)
    mi = np.sort(rng.choice(st.M, 6, replace=False))
    # the first and last rows of experts' last tiles with fewer than 256 rows (those run
    # transposed), for tails of each row-box size (up to 64, 128 and 255 rows)
    tail = np.asarray(st.counts) % 256
    for lo, hi in ((1, 64), (65, 128), (129, 255)):
        for e in np.flatnonzero((tail >= lo) & (tail <= hi))[:2]:
            t0 = ends[e] - tail[e]
            mi = np.concatenate([mi, [t0, ends[e] - 1]])
    mi = np.unique(np.concatenate([mi, [0, st.M - 1]]))
    aq, ia = _check_rows_q(st.A, st.Aq, st.Ai, mi, E4)
    ni = np.sort(rng.choice(st.N, 24, replace=False))
    nsel = torch.as_tensor(ni, device="cuda")
    for r, m in enumerate(mi):
        e = _expert_of(ends, m)
        wq, iw = oracle.quantize_rows(bits(st.Wt[e][nsel].cpu()), E4)  # per (expert, n) over K
        assert np.array_equal(codes(st.Wq[e][nsel]), wq)
        assert np.array_equal(f32_bits(st.Wi[e][nsel]), iw.view(np.uint32))
        ref, acc = oracle.gemm_fp8(aq[r:r + 1], E4, wq, E4, ia[r:r + 1], iw)
        check_gemm(st.out[int(m)][nsel].unsqueeze(0), ref, acc, True)


def test_llama4_grouped_forward_backward(fp8, bench):
    """16 experts, K=5120, N=8192, 8192 tokens (Dirichlet routing): grouped forward, grouped dX
    with per-expert W quantized over N, and dW with jagged column-wise quantization."""
    st = bench.make_step(fp8, "llama4-moe-fwdbwd")
    st.run()
    torch.cuda.synchronize()
    ends = st.ends.cpu().numpy()
    rng = np.random.default_rng(14)
    mi = np.sort(rng.choice(st.M, 6, replace=False))
    # the first and last rows of two experts' last tiles with fewer than 256 rows (the forward and
    # dX compute those tiles transposed)
    tail = np.asarray(st.counts) % 256
    for e in np.flatnonzero(tail > 0)[:2]:
        mi = np.concatenate([mi, [ends[e] - tail[e], ends[e] - 1]])
    mi = np.unique(mi)
    ni = np.sort(rng.choice(st.N, 16, replace=False))
    ki = np.sort(rng.choice(st.K, 16, replace=False))
    nsel, ksel = torch.as_tensor(ni, device="cuda"), torch.as_tensor(ki, device="cuda")
    aq, ia = _check_rows_q(st.A, st.Aq, st.Ai, mi, E4)
    dyq, idy = _check_rows_q(st.dY, st.dYq, st.dYi, mi, E5)
    for r, m in enumerate(mi):
        e = _expert_of(ends, m)
        wq, iw = oracle.quantize_rows(bits(st.Wt[e][nsel].cpu()), E4)
        ref, acc = oracle.gemm_fp8(aq[r:r + 1], E4, wq, E4, ia[r:r + 1], iw)
        check_gemm(st.out[int(m)][nsel].unsqueeze(0), ref, acc, True)
        # dX: per-expert W columns k quantized over N (column-major copy [E, K, N])
        wc, iwc = oracle.quantize_cols(bits(st.Wt[e][:, ksel].cpu()), E4)
        assert np.array_equal(codes(st.Wtq[e][ksel]), wc.T)
        assert np.array_equal(f32_bits(st.Wti[e][ksel]), iwc.view(np.uint32))
        ref, acc = oracle.gemm_fp8(dyq[r:r + 1], E5, wc, E4, idy[r:r + 1], iwc, b_trans=True)
        check_gemm(st.dX[int(m)][ksel].unsqueeze(0), ref, acc, True)
    # dW[e, n, k]: jagged column-wise codes of dY columns n and A columns k within each segment
    dq, di = oracle.quantize_jagged_cols(_cols(st.dY, ni), ends, E5)  # [M, 16] in row order, [E, 16]
    aq2, ai2 = oracle.quantize_jagged_cols(_cols(st.A, ki), ends, E4)
    assert np.array_equal(f32_bits(st.dYti[:, nsel]), di.view(np.uint32))
    assert np.array_equal(f32_bits(st.Ati[:, ksel]), ai2.view(np.uint32))
    prev, pstart = 0, 0
    for e, end in enumerate(ends):
        end = int(end)
        cnt = end - prev
        if cnt:
            # the segment-padded column-major copies hold these codes at the segment's start
            assert np.array_equal(codes(st.dYt[nsel][:, pstart:pstart + cnt]), dq[prev:end].T)
            assert np.array_equal(codes(st.At[ksel][:, pstart:pstart + cnt]), aq2[prev:end].T)
            ref, acc = oracle.gemm_fp8(dq[prev:end], E5, aq2[prev:end], E4, di[e], ai2[e], a_trans=True, b_trans=True)
        else:  # an empty expert's weight gradient is zero
            ref, acc = np.zeros((ni.size, ki.size)), np.zeros((ni.size, ki.size))
        check_gemm(st.dW[e][nsel][:, ksel], ref, acc, True)
        pstart += -(-cnt // 128) * 128
        prev = end


# ---------------------------------------------------------------------------- MXFP8 workloads

_mx_unblock_rows = mx_unblock_rows


def test_llama3_mlp_up_mx(fp8, bench):
    """The MX Linear at full size: sampled rows / columns of every quantized copy bit-exact, and
    sampled elements of y, dX and dW within the GEMM tolerance."""
    st = bench.make_step(fp8, "llama3-8b-mlp-up-mx")
    st.run()
    torch.cuda.synchronize()
    rng = np.random.default_rng(21)
    M, K, N = st.M, st.K, st.N
    mi = np.sort(rng.choice(M, 6, replace=False))
    ni = np.sort(rng.choice(N, 24, replace=False))
    ki = np.sort(rng.choice(K, 24, replace=False))
    msel, nsel, ksel = (torch.as_tensor(a, device="cuda") for a in (mi, ni, ki))
    xr, xrs = oracle.mx_quantize_rows(_rows(st.x, mi), E4)
    assert np.array_equal(codes(st.xq[msel]), xr) and np.array_equal(_mx_unblock_rows(st.xs[:st.nx], mi, K), xrs)
    wr, wrs = oracle.mx_quantize_rows(_rows(st.w, ni), E4)
    assert np.array_equal(codes(st.wq[nsel]), wr) and np.array_equal(_mx_unblock_rows(st.wsc[:st.nw], ni, K), wrs)
    dyr, dyrs = oracle.mx_quantize_rows(_rows(st.dy, mi), E5)
    wc, wcs = oracle.mx_quantize_rows(np.ascontiguousarray(_cols(st.w, ki).T), E4)  # W^T rows k, blocks along N
    assert np.array_equal(codes(st.wtq[ksel]), wc) and np.array_equal(_mx_unblock_rows(st.wsc[st.nw:], ki, N), wcs)
    ref, acc = oracle.gemm_mx(xr, E4, wr, E4, xrs, wrs)
    check_gemm(st.y[msel][:, nsel], ref, acc, True)
    ref, acc = oracle.gemm_mx(dyr, E5, wc, E4, dyrs, wcs)
    check_gemm(st.dx[msel][:, ksel], ref, acc, True)
    # dW[n, k] = sum over all M tokens of dY^T (blocks along M) and x^T (blocks along M)
    dyc, dycs = oracle.mx_quantize_rows(np.ascontiguousarray(_cols(st.dy, ni).T), E5)
    xc, xcs = oracle.mx_quantize_rows(np.ascontiguousarray(_cols(st.x, ki).T), E4)
    assert np.array_equal(codes(st.dytq[nsel]), dyc) and np.array_equal(codes(st.xtq[ksel]), xc)
    ref, acc = oracle.gemm_mx(dyc, E5, xc, E4, dycs, xcs)
    check_gemm(st.dw[nsel][:, ksel], ref, acc, True)


def test_dsv3_grouped_forward_mx(fp8, bench):
    st = bench.make_step(fp8, "dsv3-moe-fwd-mx")
    st.run()
    torch.cuda.synchronize()
    ends = st.ends.cpu().numpy()
    starts, _, pstarts, _ = oracle.mx_padded_segments(ends)
    rng = np.random.default_rng(23)
    mi = np.concatenate([np.sort(rng.choice(st.M, 6, replace=False)), [0, st.M - 1]])
    ni = np.sort(rng.choice(st.N, 24, replace=False))
    nsel = torch.as_tensor(ni, device="cuda")
    ar, ars = oracle.mx_quantize_rows(_rows(st.A, mi), E4)
    assert np.array_equal(codes(st.Aq[torch.as_tensor(mi, device="cuda")]), ar)
    for r, m in enumerate(mi):
        e = _expert_of(ends, m)
        prow = pstarts[e] + (m - starts[e])  # A's scales sit at the segment-padded row
        assert np.array_equal(_mx_unblock_rows(st.As, [prow], st.K), ars[r:r + 1])
        wq, ws = oracle.mx_quantize_rows(bits(st.Wt[e][nsel].cpu()), E4)
        assert np.array_equal(codes(st.Wq[e][nsel]), wq)
        per = st.Ws.numel() // st.E
        assert np.array_equal(_mx_unblock_rows(st.Ws[e * per:(e + 1) * per], ni, st.K), ws)
        ref, acc = oracle.gemm_mx(ar[r:r + 1], E4, wq, E4, ars[r:r + 1], ws)
        check_gemm(st.out[int(m)][nsel].unsqueeze(0), ref, acc, True)


def test_llama4_grouped_forward_backward_mx(fp8, bench):
    st = bench.make_step(fp8, "llama4-moe-fwdbwd-mx")
    st.run()
    torch.cuda.synchronize()
    ends = st.ends.cpu().numpy()
    starts, counts, pstarts, _ = oracle.mx_padded_segments(ends)
    rng = np.random.default_rng(24)
    mi = np.sort(rng.choice(st.M, 5, replace=False))
    ni = np.sort(rng.choice(st.N, 12, replace=False))
    ki = np.sort(rng.choice(st.K, 12, replace=False))
    nsel, ksel = torch.as_tensor(ni, device="cuda"), torch.as_tensor(ki, device="cuda")
    E, N, K = st.E, st.N, st.K
    sb = fp8.fp8_mx_scale_bytes
    ar, ars = oracle.mx_quantize_rows(_rows(st.A, mi), E4)
    dyr, dyrs = oracle.mx_quantize_rows(_rows(st.dY, mi), E5)
    for r, m in enumerate(mi):
        e = _expert_of(ends, m)
        wb = bits(st.Wt[e].cpu())                      # [N, K]
        wq, ws = oracle.mx_quantize_rows(wb[ni], E4)   # forward: W[e] rows n, blocks along K
        ref, acc = oracle.gemm_mx(ar[r:r + 1], E4, wq, E4, ars[r:r + 1], ws)
        check_gemm(st.out[int(m)][nsel].unsqueeze(0), ref, acc, True)
        wt, wts = oracle.mx_quantize_rows(np.ascontiguousarray(wb[:, ki].T), E4)  # W[e]^T rows k, blocks along N
        assert np.array_equal(codes(st.Wtq[e][ksel]), wt)
        base = st.nW + e * sb(K, N)
        assert np.array_equal(_mx_unblock_rows(st.W_s[base:base + sb(K, N)], ki, N), wts)
        ref, acc = oracle.gemm_mx(dyr[r:r + 1], E5, wt, E4, dyrs[r:r + 1], wts)
        check_gemm(st.dX[int(m)][ksel].unsqueeze(0), ref, acc, True)
    # dW[e, n, k]: both operands MX-quantized along the tokens of each (padded) segment
    gq, gs = oracle.mx_quantize_jagged_cols(_cols(st.dY, ni), ends, E5)
    xq, xs = oracle.mx_quantize_jagged_cols(_cols(st.A, ki), ends, E4)
    Pu = gq.shape[1]
    assert np.array_equal(codes(st.dYt[nsel])[:, :Pu], gq) and np.array_equal(codes(st.At[ksel])[:, :Pu], xq)
    assert np.array_equal(_mx_unblock_rows(st.dY_s[st.ndY:], ni, st.P)[:, :Pu // 32], gs)
    assert np.array_equal(_mx_unblock_rows(st.A_s[st.nA:], ki, st.P)[:, :Pu // 32], xs)
    padded = -(-counts // 128) * 128
    for e in range(E):
        got = st.dW[e][nsel][:, ksel]
        if counts[e] == 0:
            assert torch.count_nonzero(got).item() == 0
            continue
        ps, pe = pstarts[e], pstarts[e] + padded[e]
        ref, acc = oracle.gemm_mx(gq[:, ps:pe], E5, xq[:, ps:pe], E4, gs[:, ps // 32:pe // 32], xs[:, ps // 32:pe // 32])
        check_gemm(got, ref, acc, True)
