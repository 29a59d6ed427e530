"""GPU parity of the MXFP8 path (blocks of 32, E8M0 scales) against the oracle.

MXFP8 is named by "FP8 training on AMD GPUs with TorchTitan and TorchAO" (section "AMD FP8
format in TorchAO"; "Summary and Next Steps"); the block rule is that of the OCP Microscaling
Formats (MX) specification v1.0 (see oracle/oracle.h). Quantize: codes and E8M0 scales
bit-exact. GEMMs: within 2e-3 * sum|terms| plus half a bf16 ulp ("FP8 Training: Quantization,
Autograd, Torchao" section 2 tolerance), on inputs the oracle quantized (or random codes and
scales), never on values the GPU produced.

The GPU writes scales in the tensor-core layout of include/fp8lin.h ("MX scale layout"); the
tests move them between that layout and the oracle's plain [rows, K / 32] order with a pure
index permutation (mx_block / mx_unblock below)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_util import bits, check_gemm, codes, mx_offsets, upload_codes

pytestmark = pytest.mark.gpu

E4, E5 = oracle.E4M3, oracle.E5M2
TDT = {E4: 3, E5: 4}  # oracle format -> FP8_DT_*


@pytest.fixture(scope="module")
def fp8():
    import moe_grouped_gemm_absmax_gb300 as m
    return m


def _offsets(rows_padded, K):
    return mx_offsets(np.arange(rows_padded), K)


def mx_unblock(sf, rows, K):
    """Layout bytes -> plain [rows, K / 32] codes."""
    b = sf.cpu().numpy() if isinstance(sf, torch.Tensor) else np.asarray(sf)
    return b[_offsets(rows, K)]


def mx_block(plain, K, rows_padded=None):
    """Plain [rows, K / 32] codes -> layout bytes (rows padded to 128; the padding is 127)."""
    rows = plain.shape[0]
    rp = rows_padded or -(-rows // 128) * 128
    out = np.full(rp * K // 32, 127, np.uint8)
    out[_offsets(rows, K)] = plain
    return out


def _up(a):
    return torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _mx_rows_input(R, C, seed):
    """Normal values with outlier and all-zero blocks, a block of bf16 subnormals and a block
    that saturates (amax / X above 448)."""
    x = W.normal_bf16((R, C), 1.0, seed).float()
    g = torch.Generator().manual_seed(seed + 1)
    idx = torch.randint(0, R * C, (max(1, R * C // 500),), generator=g)
    x.view(-1)[idx] *= 300.0
    x[0, :32] = 0.0
    if R > 1:
        x[1, 32:64] = 2.0 ** -130
    if R > 2 and C >= 96:
        x[2, 64:96] = 1.0
        x[2, 64] = 480.0  # amax 480: X = 1, 480 saturates to 448
    return x.to(torch.bfloat16)


# ---------------------------------------------------------------------------- quantize

@pytest.mark.parametrize("shape,fmt", [((256, 256), E4), ((300, 384), E4), ((77, 128), E5), ((3, 128, 384), E4),
                                       ((1, 1024), E5), ((70, 7168), E4), ((40, 12288), E5), ((2, 9, 4096), E4),
                                       ((40, 16512), E4), ((2, 9, 16512), E5)])
def test_mx_quantize_rows(fp8, shape, fmt):
    """Row blocks alone; rows longer than 16384 elements take the tiled pipeline (the last two
    cases, one of them with 9-row batch entries inside a tile's 128 rows)."""
    x = _mx_rows_input(int(np.prod(shape[:-1])), shape[-1], 3).reshape(shape)
    q, _, sf, _ = fp8.mx_quantize_alloc(x.cuda(), TDT[fmt], fp8.LAYOUT_ROW_MAJOR)
    torch.cuda.synchronize()
    R, C = shape[-2], shape[-1]
    B = shape[0] if len(shape) == 3 else 1
    xb = bits(x).reshape(B, R, C)
    sfb = sf.cpu().numpy().reshape(B, -1)
    for b in range(B):
        qo, so = oracle.mx_quantize_rows(xb[b], fmt)
        assert np.array_equal(codes(q).reshape(B, R, C)[b], qo)
        assert np.array_equal(mx_unblock(sfb[b], R, C), so)


@pytest.mark.parametrize("shape,fmt,layout", [((256, 256), E5, "col"), ((384, 128), E4, "both"),
                                              ((2, 128, 256), E4, "both"), ((128, 640), E5, "col"),
                                              ((4096, 3072), E5, "both"), ((3, 1024, 2048), E4, "col")])
def test_mx_quantize_cols_and_both(fp8, shape, fmt, layout):
    """Column blocks (and row blocks from the same read) through the tiled pipeline; the last two
    cases give every CTA more tiles than its 4-stage ring holds."""
    x = _mx_rows_input(int(np.prod(shape[:-1])), shape[-1], 5).reshape(shape)
    lay = fp8.LAYOUT_COL_MAJOR if layout == "col" else fp8.LAYOUT_BOTH
    q, qt, sf, sft = fp8.mx_quantize_alloc(x.cuda(), TDT[fmt], lay)
    torch.cuda.synchronize()
    R, C = shape[-2], shape[-1]
    B = shape[0] if len(shape) == 3 else 1
    xb = bits(x).reshape(B, R, C)
    qtb = codes(qt).reshape(B, C, R)
    sftb = sft.cpu().numpy().reshape(B, -1)
    for b in range(B):
        qo, so = oracle.mx_quantize_cols(xb[b], fmt)  # codes of x^T [C, R], scales [C, R / 32]
        assert np.array_equal(qtb[b], qo)
        assert np.array_equal(mx_unblock(sftb[b], C, R), so)
        if layout == "both":
            qr, sr = oracle.mx_quantize_rows(xb[b], fmt)
            assert np.array_equal(codes(q).reshape(B, R, C)[b], qr)
            assert np.array_equal(mx_unblock(sf.cpu().numpy().reshape(B, -1)[b], R, C), sr)


@pytest.mark.parametrize("counts,C,fmt", [([40, 0, 200, 1, 130], 256, E5), ([0, 0, 128], 128, E4),
                                          ([300, 17, 0, 0, 256, 90], 384, E4),
                                          (list(W.llama4_counts(1) // 2), 2048, E5)])
def test_mx_quantize_jagged(fp8, counts, C, fmt):
    """Segments padded to 128 rows: column-major codes [C, P] and scales per (column, 32-token
    block of a segment); row-major scales at the padded rows. Both from one read."""
    M = sum(counts)
    x = _mx_rows_input(M, C, 7)
    ends = W.ends_from_counts(counts)
    q, qt, sf, sft = fp8.mx_quantize_alloc(x.cuda(), TDT[fmt], fp8.LAYOUT_BOTH, offsets=_up(ends))
    torch.cuda.synchronize()
    P = qt.shape[1]
    qo, so = oracle.mx_quantize_jagged_cols(bits(x), ends, fmt)
    used = qo.shape[1]
    assert np.array_equal(codes(qt)[:, :used], qo)
    assert np.array_equal(mx_unblock(sft, C, P)[:, :used // 32], so)
    qr, sr = oracle.mx_quantize_rows(bits(x), fmt)
    assert np.array_equal(codes(q), qr)
    sfr = mx_unblock(sf, P, C)
    starts, cnts, pstarts, _ = oracle.mx_padded_segments(ends)
    for s0, c, ps in zip(starts, cnts, pstarts):
        assert np.array_equal(sfr[ps:ps + c], sr[s0:s0 + c])


@pytest.mark.parametrize("counts,C,fmt", [([40, 0, 200, 1, 130], 256, E5), ([300, 17, 0, 0, 256, 90], 7168, E4)])
def test_mx_quantize_jagged_rows_only(fp8, counts, C, fmt):
    """The row-major output alone with segments: codes in x's rows, scales at the padded rows of
    each row's segment (the layout the jagged-M GEMM reads)."""
    M = sum(counts)
    x = _mx_rows_input(M, C, 9)
    ends = W.ends_from_counts(counts)
    q, qt, sf, sft = fp8.mx_quantize_alloc(x.cuda(), TDT[fmt], fp8.LAYOUT_ROW_MAJOR, offsets=_up(ends))
    torch.cuda.synchronize()
    assert qt is None and sft is None
    qr, sr = oracle.mx_quantize_rows(bits(x), fmt)
    assert np.array_equal(codes(q), qr)
    P = fp8.fp8_jagged_padded_rows(M, len(counts))
    sfr = mx_unblock(sf, P, C)
    starts, cnts, pstarts, _ = oracle.mx_padded_segments(ends)
    for s0, c, ps in zip(starts, cnts, pstarts):
        assert np.array_equal(sfr[ps:ps + c], sr[s0:s0 + c])


def test_mx_quantize_rejects(fp8):
    x = torch.zeros((128, 96), dtype=torch.bfloat16, device="cuda")  # C % 128 != 0
    with pytest.raises(fp8.Fp8Error):
        fp8.mx_quantize_alloc(x, 3, fp8.LAYOUT_ROW_MAJOR)
    x = torch.zeros((100, 128), dtype=torch.bfloat16, device="cuda")  # column blocks need R % 128 == 0
    with pytest.raises(fp8.Fp8Error):
        fp8.mx_quantize_alloc(x, 3, fp8.LAYOUT_COL_MAJOR)


# ---------------------------------------------------------------------------- GEMMs

def _random_mx_operand(rng, rows, K, fmt, lo=118, hi=136):
    c = rng.integers(0, 256, (rows, K)).astype(np.uint8)
    nan = (c & 0x7F) == 0x7F if fmt == E4 else (c & 0x7C) == 0x7C
    c[nan] = 0x30
    s = rng.integers(lo, hi, (rows, K // 32)).astype(np.uint8)
    return c, s


def _dense_mx(fp8, ca, fa, sa, cb, fb, sb, out_dtype):
    M, K = ca.shape
    N = cb.shape[0]
    out = torch.full((M, N), float("nan"), dtype=out_dtype, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp8.fp8_scaled_mm(upload_codes(ca, fa), upload_codes(cb, fb), _up(mx_block(sa, K)), _up(mx_block(sb, K)), out,
                      status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return out


@pytest.mark.parametrize("M,N,K,fa,fb,out_dtype", [
    (128, 192, 128, E4, E4, torch.float32),     # one tile
    (300, 500, 384, E5, E4, torch.bfloat16),    # ragged M and N, single CTAs
    (129, 200, 256, E4, E5, torch.float32),     # a 2-row block and a tile straddling two scale blocks
    (4096, 2304, 256, E4, E4, torch.bfloat16),  # CTA pairs
    (2500, 3000, 512, E5, E4, torch.float32),   # pairs, ragged
])
def test_mx_gemm_random(fp8, M, N, K, fa, fb, out_dtype):
    rng = np.random.default_rng(M + N + K)
    ca, sa = _random_mx_operand(rng, M, K, fa)
    cb, sb = _random_mx_operand(rng, N, K, fb)
    out = _dense_mx(fp8, ca, fa, sa, cb, fb, sb, out_dtype)
    rows = np.unique(np.concatenate([rng.choice(M, min(M, 64), replace=False), [0, M - 1]]))
    rows = rows if M > 256 else None
    ref, absacc = oracle.gemm_mx(ca, fa, cb, fb, sa, sb, rows=rows)
    got = out if rows is None else out[torch.as_tensor(rows, device="cuda")]
    check_gemm(got, ref, absacc, out_dtype == torch.bfloat16)


def test_mx_gemm_quantized_linear(fp8):
    """x W^T with both operands quantized to MXFP8 by the oracle (outlier channels in x)."""
    M, K, N = 512, 1024, 768
    x, w, _ = W.linear_inputs(M, K, N, seed=3, outliers=True)
    cx, sx = oracle.mx_quantize_rows(bits(x), E4)
    cw, sw = oracle.mx_quantize_rows(bits(w), E4)
    out = _dense_mx(fp8, cx, E4, sx, cw, E4, sw, torch.bfloat16)
    ref, absacc = oracle.gemm_mx(cx, E4, cw, E4, sx, sw)
    check_gemm(out, ref, absacc, True)


def _padded_rows_sf(plain, ends, K, P):
    """Row scales [M, K/32] placed at the segment-padded rows, in the MX layout of P rows."""
    starts, cnts, pstarts, _ = oracle.mx_padded_segments(ends)
    full = np.full((P, K // 32), 127, np.uint8)
    for s0, c, ps in zip(starts, cnts, pstarts):
        full[ps:ps + c] = plain[s0:s0 + c]
    return mx_block(full, K, P)


@pytest.mark.parametrize("counts,N,K,out_dtype", [
    ([100, 0, 37, 300, 1], 300, 256, torch.float32),
    ([0, 2100, 3, 0, 33], 1040, 512, torch.bfloat16),   # pairs
    ([513, 511, 1024, 0], 264, 128, torch.bfloat16),
])
def test_mx_grouped_jagged_m(fp8, counts, N, K, out_dtype):
    rng = np.random.default_rng(sum(counts))
    E, M = len(counts), sum(counts)
    A = W.normal_bf16((M, K), 1.0, 11)
    Wt = W.normal_bf16((E, N, K), 0.02, 12)
    ca, sa = oracle.mx_quantize_rows(bits(A), E4)
    cw, sw = oracle.mx_quantize_rows(bits(Wt).reshape(E * N, K), E4)
    cw, sw = cw.reshape(E, N, K), sw.reshape(E, N, K // 32)
    ends = W.ends_from_counts(counts)
    P = fp8.fp8_jagged_padded_rows(M, E)
    sfa = _padded_rows_sf(sa, ends, K, P)
    sfb = np.concatenate([mx_block(sw[e], K) for e in range(E)])
    out = torch.full((M, N), float("nan"), dtype=out_dtype, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp8.fp8_grouped_mm(upload_codes(ca, E4), upload_codes(cw, E4), _up(ends), _up(sfa), _up(sfb), out,
                       fp8.GROUPED_JAGGED_M, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rows = np.unique(np.concatenate([rng.choice(M, min(M, 48), replace=False), [0, M - 1], ends[ends < M]]))
    for r in rows:
        e = int(np.searchsorted(ends, r, side="right"))
        ref, absacc = oracle.gemm_mx(ca[r:r + 1], E4, cw[e], E4, sa[r:r + 1], sw[e])
        check_gemm(out[int(r)].unsqueeze(0), ref, absacc, out_dtype == torch.bfloat16)


@pytest.mark.parametrize("counts,N,Kd", [([40, 0, 200, 1, 130], 256, 192), ([0, 700, 300, 0], 384, 512),
                                         ([128, 128, 0], 200, 136)])
def test_mx_grouped_jagged_k(fp8, counts, N, Kd):
    """dW[e] = sum over segment e of dY^T X, both operands MX-quantized along the tokens of each
    segment (the oracle's segment-padded column codes and scales)."""
    E, M = len(counts), sum(counts)
    G = W.normal_bf16((M, N), 1e-3, 21)
    X = W.normal_bf16((M, Kd), 1.0, 22)
    ends = W.ends_from_counts(counts)
    gq, gs = oracle.mx_quantize_jagged_cols(bits(G), ends, E5)   # [N, Pu], [N, Pu / 32]
    xq, xs = oracle.mx_quantize_jagged_cols(bits(X), ends, E4)   # [Kd, Pu], [Kd, Pu / 32]
    Pu = gq.shape[1]
    P = fp8.fp8_jagged_padded_rows(M, E)
    gfull = np.zeros((N, P), np.uint8)
    gfull[:, :Pu] = gq
    xfull = np.zeros((Kd, P), np.uint8)
    xfull[:, :Pu] = xq
    gsf = np.full((N, P // 32), 127, np.uint8)
    gsf[:, :Pu // 32] = gs
    xsf = np.full((Kd, P // 32), 127, np.uint8)
    xsf[:, :Pu // 32] = xs
    out = torch.full((E, N, Kd), float("nan"), dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp8.fp8_grouped_mm(upload_codes(gfull, E5), upload_codes(xfull, E4), _up(ends), _up(mx_block(gsf, P)),
                       _up(mx_block(xsf, P)), out, fp8.GROUPED_JAGGED_K, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    _, _, pstarts, _ = oracle.mx_padded_segments(ends)
    padded = -(-np.asarray(counts) // 128) * 128
    for e in range(E):
        ps, pe = pstarts[e], pstarts[e] + padded[e]
        if padded[e] == 0:
            assert torch.count_nonzero(out[e]).item() == 0
            continue
        ref, absacc = oracle.gemm_mx(gq[:, ps:pe], E5, xq[:, ps:pe], E4, gs[:, ps // 32:pe // 32], xs[:, ps // 32:pe // 32])
        check_gemm(out[e], ref, absacc, False)


def test_mx_end_to_end_quantize_then_gemm(fp8):
    """The library's own MX quantize feeding its MX GEMM equals the oracle's quantize + GEMM
    (the codes and scales are compared bit for bit first)."""
    M, K, N = 1024, 512, 640
    x, w, _ = W.linear_inputs(M, K, N, seed=8, outliers=True)
    xq, _, xs, _ = fp8.mx_quantize_alloc(x.cuda(), 3, fp8.LAYOUT_ROW_MAJOR)
    wq, _, ws, _ = fp8.mx_quantize_alloc(w.cuda(), 3, fp8.LAYOUT_ROW_MAJOR)
    out = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    fp8.fp8_scaled_mm(xq, wq, xs, ws, out)
    torch.cuda.synchronize()
    cx, sx = oracle.mx_quantize_rows(bits(x), E4)
    cw, sw = oracle.mx_quantize_rows(bits(w), E4)
    assert np.array_equal(codes(xq), cx) and np.array_equal(mx_unblock(xs, M, K), sx)
    assert np.array_equal(codes(wq), cw) and np.array_equal(mx_unblock(ws, N, K), sw)
    ref, absacc = oracle.gemm_mx(cx, E4, cw, E4, sx, sw)
    check_gemm(out, ref, absacc, True)


# ---------------------------------------------------------------------------- Linear

@pytest.mark.parametrize("wgrad_name", ["WGRAD_FP8", "WGRAD_BF16"])
def test_mx_linear_fwd_bwd(fp8, wgrad_name):
    """The Linear with the MX recipe: x and W quantized to MX e4m3 in both layouts, dY to MX
    e5m2 in both layouts; y = x W^T, dX = dY W (W's blocks along N), dW = dY^T x (blocks along
    M) or the bf16 weight gradient."""
    wgrad = getattr(fp8, wgrad_name)
    M, K, N = 256, 384, 512
    x, w, dy = W.linear_inputs(M, K, N, seed=17, outliers=True)
    xd, wd, dyd = x.cuda(), w.cuda(), dy.cuda()
    saved, bufs = fp8.linear_saved_alloc(M, K, N, fp8.GRAN_MX, keep_xt=wgrad == fp8.WGRAD_FP8)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    dx = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    dw = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp8.fp8_linear_fwd(xd, wd, fp8.GRAN_MX, fp8.MM_FAST_ACCUM, y, saved, None, st)
    ws = torch.empty(max(fp8.fp8_workspace_size(fp8.OP_LINEAR_BWD, M, K, N, fp8.GRAN_MX, wgrad), 16),
                     dtype=torch.uint8, device="cuda")
    fp8.fp8_linear_bwd(dyd, saved, xd, wd, fp8.GRAN_MX, wgrad, dx, dw, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    x_q, x_inv, w_q, w_inv, xt_q, wt_q, xt_inv, wt_inv = bufs
    cx, sx = oracle.mx_quantize_rows(bits(x), E4)
    cw, sw = oracle.mx_quantize_rows(bits(w), E4)
    cwt, swt = oracle.mx_quantize_cols(bits(w), E4)   # W^T [K, N], blocks along N
    assert np.array_equal(codes(x_q), cx) and np.array_equal(mx_unblock(x_inv, M, K), sx)
    assert np.array_equal(codes(w_q), cw) and np.array_equal(mx_unblock(w_inv, N, K), sw)
    assert np.array_equal(codes(wt_q), cwt) and np.array_equal(mx_unblock(wt_inv, K, N), swt)
    ref, absacc = oracle.gemm_mx(cx, E4, cw, E4, sx, sw)
    check_gemm(y, ref, absacc, True)
    cdy, sdy = oracle.mx_quantize_rows(bits(dy), E5)
    ref, absacc = oracle.gemm_mx(cdy, E5, cwt, E4, sdy, swt)
    check_gemm(dx, ref, absacc, True)
    if wgrad == fp8.WGRAD_FP8:
        cxt, sxt = oracle.mx_quantize_cols(bits(x), E4)    # x^T [K, M], blocks along M
        assert np.array_equal(codes(xt_q), cxt) and np.array_equal(mx_unblock(xt_inv, K, M), sxt)
        cdyt, sdyt = oracle.mx_quantize_cols(bits(dy), E5)  # dY^T [N, M]
        ref, absacc = oracle.gemm_mx(cdyt, E5, cxt, E4, sdyt, sxt)
    else:
        ref, absacc = oracle.gemm_bf16(bits(dy), bits(x), a_trans=True, b_trans=True)
    check_gemm(dw, ref, absacc, True)
