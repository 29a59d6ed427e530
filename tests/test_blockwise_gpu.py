"""GPU parity of blockwise scaling (1 x 128 activation tiles, 128 x 128 weight tiles; "FP8 training
on AMD GPUs with TorchTitan and TorchAO", section "AMD FP8 format in TorchAO", with the tile
shapes of the reading in include/fp8lin.h) against the oracle: quantize codes and inverse scales
bit-exact; the blockwise GEMM (per-K-block partials promoted with sA * sB in fp32) within the
tolerance of "FP8 Training: Quantization, Autograd, Torchao" section 2 plus half a bf16 ulp."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_util import bits, check_gemm, codes, f32_bits, special_rows, upload_codes, upload_f32

pytestmark = pytest.mark.gpu

E4, E5 = oracle.E4M3, oracle.E5M2
TDT = {E4: 3, E5: 4}


@pytest.fixture(scope="module")
def fp8():
    import moe_grouped_gemm_absmax_gb300 as m
    return m


def _inputs(R, C, seed):
    x = W.outlier_channels_bf16((R, C), 1.0, 0.02, 60.0, seed).float()
    x[0, :128] = 0.0  # an all-zero tile row
    return x.to(torch.bfloat16)


# rows of 512-16384 elements run on the row-wise kernel's warp teams (1, 2 or 4 warps per row), the
# others on the tile kernel; the special rows probe ties, subnormals, zeros and an outlier per tile
@pytest.mark.parametrize("R,C,fmt", [(300, 384, E4), (128, 128, E5), (77, 256, E4), (300, 512, E4), (77, 4096, E5),
                                     (40, 8192, E4), (5, 16384, E5), (9, 16256, E4)])
def test_quantize_1x128(fp8, R, C, fmt):
    x = _inputs(R, C, R)
    sp = special_rows(C, 448.0 if fmt == E4 else 57344.0)
    x = torch.cat([x, sp]) if R > 16 else x
    q, _, inv, _ = fp8.blk_quantize_alloc(x.cuda(), TDT[fmt])
    torch.cuda.synchronize()
    qo, io = oracle.quantize_blocks(bits(x), fmt, 1, 128)
    assert np.array_equal(codes(q), qo) and np.array_equal(f32_bits(inv), io.view(np.uint32))


@pytest.mark.parametrize("R,C,fmt,layout", [(256, 384, E4, "both"), (130, 256, E5, "row"), (384, 128, E4, "col")])
def test_quantize_128x128(fp8, R, C, fmt, layout):
    x = _inputs(R, C, R + 1)
    lay = {"row": fp8.LAYOUT_ROW_MAJOR, "col": fp8.LAYOUT_COL_MAJOR, "both": fp8.LAYOUT_BOTH}[layout]
    q, qt, inv, inv_t = fp8.blk_quantize_alloc(x.cuda(), TDT[fmt], tile128=True, layout=lay)
    torch.cuda.synchronize()
    qo, io = oracle.quantize_blocks(bits(x), fmt, 128, 128)
    if q is not None:
        assert np.array_equal(codes(q), qo) and np.array_equal(f32_bits(inv), io.view(np.uint32))
    if qt is not None:
        assert np.array_equal(codes(qt), qo.T) and np.array_equal(f32_bits(inv_t), io.T.copy().view(np.uint32))


def _rand_codes(rng, shape):
    c = rng.integers(0, 256, shape).astype(np.uint8)
    c[(c & 0x7F) == 0x7F] = 0x33
    return c


@pytest.mark.parametrize("M,N,K,out_dtype", [(128, 256, 256, torch.float32), (300, 500, 384, torch.bfloat16),
                                             (4096, 2560, 512, torch.bfloat16), (2500, 3000, 1024, torch.float32)])
def test_blockwise_gemm(fp8, M, N, K, out_dtype):
    rng = np.random.default_rng(M + N)
    ca, cb = _rand_codes(rng, (M, K)), _rand_codes(rng, (N, K))
    sa = (rng.random((M, K // 128)) * 2 + 0.01).astype(np.float32)
    sb = (rng.random((-(-N // 128), K // 128)) * 2 + 0.01).astype(np.float32)
    out = torch.full((M, N), float("nan"), dtype=out_dtype, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp8.fp8_scaled_mm(upload_codes(ca, E4), upload_codes(cb, E4), upload_f32(sa), upload_f32(sb), out,
                      fp8.MM_BLOCKWISE, status=st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    rows = None if M <= 300 else np.unique(np.concatenate([rng.choice(M, 48, replace=False), [0, M - 1]]))
    ref, acc = oracle.gemm_blockwise(ca, E4, cb, E4, sa, sb, rows=rows)
    got = out if rows is None else out[torch.as_tensor(rows, device="cuda")]
    check_gemm(got, ref, acc, out_dtype == torch.bfloat16)


def test_blockwise_linear(fp8):
    """The Linear with the blockwise recipe: y = x W^T (x 1 x 128, W 128 x 128), dX = dY W (dY
    1 x 128, W's tiles transposed), dW in bf16."""
    M, K, N = 512, 384, 640
    x, w, dy = W.linear_inputs(M, K, N, seed=12, outliers=True)
    saved, bufs = fp8.linear_saved_alloc(M, K, N, fp8.GRAN_BLOCK_1x128, keep_xt=False)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    dx = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    dw = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    xd, wd, dyd = x.cuda(), w.cuda(), dy.cuda()
    fp8.fp8_linear_fwd(xd, wd, fp8.GRAN_BLOCK_1x128, fp8.MM_FAST_ACCUM, y, saved, None, st)
    ws = torch.empty(fp8.fp8_workspace_size(fp8.OP_LINEAR_BWD, M, K, N, fp8.GRAN_BLOCK_1x128, fp8.WGRAD_BF16),
                     dtype=torch.uint8, device="cuda")
    fp8.fp8_linear_bwd(dyd, saved, xd, wd, fp8.GRAN_BLOCK_1x128, fp8.WGRAD_BF16, dx, dw, ws, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    cx, ix = oracle.quantize_blocks(bits(x), E4, 1, 128)
    cw, iw = oracle.quantize_blocks(bits(w), E4, 128, 128)
    x_q, x_inv, w_q, w_inv, _, wt_q, _, wt_inv = bufs
    assert np.array_equal(codes(x_q), cx) and np.array_equal(f32_bits(x_inv), ix.view(np.uint32))
    assert np.array_equal(codes(w_q), cw) and np.array_equal(codes(wt_q), cw.T)
    assert np.array_equal(f32_bits(w_inv), iw.view(np.uint32)) and np.array_equal(f32_bits(wt_inv), iw.T.copy().view(np.uint32))
    ref, acc = oracle.gemm_blockwise(cx, E4, cw, E4, ix, iw)
    check_gemm(y, ref, acc, True)
    cdy, idy = oracle.quantize_blocks(bits(dy), E5, 1, 128)
    ref, acc = oracle.gemm_blockwise(cdy, E5, np.ascontiguousarray(cw.T), E4, idy, np.ascontiguousarray(iw.T))
    check_gemm(dx, ref, acc, True)
    ref, acc = oracle.gemm_bf16(bits(dy), bits(x), a_trans=True, b_trans=True)
    check_gemm(dw, ref, acc, True)
