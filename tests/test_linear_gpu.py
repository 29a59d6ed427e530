"""End-to-end FP8 Linear forward + backward through the C ABI against the oracle chain computed
from the same bf16 inputs ("FP8 Training: Quantization, Autograd, Torchao", sections 2, 4-6;
high-precision weight gradient: "FP8 training on AMD GPUs with TorchTitan and TorchAO",
Figure 1). Saved FP8 tensors and scales must be bit-exact; GEMM outputs within tolerance."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_util import bits, check_gemm, codes, f32_bits

pytestmark = pytest.mark.gpu
E4, E5 = oracle.E4M3, oracle.E5M2


@pytest.fixture(scope="module")
def fp8():
    import moe_grouped_gemm_absmax_gb300 as m
    return m


def _saved(fp8, M, K, N, gran):
    dev = "cuda"
    x_q = torch.empty((M, K), dtype=torch.float8_e4m3fn, device=dev)
    w_q = torch.empty((N, K), dtype=torch.float8_e4m3fn, device=dev)
    n_x, n_w = (1, 1) if gran == fp8.GRAN_TENSOR else (M, N)
    x_inv = torch.empty(n_x, dtype=torch.float32, device=dev)
    w_inv = torch.empty(n_w, dtype=torch.float32, device=dev)
    xt_q = wt_q = None
    if gran == fp8.GRAN_TENSOR:
        xt_q = torch.empty((K, M), dtype=torch.float8_e4m3fn, device=dev)
        wt_q = torch.empty((K, N), dtype=torch.float8_e4m3fn, device=dev)
    bufs = dict(x_q=x_q, x_inv=x_inv, w_q=w_q, w_inv=w_inv, xt_q=xt_q, wt_q=wt_q)
    return fp8.make_saved(x_q, x_inv, w_q, w_inv, xt_q, wt_q), bufs


def _run(fp8, x, w, dy, gran, wgrad, out_dtype):
    M, K = x.shape
    N = w.shape[0]
    saved, bufs = _saved(fp8, M, K, N, gran)
    xd, wd, dyd = x.cuda(), w.cuda(), dy.cuda()
    y = torch.empty((M, N), dtype=out_dtype, device="cuda")
    dx = torch.empty((M, K), dtype=out_dtype, device="cuda")
    dw = torch.empty((N, K), dtype=out_dtype, device="cuda")
    ws_f = torch.empty(max(fp8.fp8_workspace_size(fp8.OP_LINEAR_FWD, M, K, N, gran), 16), dtype=torch.uint8, device="cuda")
    ws_b = torch.empty(max(fp8.fp8_workspace_size(fp8.OP_LINEAR_BWD, M, K, N, gran, wgrad), 16), dtype=torch.uint8,
                       device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fp8.fp8_linear_fwd(xd, wd, gran, fp8.MM_FAST_ACCUM, y, saved, ws_f, st)
    fp8.fp8_linear_bwd(dyd, saved, xd, wd, gran, wgrad, dx, dw, ws_b, st)
    torch.cuda.synchronize()
    assert int(st.item()) == 0
    return y, dx, dw, bufs


@pytest.mark.parametrize("wgrad", [0, 1])
def test_tensorwise_linear_256x512(fp8, wgrad):
    """The single-Linear tensorwise workload: x [256,512] N(0,1), W [256,512] N(0,0.02),
    dY [256,256] N(0,1e-3); x, W -> e4m3, dY -> e5m2; fp32 outputs."""
    M, K, N = 256, 512, 256
    x, w, dy = W.linear_inputs(M, K, N, seed=0)
    y, dx, dw, b = _run(fp8, x, w, dy, fp8.GRAN_TENSOR, wgrad, torch.float32)
    xq, ix = oracle.quantize_tensor(bits(x), E4)
    wq, iw = oracle.quantize_tensor(bits(w), E4)
    dyq, idy = oracle.quantize_tensor(bits(dy), E5)
    assert np.array_equal(codes(b["x_q"]), xq) and np.array_equal(codes(b["xt_q"]), xq.T)
    assert np.array_equal(codes(b["w_q"]), wq) and np.array_equal(codes(b["wt_q"]), wq.T)
    assert np.array_equal(f32_bits(b["x_inv"]), ix.view(np.uint32))
    assert np.array_equal(f32_bits(b["w_inv"]), iw.view(np.uint32))
    ref, acc = oracle.gemm_fp8(xq, E4, wq, E4, ix, iw)
    check_gemm(y, ref, acc, False, 1e-2)  # forward runs with fast_accum
    ref, acc = oracle.gemm_fp8(dyq, E5, wq, E4, idy, iw, b_trans=True)
    check_gemm(dx, ref, acc, False)
    if wgrad == fp8.WGRAD_FP8:
        ref, acc = oracle.gemm_fp8(dyq, E5, xq, E4, idy, ix, a_trans=True, b_trans=True)
    else:
        ref, acc = oracle.gemm_bf16(bits(dy), bits(x), a_trans=True, b_trans=True)
    check_gemm(dw, ref, acc, False)


@pytest.mark.parametrize("wgrad", [0, 1])
@pytest.mark.parametrize("M,K,N", [(256, 512, 384), (272, 4096, 1040)])
def test_rowwise_linear(fp8, wgrad, M, K, N):
    """The Llama3-8B MLP-up recipe at reduced size: rowwise scales, x with 1% outlier channels
    x50, forward and grad-input in FP8, weight gradient in FP8 or bf16; bf16 outputs."""
    x, w, dy = W.linear_inputs(M, K, N, seed=3, outliers=True)
    y, dx, dw, b = _run(fp8, x, w, dy, fp8.GRAN_ROW, wgrad, torch.bfloat16)
    xq, ix = oracle.quantize_rows(bits(x), E4)
    wq, iw = oracle.quantize_rows(bits(w), E4)
    assert np.array_equal(codes(b["x_q"]), xq) and np.array_equal(codes(b["w_q"]), wq)
    assert np.array_equal(f32_bits(b["x_inv"]), ix.view(np.uint32))
    ref, acc = oracle.gemm_fp8(xq, E4, wq, E4, ix, iw)
    check_gemm(y, ref, acc, True, 1e-2)
    dyq, idy = oracle.quantize_rows(bits(dy), E5)
    wcq, iwc = oracle.quantize_cols(bits(w), E4)  # per input feature k, over the N rows of W
    ref, acc = oracle.gemm_fp8(dyq, E5, wcq, E4, idy, iwc, b_trans=True)
    check_gemm(dx, ref, acc, True)
    if wgrad == fp8.WGRAD_FP8:
        dycq, idyc = oracle.quantize_cols(bits(dy), E5)  # per output feature n, over the M tokens
        xcq, ixc = oracle.quantize_cols(bits(x), E4)    # per input feature k, over the M tokens
        ref, acc = oracle.gemm_fp8(dycq, E5, xcq, E4, idyc, ixc, a_trans=True, b_trans=True)
    else:
        ref, acc = oracle.gemm_bf16(bits(dy), bits(x), a_trans=True, b_trans=True)
    check_gemm(dw, ref, acc, True)
