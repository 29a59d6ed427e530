"""The autograd wrapper: Fp8LinearFunction / Fp8Linear / swap_linears ("FP8 Training:
Quantization, Autograd, Torchao", sections 5-6). Its forward output and both gradients are checked
against the oracle's chain computed from the same bf16 inputs (quantize by the recipe, then the
fp64 GEMM of the decoded codes), within the GEMM tolerance, and must also be bit-identical to
what the C-ABI entry points produce (the wrapper only allocates and wires buffers)."""
import numpy as np
import pytest
import torch

import oracle
import workloads as W
from tests.gpu_util import bits, check_gemm

E4, E5 = oracle.E4M3, oracle.E5M2

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def fp8():
    import moe_grouped_gemm_absmax_gb300 as m
    return m


def _direct(fp8, x, w, dy, gran, wgrad):
    M, K = x.shape
    N = w.shape[0]
    saved, _bufs = fp8.linear_saved_alloc(M, K, N, gran, keep_xt=wgrad == fp8.WGRAD_FP8)
    y = torch.empty((M, N), dtype=torch.bfloat16, device="cuda")
    dx = torch.empty((M, K), dtype=torch.bfloat16, device="cuda")
    dw = torch.empty((N, K), dtype=torch.bfloat16, device="cuda")
    wsf = torch.empty(max(fp8.fp8_workspace_size(fp8.OP_LINEAR_FWD, M, K, N, gran), 16), dtype=torch.uint8, device="cuda")
    wsb = torch.empty(max(fp8.fp8_workspace_size(fp8.OP_LINEAR_BWD, M, K, N, gran, wgrad), 16), dtype=torch.uint8,
                      device="cuda")
    fp8.fp8_linear_fwd(x, w, gran, fp8.MM_FAST_ACCUM, y, saved, wsf)
    fp8.fp8_linear_bwd(dy, saved, x, w, gran, wgrad, dx, dw, wsb)
    return y, dx, dw


def _oracle_linear(x, w, dy, gran_name, wgrad_name):
    """(reference, sum |a b|, tolerance) of y = x W^T, dX = dY W and dW = dY^T x by the oracle for
    the recipe of each granularity: the forward GEMM with fast accumulation (1e-2), the backward
    GEMMs with full accumulation (2e-3)."""
    xb, wb, dyb = bits(x.cpu()), bits(w.cpu()), bits(dy.cpu())
    if gran_name == "GRAN_ROW":
        xq, ix = oracle.quantize_rows(xb, E4)
        wq, iw = oracle.quantize_rows(wb, E4)
        y = oracle.gemm_fp8(xq, E4, wq, E4, ix, iw)
        dyq, idy = oracle.quantize_rows(dyb, E5)
        wcq, iwc = oracle.quantize_cols(wb, E4)  # per input feature k, over the N rows of W
        dx = oracle.gemm_fp8(dyq, E5, wcq, E4, idy, iwc, b_trans=True)
        if wgrad_name == "WGRAD_FP8":
            dycq, idyc = oracle.quantize_cols(dyb, E5)
            xcq, ixc = oracle.quantize_cols(xb, E4)
            dw = oracle.gemm_fp8(dycq, E5, xcq, E4, idyc, ixc, a_trans=True, b_trans=True)
    elif gran_name == "GRAN_TENSOR":
        xq, ix = oracle.quantize_tensor(xb, E4)
        wq, iw = oracle.quantize_tensor(wb, E4)
        dyq, idy = oracle.quantize_tensor(dyb, E5)
        y = oracle.gemm_fp8(xq, E4, wq, E4, ix, iw)
        dx = oracle.gemm_fp8(dyq, E5, wq, E4, idy, iw, b_trans=True)
        dw = oracle.gemm_fp8(dyq, E5, xq, E4, idy, ix, a_trans=True, b_trans=True)
    elif gran_name == "GRAN_MX":
        cx, sx = oracle.mx_quantize_rows(xb, E4)
        cw, sw = oracle.mx_quantize_rows(wb, E4)
        y = oracle.gemm_mx(cx, E4, cw, E4, sx, sw)
        cdy, sdy = oracle.mx_quantize_rows(dyb, E5)
        cwt, swt = oracle.mx_quantize_cols(wb, E4)  # W^T [K, N], blocks along N
        dx = oracle.gemm_mx(cdy, E5, cwt, E4, sdy, swt)
        if wgrad_name == "WGRAD_FP8":
            cxt, sxt = oracle.mx_quantize_cols(xb, E4)
            cdyt, sdyt = oracle.mx_quantize_cols(dyb, E5)
            dw = oracle.gemm_mx(cdyt, E5, cxt, E4, sdyt, sxt)
    else:  # GRAN_BLOCK_1x128: x and dY in 1 x 128 tiles, W in 128 x 128 tiles
        cx, ix = oracle.quantize_blocks(xb, E4, 1, 128)
        cw, iw = oracle.quantize_blocks(wb, E4, 128, 128)
        y = oracle.gemm_blockwise(cx, E4, cw, E4, ix, iw)
        cdy, idy = oracle.quantize_blocks(dyb, E5, 1, 128)
        dx = oracle.gemm_blockwise(cdy, E5, np.ascontiguousarray(cw.T), E4, idy, np.ascontiguousarray(iw.T))
    if wgrad_name == "WGRAD_BF16":
        dw = oracle.gemm_bf16(dyb, xb, a_trans=True, b_trans=True)
    return (y[0], y[1], 1e-2), (dx[0], dx[1], 2e-3), (dw[0], dw[1], 2e-3)


@pytest.mark.parametrize("gran_name,wgrad_name", [("GRAN_ROW", "WGRAD_BF16"), ("GRAN_ROW", "WGRAD_FP8"),
                                                  ("GRAN_TENSOR", "WGRAD_FP8"), ("GRAN_MX", "WGRAD_FP8"),
                                                  ("GRAN_MX", "WGRAD_BF16"), ("GRAN_BLOCK_1x128", "WGRAD_BF16")])
def test_function_matches_entry_points(fp8, gran_name, wgrad_name):
    from moe_grouped_gemm_absmax_gb300.autograd import Fp8LinearFunction
    gran, wgrad = getattr(fp8, gran_name), getattr(fp8, wgrad_name)
    x, w, dy = W.linear_inputs(512, 256, 384, seed=31, device="cuda", outliers=True)
    xr = x.reshape(4, 128, 256).clone().requires_grad_(True)  # a leading batch dimension
    wr = w.clone().requires_grad_(True)
    y = Fp8LinearFunction.apply(xr, wr, gran, wgrad)
    y.backward(dy.reshape(4, 128, 384))
    y0, dx0, dw0 = _direct(fp8, x, w, dy, gran, wgrad)
    assert y.shape == (4, 128, 384) and y.dtype == torch.bfloat16
    got = (y.detach().reshape(512, 384), xr.grad.reshape(512, 256), wr.grad)
    for g, (ref, acc, tol) in zip(got, _oracle_linear(x, w, dy, gran_name, wgrad_name)):
        check_gemm(g, ref, acc, True, tol)
    assert torch.equal(y.reshape(512, 384), y0)
    assert torch.equal(xr.grad.reshape(512, 256), dx0)
    assert torch.equal(wr.grad, dw0)


def test_swap_linears_in_a_model(fp8):
    from moe_grouped_gemm_absmax_gb300.autograd import Fp8Linear, swap_linears
    torch.manual_seed(0)
    model = torch.nn.Sequential(
        torch.nn.Linear(256, 512, bias=False), torch.nn.GELU(), torch.nn.Linear(512, 256, bias=False),
        torch.nn.Linear(256, 8, bias=True),  # not swapped: bias, and an output dim the filter rejects
    ).cuda().to(torch.bfloat16)
    names = swap_linears(model, module_filter=lambda fqn, lin: lin.out_features >= 16)
    assert names == ["0", "2"]
    assert isinstance(model[0], Fp8Linear) and isinstance(model[2], Fp8Linear)
    assert isinstance(model[3], torch.nn.Linear)
    x = W.normal_bf16((256, 256), 1.0, 41, device="cuda").requires_grad_(True)
    out = model(x)
    out.float().pow(2).mean().backward()
    for p in model.parameters():
        assert p.grad is not None and torch.isfinite(p.grad.float()).all()
    # the first layer's output equals the entry point's forward on the same inputs
    y_direct, _, _ = _direct(fp8, x.detach(), model[0].weight.detach(), torch.zeros((256, 512), dtype=torch.bfloat16,
                                                                                    device="cuda"),
                             fp8.GRAN_ROW, fp8.WGRAD_BF16)
    y0 = model[0](x.detach())
    assert torch.equal(y0, y_direct)
    # and the oracle's rowwise forward on the same bf16 inputs
    xq, ix = oracle.quantize_rows(bits(x.detach().cpu()), E4)
    wq, iw = oracle.quantize_rows(bits(model[0].weight.detach().cpu()), E4)
    ref, acc = oracle.gemm_fp8(xq, E4, wq, E4, ix, iw)
    check_gemm(y0, ref, acc, True, 1e-2)
