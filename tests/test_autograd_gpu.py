"""The autograd wrapper: Fp8LinearFunction / Fp8Linear / swap_linears must produce exactly what
the C-ABI entry points produce on the same inputs (the wrapper only allocates and wires buffers;
the entry points themselves are checked against the oracle in test_linear_gpu.py)."""
import pytest
import torch

import workloads as W

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
    assert torch.equal(model[0](x.detach()), y_direct)
