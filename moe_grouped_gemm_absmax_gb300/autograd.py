"""A thin training-code wrapper over the C ABI: a torch.autograd.Function for the FP8 Linear and a
module swap in the style of the pages' Float8Linear ("FP8 Training: Quantization, Autograd,
Torchao", sections 5-6: the Linear keeps a bf16 weight, quantizes x and W in the forward pass,
dY in the backward pass, and returns bf16).

Every step runs in the library's kernels through fp8_linear_fwd / fp8_linear_bwd; this module only
allocates the caller-owned buffers (FP8 copies, inverse scales, workspaces) with PyTorch and wires
them into autograd. No bias: the pages' hot path is the bias-free matmul, and a bias would add a
non-FP8 step."""
import torch

from . import (GRAN_BLOCK_1x128, GRAN_MX, GRAN_ROW, GRAN_TENSOR, MM_FAST_ACCUM, OP_LINEAR_BWD, OP_LINEAR_FWD, WGRAD_BF16,
               WGRAD_FP8, fp8_linear_bwd, fp8_linear_fwd, fp8_workspace_size, linear_saved_alloc, make_saved)


def _workspace(nbytes, device):
    return torch.empty(max(int(nbytes), 16), dtype=torch.uint8, device=device)


class Fp8LinearFunction(torch.autograd.Function):
    """y = x W^T in FP8 (forward with fast accumulation, as the pages' recipe does), dX and dW in
    the backward pass; x [..., K] bf16, W [N, K] bf16 -> y [..., N] bf16."""

    @staticmethod
    def forward(ctx, x, weight, granularity=GRAN_ROW, wgrad_mode=WGRAD_BF16):
        if x.dtype != torch.bfloat16 or weight.dtype != torch.bfloat16:
            raise TypeError("Fp8LinearFunction takes bf16 x and weight")
        K = x.shape[-1]
        N = weight.shape[0]
        x2 = x.reshape(-1, K).contiguous()
        w = weight.contiguous()
        M = x2.shape[0]
        dev = x.device
        saved, bufs = linear_saved_alloc(M, K, N, granularity, keep_xt=wgrad_mode == WGRAD_FP8, device=dev)
        y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        fp8_linear_fwd(x2, w, granularity, MM_FAST_ACCUM, y, saved,
                       _workspace(fp8_workspace_size(OP_LINEAR_FWD, M, K, N, granularity), dev))
        # the FP8 copies and scales for the backward pass (absent ones as empty placeholders)
        ctx.save_for_backward(x2, w, *(b if b is not None else x2.new_empty(0) for b in bufs))
        ctx.present = tuple(b is not None for b in bufs)
        ctx.granularity, ctx.wgrad_mode, ctx.x_shape = granularity, wgrad_mode, x.shape
        return y.reshape(*x.shape[:-1], N)

    @staticmethod
    def backward(ctx, dy):
        x2, w, *bufs = ctx.saved_tensors
        bufs = [b if keep else None for b, keep in zip(bufs, ctx.present)]
        saved = make_saved(*bufs)
        M, K = x2.shape
        N = w.shape[0]
        dy2 = dy.reshape(-1, N).to(torch.bfloat16).contiguous()
        dx = torch.empty((M, K), dtype=torch.bfloat16, device=dy.device) if ctx.needs_input_grad[0] else None
        dw = torch.empty((N, K), dtype=torch.bfloat16, device=dy.device) if ctx.needs_input_grad[1] else None
        ws = _workspace(fp8_workspace_size(OP_LINEAR_BWD, M, K, N, ctx.granularity, ctx.wgrad_mode), dy.device)
        fp8_linear_bwd(dy2, saved, x2, w, ctx.granularity, ctx.wgrad_mode, dx, dw, ws)
        return (dx.reshape(ctx.x_shape) if dx is not None else None), dw, None, None


class Fp8Linear(torch.nn.Module):
    """Drop-in for a bias-free torch.nn.Linear: the weight stays bf16; the matmuls run in FP8
    (granularity GRAN_TENSOR, GRAN_ROW, GRAN_MX or GRAN_BLOCK_1x128; MX and blockwise need
    dimensions that are multiples of 128, blockwise a bf16 weight gradient)."""

    def __init__(self, in_features, out_features, granularity=GRAN_ROW, wgrad_mode=WGRAD_BF16, weight=None,
                 device=None):
        super().__init__()
        if in_features % 16 or out_features % 16:
            raise ValueError("FP8 GEMM operands need in_features and out_features divisible by 16")
        self.in_features, self.out_features = in_features, out_features
        self.granularity, self.wgrad_mode = granularity, wgrad_mode
        if weight is None:
            weight = torch.nn.Parameter(torch.empty((out_features, in_features), dtype=torch.bfloat16, device=device))
            torch.nn.init.kaiming_uniform_(weight, a=5 ** 0.5)
        self.weight = weight

    def forward(self, x):
        return Fp8LinearFunction.apply(x.to(torch.bfloat16), self.weight, self.granularity, self.wgrad_mode)

    def extra_repr(self):
        g = {GRAN_ROW: "row", GRAN_TENSOR: "tensor", GRAN_MX: "mx", GRAN_BLOCK_1x128: "blockwise"}[self.granularity]
        w = {WGRAD_BF16: "bf16", WGRAD_FP8: "fp8"}[self.wgrad_mode]
        return f"in_features={self.in_features}, out_features={self.out_features}, scaling={g}, wgrad={w}"


def swap_linears(module, granularity=GRAN_ROW, wgrad_mode=WGRAD_BF16, module_filter=None):
    """Replace, in place, every bias-free bf16 torch.nn.Linear child (recursively) whose shape the
    FP8 GEMMs accept and that `module_filter(fqn, linear)` admits, by an Fp8Linear that shares
    its weight Parameter. Returns the names of the swapped modules."""
    swapped = []

    def visit(mod, prefix):
        for name, child in list(mod.named_children()):
            fqn = f"{prefix}.{name}" if prefix else name
            ok = (isinstance(child, torch.nn.Linear) and child.bias is None and child.weight.dtype == torch.bfloat16
                  and child.in_features % 16 == 0 and child.out_features % 16 == 0
                  and (module_filter is None or module_filter(fqn, child)))
            if ok:
                setattr(mod, name, Fp8Linear(child.in_features, child.out_features, granularity, wgrad_mode,
                                             weight=child.weight))
                swapped.append(fqn)
            else:
                visit(child, fqn)

    visit(module, "")
    return swapped
