"""Seeded synthetic inputs for the FP8 dynamic-scaling linear, shared by tests/ and bench.py.

This module only draws random numbers and rounds them to bf16; it holds none of the method's
arithmetic (no amax, scale, cast or GEMM). Shapes and value distributions follow the five
workloads the FP8 pages describe (dense Llama3-8B-shaped Linear, the column-wise backward
operand, DeepSeek-V3- and Llama4-shaped MoE layers), scaled down where a test needs the oracle
to finish in seconds.

Everything is generated in fp32 from a seeded torch generator, then rounded to bf16 (RNE) by
torch's own cast. Tensors are created on `device` (CPU by default; the full-size bench inputs
are drawn on the GPU because drawing 3.8 G values on the host takes minutes).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch


def _gen(seed: int, device) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed)
    return g


def normal_bf16(shape, std: float, seed: int, device="cpu") -> torch.Tensor:
    """~N(0, std^2) (std is the standard deviation), rounded to bf16."""
    g = _gen(seed, device)
    t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    t.mul_(std)
    return t.to(torch.bfloat16)


def outlier_channels_bf16(shape, std: float, frac: float, gain: float, seed: int, device="cpu"):
    """~N(0, std^2) with round(frac * C) seeded channels (columns) multiplied by `gain`."""
    R, C = shape
    g = _gen(seed, device)
    t = torch.randn(R, C, generator=g, device=device, dtype=torch.float32).mul_(std)
    n_out = max(1, int(round(frac * C)))
    gc = _gen(seed + 7919, "cpu")
    cols = torch.randperm(C, generator=gc)[:n_out].to(device)
    t[:, cols] *= gain
    return t.to(torch.bfloat16)


def column_gain_bf16(shape, std: float, log10_lo: float, log10_hi: float, seed: int, device="cpu"):
    """~N(0, std^2) times a per-column gain 10^U(lo, hi) (log-uniform)."""
    R, C = shape
    g = _gen(seed, device)
    t = torch.randn(R, C, generator=g, device=device, dtype=torch.float32).mul_(std)
    gc = _gen(seed + 104729, "cpu")
    u = torch.rand(C, generator=gc, dtype=torch.float64)
    gains = torch.pow(10.0, log10_lo + (log10_hi - log10_lo) * u).to(torch.float32).to(device)
    t.mul_(gains[None, :])
    return t.to(torch.bfloat16)


def zipf_counts(total: int, n_experts: int, s: float, n_forced_empty: int, seed: int,
                empty_first: bool = False, empty_last: bool = False) -> np.ndarray:
    """Per-expert row counts: p_r ~ r^-s over ranks given by a seeded permutation, counts ~
    Multinomial(total, p); then `n_forced_empty` seeded experts (plus expert 0 / the last one
    when asked) are emptied and their rows moved to the rank-1 expert."""
    rng = np.random.default_rng(seed)
    ranks = rng.permutation(n_experts) + 1
    p = ranks.astype(np.float64) ** (-s)
    p /= p.sum()
    counts = rng.multinomial(total, p).astype(np.int64)
    empty = set(rng.choice(n_experts, size=n_forced_empty, replace=False).tolist()) if n_forced_empty else set()
    if empty_first:
        empty.add(0)
    if empty_last:
        empty.add(n_experts - 1)
    top = int(np.argmin(ranks))  # rank-1 expert
    if top in empty:
        top = next(e for e in np.argsort(ranks) if e not in empty)
    for e in empty:
        counts[top] += counts[e]
        counts[e] = 0
    assert counts.sum() == total
    return counts


def dirichlet_counts(total: int, n_experts: int, alpha: float, seed: int) -> np.ndarray:
    rng = np.random.default_rng(seed)
    p = rng.dirichlet(np.full(n_experts, alpha))
    counts = rng.multinomial(total, p).astype(np.int64)
    return counts


def random_counts(total: int, n_experts: int, seed: int, n_empty: int = 0) -> np.ndarray:
    """Small-case routing: uniform-random multinomial with `n_empty` seeded empty experts."""
    rng = np.random.default_rng(seed)
    p = rng.random(n_experts) + 0.05
    empty = rng.choice(n_experts, size=n_empty, replace=False) if n_empty else []
    p[list(empty)] = 0.0
    p /= p.sum()
    return rng.multinomial(total, p).astype(np.int64)


def ends_from_counts(counts) -> np.ndarray:
    """Cumulative segment ends (int32), the offsets layout of the grouped entry points."""
    return np.cumsum(np.asarray(counts, dtype=np.int64)).astype(np.int32)


def bf16_bits(t: torch.Tensor) -> np.ndarray:
    """Raw bf16 bit patterns of a (CPU or device) bf16 tensor, as a host uint16 array."""
    return t.detach().contiguous().cpu().view(torch.int16).numpy().view(np.uint16)


# ------------------------------------------------------------------------------------------
# The five workloads, by name. Full sizes are what bench.py times; tests use scaled copies.

@dataclass
class Workload:
    name: str
    desc: str
    dims: dict = field(default_factory=dict)


WORKLOADS = {
    "linear-tensorwise-256x512": Workload(
        "linear-tensorwise-256x512",
        "single FP8 Linear fwd+bwd, tensorwise: x [256,512] N(0,1), W [256,512] N(0,0.02), "
        "dY [256,256] N(0,1e-3); x,W e4m3, dY e5m2; fp32 out",
        dict(M=256, K=512, N=256)),
    "llama3-8b-mlp-up": Workload(
        "llama3-8b-mlp-up",
        "Llama3-8B-shaped MLP-up Linear fwd+bwd, rowwise: x [8192,4096] N(0,1) with 1% channels "
        "x50, W [14336,4096] N(0,0.02), dY [8192,14336] N(0,1e-3); fwd+dX FP8 (e4m3/e5m2), dW bf16",
        dict(M=8192, K=4096, N=14336)),
    "llama3-8b-tensorwise-quant": Workload(
        "llama3-8b-tensorwise-quant",
        "tensorwise quantize with the dual output (row- and column-major codes) of the llama3-8b-mlp-up "
        "tensors: x [8192,4096] (1% channels x50) and W [14336,4096] to e4m3, dY [8192,14336] to e5m2",
        dict(M=8192, K=4096, N=14336)),
    "colwise-8192x14336": Workload(
        "colwise-8192x14336",
        "columnwise e5m2 quantize + column-major output of G [8192,14336] N(0,1e-3) x 10^U(-2,2) "
        "per column, plus rowwise e4m3 of X [8192,4096] N(0,1)",
        dict(R=8192, C=14336, RX=8192, CX=4096)),
    "dsv3-moe-fwd": Workload(
        "dsv3-moe-fwd",
        "DeepSeek-V3-shaped MoE grouped GEMM fwd: 256 experts, K=7168, N=2048, 131072 routed rows "
        "with Zipf(1.1) counts incl. 8 forced-empty experts; A N(0,1), W [256,2048,7168] N(0,0.02)",
        dict(E=256, M=131072, K=7168, N=2048)),
    "dsv3-moe-fwd-32e": Workload(
        "dsv3-moe-fwd-32e",
        "the dsv3-moe-fwd layer cut to 32 experts and 16384 routed rows (Zipf(1.1) counts, 1 forced-empty "
        "expert), same K and N: the size the full-metric profiler captures (about 2 GB on the device)",
        dict(E=32, M=16384, K=7168, N=2048)),
    "llama4-moe-fwdbwd": Workload(
        "llama4-moe-fwdbwd",
        "Llama4-shaped MoE grouped fwd+bwd: 16 experts, K=5120, N=8192, 8192 rows with "
        "Dirichlet(0.5) routing; A N(0,1), W [16,8192,5120] N(0,0.02), dY N(0,1e-3)",
        dict(E=16, M=8192, K=5120, N=8192)),
    "llama3-8b-dx-colquant-fused": Workload(
        "llama3-8b-dx-colquant-fused",
        "the llama3-8b-mlp-up grad-input GEMM dX = dY W (rowwise FP8 operands) with dX's column "
        "maxima from the GEMM epilogue, then dX quantized column-wise (e5m2, column-major) from them",
        dict(M=8192, K=4096, N=14336)),
    "llama3-8b-fwd-quant-fused": Workload(
        "llama3-8b-fwd-quant-fused",
        "the llama3-8b-mlp-up forward GEMM y = x W^T (rowwise FP8 operands) with y quantized in the GEMM "
        "epilogue (e4m3, 1 x 128 block scales: the next layer's activation operand), against the GEMM with "
        "a bf16 output followed by the 1 x 128 quantize",
        dict(M=8192, K=4096, N=14336)),
    "llama3-8b-mlp-up-blockwise": Workload(
        "llama3-8b-mlp-up-blockwise",
        "the llama3-8b-mlp-up Linear and inputs with blockwise scaling: x and dY in 1 x 128 tiles, W in "
        "128 x 128 tiles; fwd and dX blockwise FP8 GEMMs, dW bf16",
        dict(M=8192, K=4096, N=14336)),
    # the same shapes with MXFP8 (blocks of 32, E8M0 scales) for every operand of every GEMM
    "llama3-8b-mlp-up-mx": Workload(
        "llama3-8b-mlp-up-mx",
        "the llama3-8b-mlp-up Linear and inputs, MXFP8: x, W e4m3 and dY e5m2 quantized in both "
        "layouts from one read each; fwd, dX and dW all MX GEMMs",
        dict(M=8192, K=4096, N=14336)),
    "dsv3-moe-fwd-mx": Workload(
        "dsv3-moe-fwd-mx",
        "the dsv3-moe-fwd layer and inputs, MXFP8: A (segment-padded scales) and W[e] e4m3, MX "
        "grouped GEMM",
        dict(E=256, M=131072, K=7168, N=2048)),
    "llama4-moe-fwdbwd-mx": Workload(
        "llama4-moe-fwdbwd-mx",
        "the llama4-moe-fwdbwd layer and inputs, MXFP8: A, W[e] and dY each quantized once in "
        "both layouts; fwd, dX and dW MX grouped GEMMs",
        dict(E=16, M=8192, K=5120, N=8192)),
}


def linear_inputs(M: int, K: int, N: int, seed: int = 0, device="cpu", outliers: bool = False):
    """(x [M,K], W [N,K], dY [M,N]) bf16 for a dense Linear: x N(0,1) (optionally with 1% of
    channels x50), W N(0,0.02), dY N(0,1e-3)."""
    if outliers:
        x = outlier_channels_bf16((M, K), 1.0, 0.01, 50.0, seed, device)
    else:
        x = normal_bf16((M, K), 1.0, seed, device)
    W = normal_bf16((N, K), 0.02, seed + 1, device)
    dY = normal_bf16((M, N), 1e-3, seed + 2, device)
    return x, W, dY


def moe_inputs(E: int, M: int, K: int, N: int, counts, seed: int = 0, device="cpu",
               with_grad: bool = False):
    """(A [M,K] N(0,1), W [E,N,K] N(0,0.02), ends int32 [E], dY [M,N] N(0,1e-3) or None)."""
    A = normal_bf16((M, K), 1.0, seed, device)
    W = normal_bf16((E, N, K), 0.02, seed + 1, device)
    dY = normal_bf16((M, N), 1e-3, seed + 2, device) if with_grad else None
    return A, W, ends_from_counts(counts), dY


def dsv3_counts(seed: int = 0, empty_first=False, empty_last=False) -> np.ndarray:
    return zipf_counts(131072, 256, 1.1, 8, seed, empty_first, empty_last)


def dsv3_32e_counts(seed: int = 0) -> np.ndarray:
    return zipf_counts(16384, 32, 1.1, 1, seed)


def llama4_counts(seed: int = 0) -> np.ndarray:
    return dirichlet_counts(8192, 16, 0.5, seed)


def ceil_div(a: int, b: int) -> int:
    return -(-a // b)


def gemm_flops(M: int, N: int, K: int) -> float:
    return 2.0 * M * N * K

