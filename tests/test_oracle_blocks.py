"""Pins of the oracle's blockwise functions (CPU only).

Blockwise scaling is named by "FP8 training on AMD GPUs with TorchTitan and TorchAO" (section
"AMD FP8 format in TorchAO": a scale per fixed-size tile); the reading takes 1 x 128 tiles for
activations and gradients and 128 x 128 tiles for weights, each quantized by the recipe of "FP8
Training: Quantization, Autograd, Torchao" section 2. Pins: a hand-derived worked example
(tests/golden/), reductions to the already-pinned tensorwise / rowwise / columnwise recipes
(a tile equal to the tensor, a row or a column), edge tiles, and the blockwise GEMM against exact
rational arithmetic.
"""
import os
from fractions import Fraction

import numpy as np
import torch

import oracle
from oracle import E4M3, E5M2
import workloads as W

HERE = os.path.dirname(os.path.abspath(__file__))


def _bits(vals):
    return torch.tensor(vals, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def test_worked_example():
    d = {}
    with open(os.path.join(HERE, "golden", "blockwise_worked_example.txt")) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                k, v = line.split(":", 1)
                d[k.strip()] = v.split()
    row = np.zeros(256, np.float32)
    t0 = [float(v) for v in d["tile0"]]
    t1 = [float(v) for v in d["tile1"]]
    row[:len(t0)] = t0
    row[128:128 + len(t1)] = t1
    q, inv = oracle.quantize_blocks(_bits(row)[None, :], E4M3, 1, 128)
    assert q[0, :len(t0)].tolist() == [int(c, 16) for c in d["codes0"]]
    assert q[0, 128:128 + len(t1)].tolist() == [int(c, 16) for c in d["codes1"]]
    assert np.all(q[0, len(t0):128] == 0) and np.all(q[0, 128 + len(t1):] == 0)
    assert inv.view(np.uint32)[0].tolist() == [int(d["inv0"][0], 16), int(d["inv1"][0], 16)]


def test_reductions_to_pinned_recipes():
    x = W.bf16_bits(W.outlier_channels_bf16((96, 160), 1.0, 0.05, 40.0, seed=3))
    for fmt in (E4M3, E5M2):
        q, inv = oracle.quantize_blocks(x, fmt, 96, 160)        # one tile = the tensor
        qt, it = oracle.quantize_tensor(x, fmt)
        assert np.array_equal(q, qt) and np.array_equal(inv.ravel().view(np.uint32), it.view(np.uint32))
        q, inv = oracle.quantize_blocks(x, fmt, 1, 160)         # tiles = rows
        qr, ir = oracle.quantize_rows(x, fmt)
        assert np.array_equal(q, qr) and np.array_equal(inv.ravel().view(np.uint32), ir.view(np.uint32))
        q, inv = oracle.quantize_blocks(x, fmt, 96, 1)          # tiles = columns
        qc, ic = oracle.quantize_cols(x, fmt)
        assert np.array_equal(q, qc) and np.array_equal(inv.ravel().view(np.uint32), ic.view(np.uint32))


def test_tiles_and_edges():
    """Every tile (edge tiles included) equals the tensorwise recipe applied to that tile alone."""
    x = W.bf16_bits(W.normal_bf16((130, 300), 1.0, 4))
    q, inv = oracle.quantize_blocks(x, E4M3, 128, 128)
    assert inv.shape == (2, 3)
    for bi, (r0, r1) in enumerate([(0, 128), (128, 130)]):
        for bj, (c0, c1) in enumerate([(0, 128), (128, 256), (256, 300)]):
            qt, it = oracle.quantize_tensor(np.ascontiguousarray(x[r0:r1, c0:c1]), E4M3)
            assert np.array_equal(q[r0:r1, c0:c1], qt)
            assert inv[bi, bj].view(np.uint32) == it.view(np.uint32)[0]


def test_gemm_exact_rational():
    rng = np.random.default_rng(7)
    M, N, K = 3, 130, 256
    A = rng.integers(0, 256, (M, K)).astype(np.uint8)
    B = rng.integers(0, 256, (N, K)).astype(np.uint8)
    A[(A & 0x7F) == 0x7F] = 0x11
    B[(B & 0x7F) == 0x7F] = 0x22
    sA = (rng.random((M, 2)) * 4 + 0.25).astype(np.float32)
    sB = (rng.random((2, 2)) * 4 + 0.25).astype(np.float32)
    out, absacc = oracle.gemm_blockwise(A, E4M3, B, E4M3, sA, sB)
    dec = [Fraction(float(v)) for v in oracle.decode(np.arange(256, dtype=np.uint8), E4M3)[:127]] + [None] + \
          [Fraction(float(v)) for v in oracle.decode(np.arange(128, 256, dtype=np.uint8), E4M3)[:127]] + [None]
    for m in range(M):
        for n in range(0, N, 7):
            ref = sum(Fraction(float(sA[m, k // 128])) * Fraction(float(sB[n // 128, k // 128])) * dec[A[m, k]] * dec[B[n, k]]
                      for k in range(K))
            assert abs(out[m, n] - float(ref)) <= 1e-14 * absacc[m, n]
