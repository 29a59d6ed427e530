"""Pins of the oracle's MXFP8 functions against facts fixed outside them (CPU only).

MXFP8 is named by "FP8 training on AMD GPUs with TorchTitan and TorchAO" (section "AMD FP8
format in TorchAO": a scale per group stored alongside the data; "Summary and Next Steps"); the
block of 32, the E8M0 scale and the rule X = 2^(floor(log2 amax) - emax_elem) come from the OCP
Microscaling Formats (MX) specification v1.0. Each test pins one function to something other
than itself: hand-derived worked examples (tests/golden/), the range property that defines the
scale rule, torch's own CPU float8 conversion (a library routine) applied to x / X, exact
rational brute force on small GEMMs, and invariants (oddness, block locality, exact scaling by
powers of two).
"""
import os
from fractions import Fraction

import numpy as np
import pytest
import torch

import oracle
from oracle import E4M3, E5M2
import workloads as W

HERE = os.path.dirname(os.path.abspath(__file__))
TORCH_FP8 = {E4M3: torch.float8_e4m3fn, E5M2: torch.float8_e5m2}
QMAX = {E4M3: 448.0, E5M2: 57344.0}
EMAX = {E4M3: 8, E5M2: 15}  # exponent of the largest normal: 448 = 1.75 * 2^8, 57344 = 1.75 * 2^15


def bf16_bits(values):
    return torch.tensor(values, dtype=torch.float32).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def bits_to_f32(b):
    return (np.asarray(b, np.uint32) << 16).view(np.float32)


def _expand(tokens, conv):
    out = []
    for t in tokens:
        if "*" in t:
            v, n = t.split("*")
            out += [conv(v)] * int(n)
        else:
            out.append(conv(t))
    return out


def _read_golden():
    cases, cur = [], None
    with open(os.path.join(HERE, "golden", "mx_worked_examples.txt")) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, _, rest = line.partition(" ")
            if key == "case":
                name, fmt = rest.split()
                cur = {"name": name, "fmt": E4M3 if fmt == "e4m3" else E5M2}
                cases.append(cur)
            else:
                vals = rest.split(":", 1)[1].split()
                if key == "x":
                    cur["x"] = _expand(vals, float)
                elif key == "codes":
                    cur["codes"] = _expand(vals, lambda s: int(s, 16))
                else:
                    cur["scales"] = [int(s, 16) for s in vals]
    return cases


def test_golden_worked_examples():
    cases = _read_golden()
    assert len(cases) == 5
    for c in cases:
        x = bf16_bits(c["x"])
        assert np.array_equal(bits_to_f32(x), np.asarray(c["x"], np.float32)), c["name"]  # inputs are bf16-exact
        q, sc = oracle.mx_quantize_rows(x[None, :], c["fmt"])
        assert q[0].tolist() == c["codes"], c["name"]
        assert sc[0].tolist() == c["scales"], c["name"]


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_scale_rule_over_every_bf16_amax(fmt):
    """For every positive finite bf16 amax, X = 2^(code - 127) is the power of two that puts
    amax / X in [2^emax, 2^(emax + 1)), unless that power is below 2^-127 (code 0)."""
    pos = np.arange(1, 0x7F80, dtype=np.uint32)  # +min subnormal .. +max finite
    amax = bits_to_f32(pos)
    codes = np.array([oracle.mx_scale(float(a), fmt) for a in amax])
    assert codes.max() <= 254
    ratio = amax.astype(np.float64) / np.ldexp(1.0, codes.astype(np.int64) - 127)
    lo, hi = 2.0 ** EMAX[fmt], 2.0 ** (EMAX[fmt] + 1)
    clamped = codes == 0
    assert np.all((ratio[~clamped] >= lo) & (ratio[~clamped] < hi))
    assert np.all(ratio[clamped] < hi)  # a clamped scale only ever gets smaller ratios
    assert clamped.any() and not clamped[-1]
    # code 1 (X = 2^-126) starts exactly at amax = 2^(-126 + emax); below it everything is code 0
    assert amax[~clamped][0] == np.float32(2.0 ** (-126 + EMAX[fmt]))
    assert oracle.mx_scale(0.0, fmt) == 0
    assert oracle.mx_scale(float("inf"), fmt) == 0xFF and oracle.mx_scale(float("nan"), fmt) == 0xFF


def test_e8m0_decode():
    v = oracle.e8m0_decode(np.arange(255, dtype=np.uint8))
    assert np.array_equal(v, np.ldexp(1.0, np.arange(255) - 127))
    assert np.isnan(oracle.e8m0_decode([255])[0])


def _mx_inputs(R, C, seed):
    """Normal values with outlier blocks, an all-zero block and a block of tiny values."""
    x = W.normal_bf16((R, C), 1.0, seed).float().numpy()
    rng = np.random.default_rng(seed + 1)
    x[rng.integers(0, R, 8), rng.integers(0, C, 8)] *= 300.0
    x[0, :32] = 0.0
    x[min(1, R - 1), 32:64] *= 2.0 ** -125
    return bf16_bits(x)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_codes_match_torch_cast_of_scaled_block(fmt):
    """codes = torch's RNE float8 cast of clamp(x / X), X from the block's amax by the rule."""
    x = _mx_inputs(24, 256, 7 + fmt)
    q, sc = oracle.mx_quantize_rows(x, fmt)
    xf = bits_to_f32(x).astype(np.float64).reshape(24, 8, 32)
    amax = np.abs(xf).max(axis=2)
    assert np.array_equal(sc, np.array([[oracle.mx_scale(float(a), fmt) for a in row] for row in amax], np.uint8))
    X = np.ldexp(1.0, sc.astype(np.int64) - 127)[:, :, None]
    v = np.clip(xf / X, -QMAX[fmt], QMAX[fmt]).astype(np.float32)  # exact: x / X is x times a power of two
    ref = torch.from_numpy(v.reshape(24, 256)).to(TORCH_FP8[fmt]).view(torch.uint8).numpy()
    assert np.array_equal(q, ref)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_quantize_invariants(fmt):
    x = _mx_inputs(16, 128, 3)
    q, sc = oracle.mx_quantize_rows(x, fmt)
    # oddness: q(-x) = q(x) with the sign bit flipped; same scales
    qn, scn = oracle.mx_quantize_rows(x ^ np.uint16(0x8000), fmt)
    assert np.array_equal(qn, q ^ np.uint8(0x80)) and np.array_equal(scn, sc)
    # block locality: changing one block changes nothing outside it
    x2 = x.copy()
    x2[5, 64:96] = bf16_bits(np.full(32, 1000.0))
    q2, sc2 = oracle.mx_quantize_rows(x2, fmt)
    mask = np.ones_like(q, bool)
    mask[5, 64:96] = False
    assert np.array_equal(q2[mask], q[mask])
    assert sc2[5, 2] != sc[5, 2] and np.array_equal(np.delete(sc2.ravel(), 5 * 4 + 2), np.delete(sc.ravel(), 5 * 4 + 2))
    # scaling a block by 2^j shifts its scale code by j and leaves its codes alone
    x3 = bf16_bits(bits_to_f32(x[6:7]) * np.float32(2.0 ** 20))
    q3, sc3 = oracle.mx_quantize_rows(x3, fmt)
    assert np.array_equal(q3, q[6:7]) and np.array_equal(sc3.astype(int), sc[6:7].astype(int) + 20)
    # the largest element of every unclamped block lands in [2^emax, fp8_max]
    dec = np.abs(oracle.decode(q, fmt)).reshape(16, 4, 32).max(axis=2)
    live = (sc > 0) & (np.abs(bits_to_f32(x)).reshape(16, 4, 32).max(axis=2) > 0)
    assert np.all(dec[live] >= 2.0 ** EMAX[fmt]) and np.all(dec <= QMAX[fmt])


def test_quantize_rejects_partial_blocks():
    with pytest.raises(ValueError):
        oracle.mx_quantize_rows(np.zeros((2, 48), np.uint16), E4M3)


def test_columns_and_jagged_segments():
    x = _mx_inputs(96, 64, 11)
    qt, sct = oracle.mx_quantize_cols(x, E4M3)
    assert qt.shape == (64, 96) and sct.shape == (64, 3)
    # column c, block b covers rows 32b .. 32b + 31 of column c
    for c, b in [(0, 0), (5, 2), (63, 1)]:
        amax = np.abs(bits_to_f32(x[32 * b:32 * b + 32, c])).max()
        assert sct[c, b] == oracle.mx_scale(float(amax), E4M3)
    # jagged: segments of 40, 0 and 56 rows; blocks restart at each segment, padding is zero
    ends = [40, 40, 96]
    qj, scj = oracle.mx_quantize_jagged_cols(x, ends, E4M3)
    assert qj.shape == (64, 256) and scj.shape == (64, 8)
    amax_tail = np.abs(bits_to_f32(x[32:40, 7])).max()  # the second block of segment 0 holds 8 rows
    assert scj[7, 1] == oracle.mx_scale(float(amax_tail), E4M3)
    assert np.all(scj[:, 2:4] == 0) and np.all(qj[:, 40:128] == 0)  # padding of segment 0
    q2, s2 = oracle.mx_quantize_cols(np.concatenate([x[40:96], np.zeros((8, 64), np.uint16)]), E4M3)
    assert np.array_equal(qj[:, 128:192], q2) and np.array_equal(scj[:, 4:6], s2)


def _rational_mx_gemm(A, fa, B, fb, sA, sB):
    M, K = A.shape
    N = B.shape[0]
    codes = np.arange(256, dtype=np.uint8)
    da = [None if not np.isfinite(v) else Fraction(float(v)) for v in oracle.decode(codes, fa)]
    db = [None if not np.isfinite(v) else Fraction(float(v)) for v in oracle.decode(codes, fb)]
    out = np.empty((M, N))
    for m in range(M):
        for n in range(N):
            s = Fraction(0)
            for k in range(K):
                s += Fraction(2) ** (int(sA[m, k // 32]) + int(sB[n, k // 32]) - 254) * da[A[m, k]] * db[B[n, k]]
            out[m, n] = float(s)
    return out


def _finite_codes(rng, shape, fmt):
    c = rng.integers(0, 256, shape).astype(np.uint8)
    nan = (c & 0x7F) == 0x7F if fmt == E4M3 else (c & 0x7C) == 0x7C
    c[nan] = 0x10
    return c


@pytest.mark.parametrize("fa,fb", [(E4M3, E4M3), (E5M2, E4M3)])
def test_gemm_exact_rational(fa, fb):
    rng = np.random.default_rng(5)
    M, N, K = 3, 4, 96
    A, B = _finite_codes(rng, (M, K), fa), _finite_codes(rng, (N, K), fb)
    sA = rng.integers(110, 140, (M, 3)).astype(np.uint8)
    sB = rng.integers(110, 140, (N, 3)).astype(np.uint8)
    out, absacc = oracle.gemm_mx(A, fa, B, fb, sA, sB)
    ref = _rational_mx_gemm(A, fa, B, fb, sA, sB)
    assert np.all(np.abs(out - ref) <= 1e-14 * absacc)
    # rows subset
    out2, _ = oracle.gemm_mx(A, fa, B, fb, sA, sB, rows=[2, 0])
    assert np.array_equal(out2, out[[2, 0]])


def test_gemm_unit_scales_reduce_to_scaled_gemm():
    """With every E8M0 code 127 (X = 1) the MX GEMM is the plain FP8 GEMM with unit scales;
    raising one row's codes by j multiplies that row by 2^j exactly."""
    rng = np.random.default_rng(9)
    A, B = _finite_codes(rng, (8, 128), E4M3), _finite_codes(rng, (16, 128), E4M3)
    ones_a, ones_b = np.full((8, 4), 127, np.uint8), np.full((16, 4), 127, np.uint8)
    mx, _ = oracle.gemm_mx(A, E4M3, B, E4M3, ones_a, ones_b)
    ref, _ = oracle.gemm_fp8(A, E4M3, B, E4M3, np.float32(1.0), np.float32(1.0))
    assert np.array_equal(mx, ref)
    sa = ones_a.copy()
    sa[3] += 5
    mx2, _ = oracle.gemm_mx(A, E4M3, B, E4M3, sa, ones_b)
    assert np.array_equal(mx2[3], ref[3] * 32.0) and np.array_equal(np.delete(mx2, 3, 0), np.delete(ref, 3, 0))
    # a scale of block b touches only k in [32b, 32b + 32): zero that slice of A, then any
    # code there changes nothing
    A0 = A.copy()
    A0[:, 64:96] = 0
    sb = ones_b.copy()
    sb[:, 2] = 3
    r1, _ = oracle.gemm_mx(A0, E4M3, B, E4M3, ones_a, ones_b)
    r2, _ = oracle.gemm_mx(A0, E4M3, B, E4M3, ones_a, sb)
    assert np.array_equal(r1, r2)
