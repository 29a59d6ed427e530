"""Pins of the CPU oracle against facts fixed outside it (CPU only, no GPU).

Each test pins one oracle function to something other than itself: closed forms of the two
FP8 formats, torch's own CPU float8 conversions (a library routine), an independent
nearest-value search, exact rational brute force on tiny GEMMs, numpy matmul, hand-derived
worked examples (tests/golden/), and invariants of the recipe (oddness, amax -> fp8_max,
rank-1 agreement, error bounds).

Sources: "FP8 Training: Quantization, Autograd, Torchao" sections 2-5; "FP8 training on AMD
GPUs with TorchTitan and TorchAO", "Scaling FP8 to MoE Architectures" and Figure 3.
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


def torch_decode(codes, fmt):
    return torch.from_numpy(np.asarray(codes, np.uint8)).view(TORCH_FP8[fmt]).to(torch.float64).numpy()


def f32_from_bits(b):
    return np.asarray(b, np.uint32).view(np.float32)


# --------------------------------------------------------------------------------------------
# Formats (section 3 of the nanochat FP8 page)

@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_decode_all_codes_match_torch(fmt):
    codes = np.arange(256, dtype=np.uint8)
    ours = oracle.decode(codes, fmt)
    ref = torch_decode(codes, fmt)
    both_nan = np.isnan(ours) & np.isnan(ref)
    assert np.all(both_nan | (ours == ref))
    assert np.array_equal(np.isnan(ours), np.isnan(ref))
    # signs of zeros
    assert np.signbit(ours[0x80]) and not np.signbit(ours[0x00])


def test_decode_closed_forms():
    assert oracle.fp8_max(E4M3) == 448.0
    assert oracle.fp8_max(E5M2) == 57344.0
    assert oracle.decode([0x7E], E4M3)[0] == 448.0
    assert oracle.decode([0xFE], E4M3)[0] == -448.0
    assert np.isnan(oracle.decode([0x7F], E4M3)[0]) and np.isnan(oracle.decode([0xFF], E4M3)[0])
    assert oracle.decode([0x01], E4M3)[0] == 2.0 ** -9       # smallest subnormal
    assert oracle.decode([0x08], E4M3)[0] == 2.0 ** -6       # smallest normal
    assert oracle.decode([0x7B], E5M2)[0] == 57344.0
    assert oracle.decode([0x01], E5M2)[0] == 2.0 ** -16
    assert oracle.decode([0x04], E5M2)[0] == 2.0 ** -14
    assert np.isinf(oracle.decode([0x7C], E5M2)[0])
    for c in (0x7D, 0x7E, 0x7F):
        assert np.isnan(oracle.decode([c], E5M2)[0])
    # positive finite codes are strictly increasing
    for fmt, last in ((E4M3, 0x7E), (E5M2, 0x7B)):
        v = oracle.decode(np.arange(last + 1), fmt)
        assert np.all(np.diff(v) > 0)


def _structured_f32(fmt):
    """fp32 values in [-qmax, qmax] that exercise every rounding position of the target: each
    fp32 exponent from 0 to that of qmax, every top-8 mantissa pattern, and low bits at the
    interesting points (0, 1, tie-1, tie, tie+1, all ones)."""
    top_exp = 127 + (8 if fmt == E4M3 else 15)
    exps = np.arange(0, top_exp + 1, dtype=np.uint32)
    tops = np.arange(256, dtype=np.uint32) << 15
    lows = np.array([0, 1, 0x3FFF, 0x4000, 0x4001, 0x7FFF, 0x1234, 0x6543], np.uint32)
    bits = (exps[:, None, None] << 23) | tops[None, :, None] | lows[None, None, :]
    bits = bits.reshape(-1)
    bits = np.concatenate([bits, bits | np.uint32(0x80000000)])
    v = f32_from_bits(bits)
    return v[np.abs(v) <= QMAX[fmt]]


def _random_f32(fmt, n, seed):
    rng = np.random.default_rng(seed)
    bits = rng.integers(0, 2 ** 32, size=n, dtype=np.uint64).astype(np.uint32)
    v = f32_from_bits(bits)
    return v[np.isfinite(v) & (np.abs(v) <= QMAX[fmt])]


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_encode_matches_torch_cast(fmt):
    v = np.concatenate([_structured_f32(fmt), _random_f32(fmt, 3_000_000, 11 + fmt)])
    ours = oracle.encode(v, fmt)
    ref = torch.from_numpy(v).to(TORCH_FP8[fmt]).view(torch.uint8).numpy()
    bad = np.nonzero(ours != ref)[0]
    assert bad.size == 0, [(float(v[i]), hex(ours[i]), hex(ref[i])) for i in bad[:8]]


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_encode_is_nearest_ties_even(fmt):
    """Independent route: nearest value among all finite codes, ties to the even code."""
    codes = np.arange(0, 0x7F if fmt == E4M3 else 0x7C, dtype=np.uint8)  # +0 .. +max
    vals = torch_decode(codes, fmt)
    v = np.concatenate([_structured_f32(fmt), _random_f32(fmt, 200_000, 5)])
    a = np.abs(v.astype(np.float64))
    hi = np.clip(np.searchsorted(vals, a, side="left"), 1, len(vals) - 1)
    lo = hi - 1
    dlo = a - vals[lo]
    dhi = vals[hi] - a
    pick = np.where(dlo < dhi, lo, np.where(dhi < dlo, hi, np.where(lo % 2 == 0, lo, hi)))
    pick = np.where(a >= vals[-1], len(vals) - 1, pick)
    expect = codes[pick] | np.where(np.signbit(v), 0x80, 0).astype(np.uint8)
    ours = oracle.encode(v, fmt)
    assert np.array_equal(ours, expect)


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_encode_saturates_and_roundtrips(fmt):
    maxc = 0x7E if fmt == E4M3 else 0x7B
    big = np.array([QMAX[fmt] * 1.0001, 1e30, np.inf, -1e30, -np.inf], np.float32)
    assert list(oracle.encode(big, fmt)) == [maxc, maxc, maxc, maxc | 0x80, maxc | 0x80]
    codes = np.array([c for c in range(256) if np.isfinite(torch_decode([c], fmt)[0])], np.uint8)
    vals = torch_decode(codes, fmt).astype(np.float32)
    assert np.array_equal(oracle.encode(vals, fmt), codes)


# --------------------------------------------------------------------------------------------
# The scale step (section 2 of the nanochat FP8 page)

def test_scale_closed_forms():
    s64, s32, i32 = oracle.scale(448.0, E4M3)
    assert (s64, float(s32), float(i32)) == (1.0, 1.0, 1.0)
    s64, s32, i32 = oracle.scale(1.0, E5M2)
    assert s64 == 57344.0 and float(s32) == 57344.0 and float(i32) == float(np.float32(1.0 / 57344.0))
    # an all-zero group: amax clamps to eps = 1e-12
    s64, s32, i32 = oracle.scale(0.0, E4M3)
    assert s64 == 448.0 / 1e-12
    assert float(s32) == float(np.float32(448.0 / 1e-12))
    assert float(i32) == float(np.float32(1.0 / (448.0 / 1e-12)))


def test_scale_inverse_product_is_one():
    rng = np.random.default_rng(3)
    amaxes = (10.0 ** rng.uniform(-30, 30, 20000)).astype(np.float32)
    for fmt in (E4M3, E5M2):
        for a in amaxes[:4000]:
            s64, s32, i32 = oracle.scale(float(a), fmt)
            assert abs(s64 * (1.0 / s64) - 1.0) <= 2.0 ** -52
            assert abs(float(s32) * float(i32) - 1.0) <= 2.0 ** -22
            assert s64 == QMAX[fmt] / max(float(a), 1e-12)


# --------------------------------------------------------------------------------------------
# Quantize (section 2)

def _read_golden():
    cases = {}
    cur = None
    with open(os.path.join(HERE, "golden", "quantize_worked_examples.txt")) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if not line:
                continue
            if line.startswith("case"):
                _, name, fmt, gran = line.split()
                cur = cases[name] = dict(fmt=E4M3 if fmt == "e4m3" else E5M2, gran=gran, x={}, codes={}, inv={})
                continue
            key, rest = line.split(" ", 1)
            row, vals = rest.split(":")
            row = int(row)
            if key == "x":
                cur["x"][row] = [float(t) for t in vals.split()]
            elif key == "codes":
                cur["codes"][row] = [int(t, 16) for t in vals.split()]
            elif key == "inv":
                cur["inv"][row] = int(vals.strip(), 16)
    return cases


def test_golden_worked_examples():
    cases = _read_golden()
    assert set(cases) == {"e4m3_tensor", "e5m2_rows"}
    for case in cases.values():
        rows = [case["x"][r] for r in sorted(case["x"])]
        x = torch.tensor(rows, dtype=torch.float32)
        assert torch.equal(x.to(torch.bfloat16).float(), x)  # inputs are bf16-exact
        bits = W.bf16_bits(x.to(torch.bfloat16))
        if case["gran"] == "tensor":
            q, inv = oracle.quantize_tensor(bits, case["fmt"])
            inv_rows = [inv[0]]
        else:
            q, inv = oracle.quantize_rows(bits, case["fmt"])
            inv_rows = list(inv)
        for r in sorted(case["codes"]):
            assert list(q[r]) == case["codes"][r]
        for r in sorted(case["inv"]):
            assert int(np.float32(inv_rows[r]).view(np.uint32)) == case["inv"][r]


def _ulp_fp8(y, fmt):
    y = np.abs(y)
    emin = -6 if fmt == E4M3 else -14
    p = 3 if fmt == E4M3 else 2
    e = np.floor(np.log2(np.maximum(y, 2.0 ** emin)))
    return 2.0 ** (e - p)


def _bits(shape, std, seed):
    return W.bf16_bits(W.normal_bf16(shape, std, seed))


@pytest.mark.parametrize("fmt", [E4M3, E5M2])
def test_quantize_rows_invariants(fmt):
    x = _bits((64, 300), 1.0, 21)
    xf = x.astype(np.uint32) << 16
    xf = xf.view(np.float32).astype(np.float64)
    q, inv = oracle.quantize_rows(x, fmt)
    maxc = 0x7E if fmt == E4M3 else 0x7B
    # the amax element of each row maps to +-fp8_max exactly
    am = np.argmax(np.abs(xf), axis=1)
    for r in range(x.shape[0]):
        assert q[r, am[r]] & 0x7F == maxc
        assert (q[r, am[r]] >> 7) == (1 if xf[r, am[r]] < 0 else 0)
    # oddness: q(-x) = q(x) with the sign bit flipped
    qn, invn = oracle.quantize_rows(x ^ np.uint16(0x8000), fmt)
    assert np.array_equal(qn, q ^ np.uint8(0x80)) and np.array_equal(inv, invn)
    # error bound per element and the coarse half-ulp-of-max bound
    dq = oracle.decode(q, fmt) * inv[:, None].astype(np.float64)
    y = xf / inv[:, None].astype(np.float64)
    err = np.abs(dq - xf)
    bound = inv[:, None] * 0.5 * _ulp_fp8(y, fmt) + 2.0 ** -22 * np.abs(xf)
    assert np.all(err <= bound)
    half_ulp_max = 16.0 if fmt == E4M3 else 4096.0
    amax = np.abs(xf).max(axis=1)
    assert np.all(err.max(axis=1) <= half_ulp_max * amax / QMAX[fmt] * (1 + 2.0 ** -20))


def test_rank1_agreement():
    rng = np.random.default_rng(7)
    v = W.normal_bf16((40,), 1.0, 9).float()
    j = rng.integers(-5, 6, 24)
    sgn = rng.choice([-1.0, 1.0], 24)
    u = torch.tensor(sgn * 2.0 ** j, dtype=torch.float32)
    x = (u[:, None] * v[None, :]).to(torch.bfloat16)
    assert torch.equal(x.float(), u[:, None] * v[None, :])  # exact in bf16
    bits = W.bf16_bits(x)
    for fmt in (E4M3, E5M2):
        qr, invr = oracle.quantize_rows(bits, fmt)
        # rowwise codes are the same for every row up to the sign of u_i
        base = qr[0] ^ np.uint8(0x80 if sgn[0] < 0 else 0)
        for i in range(24):
            flip = np.uint8(0x80 if sgn[i] < 0 else 0)
            nz = oracle.decode(base, fmt) != 0
            assert np.array_equal((qr[i] ^ flip)[nz], base[nz])
        # ... and equal the tensorwise codes of the row with the largest |u_i|
        qt, invt = oracle.quantize_tensor(bits, fmt)
        imax = int(np.argmax(np.abs(u.numpy())))
        assert np.array_equal(qt.reshape(x.shape)[imax], qr[imax])
        assert invt[0] == invr[imax]
        # colwise of x equals rowwise of x^T
        qc, invc = oracle.quantize_cols(bits, fmt)
        qrt, invrt = oracle.quantize_rows(np.ascontiguousarray(bits.T), fmt)
        assert np.array_equal(qc, qrt.T) and np.array_equal(invc, invrt)
        # general rank-1: every granularity dequantizes to x within the coarse bound
        xf = x.double().numpy()
        half = 16.0 if fmt == E4M3 else 4096.0
        for deq in (oracle.decode(qr, fmt) * invr[:, None], oracle.decode(qt.reshape(x.shape), fmt) * invt[0],
                    oracle.decode(qc, fmt) * invc[None, :]):
            assert np.all(np.abs(deq - xf) <= half * np.abs(xf).max() / QMAX[fmt] * (1 + 2.0 ** -20))


def test_quantize_cols_batched_and_jagged():
    x3 = _bits((3, 50, 70), 1.0, 31)
    q3, inv3 = oracle.quantize_cols(x3, E4M3)
    for b in range(3):
        q2, inv2 = oracle.quantize_cols(x3[b], E4M3)
        assert np.array_equal(q3[b], q2) and np.array_equal(inv3[b], inv2)
    x = _bits((100, 40), 1e-3, 32)
    # one segment covering all rows equals plain colwise
    qj, invj = oracle.quantize_jagged_cols(x, [100], E5M2)
    qc, invc = oracle.quantize_cols(x, E5M2)
    assert np.array_equal(qj, qc) and np.array_equal(invj[0], invc)
    # segments (with empty ones) equal colwise on each slice; empty -> all-zero scales
    ends = [0, 17, 17, 60, 100, 100]
    qj, invj = oracle.quantize_jagged_cols(x, ends, E5M2)
    prev = 0
    zero_inv = oracle.scale(0.0, E5M2)[2]
    for e, end in enumerate(ends):
        if end > prev:
            qs, invs = oracle.quantize_cols(x[prev:end], E5M2)
            assert np.array_equal(qj[prev:end], qs) and np.array_equal(invj[e], invs)
        else:
            assert np.all(invj[e] == zero_inv)
        prev = end
    with pytest.raises(ValueError):
        oracle.quantize_jagged_cols(x, [50, 40, 100], E5M2)
    with pytest.raises(ValueError):
        oracle.quantize_jagged_cols(x, [50, 99], E5M2)


def test_all_zero_group():
    x = np.zeros((4, 32), np.uint16)
    x[1, 3] = 0x8000  # -0.0
    q, inv = oracle.quantize_rows(x, E4M3)
    assert np.all(q[0] == 0) and q[1, 3] == 0x80
    assert np.all(inv == np.float32(1.0 / (448.0 / 1e-12)))


# --------------------------------------------------------------------------------------------
# GEMMs (sections 2, 4 and 5; grouped contract of the MoE section of the AMD page)

def _random_codes(shape, fmt, seed, finite=True):
    rng = np.random.default_rng(seed)
    c = rng.integers(0, 256, size=shape, dtype=np.uint8)
    if finite:
        bad = ~np.isfinite(torch_decode(c.reshape(-1), fmt).reshape(shape))
        c[bad] = 0x38
    return c


def _exact(code, fmt):
    return Fraction(float(torch_decode([code], fmt)[0]))


@pytest.mark.parametrize("fa,fb", [(E4M3, E4M3), (E5M2, E4M3)])
def test_gemm_bruteforce_4x4x8(fa, fb):
    A = _random_codes((4, 8), fa, 1)
    B = _random_codes((4, 8), fb, 2)
    sA = np.array([0.5, 2.0, 0.125, 4.0], np.float32)
    sB = np.array([1.0, 0.25, 8.0, 0.5], np.float32)
    out, absacc = oracle.gemm_fp8(A, fa, B, fb, sA, sB)
    for m in range(4):
        for n in range(4):
            s = sum(_exact(A[m, k], fa) * _exact(B[n, k], fb) for k in range(8))
            exact = Fraction(float(sA[m])) * Fraction(float(sB[n])) * s
            if fa == fb == E4M3:
                assert Fraction(out[m, n]) == exact  # all partial sums fit in fp64
            else:
                assert abs(Fraction(out[m, n]) - exact) <= abs(exact) * Fraction(2) ** -50 + Fraction(2) ** -60
            aexact = abs(Fraction(float(sA[m])) * Fraction(float(sB[n]))) * sum(
                abs(_exact(A[m, k], fa) * _exact(B[n, k], fb)) for k in range(8))
            assert abs(Fraction(absacc[m, n]) - aexact) <= aexact * Fraction(2) ** -50


def test_gemm_layouts_against_numpy():
    A = _random_codes((3, 37), E4M3, 3)
    B = _random_codes((5, 37), E5M2, 4)
    sA = np.array([0.5, 1.5, 3.0], np.float32)
    sB = np.array([2.0], np.float32)
    ref = (oracle.decode(A, E4M3) * sA[:, None]) @ (oracle.decode(B, E5M2) * sB[0]).T
    out, _ = oracle.gemm_fp8(A, E4M3, B, E5M2, sA, sB)
    np.testing.assert_allclose(out, ref, rtol=1e-12, atol=1e-12 * np.abs(ref).max())
    # the same operands stored transposed (MN-major)
    out_t, _ = oracle.gemm_fp8(np.ascontiguousarray(A.T), E4M3, np.ascontiguousarray(B.T), E5M2, sA, sB,
                               a_trans=True, b_trans=True)
    assert np.array_equal(out, out_t)
    # row sampling returns the same rows
    out_r, _ = oracle.gemm_fp8(A, E4M3, B, E5M2, sA, sB, rows=[2, 0])
    assert np.array_equal(out_r, out[[2, 0]])


def test_gemm_scale_direction_and_factorization():
    """The GEMM multiplies by sA * sB (the inverse scales); getting it backwards is off by
    scale^2. Rowwise with all-equal scales equals tensorwise."""
    A = np.full((2, 4), 0x38, np.uint8)  # e4m3 1.0
    B = np.full((3, 4), 0x40, np.uint8)  # e4m3 2.0
    out, _ = oracle.gemm_fp8(A, E4M3, B, E4M3, [0.25], [3.0])
    assert np.all(out == 0.25 * 3.0 * 4 * 2.0)
    A = _random_codes((6, 33), E4M3, 8)
    B = _random_codes((7, 33), E4M3, 9)
    o1, _ = oracle.gemm_fp8(A, E4M3, B, E4M3, np.full(6, 0.375, np.float32), np.full(7, 1.25, np.float32))
    o2, _ = oracle.gemm_fp8(A, E4M3, B, E4M3, [0.375], [1.25])
    assert np.array_equal(o1, o2)


def test_quantized_gemm_approximates_float_product():
    """quantize -> scaled GEMM reproduces x @ w^T within the propagated quantization error:
    a wrong scale direction or a dropped scale fails by orders of magnitude."""
    x = _bits((16, 64), 1.0, 41)
    w = _bits((24, 64), 0.02, 42)
    xf = (x.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    wf = (w.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    qx, ix = oracle.quantize_rows(x, E4M3)
    qw, iw = oracle.quantize_rows(w, E4M3)
    out, _ = oracle.gemm_fp8(qx, E4M3, qw, E4M3, ix, iw)
    ex = oracle.decode(qx, E4M3) * ix[:, None] - xf
    ew = oracle.decode(qw, E4M3) * iw[:, None] - wf
    bound = np.abs(ex) @ np.abs(wf).T + np.abs(xf) @ np.abs(ew).T + np.abs(ex) @ np.abs(ew).T
    assert np.all(np.abs(out - xf @ wf.T) <= bound * (1 + 1e-9) + 1e-300)


def test_gemm_bf16_against_numpy():
    a = _bits((9, 31), 1.0, 51)
    b = _bits((31, 11), 1.0, 52)  # stored [K, N]
    af = (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    bf = (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
    out, _ = oracle.gemm_bf16(a, b, b_trans=True)
    np.testing.assert_allclose(out, af @ bf, rtol=1e-12, atol=1e-12)
    out2, _ = oracle.gemm_bf16(np.ascontiguousarray(a.T), b, a_trans=True, b_trans=True)
    assert np.array_equal(out, out2)


def test_grouped_m_reductions():
    E, M, N, K = 4, 40, 12, 48
    A = _random_codes((M, K), E4M3, 61)
    Wt = _random_codes((E, N, K), E4M3, 62)
    sA = np.linspace(0.5, 2, M).astype(np.float32)
    sB = np.linspace(0.1, 3, E * N).astype(np.float32).reshape(E, N)
    # one expert holding every row = the dense GEMM
    out1, _ = oracle.grouped_gemm_m(A, E4M3, Wt[:1], E4M3, sA, sB[:1], [M])
    dense, _ = oracle.gemm_fp8(A, E4M3, Wt[0], E4M3, sA, sB[0])
    assert np.array_equal(out1, dense)
    # ragged segments with empty experts = the dense GEMM of each segment
    ends = [0, 13, 13, 40]
    out, _ = oracle.grouped_gemm_m(A, E4M3, Wt, E4M3, sA, sB, ends)
    prev = 0
    for e, end in enumerate(ends):
        if end > prev:
            d, _ = oracle.gemm_fp8(A[prev:end], E4M3, Wt[e], E4M3, sA[prev:end], sB[e])
            assert np.array_equal(out[prev:end], d)
        prev = end
    rows = [39, 0, 13, 12]
    out_r, _ = oracle.grouped_gemm_m(A, E4M3, Wt, E4M3, sA, sB, ends, rows=rows)
    assert np.array_equal(out_r, out[rows])
    with pytest.raises(ValueError):
        oracle.grouped_gemm_m(A, E4M3, Wt, E4M3, sA, sB, [0, 13, 12, 40])


def test_grouped_k_reductions():
    E, M, N, K = 3, 30, 10, 14
    G = _random_codes((M, N), E5M2, 71)
    X = _random_codes((M, K), E4M3, 72)
    sG = np.linspace(0.5, 2, E * N).astype(np.float32).reshape(E, N)
    sX = np.linspace(0.25, 1, E * K).astype(np.float32).reshape(E, K)
    ends = [11, 11, 30]
    out, _ = oracle.grouped_gemm_k(G, E5M2, X, E4M3, sG, sX, ends)
    assert out.shape == (E, N, K)
    prev = 0
    for e, end in enumerate(ends):
        if end > prev:
            d, _ = oracle.gemm_fp8(np.ascontiguousarray(G[prev:end].T), E5M2, np.ascontiguousarray(X[prev:end].T),
                                   E4M3, sG[e], sX[e])
            assert np.array_equal(out[e], d)
        else:
            assert np.all(out[e] == 0)
        prev = end
    out_s, _ = oracle.grouped_gemm_k(G, E5M2, X, E4M3, sG, sX, ends, nsel=[9, 2])
    assert np.array_equal(out_s, out[:, [9, 2]])


def test_oracle_results_do_not_depend_on_its_thread_count():
    """The 1-core baseline times the same arithmetic: quantize and GEMM give the same bits on one
    thread as on all of them (each output element is computed by one thread, in a fixed order)."""
    import workloads as W
    x = W.bf16_bits(W.normal_bf16((96, 160), 1.0, 31))
    w = W.bf16_bits(W.normal_bf16((64, 160), 0.02, 32))
    n = oracle.num_threads()

    def chain():
        xq, xi = oracle.quantize_rows(x, oracle.E4M3)
        wq, wi = oracle.quantize_cols(w.T.copy(), oracle.E4M3)
        out, _ = oracle.gemm_fp8(xq, oracle.E4M3, wq.T.copy(), oracle.E4M3, xi, wi)
        return xq, xi, wq, wi, out

    try:
        oracle.set_num_threads(1)
        one = chain()
    finally:
        oracle.set_num_threads(n)
    many = chain()
    for a, b in zip(one, many):
        assert np.array_equal(np.asarray(a).view(np.uint8), np.asarray(b).view(np.uint8))
