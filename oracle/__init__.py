"""Python access to the CPU oracle (oracle.c) through ctypes, with numpy arrays.

TEST INFRASTRUCTURE ONLY: tests/, __graft_entry__.smoke() and bench.py's CPU baseline /
reference leg may import this module; the product package never does.

Conventions: bf16 tensors are numpy uint16 arrays of raw bit patterns; FP8 tensors are uint8
arrays of raw codes; scales are float32; GEMM results are float64 (the exact-as-possible value,
before any output rounding). Formats: E4M3 = 0, E5M2 = 1.
"""
import ctypes
import os

import numpy as np

from . import build as _build

E4M3 = 0
E5M2 = 1

_lib = None


def lib():
    global _lib
    if _lib is None:
        # FP8LIN_ORACLE_LIB: a deliberately broken copy of the oracle, built by the mutation test
        # (tests/test_oracle_mutations.py) to show that the pins catch it.
        path = os.environ.get("FP8LIN_ORACLE_LIB") or _build.build()
        L = ctypes.CDLL(path)
        P = ctypes.c_void_p
        I64 = ctypes.c_int64
        I = ctypes.c_int
        L.orc_fp8_max.restype = ctypes.c_double
        L.orc_fp8_max.argtypes = [I]
        L.orc_fp8_decode.restype = ctypes.c_double
        L.orc_fp8_decode.argtypes = [ctypes.c_uint8, I]
        L.orc_fp8_encode.restype = ctypes.c_uint8
        L.orc_fp8_encode.argtypes = [ctypes.c_float, I]
        L.orc_fp8_encode_array.argtypes = [P, I64, I, P]
        L.orc_fp8_decode_array.argtypes = [P, I64, I, P]
        L.orc_scale.argtypes = [ctypes.c_float, I, P, P, P]
        L.orc_quantize_tensor.argtypes = [P, I64, I, P, P]
        L.orc_quantize_rows.argtypes = [P, I64, I64, I, P, P]
        L.orc_quantize_cols.argtypes = [P, I64, I64, I64, I, P, P]
        L.orc_quantize_jagged_cols.restype = I
        L.orc_quantize_jagged_cols.argtypes = [P, I64, I64, P, I64, I, P, P]
        L.orc_gemm_fp8.argtypes = [P, I, I64, I64, P, I, I64, I64, P, I64, P, I64, I64, I64, I64,
                                   P, I64, P, P]
        L.orc_gemm_bf16.argtypes = [P, I64, I64, P, I64, I64, I64, I64, I64, P, I64, P, P]
        L.orc_grouped_gemm_m.restype = I
        L.orc_grouped_gemm_m.argtypes = [P, I, P, I, P, P, P, I64, I64, I64, I64, P, I64, P, P]
        L.orc_grouped_gemm_k.restype = I
        L.orc_grouped_gemm_k.argtypes = [P, I, P, I, P, P, P, I64, I64, I64, I64, P, I64, P, P]
        L.orc_mx_scale.restype = ctypes.c_uint8
        L.orc_mx_scale.argtypes = [ctypes.c_float, I]
        L.orc_e8m0_decode.restype = ctypes.c_double
        L.orc_e8m0_decode.argtypes = [ctypes.c_uint8]
        L.orc_mx_quantize_rows.restype = I
        L.orc_mx_quantize_rows.argtypes = [P, I64, I64, I, P, P]
        L.orc_gemm_mx.restype = I
        L.orc_gemm_mx.argtypes = [P, I, P, I, P, P, I64, I64, I64, P, I64, P, P]
        L.orc_quantize_blocks.argtypes = [P, I64, I64, I64, I64, I, P, P]
        L.orc_gemm_blockwise.argtypes = [P, I, P, I, P, P, I64, I64, I64, P, I64, P, P]
        L.orc_num_threads.restype = I
        L.orc_set_num_threads.argtypes = [I]
        L.orc_set_num_threads.restype = None
        _lib = L
    return _lib


def _p(a):
    return None if a is None else ctypes.c_void_p(a.ctypes.data)


def _c(a, dtype):
    return np.ascontiguousarray(a, dtype=dtype)


def num_threads() -> int:
    return lib().orc_num_threads()


def set_num_threads(n: int) -> None:
    """Threads of the oracle's parallel loops from now on (timing only)."""
    lib().orc_set_num_threads(int(n))


def fp8_max(fmt: int) -> float:
    return lib().orc_fp8_max(fmt)


def decode(codes, fmt: int) -> np.ndarray:
    c = _c(codes, np.uint8)
    out = np.empty(c.shape, np.float64)
    lib().orc_fp8_decode_array(_p(c), c.size, fmt, _p(out))
    return out


def encode(values, fmt: int) -> np.ndarray:
    v = _c(values, np.float32)
    out = np.empty(v.shape, np.uint8)
    lib().orc_fp8_encode_array(_p(v), v.size, fmt, _p(out))
    return out


def scale(amax: float, fmt: int):
    """(scale64, scale32, inv32) for one group's amax."""
    s64 = ctypes.c_double()
    s32 = ctypes.c_float()
    i32 = ctypes.c_float()
    lib().orc_scale(ctypes.c_float(amax), fmt, ctypes.byref(s64), ctypes.byref(s32), ctypes.byref(i32))
    return s64.value, np.float32(s32.value), np.float32(i32.value)


def quantize_tensor(x_bits, fmt: int):
    x = _c(x_bits, np.uint16)
    q = np.empty(x.shape, np.uint8)
    inv = np.empty(1, np.float32)
    lib().orc_quantize_tensor(_p(x), x.size, fmt, _p(q), _p(inv))
    return q, inv


def quantize_rows(x_bits, fmt: int):
    x = _c(x_bits, np.uint16)
    R, C = x.shape
    q = np.empty((R, C), np.uint8)
    inv = np.empty(R, np.float32)
    lib().orc_quantize_rows(_p(x), R, C, fmt, _p(q), _p(inv))
    return q, inv


def quantize_cols(x_bits, fmt: int):
    """x [R, C] or [B, R, C]; one scale per (batch, column). Codes come back in x's order."""
    x = _c(x_bits, np.uint16)
    squeeze = x.ndim == 2
    if squeeze:
        x = x[None]
    B, R, C = x.shape
    q = np.empty((B, R, C), np.uint8)
    inv = np.empty((B, C), np.float32)
    lib().orc_quantize_cols(_p(x), B, R, C, fmt, _p(q), _p(inv))
    if squeeze:
        return q[0], inv[0]
    return q, inv


def quantize_jagged_cols(x_bits, ends, fmt: int):
    x = _c(x_bits, np.uint16)
    e = _c(ends, np.int32)
    R, C = x.shape
    q = np.empty((R, C), np.uint8)
    inv = np.empty((e.size, C), np.float32)
    rc = lib().orc_quantize_jagged_cols(_p(x), R, C, _p(e), e.size, fmt, _p(q), _p(inv))
    if rc:
        raise ValueError("bad segment ends")
    return q, inv


def gemm_fp8(A, fmtA, B, fmtB, sA, sB, rows=None, a_trans=False, b_trans=False):
    """out[i, n] = sA[m] sB[n] sum_k dec(A[m, k]) dec(B[n, k]).

    A is [M, K] (or [K, M] when a_trans); B is [N, K] (or [K, N] when b_trans).
    Returns (out float64 [len(rows) or M, N], absacc of the same shape)."""
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    if a_trans:
        K, M = A.shape
        a_sm, a_sk = 1, M
    else:
        M, K = A.shape
        a_sm, a_sk = K, 1
    if b_trans:
        K2, N = B.shape
        b_sn, b_sk = 1, N
    else:
        N, K2 = B.shape
        b_sn, b_sk = K2, 1
    assert K == K2
    sA = _c(np.atleast_1d(sA), np.float32)
    sB = _c(np.atleast_1d(sB), np.float32)
    r = None if rows is None else _c(rows, np.int64)
    cnt = M if r is None else r.size
    out = np.empty((cnt, N), np.float64)
    absacc = np.empty((cnt, N), np.float64)
    lib().orc_gemm_fp8(_p(A), fmtA, a_sm, a_sk, _p(B), fmtB, b_sn, b_sk, _p(sA), sA.size, _p(sB),
                       sB.size, M, N, K, _p(r), 0 if r is None else r.size, _p(out), _p(absacc))
    return out, absacc


def gemm_bf16(A, B, rows=None, a_trans=False, b_trans=False):
    """out[i, n] = sum_k A(m, k) B(n, k) on bf16 bit patterns, fp64 accumulation."""
    A = _c(A, np.uint16)
    B = _c(B, np.uint16)
    if a_trans:
        K, M = A.shape
        a_sm, a_sk = 1, M
    else:
        M, K = A.shape
        a_sm, a_sk = K, 1
    if b_trans:
        K2, N = B.shape
        b_sn, b_sk = 1, N
    else:
        N, K2 = B.shape
        b_sn, b_sk = K2, 1
    assert K == K2
    r = None if rows is None else _c(rows, np.int64)
    cnt = M if r is None else r.size
    out = np.empty((cnt, N), np.float64)
    absacc = np.empty((cnt, N), np.float64)
    lib().orc_gemm_bf16(_p(A), a_sm, a_sk, _p(B), b_sn, b_sk, M, N, K, _p(r),
                        0 if r is None else r.size, _p(out), _p(absacc))
    return out, absacc


def grouped_gemm_m(A, fmtA, W, fmtW, sA, sB, ends, rows=None):
    A = _c(A, np.uint8)
    W = _c(W, np.uint8)
    sA = _c(sA, np.float32)
    sB = _c(sB, np.float32)
    e = _c(ends, np.int32)
    M, K = A.shape
    E, N, K2 = W.shape
    assert K == K2 and E == e.size
    r = None if rows is None else _c(rows, np.int64)
    cnt = M if r is None else r.size
    out = np.empty((cnt, N), np.float64)
    absacc = np.empty((cnt, N), np.float64)
    rc = lib().orc_grouped_gemm_m(_p(A), fmtA, _p(W), fmtW, _p(sA), _p(sB), _p(e), E, M, N, K,
                                  _p(r), 0 if r is None else r.size, _p(out), _p(absacc))
    if rc:
        raise ValueError("bad segment ends")
    return out, absacc


def grouped_gemm_k(G, fmtG, X, fmtX, sG, sX, ends, nsel=None):
    """out[e, i, k] = sG[e, n] sX[e, k] sum_{r in segment e} dec(G[r, n]) dec(X[r, k])."""
    G = _c(G, np.uint8)
    X = _c(X, np.uint8)
    sG = _c(sG, np.float32)
    sX = _c(sX, np.float32)
    e = _c(ends, np.int32)
    M, N = G.shape
    M2, K = X.shape
    assert M == M2
    E = e.size
    ns = None if nsel is None else _c(nsel, np.int64)
    cnt = N if ns is None else ns.size
    out = np.empty((E, cnt, K), np.float64)
    absacc = np.empty((E, cnt, K), np.float64)
    rc = lib().orc_grouped_gemm_k(_p(G), fmtG, _p(X), fmtX, _p(sG), _p(sX), _p(e), E, M, N, K,
                                  _p(ns), 0 if ns is None else ns.size, _p(out), _p(absacc))
    if rc:
        raise ValueError("bad segment ends")
    return out, absacc


# ---- MXFP8 (blocks of 32 along the contraction, E8M0 power-of-two scales) ----

MX_BLOCK = 32


def mx_scale(amax: float, fmt: int) -> int:
    """E8M0 code of the shared scale of a block whose largest magnitude is amax."""
    return int(lib().orc_mx_scale(ctypes.c_float(amax), fmt))


def e8m0_decode(codes) -> np.ndarray:
    c = np.asarray(codes, np.uint8)
    return np.array([lib().orc_e8m0_decode(int(v)) for v in c.ravel()], np.float64).reshape(c.shape)


def mx_quantize_rows(x_bits, fmt: int):
    """x [R, C] (C % 32 == 0): blocks of 32 along each row -> codes [R, C], E8M0 [R, C // 32]."""
    x = _c(x_bits, np.uint16)
    R, C = x.shape
    q = np.empty((R, C), np.uint8)
    sc = np.empty((R, C // MX_BLOCK), np.uint8)
    if lib().orc_mx_quantize_rows(_p(x), R, C, fmt, _p(q), _p(sc)):
        raise ValueError("the row length must be a multiple of 32")
    return q, sc


def mx_quantize_cols(x_bits, fmt: int):
    """x [R, C] (R % 32 == 0): blocks of 32 rows down each column, i.e. the row blocks of x^T.
    Returns the codes of x^T [C, R] (the column-major copy) and E8M0 [C, R // 32]."""
    return mx_quantize_rows(np.ascontiguousarray(np.asarray(x_bits, np.uint16).T), fmt)


def mx_padded_segments(ends, pad: int = 128):
    """(start, count, padded start) of each segment when every segment is padded to `pad` rows."""
    ends = np.asarray(ends, np.int64)
    starts = np.concatenate([[0], ends[:-1]])
    counts = ends - starts
    padded = -(-counts // pad) * pad
    pstarts = np.concatenate([[0], np.cumsum(padded)[:-1]])
    return starts, counts, pstarts, int(padded.sum())


def mx_quantize_jagged_cols(x_bits, ends, fmt: int, pad: int = 128):
    """x [M, C] with rows in segments ending at `ends`: each segment's rows, padded with zeros to
    a multiple of `pad`, are laid side by side along the token axis of x^T [C, P]; blocks of 32
    tokens start at each segment's start. Returns the codes of that padded x^T [C, P] and
    E8M0 [C, P // 32] (padding blocks are all-zero blocks)."""
    x = np.asarray(x_bits, np.uint16)
    M, C = x.shape
    starts, counts, pstarts, P = mx_padded_segments(ends, pad)
    if int(counts.sum()) != M or (counts < 0).any():
        raise ValueError("bad segment ends")
    xt = np.zeros((C, P), np.uint16)
    for s, c, ps in zip(starts, counts, pstarts):
        xt[:, ps:ps + c] = x[s:s + c].T
    return mx_quantize_rows(xt, fmt)


def gemm_mx(A, fmtA, B, fmtB, sA, sB, rows=None):
    """out[i, n] = sum_k X_A[m, k // 32] X_B[n, k // 32] dec(A[m, k]) dec(B[n, k]); A [M, K],
    B [N, K] codes, sA [M, K // 32], sB [N, K // 32] E8M0. Returns (out, absacc) in float64."""
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    sA = _c(sA, np.uint8)
    sB = _c(sB, np.uint8)
    M, K = A.shape
    N, K2 = B.shape
    assert K == K2 and sA.shape == (M, K // MX_BLOCK) and sB.shape == (N, K // MX_BLOCK)
    r = None if rows is None else _c(rows, np.int64)
    cnt = M if r is None else r.size
    out = np.empty((cnt, N), np.float64)
    absacc = np.empty((cnt, N), np.float64)
    if lib().orc_gemm_mx(_p(A), fmtA, _p(B), fmtB, _p(sA), _p(sB), M, N, K, _p(r), 0 if r is None else r.size,
                         _p(out), _p(absacc)):
        raise ValueError("the contraction length must be a multiple of 32")
    return out, absacc


# ---- blockwise (1 x 128 activation tiles, 128 x 128 weight tiles) ----

def quantize_blocks(x_bits, fmt: int, br: int, bc: int):
    """Tiles of br x bc, each quantized by the recipe: codes [R, C], inv [ceil(R/br), ceil(C/bc)]."""
    x = _c(x_bits, np.uint16)
    R, C = x.shape
    q = np.empty((R, C), np.uint8)
    inv = np.empty((-(-R // br), -(-C // bc)), np.float32)
    lib().orc_quantize_blocks(_p(x), R, C, br, bc, fmt, _p(q), _p(inv))
    return q, inv


def gemm_blockwise(A, fmtA, B, fmtB, sA, sB, rows=None):
    """out[i, n] = sum_k sA[m, k // 128] sB[n // 128, k // 128] dec(A[m, k]) dec(B[n, k])."""
    A = _c(A, np.uint8)
    B = _c(B, np.uint8)
    sA = _c(sA, np.float32)
    sB = _c(sB, np.float32)
    M, K = A.shape
    N, K2 = B.shape
    kb = -(-K // 128)
    assert K == K2 and sA.shape == (M, kb) and sB.shape == (-(-N // 128), kb)
    r = None if rows is None else _c(rows, np.int64)
    cnt = M if r is None else r.size
    out = np.empty((cnt, N), np.float64)
    absacc = np.empty((cnt, N), np.float64)
    lib().orc_gemm_blockwise(_p(A), fmtA, _p(B), fmtB, _p(sA), _p(sB), M, N, K, _p(r), 0 if r is None else r.size,
                             _p(out), _p(absacc))
    return out, absacc
