"""The allocation-free tensorwise quantize (fp8_quantize_tensor_noalloc).

Some callers cannot allocate device memory: plugin or callback interfaces that give the library
only its inputs and outputs, and runtimes that reserve all device memory up front and forbid
cudaMalloc afterwards. For them the library keeps the amax reduction's scratch in a fixed device
array of its own instead of a caller workspace. These tests call that entry point through the C
ABI and check it against the oracle's tensorwise recipe ("FP8 Training: Quantization, Autograd,
Torchao", section 2) on the same bf16 inputs, bit for bit, and against the ordinary entry point
(fp8_quantize with tensor granularity and a caller workspace).

This file is collected last so that a run stopping at the first failure has run everything else.
"""
import ctypes

import numpy as np
import pytest
import torch

import oracle
import workloads as W


@pytest.fixture(scope="module")
def fp8():
    import moe_grouped_gemm_absmax_gb300 as m
    return m


def _call(fp8, x, inv, dt=3, q=None, qt=None, layout=1):
    q = q if q is not None else x
    return fp8.lib.fp8_quantize_tensor_noalloc(ctypes.byref(x), dt, layout, ctypes.byref(q),
                                               ctypes.byref(qt) if qt is not None else None, ctypes.byref(inv), None)


def _desc(fp8, dtype, shape, ptr=256):
    d = fp8.Fp8Tensor()
    d.ptr, d.dtype, d.ndim = ptr, dtype, len(shape)
    for i, n in enumerate(shape):
        d.shape[i] = n
    return d


def test_rejects_more_than_the_fixed_scratch_holds(fp8):
    """Host-side checks, before any device work: more elements than the fixed array's partial
    maxima can cover is an error (FP8_ERR_UNSUPPORTED), not an overflow; so are extents whose
    product would overflow; a malformed inverse-scale descriptor is FP8_ERR_INVALID_ARG."""
    limit = 16384 * 32768
    inv = _desc(fp8, fp8.DT_F32, (1,))
    assert _call(fp8, _desc(fp8, fp8.DT_BF16, (limit // 4096 + 1, 4096)), inv) == 2  # one row past the limit
    assert _call(fp8, _desc(fp8, fp8.DT_BF16, (1 << 40, 1 << 40)), inv) == 2  # product overflows int64
    assert _call(fp8, _desc(fp8, fp8.DT_BF16, (1 << 31, 8)), inv) == 2
    assert _call(fp8, _desc(fp8, fp8.DT_BF16, (8, limit + 8)), inv) == 2
    x = _desc(fp8, fp8.DT_BF16, (64, 64))
    bad = _desc(fp8, fp8.DT_F32, (1,))
    bad.ndim = 4  # the descriptor holds three extents
    assert _call(fp8, x, bad) == 1
    assert _call(fp8, x, _desc(fp8, fp8.DT_F32, (1, -1))) == 1
    assert _call(fp8, x, _desc(fp8, fp8.DT_F32, (2,))) == 1


def _noalloc(fp8, x, dt):
    R, C = x.shape
    fdt = fp8.FP8_TORCH[dt]
    q = torch.empty((R, C), dtype=fdt, device="cuda")
    qt = torch.empty((C, R), dtype=fdt, device="cuda")
    inv = torch.empty(1, dtype=torch.float32, device="cuda")
    rc = fp8.lib.fp8_quantize_tensor_noalloc(ctypes.byref(fp8.desc(x)), dt, fp8.LAYOUT_BOTH,
                                             ctypes.byref(fp8.desc(q)), ctypes.byref(fp8.desc(qt)),
                                             ctypes.byref(fp8.desc(inv)),
                                             ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, fp8.status_string(rc)
    return q, qt, inv


def _codes(t):
    return t.view(torch.uint8).cpu().numpy()


def _check(fp8, x, dt, got):
    """Bit-exact against the oracle's tensorwise recipe on the same bf16 input, and against the
    ordinary entry point with a workspace."""
    fmt = oracle.E4M3 if dt == fp8.DT_E4M3 else oracle.E5M2
    qo, io = oracle.quantize_tensor(W.bf16_bits(x.cpu()), fmt)
    q, qt, inv = got
    assert np.array_equal(_codes(q), qo)
    assert np.array_equal(_codes(qt), qo.T)
    assert np.array_equal(inv.cpu().numpy().view(np.uint32), io.view(np.uint32))
    ref = fp8.quantize_alloc(x, fp8.GRAN_TENSOR, dt, layout=fp8.LAYOUT_BOTH)
    torch.cuda.synchronize()
    for g, r in zip(got, ref):
        assert np.array_equal(_codes(g), _codes(r))


@pytest.mark.gpu
def test_matches_oracle_and_workspace_entry_point_on_calls_in_a_row(fp8):
    """Calls in a row share the array. Each case would go wrong if a call read a slot it had not
    written: the first leaves 4096 partial maxima with a large one near the end; the second has a
    ragged tail (1029 full partials and one of 16 vectors) and a smaller amax, so a read past its
    own partials or of the first call's final word would change its scale; the third has more
    than 1024 partials (the final reduction's strided loop runs four times) with its outlier in
    the last partial's range; the fourth is empty (no partials: amax 0, the eps scale)."""
    x1 = W.normal_bf16((8192, 16384), 1.0, 91, device="cuda")
    x1[8000, 100] = 5000.0
    x2 = W.normal_bf16((4112, 8200), 0.02, 92, device="cuda")
    x3 = W.normal_bf16((8192, 16384), 1.0, 93, device="cuda")
    x3[8191, 16383] = -300.0
    x4 = torch.empty((0, 64), dtype=torch.bfloat16, device="cuda")
    for x, dt in ((x1, fp8.DT_E4M3), (x2, fp8.DT_E5M2), (x3, fp8.DT_E4M3), (x4, fp8.DT_E4M3)):
        got = _noalloc(fp8, x, dt)
        torch.cuda.synchronize()
        _check(fp8, x, dt, got)
