"""The allocation-free tensorwise quantize (fp8_quantize_tensor_noalloc).

Some callers cannot allocate device memory: plugin or callback interfaces that give the library
only its inputs and outputs, and runtimes that reserve all device memory up front and forbid
cudaMalloc afterwards. For them the library keeps the amax reduction's scratch in a fixed device
array of its own instead of a caller workspace. These tests call that entry point through the C
ABI and check it against the ordinary entry point (fp8_quantize with tensor granularity), which
the other test files pin to the oracle; results must be bit-identical.

This file is collected last so that a run stopping at the first failure has run everything else.
"""
import ctypes

import numpy as np
import pytest
import torch

import workloads as W


@pytest.fixture(scope="module")
def fp8():
    import moe_grouped_gemm_absmax_gb300 as m
    return m


def test_rejects_more_than_the_fixed_scratch_holds(fp8):
    """Host-side check, before any device work: more elements than the fixed array's partial
    maxima can cover is an error (FP8_ERR_UNSUPPORTED), not an overflow."""
    limit = 16384 * 32768
    x = fp8.Fp8Tensor()
    x.ptr, x.dtype, x.ndim = 256, fp8.DT_BF16, 2
    x.shape[0], x.shape[1] = limit // 4096 + 1, 4096  # one row past the limit
    inv = fp8.Fp8Tensor()
    inv.ptr, inv.dtype, inv.ndim = 256, fp8.DT_F32, 1
    inv.shape[0] = 1
    rc = fp8.lib.fp8_quantize_tensor_noalloc(ctypes.byref(x), fp8.DT_E4M3, fp8.LAYOUT_ROW_MAJOR, ctypes.byref(x),
                                             None, ctypes.byref(inv), None)
    assert rc == 2


def _reference(fp8, x, dt):
    """The ordinary entry point, with a caller workspace."""
    q, qt, inv = fp8.quantize_alloc(x, fp8.GRAN_TENSOR, dt, layout=fp8.LAYOUT_BOTH)
    return q, qt, inv


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


def _same(a, b):
    return np.array_equal(a.view(torch.uint8).cpu().numpy(), b.view(torch.uint8).cpu().numpy())


@pytest.mark.gpu
def test_matches_workspace_entry_point_on_two_calls_in_a_row(fp8):
    # First call: a large tensor (1024 partial maxima) with one big outlier. Second call: a small
    # tensor with a smaller amax, so stale partials or a stale final word from the first call
    # would change its scale.
    x1 = W.normal_bf16((4096, 8192), 1.0, 91, device="cuda")
    x1[1234, 567] = 1000.0
    x2 = W.normal_bf16((256, 512), 0.02, 92, device="cuda")
    for x, dt in ((x1, fp8.DT_E4M3), (x2, fp8.DT_E5M2)):
        got = _noalloc(fp8, x, dt)
        ref = _reference(fp8, x, dt)
        torch.cuda.synchronize()
        for g, r in zip(got, ref):
            assert _same(g, r)
