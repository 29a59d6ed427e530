"""The C-ABI library loads and exports every entry point include/fp8lin.h declares; host-only
helpers (no GPU compute) behave as documented. Runs on CPU."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def fp8():
    import moe_grouped_gemm_absmax_gb300 as m
    return m


def _declared():
    src = open(os.path.join(ROOT, "include", "fp8lin.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(fp8_[a-z0-9_]+)\s*\(", src)))


def test_header_declarations_are_exported(fp8):
    names = _declared()
    assert len(names) >= 9
    for n in names:
        assert hasattr(fp8.lib, n), n  # ctypes resolves the symbol in the .so
    assert set(names) == set(fp8.EXPORTS)


def test_host_helpers(fp8):
    for R, E in [(0, 1), (1, 1), (100, 3), (8192, 16), (131072, 256)]:
        P = fp8.fp8_jagged_padded_rows(R, E)
        assert P % 128 == 0 and R + 127 * E <= P < R + 127 * E + 128
    assert fp8.fp8_workspace_size(fp8.OP_QUANTIZE, granularity=fp8.GRAN_TENSOR) == 8
    assert fp8.fp8_workspace_size(fp8.OP_QUANTIZE, granularity=fp8.GRAN_ROW) == 0
    # one 128-byte partial (64 column maxima) per 256-row x 64-column unit: (rows / 256 + groups)
    # row tiles bound the units of every 64-column strip
    assert fp8.fp8_workspace_size(fp8.OP_QUANTIZE, 16, 5120, 16 * 8192, granularity=fp8.GRAN_COL) == (512 + 16) * 80 * 128
    assert fp8.fp8_workspace_size(fp8.OP_QUANTIZE, 1, 70, 300, granularity=fp8.GRAN_COL) == (2 + 1) * 2 * 128
    M, K, N = 256, 512, 128
    ws_row_bf16 = fp8.fp8_workspace_size(fp8.OP_LINEAR_BWD, M, K, N, fp8.GRAN_ROW, fp8.WGRAD_BF16)
    ws_row_fp8 = fp8.fp8_workspace_size(fp8.OP_LINEAR_BWD, M, K, N, fp8.GRAN_ROW, fp8.WGRAD_FP8)
    assert ws_row_bf16 >= M * N + K * N and ws_row_fp8 >= ws_row_bf16 + N * M + K * M
    for code in (0, 1, 2, 3, 4, 5, 6, fp8.DEV_BAD_OFFSETS, fp8.DEV_TIMEOUT):
        assert fp8.status_string(code) != "unknown status"
    old = fp8.fp8_set_wait_limit_ns(123)
    assert fp8.fp8_set_wait_limit_ns(old) == 123


def test_no_device_is_an_error_not_a_crash(fp8):
    import torch
    if torch.cuda.is_available():
        pytest.skip("a GPU is present")
    x = fp8.Fp8Tensor()
    x.ptr, x.dtype, x.ndim = 16, fp8.DT_BF16, 2
    x.shape[0], x.shape[1] = 4, 8
    rc = fp8.lib.fp8_quantize(ctypes.byref(x), 1, fp8.DT_E4M3, 1, ctypes.byref(x), None, ctypes.byref(x), None,
                              None, 0, None, None)
    assert rc == 6  # FP8_ERR_DEVICE
