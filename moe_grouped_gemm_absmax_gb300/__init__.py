"""Python binding of the fp8lin C ABI (include/fp8lin.h): argument marshalling only.

Every function named like a C entry point takes torch tensors (device memory), turns each into
an fp8_tensor descriptor and calls the shared library; all arithmetic runs in the library's CUDA
kernels. Outputs are caller-provided; the `*_alloc` helpers only allocate torch buffers of the
right shape before calling the same entry points.

The library is built in-tree by `build.py` (`_lib/libfp8lin.so`). Importing this module raises
if it is missing: there is no fallback path.
"""
from __future__ import annotations

import ctypes
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libfp8lin.so")

# enums of include/fp8lin.h
DT_BF16, DT_F32, DT_E4M3, DT_E5M2, DT_I32, DT_E8M0 = 1, 2, 3, 4, 5, 6
GRAN_TENSOR, GRAN_ROW, GRAN_COL, GRAN_MX, GRAN_BLOCK_1x128, GRAN_BLOCK_128x128 = 0, 1, 2, 3, 4, 5
LAYOUT_ROW_MAJOR, LAYOUT_COL_MAJOR, LAYOUT_BOTH = 1, 2, 3
MM_FAST_ACCUM, MM_A_MN_MAJOR, MM_B_MN_MAJOR, MM_BLOCKWISE = 1, 2, 4, 8
GROUPED_JAGGED_M, GROUPED_JAGGED_K = 0, 1
WGRAD_FP8, WGRAD_BF16 = 0, 1
OP_QUANTIZE, OP_LINEAR_FWD, OP_LINEAR_BWD = 0, 1, 2
OK = 0
DEV_BAD_OFFSETS = 1 << 8
DEV_TIMEOUT = 1 << 9

_TORCH_DT = {
    torch.bfloat16: DT_BF16,
    torch.float32: DT_F32,
    torch.float8_e4m3fn: DT_E4M3,
    torch.float8_e5m2: DT_E5M2,
    torch.int32: DT_I32,
    torch.uint8: DT_E8M0,  # MX scale codes travel as raw bytes
}
FP8_TORCH = {DT_E4M3: torch.float8_e4m3fn, DT_E5M2: torch.float8_e5m2}


class Fp8Tensor(ctypes.Structure):
    _fields_ = [("ptr", ctypes.c_void_p), ("dtype", ctypes.c_int32), ("ndim", ctypes.c_int32),
                ("shape", ctypes.c_int64 * 3)]


class Fp8LinearSaved(ctypes.Structure):
    _fields_ = [(n, Fp8Tensor) for n in ("x_q", "x_inv", "w_q", "w_inv", "xt_q", "wt_q", "xt_inv", "wt_inv")]


class Fp8Error(RuntimeError):
    def __init__(self, code: int, where: str):
        super().__init__(f"{where}: {status_string(code)} (code {code})")
        self.code = code


def _load():
    if not os.path.exists(LIB_PATH):
        raise ImportError(f"fp8lin library not built: {LIB_PATH} missing (run __graft_entry__.build())")
    L = ctypes.CDLL(LIB_PATH)
    P = ctypes.c_void_p
    T = ctypes.POINTER(Fp8Tensor)
    L.fp8_quantize.argtypes = [T, ctypes.c_int, ctypes.c_int, ctypes.c_int, T, T, T, T, P, ctypes.c_size_t, P, P]
    L.fp8_scaled_mm.argtypes = [T, T, T, T, T, ctypes.c_int, P, P]
    L.fp8_grouped_mm.argtypes = [T, T, T, T, T, T, ctypes.c_int, ctypes.c_int, P, P]
    L.fp8_linear_fwd.argtypes = [T, T, ctypes.c_int, ctypes.c_int, T, ctypes.POINTER(Fp8LinearSaved), P,
                                 ctypes.c_size_t, P, P]
    L.fp8_linear_bwd.argtypes = [T, ctypes.POINTER(Fp8LinearSaved), T, T, ctypes.c_int, ctypes.c_int, T, T, P,
                                 ctypes.c_size_t, P, P]
    L.fp8_workspace_size.argtypes = [ctypes.c_int, ctypes.c_int64, ctypes.c_int64, ctypes.c_int64, ctypes.c_int,
                                     ctypes.c_int]
    L.fp8_workspace_size.restype = ctypes.c_size_t
    L.fp8_jagged_padded_rows.argtypes = [ctypes.c_int64, ctypes.c_int64]
    L.fp8_jagged_padded_rows.restype = ctypes.c_int64
    L.fp8_mx_scale_bytes.argtypes = [ctypes.c_int64, ctypes.c_int64]
    L.fp8_mx_scale_bytes.restype = ctypes.c_int64
    L.fp8_status_string.argtypes = [ctypes.c_int]
    L.fp8_status_string.restype = ctypes.c_char_p
    L.fp8_set_wait_limit_ns.argtypes = [ctypes.c_uint64]
    L.fp8_set_wait_limit_ns.restype = ctypes.c_uint64
    L.fp8_quantize_tensor_noalloc.argtypes = [T, ctypes.c_int, ctypes.c_int, T, T, T, P]
    L.fp8_scaled_mm_amax.argtypes = [T, T, T, T, T, ctypes.c_int, T, T, P, P]
    L.fp8_quantize_from_amax.argtypes = [T, ctypes.c_int, ctypes.c_int, ctypes.c_int, T, T, T, T, P, P]
    L.fp8_set_test_stall.argtypes = [ctypes.c_int]
    L.fp8_test_cast_bits.argtypes = [ctypes.c_uint32, ctypes.c_int64, ctypes.c_int, P, P]
    L.fp8_scaled_mm_quant.argtypes = [T, T, T, T, ctypes.c_int, ctypes.c_int, T, T, P, P]
    L.fp8_set_test_stall.restype = ctypes.c_int
    return L


lib = _load()

# Symbols include/fp8lin.h declares (checked by the CPU tests against the header and the .so).
EXPORTS = ("fp8_quantize", "fp8_scaled_mm", "fp8_grouped_mm", "fp8_linear_fwd", "fp8_linear_bwd",
           "fp8_workspace_size", "fp8_jagged_padded_rows", "fp8_status_string", "fp8_set_wait_limit_ns",
           "fp8_quantize_tensor_noalloc", "fp8_set_test_stall", "fp8_mx_scale_bytes", "fp8_scaled_mm_amax",
           "fp8_quantize_from_amax", "fp8_test_cast_bits", "fp8_scaled_mm_quant")


def status_string(code: int) -> str:
    return lib.fp8_status_string(int(code)).decode()


def desc(t: torch.Tensor | None, dtype: int | None = None):
    """fp8_tensor descriptor of a dense torch tensor (None -> NULL)."""
    if t is None:
        return None
    if not t.is_contiguous():
        raise ValueError("tensors passed to fp8lin must be contiguous")
    if t.dim() < 1 or t.dim() > 3:
        raise ValueError("fp8lin tensors have 1 to 3 dimensions")
    d = Fp8Tensor()
    d.ptr = t.data_ptr() if t.numel() else 0
    d.dtype = dtype if dtype is not None else _TORCH_DT[t.dtype]
    d.ndim = t.dim()
    for i, s in enumerate(t.shape):
        d.shape[i] = s
    return d


def _ref(d):
    return None if d is None else ctypes.byref(d)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream):
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(rc: int, where: str):
    if rc != OK:
        raise Fp8Error(rc, where)


def fp8_quantize(x, granularity, out_dtype, layout, out=None, out_t=None, inv_scales=None, offsets=None,
                 workspace=None, status=None, stream=None):
    rc = lib.fp8_quantize(_ref(desc(x)), granularity, out_dtype, layout, _ref(desc(out)), _ref(desc(out_t)),
                          _ref(desc(inv_scales)), _ref(desc(offsets)), _ptr(workspace),
                          0 if workspace is None else workspace.numel() * workspace.element_size(),
                          _ptr(status), _stream(stream))
    _check(rc, "fp8_quantize")


def fp8_scaled_mm(A, B, sA, sB, out, flags=0, status=None, stream=None):
    rc = lib.fp8_scaled_mm(_ref(desc(A)), _ref(desc(B)), _ref(desc(sA)), _ref(desc(sB)), _ref(desc(out)), flags,
                           _ptr(status), _stream(stream))
    _check(rc, "fp8_scaled_mm")


def fp8_scaled_mm_amax(A, B, sA, sB, out, flags=0, row_amax=None, col_amax=None, status=None, stream=None):
    """fp8_scaled_mm plus max |out| per row / per column (fp32 tensors [M] / [N]) from the epilogue."""
    rc = lib.fp8_scaled_mm_amax(_ref(desc(A)), _ref(desc(B)), _ref(desc(sA)), _ref(desc(sB)), _ref(desc(out)), flags,
                                _ref(desc(row_amax)), _ref(desc(col_amax)), _ptr(status), _stream(stream))
    _check(rc, "fp8_scaled_mm_amax")


def fp8_scaled_mm_quant(A, B, sA, sB, out_q, out_scales, out_granularity, flags=0, status=None, stream=None):
    """fp8_scaled_mm whose epilogue writes the result's next quantization: codes out_q [M, N] and
    1 x 128 (fp32 [M, N/128]) or MX (E8M0 bytes) scales out_scales."""
    sdt = DT_E8M0 if out_granularity == GRAN_MX else None
    rc = lib.fp8_scaled_mm_quant(_ref(desc(A)), _ref(desc(B)), _ref(desc(sA)), _ref(desc(sB)), flags, out_granularity,
                                 _ref(desc(out_q)), _ref(desc(out_scales, sdt)), _ptr(status), _stream(stream))
    _check(rc, "fp8_scaled_mm_quant")


def fp8_quantize_from_amax(x, granularity, out_dtype, layout, out=None, out_t=None, inv_scales=None, amax=None,
                           status=None, stream=None):
    """The scale and cast steps of fp8_quantize with the amax given (tensor [1] or column [C])."""
    rc = lib.fp8_quantize_from_amax(_ref(desc(x)), granularity, out_dtype, layout, _ref(desc(out)),
                                    _ref(desc(out_t)), _ref(desc(inv_scales)), _ref(desc(amax)), _ptr(status),
                                    _stream(stream))
    _check(rc, "fp8_quantize_from_amax")


def fp8_grouped_mm(A, B, offsets, sA, sB, out, mode, flags=0, status=None, stream=None):
    rc = lib.fp8_grouped_mm(_ref(desc(A)), _ref(desc(B)), _ref(desc(offsets)), _ref(desc(sA)), _ref(desc(sB)),
                            _ref(desc(out)), mode, flags, _ptr(status), _stream(stream))
    _check(rc, "fp8_grouped_mm")


def make_saved(x_q, x_inv, w_q, w_inv, xt_q=None, wt_q=None, xt_inv=None, wt_inv=None) -> Fp8LinearSaved:
    s = Fp8LinearSaved()
    s.x_q, s.x_inv, s.w_q, s.w_inv = desc(x_q), desc(x_inv), desc(w_q), desc(w_inv)
    for name, t in (("xt_q", xt_q), ("wt_q", wt_q), ("xt_inv", xt_inv), ("wt_inv", wt_inv)):
        if t is not None:
            setattr(s, name, desc(t))
    return s


def linear_saved_alloc(M: int, K: int, N: int, granularity: int, keep_xt: bool = True, device="cuda"):
    """Caller-owned buffers of fp8_linear_saved for a granularity; returns (saved, tensors) where
    `tensors` keeps the torch buffers alive (x_q, x_inv, w_q, w_inv, xt_q, wt_q, xt_inv, wt_inv)."""
    e4 = torch.float8_e4m3fn
    x_q = torch.empty((M, K), dtype=e4, device=device)
    w_q = torch.empty((N, K), dtype=e4, device=device)
    xt_q = wt_q = xt_inv = wt_inv = None
    if granularity == GRAN_BLOCK_1x128:  # 1 x 128 tiles of x, 128 x 128 tiles of W (both layouts)
        f32 = torch.float32
        x_inv = torch.empty((M, K // 128), dtype=f32, device=device)
        w_inv = torch.empty((N // 128, K // 128), dtype=f32, device=device)
        wt_q = torch.empty((K, N), dtype=e4, device=device)
        wt_inv = torch.empty((K // 128, N // 128), dtype=f32, device=device)
    elif granularity == GRAN_MX:
        u8 = torch.uint8
        x_inv = torch.empty(fp8_mx_scale_bytes(M, K), dtype=u8, device=device)
        w_inv = torch.empty(fp8_mx_scale_bytes(N, K), dtype=u8, device=device)
        wt_q = torch.empty((K, N), dtype=e4, device=device)
        wt_inv = torch.empty(fp8_mx_scale_bytes(K, N), dtype=u8, device=device)
        if keep_xt:
            xt_q = torch.empty((K, M), dtype=e4, device=device)
            xt_inv = torch.empty(fp8_mx_scale_bytes(K, M), dtype=u8, device=device)
    else:
        tens = granularity == GRAN_TENSOR
        x_inv = torch.empty(1 if tens else M, dtype=torch.float32, device=device)
        w_inv = torch.empty(1 if tens else N, dtype=torch.float32, device=device)
        if tens:
            wt_q = torch.empty((K, N), dtype=e4, device=device)
            if keep_xt:
                xt_q = torch.empty((K, M), dtype=e4, device=device)
    tensors = (x_q, x_inv, w_q, w_inv, xt_q, wt_q, xt_inv, wt_inv)
    return make_saved(*tensors), tensors


def fp8_linear_fwd(x, w, granularity, flags, y, saved: Fp8LinearSaved, workspace=None, status=None, stream=None):
    rc = lib.fp8_linear_fwd(_ref(desc(x)), _ref(desc(w)), granularity, flags, _ref(desc(y)), ctypes.byref(saved),
                            _ptr(workspace), 0 if workspace is None else workspace.numel() * workspace.element_size(),
                            _ptr(status), _stream(stream))
    _check(rc, "fp8_linear_fwd")


def fp8_linear_bwd(dy, saved: Fp8LinearSaved, x, w, granularity, wgrad_mode, dx, dw, workspace=None, status=None,
                   stream=None):
    rc = lib.fp8_linear_bwd(_ref(desc(dy)), ctypes.byref(saved), _ref(desc(x)), _ref(desc(w)), granularity,
                            wgrad_mode, _ref(desc(dx)), _ref(desc(dw)), _ptr(workspace),
                            0 if workspace is None else workspace.numel() * workspace.element_size(),
                            _ptr(status), _stream(stream))
    _check(rc, "fp8_linear_bwd")


def fp8_quantize_tensor_noalloc(x, out_dtype, layout, out=None, out_t=None, inv_scale=None, stream=None):
    """Tensorwise quantize without a workspace (the library's fixed device array holds the amax
    reduction); for callers that cannot allocate. Same results as fp8_quantize(GRAN_TENSOR)."""
    rc = lib.fp8_quantize_tensor_noalloc(_ref(desc(x)), out_dtype, layout, _ref(desc(out)), _ref(desc(out_t)),
                                         _ref(desc(inv_scale)), _stream(stream))
    _check(rc, "fp8_quantize_tensor_noalloc")


def fp8_workspace_size(op, d0=0, d1=0, d2=0, granularity=0, wgrad_mode=0) -> int:
    return int(lib.fp8_workspace_size(op, d0, d1, d2, granularity, wgrad_mode))


def fp8_jagged_padded_rows(rows: int, n_segments: int) -> int:
    return int(lib.fp8_jagged_padded_rows(rows, n_segments))


def fp8_mx_scale_bytes(rows: int, k: int) -> int:
    return int(lib.fp8_mx_scale_bytes(rows, k))


def fp8_set_wait_limit_ns(ns: int) -> int:
    return int(lib.fp8_set_wait_limit_ns(ns))


def fp8_set_test_stall(enable: bool) -> int:
    return int(lib.fp8_set_test_stall(1 if enable else 0))


# ------------------------------------------------------------------------------------------
# allocation helpers (torch buffers of the right shapes, then the entry points above)

def col_workspace(groups: int, cols: int, rows: int, device) -> torch.Tensor:
    """Workspace of a column-granularity fp8_quantize of `rows` rows (all groups) x `cols` columns."""
    n = fp8_workspace_size(OP_QUANTIZE, groups, cols, rows, granularity=GRAN_COL)
    return torch.empty(max(n // 4, 4), dtype=torch.int32, device=device)


def quantize_alloc(x, granularity, out_dtype, layout=None, offsets=None, padded_rows=None, status=None,
                   stream=None):
    """Returns (out or None, out_t or None, inv_scales). Shapes follow include/fp8lin.h."""
    dev = x.device
    if layout is None:
        layout = LAYOUT_COL_MAJOR if granularity == GRAN_COL else LAYOUT_ROW_MAJOR
    fdt = FP8_TORCH[out_dtype]
    R, C = x.shape[-2], x.shape[-1]
    B = x.shape[0] if x.dim() == 3 else 1
    out = torch.empty(x.shape, dtype=fdt, device=dev) if layout & LAYOUT_ROW_MAJOR else None
    out_t = None
    ws = None
    if granularity == GRAN_TENSOR:
        inv = torch.empty(1, dtype=torch.float32, device=dev)
        ws = torch.empty(2, dtype=torch.int32, device=dev)  # amax word, grid-barrier count
        if layout & LAYOUT_COL_MAJOR:
            out_t = torch.empty((C, R), dtype=fdt, device=dev)
    elif granularity == GRAN_ROW:
        inv = torch.empty(x.shape[:-1], dtype=torch.float32, device=dev)
    else:
        if offsets is not None:
            E = offsets.numel()
            P = padded_rows or fp8_jagged_padded_rows(R, E)
            out_t = torch.empty((C, P), dtype=fdt, device=dev)
            inv = torch.empty((E, C), dtype=torch.float32, device=dev)
            groups = E
        else:
            out_t = torch.empty((B, C, R) if x.dim() == 3 else (C, R), dtype=fdt, device=dev)
            inv = torch.empty((B, C) if x.dim() == 3 else (C,), dtype=torch.float32, device=dev)
            groups = B
        ws = col_workspace(groups, C, B * R, dev)
    fp8_quantize(x, granularity, out_dtype, layout, out, out_t, inv, offsets, ws, status=status, stream=stream)
    return out, out_t, inv


def mx_quantize_alloc(x, out_dtype, layout=LAYOUT_ROW_MAJOR, offsets=None, padded_rows=None, status=None,
                      stream=None):
    """MXFP8 quantize (blocks of 32, E8M0 scales). Returns (out or None, out_t or None,
    row-major scales or None, column-major scales or None); scales are uint8 tensors in the MX
    scale layout of include/fp8lin.h."""
    dev = x.device
    fdt = FP8_TORCH[out_dtype]
    R, C = x.shape[-2], x.shape[-1]
    B = x.shape[0] if x.dim() == 3 else 1
    out = torch.empty(x.shape, dtype=fdt, device=dev) if layout & LAYOUT_ROW_MAJOR else None
    ws = None
    if offsets is not None:
        E = offsets.numel()
        P = padded_rows or fp8_jagged_padded_rows(R, E)
        out_t = torch.empty((C, P), dtype=fdt, device=dev) if layout & LAYOUT_COL_MAJOR else None
        row_bytes = fp8_mx_scale_bytes(P, C) if layout & LAYOUT_ROW_MAJOR else 0
        col_bytes = fp8_mx_scale_bytes(C, P) if layout & LAYOUT_COL_MAJOR else 0
        ws = torch.empty(max(fp8_workspace_size(OP_QUANTIZE, E, C, granularity=GRAN_MX) // 4, 4), dtype=torch.int32,
                         device=dev)
    else:
        out_t = None
        if layout & LAYOUT_COL_MAJOR:
            out_t = torch.empty((B, C, R) if x.dim() == 3 else (C, R), dtype=fdt, device=dev)
        row_bytes = B * fp8_mx_scale_bytes(R, C) if layout & LAYOUT_ROW_MAJOR else 0
        col_bytes = B * fp8_mx_scale_bytes(C, R) if layout & LAYOUT_COL_MAJOR else 0
    row_bytes, col_bytes = max(row_bytes, 0), max(col_bytes, 0)  # bad shapes: the library rejects them
    sf = torch.empty(row_bytes + col_bytes, dtype=torch.uint8, device=dev)
    fp8_quantize(x, GRAN_MX, out_dtype, layout, out, out_t, sf, offsets, ws, status=status, stream=stream)
    return out, out_t, (sf[:row_bytes] if row_bytes else None), (sf[row_bytes:] if col_bytes else None)


def blk_quantize_alloc(x, out_dtype, tile128=False, layout=LAYOUT_ROW_MAJOR, status=None, stream=None):
    """Blockwise quantize: 1 x 128 tiles (row-major) or 128 x 128 tiles (row- and/or column-major).
    Returns (out or None, out_t or None, inverse scales of out or None, of out_t or None)."""
    dev = x.device
    fdt = FP8_TORCH[out_dtype]
    R, C = x.shape
    out = torch.empty((R, C), dtype=fdt, device=dev) if layout & LAYOUT_ROW_MAJOR else None
    out_t = torch.empty((C, R), dtype=fdt, device=dev) if layout & LAYOUT_COL_MAJOR else None
    if not tile128:
        inv = torch.empty((R, max(C // 128, 1)), dtype=torch.float32, device=dev)
        fp8_quantize(x, GRAN_BLOCK_1x128, out_dtype, layout, out, out_t, inv, status=status, stream=stream)
        return out, out_t, inv, None
    nr = -(-R // 128) * (C // 128) if out is not None else 0
    nc = (C // 128) * (R // 128) if out_t is not None else 0
    inv = torch.empty(max(nr + nc, 1), dtype=torch.float32, device=dev)
    fp8_quantize(x, GRAN_BLOCK_128x128, out_dtype, layout, out, out_t, inv[:nr + nc] if nr + nc else inv,
                 status=status, stream=stream)
    return (out, out_t, inv[:nr].view(-1, C // 128) if nr else None,
            inv[nr:nr + nc].view(C // 128, R // 128) if nc else None)
