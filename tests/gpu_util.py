"""Helpers shared by the GPU parity tests (host-side plumbing only)."""
import numpy as np
import torch

import workloads as W


def dev_bf16(t_cpu: torch.Tensor) -> torch.Tensor:
    return t_cpu.to("cuda")


def codes(t: torch.Tensor) -> np.ndarray:
    return t.view(torch.uint8).cpu().numpy()


def f32_bits(t: torch.Tensor) -> np.ndarray:
    return t.float().cpu().numpy().view(np.uint32)


def bits(t_cpu: torch.Tensor) -> np.ndarray:
    return W.bf16_bits(t_cpu)


def special_rows(C: int, fmt_max: float) -> torch.Tensor:
    """Rows that probe the cast: exact fp8 ties at scale 1 (amax = fp8_max), fp8 subnormal ties,
    a single huge outlier, all zeros, negative zeros, tiny values that underflow."""
    rows = []
    r = torch.zeros(C)
    r[0] = fmt_max
    ties = torch.tensor([1.0625, 1.1875, -1.3125, 2.125, -3.25, 0.0078125 * 1.5, 2.0 ** -10, 3 * 2.0 ** -10,
                         -(2.0 ** -10), 2.0 ** -17, 3 * 2.0 ** -17, 5 * 2.0 ** -18])
    n = min(C - 1, ties.numel())
    r[1:1 + n] = ties[:n]
    rows.append(r)
    r = torch.randn(C, generator=torch.Generator().manual_seed(5)) * 1e-3
    r[C // 2] = 3.0e4
    rows.append(r)
    rows.append(torch.zeros(C))
    r = torch.zeros(C)
    r[::3] = -0.0
    rows.append(r)
    r = torch.full((C,), 1e-30)
    r[-1] = 1.0
    rows.append(r)
    return torch.stack(rows).to(torch.bfloat16)


FP8_TORCH = {0: torch.float8_e4m3fn, 1: torch.float8_e5m2}  # oracle fmt -> torch dtype


def upload_codes(c: np.ndarray, fmt: int) -> torch.Tensor:
    """Oracle-produced FP8 codes as a device tensor of the matching float8 dtype."""
    return torch.from_numpy(np.ascontiguousarray(c)).view(FP8_TORCH[fmt]).cuda()


def upload_f32(a: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(np.ascontiguousarray(a, dtype=np.float32)).cuda()


def check_gemm(got, ref, absacc, out_bf16, tol=2e-3):
    """|got - ref| <= tol * absacc (+ half a bf16 ulp of ref when the output is bf16)."""
    got = got.detach().double().cpu().numpy() if isinstance(got, torch.Tensor) else got
    bound = tol * absacc + (2.0 ** -8 * np.abs(ref) if out_bf16 else 0.0) + 1e-30
    err = np.abs(got - ref)
    bad = err > bound
    assert not bad.any(), (f"{bad.sum()} of {bad.size} outside the bound; worst excess "
                           f"{(err - bound).max():.3e} at {np.unravel_index(np.argmax(err - bound), err.shape)}")


def segpad_cols(q_rows: np.ndarray, ends, P: int) -> np.ndarray:
    """Row-major codes [R, C] -> the segment-padded column-major layout [C, P]: segment e starts
    at the sum of the previous segments' lengths rounded up to 128, zeros fill the gaps."""
    R, C = q_rows.shape
    out = np.zeros((C, P), np.uint8)
    prev, pos = 0, 0
    for e in ends:
        e = int(e)
        out[:, pos:pos + e - prev] = q_rows[prev:e].T
        pos += -(-(e - prev) // 128) * 128
        prev = e
    return out


def mx_offsets(rows, K):
    """Byte offsets of (row r, K block j) in the MX scale layout of include/fp8lin.h, for the
    given rows (an index array) and every j < K / 32: a pure index permutation."""
    r = np.asarray(rows, np.int64)[:, None]
    j = np.arange(K // 32, dtype=np.int64)[None, :]
    return ((r // 128) * (K // 128) + j // 4) * 512 + (r % 32) * 16 + ((r // 32) % 4) * 4 + j % 4


def mx_unblock_rows(sf, rows, K):
    """Plain E8M0 codes [len(rows), K / 32] of the given rows, read from layout bytes (a device
    tensor is indexed on the device; only the selected codes come back)."""
    off = mx_offsets(rows, K)
    if isinstance(sf, torch.Tensor):
        return sf[torch.as_tensor(off.ravel(), device=sf.device)].cpu().numpy().reshape(off.shape)
    return np.asarray(sf)[off]
