"""The cast step of every quantize kernel, exhaustively ("FP8 Training: Quantization, Autograd,
Torchao", section 2: the scaled value is cast round-to-nearest-even and saturated; section 3: the
e4m3 and e5m2 formats).

Every fp32 value in [-fp8_max, fp8_max] goes through the library's own cast on the GPU
(fp8_test_cast_bits runs the cvt the kernels use) and is compared with the oracle's bit-level
encoder on the same value. Values beyond fp8_max, up to infinity, must give the code of +-fp8_max,
which is what the recipe's clamp before the cast gives (the kernels rely on the saturating cvt in
place of that clamp). The bit patterns are generated on both sides from their index; no value
passes from the GPU to the oracle."""
import ctypes

import numpy as np
import pytest
import torch

import oracle

pytestmark = pytest.mark.gpu
CHUNK = 1 << 28


@pytest.fixture(scope="module")
def fp8():
    import moe_grouped_gemm_absmax_gb300 as m
    return m


def _gpu_codes(fp8, first, n, dt, out):
    rc = fp8.lib.fp8_test_cast_bits(first, n, dt, ctypes.c_void_p(out.data_ptr()),
                                    ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert rc == 0, fp8.status_string(rc)
    return out[:n].cpu().numpy()


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_every_fp32_up_to_fp8_max(fp8, fmt):
    dt = fp8.DT_E4M3 if fmt == oracle.E4M3 else fp8.DT_E5M2
    top = int(np.float32(oracle.fp8_max(fmt)).view(np.uint32))  # the bit pattern of +fp8_max
    base = np.arange(CHUNK, dtype=np.uint32)
    pat = np.empty(CHUNK, np.uint32)
    out = torch.empty(CHUNK, dtype=torch.uint8, device="cuda")
    for sign in (0, 0x80000000):
        end = sign + top + 1
        for a in range(sign, end, CHUNK):
            n = min(CHUNK, end - a)
            got = _gpu_codes(fp8, a, n, dt, out)
            np.add(base[:n], np.uint32(a), out=pat[:n])
            ref = oracle.encode(pat[:n].view(np.float32), fmt)
            bad = np.flatnonzero(got != ref)
            assert bad.size == 0, (f"{bad.size} codes differ; first at bits {a + int(bad[0]):#010x}: "
                                   f"gpu {got[bad[0]]:#04x} oracle {ref[bad[0]]:#04x}")


@pytest.mark.parametrize("fmt", [oracle.E4M3, oracle.E5M2])
def test_beyond_fp8_max_saturates_like_the_clamp(fp8, fmt):
    """Every 4099th fp32 above fp8_max up to +-inf (and the patterns right above fp8_max): the
    code of the clamped value, i.e. the largest finite code with the value's sign."""
    dt = fp8.DT_E4M3 if fmt == oracle.E4M3 else fp8.DT_E5M2
    qmax = np.float32(oracle.fp8_max(fmt))
    top = int(qmax.view(np.uint32))
    inf = 0x7F800000
    out = torch.empty(1 << 20, dtype=torch.uint8, device="cuda")
    for sign in (0, 0x80000000):
        firsts = [sign + top + 1] + list(range(sign + top + 4096, sign + inf + 1, 4099 * 4096))
        want = oracle.encode(np.array([qmax if sign == 0 else -qmax], np.float32), fmt)[0]
        for a in firsts:
            n = min(4096, sign + inf + 1 - a)
            got = _gpu_codes(fp8, a, n, dt, out)
            assert (got == want).all(), f"bits {a:#010x}: codes {np.unique(got)} vs {want:#04x}"
