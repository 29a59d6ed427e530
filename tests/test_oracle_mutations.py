"""The pins have teeth: each plausible mistake below is planted in a copy of the oracle (the C
source, on the CPU), the copy is compiled, and the oracle's pin tests (tests/test_oracle.py,
tests/test_oracle_mx.py and tests/test_oracle_blocks.py) are run against it in a subprocess;
every mutant must make at least one pin fail. The mistakes cover each step of the recipe and of the GEMMs: rounding ties, the subnormal binade, the eps clamp,
the direction of the scale, the inverse scale's rounding, a dropped product in the contraction,
a segment boundary, the column of a transposed operand; for MXFP8 the scale rule's exponent,
floor and clamp, the block amax, and the block index of a scale in the GEMM; for blockwise
scaling a tile's edge and the K block of each operand's scale."""
import os
import re
import subprocess
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
SRC = os.path.join(ROOT, "oracle", "oracle.c")

MUTANTS = {
    # round half away from zero instead of half to even
    "ties_away": ("if (rem > half || (rem == half && (n & 1u))) n += 1;", "if (rem >= half) n += 1;"),
    # no floor at the smallest normal binade: subnormal results get the wrong quantum
    "subnormal_binade": ("int E8 = lg > f.emin ? lg : f.emin;", "int E8 = lg;"),
    # another eps
    "eps": ("static const double ORC_EPS = 1e-12;", "static const double ORC_EPS = 1e-10;"),
    # the scale upside down
    "scale_direction": ("double s = fp8_max / a;", "double s = a / fp8_max;"),
    # the inverse taken from the fp32 scale instead of the fp64 one
    "inverse_from_fp32": ("if (inv32) *inv32 = (float)(1.0 / s);", "if (inv32) *inv32 = 1.0f / (float)s;"),
    # the last product of every FP8 dot product dropped
    "dropped_product": ("double p = ta[A[m * a_sm + k * a_sk]] * tb[B[n * b_sn + k * b_sk]];",
                        "double p = k + 1 < K ? ta[A[m * a_sm + k * a_sk]] * tb[B[n * b_sn + k * b_sk]] : 0.0;"),
    # a jagged segment starting one row late
    "segment_edge": ("int64_t r0 = e ? ends[e - 1] : 0, r1 = ends[e];\n    /* an empty segment",
                     "int64_t r0 = e ? ends[e - 1] + 1 : 0, r1 = ends[e];\n    if (r0 > r1) r0 = r1;\n    /* an empty segment"),
    # B read with A's column stride (a transposed-operand mix-up)
    "operand_stride": ("tb[B[n * b_sn + k * b_sk]]", "tb[B[n * b_sn + k * a_sk]]"),
    # MX: e4m3's largest-normal exponent off by one
    "mx_emax": ("return fmt == ORC_E4M3 ? 8 : 15;", "return fmt == ORC_E4M3 ? 7 : 15;"),
    # MX: ceil(log2 amax) where the rule takes the floor
    "mx_ceil_log2": ("e = (ex - 1) - mx_emax_elem(fmt);", "e = ex - mx_emax_elem(fmt);"),
    # MX: no clamp of the scale exponent at -127
    "mx_no_clamp": ("if (e < -127) e = -127;\n    if (e > 127)", "if (e > 127)"),
    # MX: block amax taken over signed values, not magnitudes
    "mx_signed_amax": ("float a = fabsf(bf16_to_float(xb[i]));", "float a = bf16_to_float(xb[i]);"),
    # MX GEMM: B's first block scale used for every block
    "mx_block_index": ("ts[sB[n * nb + k / 32]]", "ts[sB[n * nb]]"),
    # blockwise: a tile's last row left out
    "blk_tile_edge": ("int64_t r1 = r0 + br < R ? r0 + br : R, c1", "int64_t r1 = r0 + br - 1 < R ? r0 + br - 1 : R, c1"),
    # blockwise GEMM: the weight tile's scale taken from the first K block only
    "blk_weight_kblock": ("(double)sB[(n / 128) * kb + k / 128]", "(double)sB[(n / 128) * kb]"),
    # blockwise GEMM: the activation's scale from 256-wide K blocks
    "blk_act_kblock": ("(double)sA[m * kb + k / 128]", "(double)sA[m * kb + k / 256]"),
}


def _build_mutant(name, tmp_path):
    src = open(SRC).read()
    if name != "unchanged":
        old, new = MUTANTS[name]
        assert src.count(old) >= 1, f"mutation site of {name} not found"
        src = src.replace(old, new)
    path_c = tmp_path / f"oracle_{name}.c"
    path_c.write_text(src)
    so = tmp_path / f"liboracle_{name}.so"
    subprocess.run(["gcc", "-std=c11", "-O2", "-fopenmp", "-ffp-contract=off", "-fno-fast-math", "-fPIC",
                    "-shared", "-I", os.path.join(ROOT, "oracle"), "-o", str(so), str(path_c), "-lm"], check=True)
    return so


def _run_pins(so):
    env = dict(os.environ, FP8LIN_ORACLE_LIB=str(so))
    return subprocess.run([sys.executable, "-m", "pytest", os.path.join(ROOT, "tests", "test_oracle.py"),
                           os.path.join(ROOT, "tests", "test_oracle_mx.py"), os.path.join(ROOT, "tests", "test_oracle_blocks.py"),
                           "-x", "-q", "-p", "no:cacheprovider"],
                          cwd=ROOT, env=env, capture_output=True, text=True, timeout=600)


def test_unchanged_copy_passes(tmp_path):
    """Control: an unmodified copy built the same way passes every pin."""
    r = _run_pins(_build_mutant("unchanged", tmp_path))
    assert r.returncode == 0, r.stdout[-2000:]


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_pins_catch_mutant(name, tmp_path):
    r = _run_pins(_build_mutant(name, tmp_path))
    summary = r.stdout.strip().splitlines()[-1] if r.stdout.strip() else ""
    # a pin failed (not a collection or import error)
    assert r.returncode == 1 and re.match(r"\d+ failed", summary) and "error" not in summary, \
        f"mutant {name} was not caught by a failing pin:\n{r.stdout[-2000:]}"
