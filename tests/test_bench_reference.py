"""The bench's reference arm and CPU baselines (CPU only): the oracle on host-drawn samples of
every workload, and the reference arm's JSON line."""
import json
import os
import subprocess
import sys

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)

import bench  # noqa: E402
import workloads as W  # noqa: E402


def _small_rows(name):
    if name == "llama3-8b-mlp-up-mx":
        return 32  # MX blocks of 32 along the tokens for the weight gradient's operands
    if name in ("colwise-8192x14336", "llama3-8b-tensorwise-quant"):
        return 256
    return 1


def test_every_workload_has_a_host_sample():
    """Each workload's host-drawn sample runs through the oracle and counts positive work in the
    workload's unit (bytes for the quantize-only workloads, GEMM FLOPs otherwise)."""
    for name in W.WORKLOADS:
        assert name in bench.SAMPLE_ROWS or name == "linear-tensorwise-256x512", name
        run, work, sample = bench.host_cpu_sample(name, _small_rows(name))
        run()
        assert work > 0 and sample, name
        assert bench.workload_unit(name) in ("GB/s", "TFLOP/s")


def test_sample_work_counts():
    """Work of a few samples by hand: the tensorwise Linear is three GEMMs of 256 x 256 x 512; the
    Llama4 sample is two GEMM rows per routed row plus the 64 x 64 weight-gradient block of its
    expert's segment."""
    _, work, _ = bench.host_cpu_sample("linear-tensorwise-256x512")
    assert work == 3 * 2.0 * 256 * 256 * 512
    _, work, sample = bench.host_cpu_sample("llama4-moe-fwdbwd", 1)
    counts = W.llama4_counts(0)
    row = np.random.default_rng(0).choice(8192, 1, replace=False)
    e = int(np.searchsorted(W.ends_from_counts(counts), row, side="right")[0])
    c0 = int(counts[e])
    assert sample.endswith(f"expert {e} ({c0} rows)")
    assert work == 2 * 2.0 * 8192 * 5120 + 2.0 * c0 * 64 * 64
    _, work, _ = bench.host_cpu_sample("colwise-8192x14336", 256)
    assert work == 3.0 * 8192 * 256 + 4 * 256 + 3.0 * 256 * 4096 + 4 * 256


def test_reference_line_contract():
    """`bench.py --impl reference` prints one JSON line: the oracle's throughput in the workload's
    metric and unit, with itself as the CPU baseline and no host-device bytes."""
    p = subprocess.run([sys.executable, "bench.py", "--impl", "reference", "--workload", "linear-tensorwise-256x512",
                        "--steps", "1", "--warmup", "3"], capture_output=True, text=True, cwd=ROOT, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    d = json.loads(p.stdout.strip().splitlines()[-1])
    assert d["impl"] == "reference" and d["metric"] == bench.METRIC and d["unit"] == "TFLOP/s"
    assert d["value"] > 0 and d["higher_is_better"] is True and d["steps"] == 1 and d["warmup"] == 3
    assert d["config"]["workload"] == "linear-tensorwise-256x512"
    cb = d["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == d["value"] and cb["cores"] >= 1 and cb["sample"]
    assert d["e2e"] == {"value": d["value"], "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}


def test_full_tensor_quantize_line():
    """`bench.py --cpu-full-quantize` times the oracle's quantize of each full-size tensor of a
    workload: one entry per tensor with its element count, rate and seconds."""
    p = subprocess.run([sys.executable, "bench.py", "--cpu-full-quantize", "--workload", "linear-tensorwise-256x512"],
                       capture_output=True, text=True, cwd=ROOT, timeout=600)
    assert p.returncode == 0, p.stderr[-2000:]
    d = json.loads(p.stdout.strip().splitlines()[-1])
    assert d["kind"] == "oracle full-tensor quantize" and d["cores"] >= 1
    assert [t["tensor"] for t in d["tensors"]] == ["x e4m3 tensorwise", "W e4m3 tensorwise", "dY e5m2 tensorwise"]
    assert [t["elements"] for t in d["tensors"]] == [256 * 512, 256 * 512, 256 * 256]
    assert all(t["GB/s"] > 0 and t["seconds"] >= 0 for t in d["tensors"])
