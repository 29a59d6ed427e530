"""Benchmark of the FP8 dynamic-scaling linear on one or more GB300s (one process per GPU).

Default workload: the DeepSeek-V3-shaped MoE layer forward (dsv3-moe-fwd): 256 experts, hidden
K=7168, expert intermediate N=2048, 16384 tokens top-8 = 131072 routed rows with seeded Zipf(1.1)
expert counts including 8 empty experts. One step = quantize the routed activations A
[131072, 7168] rowwise (e4m3), quantize the expert weights W [256, 2048, 7168] per expert column
(e4m3), and the grouped FP8 GEMM routed by the offsets (jagged M): 3 kernels, 3.85 TFLOP.

Other workloads (`--workload`): llama3-8b-mlp-up (the Llama3-8B-shaped dense MLP-up Linear,
forward + backward, rowwise), linear-tensorwise-256x512, colwise-8192x14336, llama4-moe-fwdbwd,
llama3-8b-dx-colquant-fused, llama3-8b-mlp-up-blockwise, llama3-8b-mlp-up-mx, dsv3-moe-fwd-mx,
llama4-moe-fwdbwd-mx.

`value` = whole-job throughput with inputs resident in HBM (CUDA events around each step on the
launching stream, L2 flushed between steps outside the events: a 256 MiB write, then a 256 MiB
read of a second buffer, so the cache is cold and holds no dirty lines of the flush, then a ~50 us
GPU spin while the flush's write-backs drain; a GPU spin before the first step gives the host a
head start, so that no timed kernel waits for its own launch);
`e2e` = the same metric through the public entry points with host buffers (pinned host->device
copies of the step's inputs and device->host copies of its outputs inside the timed region).
`--impl reference` times the CPU oracle (the plain C restatement used by the tests) on a bounded
sample of the same workload; it is a deliberately slow reference, not a target.

Under torchrun (WORLD_SIZE > 1) every rank runs an independent replica of the workload on its
own GPU (the path shards by tokens / experts with no data exchange): weak scaling, the timing is
the max over ranks, and `value` counts the work of all ranks.
"""
from __future__ import annotations

import argparse
import datetime
import hashlib
import json
import os
import statistics
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import workloads as W  # noqa: E402

METRIC = "quantize GB/s & FP8 (grouped) GEMM TFLOPS at 1 GB300; % of roofline"
L2_FLUSH_BYTES = 256 << 20
# nominal GB300 figures (dense): HBM3e 7.9 TB/s, FP8 4.5 PFLOP/s, BF16 2.25 PFLOP/s; reported beside
# the fractions of the measured peaks, which are the ones the roofline uses
NOMINAL_PEAK = {"hbm": 7900.0, "fp8": 4500.0, "bf16": 2250.0}


def grouped_attainable_ms(counts, N, K, out_bytes, peak_tflops, bw_gbs, jagged_k=False):
    """The grouped GEMM's attainable time: the sum over experts of max(2 m N K / peak, bytes / BW),
    bytes = the expert's FP8 operands plus its output (rows jagged: W_e [N, K] + A_e [m, K] +
    out [m, N]; contraction jagged: dY_e^T [N, m] + X_e^T [K, m] + dW_e [N, K])."""
    t = 0.0
    for m in counts:
        m = int(m)
        flops = 2.0 * m * N * K
        if jagged_k:
            nbytes = m * (N + K) + out_bytes * N * K
        else:
            nbytes = N * K + m * K + out_bytes * m * N
        t += max(flops / (peak_tflops * 1e9), nbytes / (bw_gbs * 1e6))  # ms
    return t


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        d = json.load(open(p))
        return dict(hbm=float(d["hbm_gbs"]), bf16=float(d["bf16_tflops"]),
                    bf16_sust=float(d.get("bf16_tflops_sustained", d["bf16_tflops"])), src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sust=1700.0, src="fallback")


# ------------------------------------------------------------------------------------------
# Workload steps. Each builds its buffers once; run(mark) launches the step's kernels in order,
# calling mark(label) before each launch (used to drop CUDA events between kernels).

class Step:
    name = ""
    unit = "TFLOP/s"
    kernels: list = []  # (label, kind "tensor"|"hbm", amount per launch (flop or byte), peak key)

    def total_units(self):  # flop (TFLOP/s metrics) or byte (GB/s metrics) per step
        raise NotImplementedError


class DenseLinearStep(Step):
    """Linear fwd+bwd, rowwise FP8 (fwd, dX) and bf16 dW."""

    def __init__(self, fp8, M, K, N, seed=0, device="cuda"):
        self.fp8, self.M, self.K, self.N = fp8, M, K, N
        self.name = "llama3-8b-mlp-up" if (M, K, N) == (8192, 4096, 14336) else f"linear-rowwise-{M}x{K}x{N}"
        self.x, self.w, self.dy = W.linear_inputs(M, K, N, seed=seed, device=device, outliers=True)
        d = device
        e4, e5 = torch.float8_e4m3fn, torch.float8_e5m2
        self.xq = torch.empty((M, K), dtype=e4, device=d)
        self.xi = torch.empty(M, device=d)
        self.wq = torch.empty((N, K), dtype=e4, device=d)
        self.wi = torch.empty(N, device=d)
        self.y = torch.empty((M, N), dtype=torch.bfloat16, device=d)
        self.dyq = torch.empty((M, N), dtype=e5, device=d)
        self.dyi = torch.empty(M, device=d)
        self.wtq = torch.empty((K, N), dtype=e4, device=d)
        self.wti = torch.empty(K, device=d)
        self.wsc = fp8.col_workspace(1, K, N, d)  # W [N, K] column-wise
        self.dx = torch.empty((M, K), dtype=torch.bfloat16, device=d)
        self.dw = torch.empty((N, K), dtype=torch.bfloat16, device=d)
        f = 2.0 * M * N * K
        self.kernels = [
            ("quantize_rows x e4m3", "hbm", 3 * M * K + 4 * M, "hbm"),
            ("quantize_rows W e4m3", "hbm", 3 * N * K + 4 * N, "hbm"),
            ("gemm_fp8 fwd", "tensor", f, "fp8"),
            ("quantize_rows dY e5m2", "hbm", 3 * M * N + 4 * M, "hbm"),
            ("quantize_cols W e4m3 col-major", "hbm", 3 * N * K + 4 * K, "hbm"),
            ("gemm_fp8 dX", "tensor", f, "fp8"),
            ("gemm_bf16 dW", "tensor", f, "bf16"),
        ]

    def total_units(self):
        return 3 * 2.0 * self.M * self.N * self.K

    def run(self, mark=lambda s: None):
        f = self.fp8
        mark(0)
        f.fp8_quantize(self.x, f.GRAN_ROW, f.DT_E4M3, f.LAYOUT_ROW_MAJOR, self.xq, None, self.xi)
        mark(1)
        f.fp8_quantize(self.w, f.GRAN_ROW, f.DT_E4M3, f.LAYOUT_ROW_MAJOR, self.wq, None, self.wi)
        mark(2)
        f.fp8_scaled_mm(self.xq, self.wq, self.xi, self.wi, self.y, f.MM_FAST_ACCUM)
        mark(3)
        f.fp8_quantize(self.dy, f.GRAN_ROW, f.DT_E5M2, f.LAYOUT_ROW_MAJOR, self.dyq, None, self.dyi)
        mark(4)
        f.fp8_quantize(self.w, f.GRAN_COL, f.DT_E4M3, f.LAYOUT_COL_MAJOR, None, self.wtq, self.wti, None, self.wsc)
        mark(5)
        f.fp8_scaled_mm(self.dyq, self.wtq, self.dyi, self.wti, self.dx, 0)
        mark(6)
        f.fp8_scaled_mm(self.dy, self.x, None, None, self.dw, f.MM_A_MN_MAJOR | f.MM_B_MN_MAJOR)

    # e2e: the public Linear entry points with host buffers. Inputs and outputs are
    # double-buffered on the device so that the copies of step i+1 (host -> device) and of
    # step i-1 (device -> host) run on the copy engines while step i computes.
    def e2e_setup(self):
        f = self.fp8
        dev = self.x.device
        self.h_in = [t.cpu().pin_memory() for t in (self.x, self.w, self.dy)]
        self.h_out = [torch.empty(t.shape, dtype=t.dtype).pin_memory() for t in (self.y, self.dx, self.dw)]
        self.d_in = [[torch.empty_like(t) for t in (self.x, self.w, self.dy)] for _ in range(2)]
        self.d_out = [[torch.empty_like(t) for t in (self.y, self.dx, self.dw)] for _ in range(2)]
        self.e2e_buffers(dev)
        self.s_in, self.s_out = torch.cuda.Stream(), torch.cuda.Stream()
        return sum(t.numel() * t.element_size() for t in self.h_in), \
            sum(t.numel() * t.element_size() for t in self.h_out)

    def e2e_buffers(self, dev):
        """Saved FP8 copies and the backward workspace of the public Linear entry points."""
        f = self.fp8
        self.e2e_gran, self.e2e_wgrad = f.GRAN_ROW, f.WGRAD_BF16
        self.saved = f.make_saved(self.xq, self.xi, self.wq, self.wi)
        self.ws = torch.empty(max(f.fp8_workspace_size(f.OP_LINEAR_BWD, self.M, self.K, self.N, f.GRAN_ROW,
                                                       f.WGRAD_BF16), 256), dtype=torch.uint8, device=dev)

    def e2e_run_steps(self, n):
        """n steps through fp8_linear_fwd / fp8_linear_bwd, each with its host->device input copy
        and device->host output copy; returns (start, end) CUDA events spanning all of it."""
        f = self.fp8
        comp = torch.cuda.current_stream()
        ev = lambda: torch.cuda.Event(enable_timing=True)
        in_ready = [ev(), ev()]
        done = [ev(), ev()]
        out_done = [ev(), ev()]
        start, end = ev(), ev()
        start.record(self.s_in)

        def copy_in(i):
            s = i % 2
            with torch.cuda.stream(self.s_in):
                if i >= 2:
                    self.s_in.wait_event(done[s])  # the step that read these inputs has finished
                for d, h in zip(self.d_in[s], self.h_in):
                    d.copy_(h, non_blocking=True)
                in_ready[s].record(self.s_in)

        copy_in(0)
        for i in range(n):
            s = i % 2
            if i + 1 < n:
                copy_in(i + 1)
            comp.wait_event(in_ready[s])
            if i >= 2:
                comp.wait_event(out_done[s])  # these outputs have been copied out
            x, w, dy = self.d_in[s]
            y, dx, dw = self.d_out[s]
            f.fp8_linear_fwd(x, w, self.e2e_gran, f.MM_FAST_ACCUM, y, self.saved)
            f.fp8_linear_bwd(dy, self.saved, x, w, self.e2e_gran, self.e2e_wgrad, dx, dw, self.ws)
            done[s].record(comp)
            with torch.cuda.stream(self.s_out):
                self.s_out.wait_event(done[s])
                for d, h in zip(self.d_out[s], self.h_out):
                    h.copy_(d, non_blocking=True)
                out_done[s].record(self.s_out)
        self.s_out.wait_stream(comp)
        end.record(self.s_out)
        return start, end

    def cpu_sample(self, rows):
        return dense_cpu_sample(self.x[:rows].cpu(), self.w.cpu(), self.dy[:rows].cpu(), self.M)


def dense_cpu_sample(x, w, dy, full_rows):
    """The oracle (as it stands) on the first rows of x / dY and all of W: the same quantize and
    GEMM steps as one dense Linear step, on fewer tokens."""
    import oracle
    M, K = x.shape
    N = w.shape[0]
    xb, wb, db = W.bf16_bits(x), W.bf16_bits(w), W.bf16_bits(dy)

    def run():
        xq, xi = oracle.quantize_rows(xb, oracle.E4M3)
        wq, wi = oracle.quantize_rows(wb, oracle.E4M3)
        oracle.gemm_fp8(xq, oracle.E4M3, wq, oracle.E4M3, xi, wi)
        dq, di = oracle.quantize_rows(db, oracle.E5M2)
        wc, wci = oracle.quantize_cols(wb, oracle.E4M3)
        oracle.gemm_fp8(dq, oracle.E5M2, wc, oracle.E4M3, di, wci, b_trans=True)
        oracle.gemm_bf16(db, xb, a_trans=True, b_trans=True)
    return run, 3 * 2.0 * M * N * K, f"llama3-8b-mlp-up step on the first {M} of {full_rows} tokens (all of W)"


class TensorwiseLinearStep(Step):
    """Single Linear fwd+bwd, tensorwise, fp32 outputs (latency-bound)."""

    def __init__(self, fp8, M=256, K=512, N=256, seed=0, device="cuda"):
        self.fp8, self.M, self.K, self.N = fp8, M, K, N
        self.name = "linear-tensorwise-256x512"
        self.x, self.w, self.dy = W.linear_inputs(M, K, N, seed=seed, device=device)
        e4 = torch.float8_e4m3fn
        d = device
        self.xq, self.xtq = torch.empty((M, K), dtype=e4, device=d), torch.empty((K, M), dtype=e4, device=d)
        self.wq, self.wtq = torch.empty((N, K), dtype=e4, device=d), torch.empty((K, N), dtype=e4, device=d)
        self.xi, self.wi = torch.empty(1, device=d), torch.empty(1, device=d)
        self.saved = fp8.make_saved(self.xq, self.xi, self.wq, self.wi, self.xtq, self.wtq)
        self.y = torch.empty((M, N), device=d)
        self.dx = torch.empty((M, K), device=d)
        self.dw = torch.empty((N, K), device=d)
        self.wsf = torch.empty(256, dtype=torch.uint8, device=d)
        self.wsb = torch.empty(fp8.fp8_workspace_size(fp8.OP_LINEAR_BWD, M, K, N, fp8.GRAN_TENSOR, fp8.WGRAD_FP8),
                               dtype=torch.uint8, device=d)
        f = 2.0 * M * N * K
        self.kernels = [("linear_fwd (2x quantize tensor dual, gemm)", "tensor", f, "fp8"),
                        ("linear_bwd (quantize dY dual, gemm dX, gemm dW)", "tensor", 2 * f, "fp8")]

    def total_units(self):
        return 3 * 2.0 * self.M * self.N * self.K

    def run(self, mark=lambda s: None):
        f = self.fp8
        mark(0)
        f.fp8_linear_fwd(self.x, self.w, f.GRAN_TENSOR, f.MM_FAST_ACCUM, self.y, self.saved, self.wsf)
        mark(1)
        f.fp8_linear_bwd(self.dy, self.saved, self.x, self.w, f.GRAN_TENSOR, f.WGRAD_FP8, self.dx, self.dw, self.wsb)

    def launches_per_step(self):
        return 9  # three tensorwise quantizes (amax + cast kernels each) and three GEMMs

    def cpu_sample(self, rows):
        return tensorwise_linear_cpu_sample(self.x.cpu(), self.w.cpu(), self.dy.cpu())


def tensorwise_linear_cpu_sample(x, w, dy):
    """The whole tensorwise Linear step in the oracle (it is small): one scale per tensor, fwd, dX
    and dW FP8 GEMMs."""
    import oracle
    M, K = x.shape
    N = w.shape[0]
    xb, wb, db = W.bf16_bits(x), W.bf16_bits(w), W.bf16_bits(dy)

    def run():
        xq, xi = oracle.quantize_tensor(xb, oracle.E4M3)
        wq, wi = oracle.quantize_tensor(wb, oracle.E4M3)
        oracle.gemm_fp8(xq, oracle.E4M3, wq, oracle.E4M3, xi, wi)
        dq, di = oracle.quantize_tensor(db, oracle.E5M2)
        oracle.gemm_fp8(dq, oracle.E5M2, wq, oracle.E4M3, di, wi, b_trans=True)
        oracle.gemm_fp8(dq, oracle.E5M2, xq, oracle.E4M3, di, xi, a_trans=True, b_trans=True)
    return run, 3 * 2.0 * M * N * K, "the whole step"


class ColwiseStep(Step):
    unit = "GB/s"

    def __init__(self, fp8, R=8192, C=14336, RX=8192, CX=4096, seed=0, device="cuda"):
        self.fp8 = fp8
        self.name = "colwise-8192x14336"
        self.g = W.column_gain_bf16((R, C), 1e-3, -2, 2, seed, device)
        self.xx = W.normal_bf16((RX, CX), 1.0, seed + 1, device)
        self.gt = torch.empty((C, R), dtype=torch.float8_e5m2, device=device)
        self.gi = torch.empty(C, device=device)
        self.gsc = fp8.col_workspace(1, C, R, device)
        self.xq = torch.empty((RX, CX), dtype=torch.float8_e4m3fn, device=device)
        self.xi = torch.empty(RX, device=device)
        self.R, self.C, self.RX, self.CX = R, C, RX, CX
        self.kernels = [("quantize_cols G e5m2 col-major", "hbm", 3 * R * C + 4 * C, "hbm"),
                        ("quantize_rows X e4m3", "hbm", 3 * RX * CX + 4 * RX, "hbm")]

    def total_units(self):
        return float(sum(k[2] for k in self.kernels))

    def cpu_sample(self, rows):
        """The oracle's column quantize on the first 1024 columns of G (all 8192 rows) and its row
        quantize on the first 1024 rows of X."""
        return colwise_cpu_sample(self.g[:, :1024].cpu(), self.xx[:1024].cpu())

    def run(self, mark=lambda s: None):
        f = self.fp8
        mark(0)
        f.fp8_quantize(self.g, f.GRAN_COL, f.DT_E5M2, f.LAYOUT_COL_MAJOR, None, self.gt, self.gi, None, self.gsc)
        mark(1)
        f.fp8_quantize(self.xx, f.GRAN_ROW, f.DT_E4M3, f.LAYOUT_ROW_MAJOR, self.xq, None, self.xi)


def colwise_cpu_sample(g, x):
    """The oracle's column-wise e5m2 quantize of G's columns (over all their rows) and its row-wise
    e4m3 quantize of X's rows, counted in algorithmic bytes."""
    import oracle
    gb, xb = W.bf16_bits(g), W.bf16_bits(x)

    def run():
        oracle.quantize_cols(gb, oracle.E5M2)
        oracle.quantize_rows(xb, oracle.E4M3)
    work = 3.0 * gb.size + 4 * gb.shape[1] + 3.0 * xb.size + 4 * xb.shape[0]
    return run, work, f"column quantize of G[:, :{gb.shape[1]}] and row quantize of X[:{xb.shape[0]}]"


class TensorwiseQuantStep(Step):
    """Tensorwise quantization of the llama3-8b-mlp-up tensors with the dual output (row-major and
    column-major codes from one quantize, as the tensorwise Linear saves them for backward):
    x [8192, 4096] and W [14336, 4096] to e4m3, dY [8192, 14336] to e5m2."""
    unit = "GB/s"

    def __init__(self, fp8, seed=0, device="cuda"):
        self.fp8 = fp8
        self.name = "llama3-8b-tensorwise-quant"
        d = W.WORKLOADS[self.name].dims
        M, K, N = d["M"], d["K"], d["N"]
        self.x, self.w, self.dy = W.linear_inputs(M, K, N, seed=seed, device=device, outliers=True)
        e4, e5 = torch.float8_e4m3fn, torch.float8_e5m2
        self.bufs = []
        for t, dt in ((self.x, e4), (self.w, e4), (self.dy, e5)):
            R, C = t.shape
            self.bufs.append((torch.empty((R, C), dtype=dt, device=device), torch.empty((C, R), dtype=dt, device=device),
                              torch.empty(1, device=device), torch.empty(4, dtype=torch.int32, device=device)))
        self.M, self.K, self.N = M, K, N
        self.kernels = [("quantize_tensor x e4m3 dual", "hbm", 4 * M * K + 4, "hbm"),
                        ("quantize_tensor W e4m3 dual", "hbm", 4 * N * K + 4, "hbm"),
                        ("quantize_tensor dY e5m2 dual", "hbm", 4 * M * N + 4, "hbm")]

    def total_units(self):
        return float(sum(k[2] for k in self.kernels))

    def launches_per_step(self):
        return 2 * len(self.kernels)  # amax pass and cast pass per tensor

    def cpu_sample(self, rows):
        """The oracle's tensorwise quantize of x[:rows] (all columns)."""
        return tensorwise_quant_cpu_sample(self.x[:rows].cpu())

    def run(self, mark=lambda s: None):
        f = self.fp8
        for i, (t, dt) in enumerate(((self.x, f.DT_E4M3), (self.w, f.DT_E4M3), (self.dy, f.DT_E5M2))):
            q, qt, inv, ws = self.bufs[i]
            mark(i)
            f.fp8_quantize(t, f.GRAN_TENSOR, dt, f.LAYOUT_BOTH, q, qt, inv, None, ws)


def tensorwise_quant_cpu_sample(x):
    """The oracle's tensorwise e4m3 quantize of x, counted in the dual output's bytes."""
    import oracle
    xb = W.bf16_bits(x)

    def run():
        oracle.quantize_tensor(xb, oracle.E4M3)
    return run, 4.0 * xb.size + 4, f"tensorwise quantize of x[:{xb.shape[0]}] (dual-output bytes)"


class MoeFwdStep(Step):
    """DeepSeek-V3-shaped grouped GEMM forward: quantize A rowwise, W per (expert, n), grouped GEMM."""

    def __init__(self, fp8, seed=0, device="cuda", name="dsv3-moe-fwd"):
        self.fp8 = fp8
        self.name = name
        d = W.WORKLOADS[self.name].dims
        E, M, K, N = d["E"], d["M"], d["K"], d["N"]
        counts = W.dsv3_counts(seed) if name == "dsv3-moe-fwd" else W.dsv3_32e_counts(seed)
        self.A, self.Wt, ends, _ = W.moe_inputs(E, M, K, N, counts, seed=seed, device=device)
        self.ends = torch.from_numpy(ends).to(device)
        self.counts = counts
        self.Aq = torch.empty((M, K), dtype=torch.float8_e4m3fn, device=device)
        self.Ai = torch.empty(M, device=device)
        self.Wq = torch.empty((E, N, K), dtype=torch.float8_e4m3fn, device=device)
        self.Wi = torch.empty((E, N), device=device)
        self.out = torch.empty((M, N), dtype=torch.bfloat16, device=device)
        self.E, self.M, self.K, self.N = E, M, K, N
        f = 2.0 * M * N * K
        self.kernels = [("quantize_rows A e4m3", "hbm", 3 * M * K + 4 * M, "hbm"),
                        ("quantize_rows W[e] e4m3 (per expert column)", "hbm", 3 * E * N * K + 4 * E * N, "hbm"),
                        ("grouped_gemm_fp8 jagged-M", "tensor", f, "fp8")]

    def total_units(self):
        return 2.0 * self.M * self.N * self.K

    @property
    def attainable_ms(self):
        pk = self.peak_of
        return {"grouped_gemm_fp8 jagged-M": grouped_attainable_ms(self.counts, self.N, self.K, 2, pk["fp8"], pk["hbm"])}

    def cpu_sample(self, rows):
        """The oracle on `rows` routed rows (their row quantize, their experts' weights quantized
        per column, their grouped-GEMM outputs), counted in grouped-GEMM FLOPs."""
        import oracle
        ends = self.ends.cpu().numpy()
        ridx = np.sort(np.random.default_rng(0).choice(self.M, rows, replace=False))
        experts = np.unique(np.searchsorted(ends, ridx, side="right"))
        ab = W.bf16_bits(self.A[torch.as_tensor(ridx, device=self.A.device)].cpu())
        wb = {int(e): W.bf16_bits(self.Wt[int(e)].cpu()) for e in experts}

        def run():
            aq, ai = oracle.quantize_rows(ab, oracle.E4M3)
            for i, r in enumerate(ridx):
                e = int(np.searchsorted(ends, r, side="right"))
                wq, wi = oracle.quantize_rows(wb[e], oracle.E4M3)
                oracle.gemm_fp8(aq[i:i + 1], oracle.E4M3, wq, oracle.E4M3, ai[i:i + 1], wi)
        return run, 2.0 * rows * self.N * self.K, f"{rows} routed rows: their quantize, their experts' weights, their outputs"

    def run(self, mark=lambda s: None):
        f = self.fp8
        mark(0)
        f.fp8_quantize(self.A, f.GRAN_ROW, f.DT_E4M3, f.LAYOUT_ROW_MAJOR, self.Aq, None, self.Ai)
        mark(1)
        f.fp8_quantize(self.Wt, f.GRAN_ROW, f.DT_E4M3, f.LAYOUT_ROW_MAJOR, self.Wq, None, self.Wi)
        mark(2)
        f.fp8_grouped_mm(self.Aq, self.Wq, self.ends, self.Ai, self.Wi, self.out, f.GROUPED_JAGGED_M)

    # e2e: the layer through the public entry points (fp8_quantize, fp8_grouped_mm) with host
    # buffers. Every step copies its inputs host -> device (A, the expert weights W and the
    # offsets, from pinned memory) and its output device -> host; inputs and outputs are
    # double-buffered on the device so the copies of the neighbouring steps run on the copy
    # engines while a step computes.
    def e2e_setup(self):
        dev = self.A.device
        ins = (self.A, self.Wt, self.ends)
        self.h_in = [t.cpu().pin_memory() for t in ins]
        self.h_out = [torch.empty(self.out.shape, dtype=self.out.dtype).pin_memory()]
        self.d_in = [[torch.empty_like(t) for t in ins] for _ in range(2)]
        self.d_out = [[torch.empty_like(self.out)] for _ in range(2)]
        self.s_in, self.s_out = torch.cuda.Stream(device=dev), torch.cuda.Stream(device=dev)
        return sum(t.numel() * t.element_size() for t in self.h_in), \
            sum(t.numel() * t.element_size() for t in self.h_out)

    def e2e_compute(self, d_in, d_out):
        f = self.fp8
        A, Wt, ends = d_in
        f.fp8_quantize(A, f.GRAN_ROW, f.DT_E4M3, f.LAYOUT_ROW_MAJOR, self.Aq, None, self.Ai)
        f.fp8_quantize(Wt, f.GRAN_ROW, f.DT_E4M3, f.LAYOUT_ROW_MAJOR, self.Wq, None, self.Wi)
        f.fp8_grouped_mm(self.Aq, self.Wq, ends, self.Ai, self.Wi, d_out[0], f.GROUPED_JAGGED_M)

    def e2e_run_steps(self, n):
        return pipelined_e2e(self, n)


def pipelined_e2e(step, n):
    """n steps of step.e2e_compute, each with the host->device copy of its inputs (s_in) and the
    device->host copy of its outputs (s_out), double-buffered; returns (start, end) CUDA events
    spanning all of it."""
    comp = torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event(enable_timing=True)
    in_ready, done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    start, end = ev(), ev()
    start.record(step.s_in)

    def copy_in(i):
        s = i % 2
        with torch.cuda.stream(step.s_in):
            if i >= 2:
                step.s_in.wait_event(done[s])  # the step that read these inputs has finished
            for d, h in zip(step.d_in[s], step.h_in):
                d.copy_(h, non_blocking=True)
            in_ready[s].record(step.s_in)

    copy_in(0)
    for i in range(n):
        s = i % 2
        if i + 1 < n:
            copy_in(i + 1)
        comp.wait_event(in_ready[s])
        if i >= 2:
            comp.wait_event(out_done[s])  # these outputs have been copied out
        step.e2e_compute(step.d_in[s], step.d_out[s])
        done[s].record(comp)
        with torch.cuda.stream(step.s_out):
            step.s_out.wait_event(done[s])
            for d, h in zip(step.d_out[s], step.h_out):
                h.copy_(d, non_blocking=True)
            out_done[s].record(step.s_out)
    step.s_out.wait_stream(comp)
    end.record(step.s_out)
    return start, end


def moe_fwd_cpu_sample(rows, seed=0, name="dsv3-moe-fwd", mx=False):
    """The oracle (as it stands) on `rows` routed rows of a DeepSeek-V3-shaped MoE forward layer:
    the rows' quantize (rowwise, or MX blocks of 32 along K), their experts' weights quantized the
    same way per expert row, and the rows' grouped-GEMM outputs. The sampled rows and their
    experts' weights are drawn on the host from the workload's distributions (A N(0,1),
    W N(0,0.02)), seeded; counted in grouped-GEMM FLOPs."""
    import oracle
    d = W.WORKLOADS[name].dims
    E, M, K, N = d["E"], d["M"], d["K"], d["N"]
    counts = W.dsv3_32e_counts(seed) if name == "dsv3-moe-fwd-32e" else W.dsv3_counts(seed)
    ends = W.ends_from_counts(counts)
    ridx = np.sort(np.random.default_rng(seed).choice(M, rows, replace=False))
    rexp = np.searchsorted(ends, ridx, side="right")
    ab = W.bf16_bits(W.normal_bf16((rows, K), 1.0, seed + 11))
    wb = {int(e): W.bf16_bits(W.normal_bf16((N, K), 0.02, seed + 1000 + int(e))) for e in np.unique(rexp)}
    quant, gemm = (oracle.mx_quantize_rows, oracle.gemm_mx) if mx else (oracle.quantize_rows, oracle.gemm_fp8)

    def run():
        aq, ai = quant(ab, oracle.E4M3)
        wq = {e: quant(b, oracle.E4M3) for e, b in wb.items()}
        for i, e in enumerate(rexp):
            cw, iw = wq[int(e)]
            gemm(aq[i:i + 1], oracle.E4M3, cw, oracle.E4M3, ai[i:i + 1], iw)
    return run, 2.0 * rows * N * K, (f"{rows} of {M} routed rows (their experts: {len(wb)} of {E}): the rows' "
                                     f"{'MX ' if mx else ''}quantize, their experts' weights quantized "
                                     f"{'in blocks of 32 along K' if mx else 'per expert column'}, their "
                                     f"grouped-GEMM outputs")


def moe_fwdbwd_cpu_sample(rows, seed=0, mx=False):
    """The oracle (as it stands) on a sample of the Llama4-shaped MoE fwd + bwd layer: `rows` routed
    rows (their quantize, their experts' weights quantized for the forward and, over N, for the
    grad-input GEMM, the rows' forward and grad-input outputs), and a 64 x 64 block of the weight
    gradient of the sampled expert with the fewest rows (its segment's dY and A columns quantized
    per segment column, then the contraction over the segment). Inputs drawn on the host from the
    workload's distributions, seeded; counted in GEMM FLOPs."""
    import oracle
    name = "llama4-moe-fwdbwd-mx" if mx else "llama4-moe-fwdbwd"
    d = W.WORKLOADS[name].dims
    E, M, K, N = d["E"], d["M"], d["K"], d["N"]
    counts = W.llama4_counts(seed)
    ends = W.ends_from_counts(counts)
    ridx = np.sort(np.random.default_rng(seed).choice(M, rows, replace=False))
    rexp = np.searchsorted(ends, ridx, side="right")
    ab = W.bf16_bits(W.normal_bf16((rows, K), 1.0, seed + 11))
    db = W.bf16_bits(W.normal_bf16((rows, N), 1e-3, seed + 12))
    wb = {int(e): W.bf16_bits(W.normal_bf16((N, K), 0.02, seed + 1000 + int(e))) for e in np.unique(rexp)}
    e0 = min(wb, key=lambda e: int(counts[e]))
    c0, nb = int(counts[e0]), 64
    gb = W.bf16_bits(W.normal_bf16((c0, nb), 1e-3, seed + 13))
    xb = W.bf16_bits(W.normal_bf16((c0, nb), 1.0, seed + 14))
    seg = np.array([c0], np.int32)
    E4, E5 = oracle.E4M3, oracle.E5M2

    def run():
        if mx:
            aq, as_ = oracle.mx_quantize_rows(ab, E4)
            dq, ds = oracle.mx_quantize_rows(db, E5)
            wq = {e: (oracle.mx_quantize_rows(b, E4), oracle.mx_quantize_cols(b, E4)) for e, b in wb.items()}
            for i, e in enumerate(rexp):
                (cw, sw), (ct, st) = wq[int(e)]
                oracle.gemm_mx(aq[i:i + 1], E4, cw, E4, as_[i:i + 1], sw)
                oracle.gemm_mx(dq[i:i + 1], E5, ct, E4, ds[i:i + 1], st)
            gq, gs = oracle.mx_quantize_jagged_cols(gb, seg, E5)
            xq, xs = oracle.mx_quantize_jagged_cols(xb, seg, E4)
            oracle.gemm_mx(gq, E5, xq, E4, gs, xs)
        else:
            aq, ai = oracle.quantize_rows(ab, E4)
            dq, di = oracle.quantize_rows(db, E5)
            wq = {e: (oracle.quantize_rows(b, E4), oracle.quantize_cols(b, E4)) for e, b in wb.items()}
            for i, e in enumerate(rexp):
                (cw, iw), (cc, ic) = wq[int(e)]
                oracle.gemm_fp8(aq[i:i + 1], E4, cw, E4, ai[i:i + 1], iw)
                oracle.gemm_fp8(dq[i:i + 1], E5, cc, E4, di[i:i + 1], ic, b_trans=True)
            gq, gi = oracle.quantize_jagged_cols(gb, seg, E5)
            xq, xi = oracle.quantize_jagged_cols(xb, seg, E4)
            oracle.grouped_gemm_k(gq, E5, xq, E4, gi, xi, seg)
    work = 2 * 2.0 * rows * N * K + 2.0 * c0 * nb * nb
    return run, work, (f"{rows} of {M} routed rows (their experts: {len(wb)} of {E}): their {'MX ' if mx else ''}"
                       f"quantize, their experts' weights in both layouts, their fwd and dX outputs; the "
                       f"{nb} x {nb} dW block of expert {e0} ({c0} rows)")


class MoeFwdBwdStep(Step):
    """Llama4-shaped grouped fwd + bwd: fwd, dX (per-expert W quantized over N, column-major),
    dW with jagged column-wise quantization of dY and x inside each segment."""

    def __init__(self, fp8, seed=0, device="cuda"):
        self.fp8 = fp8
        self.name = "llama4-moe-fwdbwd"
        d = W.WORKLOADS[self.name].dims
        E, M, K, N = d["E"], d["M"], d["K"], d["N"]
        counts = W.llama4_counts(seed)
        self.counts = counts
        self.A, self.Wt, ends, self.dY = W.moe_inputs(E, M, K, N, counts, seed=seed, device=device, with_grad=True)
        self.ends = torch.from_numpy(ends).to(device)
        e4, e5 = torch.float8_e4m3fn, torch.float8_e5m2
        P = fp8.fp8_jagged_padded_rows(M, E)
        self.Aq, self.Ai = torch.empty((M, K), dtype=e4, device=device), torch.empty(M, device=device)
        self.Wq, self.Wi = torch.empty((E, N, K), dtype=e4, device=device), torch.empty((E, N), device=device)
        self.out = torch.empty((M, N), dtype=torch.bfloat16, device=device)
        self.dYq, self.dYi = torch.empty((M, N), dtype=e5, device=device), torch.empty(M, device=device)
        self.Wtq, self.Wti = torch.empty((E, K, N), dtype=e4, device=device), torch.empty((E, K), device=device)
        self.dX = torch.empty((M, K), dtype=torch.bfloat16, device=device)
        self.dYt, self.dYti = torch.empty((N, P), dtype=e5, device=device), torch.empty((E, N), device=device)
        self.At, self.Ati = torch.empty((K, P), dtype=e4, device=device), torch.empty((E, K), device=device)
        self.dW = torch.empty((E, N, K), dtype=torch.bfloat16, device=device)
        self.ws_w = fp8.col_workspace(E, K, E * N, device)
        self.ws_dy = fp8.col_workspace(E, N, M, device)
        self.ws_a = fp8.col_workspace(E, K, M, device)
        self.E, self.M, self.K, self.N = E, M, K, N
        f = 2.0 * M * N * K
        self.kernels = [("quantize_rows A e4m3", "hbm", 3 * M * K + 4 * M, "hbm"),
                        ("quantize_rows W[e] e4m3", "hbm", 3 * E * N * K + 4 * E * N, "hbm"),
                        ("grouped_gemm_fp8 fwd jagged-M", "tensor", f, "fp8"),
                        ("quantize_rows dY e5m2", "hbm", 3 * M * N + 4 * M, "hbm"),
                        ("quantize_cols W[e] e4m3 col-major (over N)", "hbm", 3 * E * N * K + 4 * E * K, "hbm"),
                        ("grouped_gemm_fp8 dX jagged-M", "tensor", f, "fp8"),
                        ("quantize_cols jagged dY e5m2", "hbm", 3 * M * N + 4 * E * N, "hbm"),
                        ("quantize_cols jagged A e4m3", "hbm", 3 * M * K + 4 * E * K, "hbm"),
                        ("grouped_gemm_fp8 dW jagged-K", "tensor", f, "fp8")]

    def total_units(self):
        return 3 * 2.0 * self.M * self.N * self.K

    @property
    def attainable_ms(self):
        pk = self.peak_of
        c, N, K = self.counts, self.N, self.K
        return {"grouped_gemm_fp8 fwd jagged-M": grouped_attainable_ms(c, N, K, 2, pk["fp8"], pk["hbm"]),
                "grouped_gemm_fp8 dX jagged-M": grouped_attainable_ms(c, K, N, 2, pk["fp8"], pk["hbm"]),
                "grouped_gemm_fp8 dW jagged-K": grouped_attainable_ms(c, N, K, 2, pk["fp8"], pk["hbm"], jagged_k=True)}

    def run(self, mark=lambda s: None):
        f = self.fp8
        mark(0)
        f.fp8_quantize(self.A, f.GRAN_ROW, f.DT_E4M3, f.LAYOUT_ROW_MAJOR, self.Aq, None, self.Ai)
        mark(1)
        f.fp8_quantize(self.Wt, f.GRAN_ROW, f.DT_E4M3, f.LAYOUT_ROW_MAJOR, self.Wq, None, self.Wi)
        mark(2)
        f.fp8_grouped_mm(self.Aq, self.Wq, self.ends, self.Ai, self.Wi, self.out, f.GROUPED_JAGGED_M)
        mark(3)
        f.fp8_quantize(self.dY, f.GRAN_ROW, f.DT_E5M2, f.LAYOUT_ROW_MAJOR, self.dYq, None, self.dYi)
        mark(4)
        f.fp8_quantize(self.Wt, f.GRAN_COL, f.DT_E4M3, f.LAYOUT_COL_MAJOR, None, self.Wtq, self.Wti, None, self.ws_w)
        mark(5)
        f.fp8_grouped_mm(self.dYq, self.Wtq, self.ends, self.dYi, self.Wti, self.dX, f.GROUPED_JAGGED_M)
        mark(6)
        f.fp8_quantize(self.dY, f.GRAN_COL, f.DT_E5M2, f.LAYOUT_COL_MAJOR, None, self.dYt, self.dYti, self.ends,
                       self.ws_dy)
        mark(7)
        f.fp8_quantize(self.A, f.GRAN_COL, f.DT_E4M3, f.LAYOUT_COL_MAJOR, None, self.At, self.Ati, self.ends,
                       self.ws_a)
        mark(8)
        f.fp8_grouped_mm(self.dYt, self.At, self.ends, self.dYti, self.Ati, self.dW, f.GROUPED_JAGGED_K)


class DenseMxLinearStep(DenseLinearStep):
    """Linear fwd+bwd with MXFP8 everywhere: x, W (e4m3) and dY (e5m2) each quantized once into
    both layouts (blocks of 32 along K for the row-major copies, along M / N for the column-major
    ones); fwd, dX and dW are block-scaled FP8 GEMMs."""
    dtype = "mxfp8 e4m3/e5m2 (E8M0 scales per 32, fp32 accumulate)"

    def __init__(self, fp8, M, K, N, seed=0, device="cuda"):
        self.fp8, self.M, self.K, self.N = fp8, M, K, N
        self.name = "llama3-8b-mlp-up-mx" if (M, K, N) == (8192, 4096, 14336) else f"linear-mx-{M}x{K}x{N}"
        self.x, self.w, self.dy = W.linear_inputs(M, K, N, seed=seed, device=device, outliers=True)
        d = device
        e4, e5, u8 = torch.float8_e4m3fn, torch.float8_e5m2, torch.uint8
        sb = fp8.fp8_mx_scale_bytes
        # codes in both layouts; each scale buffer holds the row-major scales, then the column-major ones
        self.xq, self.xtq = torch.empty((M, K), dtype=e4, device=d), torch.empty((K, M), dtype=e4, device=d)
        self.wq, self.wtq = torch.empty((N, K), dtype=e4, device=d), torch.empty((K, N), dtype=e4, device=d)
        self.dyq, self.dytq = torch.empty((M, N), dtype=e5, device=d), torch.empty((N, M), dtype=e5, device=d)
        self.xs = torch.empty(sb(M, K) + sb(K, M), dtype=u8, device=d)
        self.wsc = torch.empty(sb(N, K) + sb(K, N), dtype=u8, device=d)
        self.dys = torch.empty(sb(M, N) + sb(N, M), dtype=u8, device=d)
        self.nx, self.nw, self.nd = sb(M, K), sb(N, K), sb(M, N)
        self.y = torch.empty((M, N), dtype=torch.bfloat16, device=d)
        self.dx = torch.empty((M, K), dtype=torch.bfloat16, device=d)
        self.dw = torch.empty((N, K), dtype=torch.bfloat16, device=d)
        f = 2.0 * M * N * K
        dual = lambda r, c: 4 * r * c + 2 * (r * c // 32)  # bf16 read, two code copies, two scale sets
        self.kernels = [
            ("mx_quantize x e4m3 rows+cols", "hbm", dual(M, K), "hbm"),
            ("mx_quantize W e4m3 rows+cols", "hbm", dual(N, K), "hbm"),
            ("gemm_mx fwd", "tensor", f, "fp8"),
            ("mx_quantize dY e5m2 rows+cols", "hbm", dual(M, N), "hbm"),
            ("gemm_mx dX", "tensor", f, "fp8"),
            ("gemm_mx dW", "tensor", f, "fp8"),
        ]

    def run(self, mark=lambda s: None):
        f = self.fp8
        mark(0)
        f.fp8_quantize(self.x, f.GRAN_MX, f.DT_E4M3, f.LAYOUT_BOTH, self.xq, self.xtq, self.xs)
        mark(1)
        f.fp8_quantize(self.w, f.GRAN_MX, f.DT_E4M3, f.LAYOUT_BOTH, self.wq, self.wtq, self.wsc)
        mark(2)
        f.fp8_scaled_mm(self.xq, self.wq, self.xs[:self.nx], self.wsc[:self.nw], self.y, f.MM_FAST_ACCUM)
        mark(3)
        f.fp8_quantize(self.dy, f.GRAN_MX, f.DT_E5M2, f.LAYOUT_BOTH, self.dyq, self.dytq, self.dys)
        mark(4)
        f.fp8_scaled_mm(self.dyq, self.wtq, self.dys[:self.nd], self.wsc[self.nw:], self.dx, 0)
        mark(5)
        f.fp8_scaled_mm(self.dytq, self.xtq, self.dys[self.nd:], self.xs[self.nx:], self.dw, 0)

    def e2e_buffers(self, dev):
        f = self.fp8
        self.e2e_gran, self.e2e_wgrad = f.GRAN_MX, f.WGRAD_FP8
        self.saved, self.saved_bufs = f.linear_saved_alloc(self.M, self.K, self.N, f.GRAN_MX, keep_xt=True, device=dev)
        self.ws = torch.empty(max(f.fp8_workspace_size(f.OP_LINEAR_BWD, self.M, self.K, self.N, f.GRAN_MX,
                                                       f.WGRAD_FP8), 256), dtype=torch.uint8, device=dev)

    def cpu_sample(self, rows):
        return dense_mx_cpu_sample(self.x[:rows].cpu(), self.w.cpu(), self.dy[:rows].cpu(), self.M)


def dense_mx_cpu_sample(x, w, dy, full_rows):
    """The oracle's MX quantize and MX GEMMs of one Linear step on the first rows of x / dY."""
    import oracle
    M, K = x.shape
    N = w.shape[0]
    xb, wb, db = W.bf16_bits(x), W.bf16_bits(w), W.bf16_bits(dy)

    def run():
        xq, xs = oracle.mx_quantize_rows(xb, oracle.E4M3)
        wq, ws = oracle.mx_quantize_rows(wb, oracle.E4M3)
        oracle.gemm_mx(xq, oracle.E4M3, wq, oracle.E4M3, xs, ws)
        dq, ds = oracle.mx_quantize_rows(db, oracle.E5M2)
        wtq, wts = oracle.mx_quantize_cols(wb, oracle.E4M3)
        oracle.gemm_mx(dq, oracle.E5M2, wtq, oracle.E4M3, ds, wts)
        dtq, dts = oracle.mx_quantize_cols(db, oracle.E5M2)
        xtq, xts = oracle.mx_quantize_cols(xb, oracle.E4M3)
        oracle.gemm_mx(dtq, oracle.E5M2, xtq, oracle.E4M3, dts, xts)
    return run, 3 * 2.0 * M * N * K, f"llama3-8b-mlp-up-mx step on the first {M} of {full_rows} tokens (all of W)"


class MoeFwdMxStep(MoeFwdStep):
    """The DeepSeek-V3-shaped grouped forward with MXFP8: A quantized with its scales in the
    segment-padded row space, W[e] per expert, one block-scaled grouped GEMM."""
    dtype = "mxfp8 e4m3 (E8M0 scales per 32, fp32 accumulate)"

    def __init__(self, fp8, seed=0, device="cuda"):
        self.fp8 = fp8
        self.name = "dsv3-moe-fwd-mx"
        d = W.WORKLOADS[self.name].dims
        E, M, K, N = d["E"], d["M"], d["K"], d["N"]
        counts = W.dsv3_counts(seed)
        self.A, self.Wt, ends, _ = W.moe_inputs(E, M, K, N, counts, seed=seed, device=device)
        self.ends = torch.from_numpy(ends).to(device)
        self.counts = counts
        sb = fp8.fp8_mx_scale_bytes
        self.P = fp8.fp8_jagged_padded_rows(M, E)
        self.Aq = torch.empty((M, K), dtype=torch.float8_e4m3fn, device=device)
        self.As = torch.empty(sb(self.P, K), dtype=torch.uint8, device=device)
        self.Wq = torch.empty((E, N, K), dtype=torch.float8_e4m3fn, device=device)
        self.Ws = torch.empty(E * sb(N, K), dtype=torch.uint8, device=device)
        self.ws_a = torch.empty(max(fp8.fp8_workspace_size(fp8.OP_QUANTIZE, E, K, granularity=fp8.GRAN_MX) // 4, 4),
                                dtype=torch.int32, device=device)
        self.out = torch.empty((M, N), dtype=torch.bfloat16, device=device)
        self.E, self.M, self.K, self.N = E, M, K, N
        f = 2.0 * M * N * K
        self.kernels = [("mx_quantize A e4m3 rows", "hbm", 3 * M * K + M * K // 32, "hbm"),
                        ("mx_quantize W[e] e4m3 rows", "hbm", 3 * E * N * K + E * N * K // 32, "hbm"),
                        ("grouped_gemm_mx jagged-M", "tensor", f, "fp8")]

    @property
    def attainable_ms(self):
        pk = self.peak_of
        return {"grouped_gemm_mx jagged-M": grouped_attainable_ms(self.counts, self.N, self.K, 2, pk["fp8"], pk["hbm"])}

    def cpu_sample(self, rows):
        import oracle
        ends = self.ends.cpu().numpy()
        ridx = np.sort(np.random.default_rng(0).choice(self.M, 64, replace=False))
        experts = np.unique(np.searchsorted(ends, ridx, side="right"))
        ab = W.bf16_bits(self.A[torch.as_tensor(ridx, device=self.A.device)].cpu())
        wb = {int(e): W.bf16_bits(self.Wt[int(e)].cpu()) for e in experts}

        def run():
            aq, as_ = oracle.mx_quantize_rows(ab, oracle.E4M3)
            for i, r in enumerate(ridx):
                e = int(np.searchsorted(ends, r, side="right"))
                wq, ws = oracle.mx_quantize_rows(wb[e], oracle.E4M3)
                oracle.gemm_mx(aq[i:i + 1], oracle.E4M3, wq, oracle.E4M3, as_[i:i + 1], ws)
        return run, 2.0 * 64 * self.N * self.K, "64 routed rows: their MX quantize, their experts' weights, their outputs"

    def run(self, mark=lambda s: None):
        f = self.fp8
        mark(0)
        f.fp8_quantize(self.A, f.GRAN_MX, f.DT_E4M3, f.LAYOUT_ROW_MAJOR, self.Aq, None, self.As, self.ends, self.ws_a)
        mark(1)
        f.fp8_quantize(self.Wt, f.GRAN_MX, f.DT_E4M3, f.LAYOUT_ROW_MAJOR, self.Wq, None, self.Ws)
        mark(2)
        f.fp8_grouped_mm(self.Aq, self.Wq, self.ends, self.As, self.Ws, self.out, f.GROUPED_JAGGED_M)

    def e2e_compute(self, d_in, d_out):
        f = self.fp8
        A, Wt, ends = d_in
        f.fp8_quantize(A, f.GRAN_MX, f.DT_E4M3, f.LAYOUT_ROW_MAJOR, self.Aq, None, self.As, ends, self.ws_a)
        f.fp8_quantize(Wt, f.GRAN_MX, f.DT_E4M3, f.LAYOUT_ROW_MAJOR, self.Wq, None, self.Ws)
        f.fp8_grouped_mm(self.Aq, self.Wq, ends, self.As, self.Ws, d_out[0], f.GROUPED_JAGGED_M)


class MoeFwdBwdMxStep(MoeFwdBwdStep):
    """The Llama4-shaped grouped fwd + bwd with MXFP8: A, W[e] and dY are each read once and
    quantized into both layouts (row-major for the jagged-M GEMMs, column-major for dX's
    weights and for the jagged-K weight gradient); three block-scaled grouped GEMMs."""
    dtype = "mxfp8 e4m3/e5m2 (E8M0 scales per 32, fp32 accumulate)"

    def __init__(self, fp8, seed=0, device="cuda"):
        self.fp8 = fp8
        self.name = "llama4-moe-fwdbwd-mx"
        d = W.WORKLOADS[self.name].dims
        E, M, K, N = d["E"], d["M"], d["K"], d["N"]
        counts = W.llama4_counts(seed)
        self.counts = counts
        self.A, self.Wt, ends, self.dY = W.moe_inputs(E, M, K, N, counts, seed=seed, device=device, with_grad=True)
        self.ends = torch.from_numpy(ends).to(device)
        e4, e5, u8 = torch.float8_e4m3fn, torch.float8_e5m2, torch.uint8
        sb = fp8.fp8_mx_scale_bytes
        P = self.P = fp8.fp8_jagged_padded_rows(M, E)
        dev = device
        self.Aq, self.At = torch.empty((M, K), dtype=e4, device=dev), torch.empty((K, P), dtype=e4, device=dev)
        self.A_s = torch.empty(sb(P, K) + sb(K, P), dtype=u8, device=dev)      # rows (padded), then A^T
        self.Wq, self.Wtq = torch.empty((E, N, K), dtype=e4, device=dev), torch.empty((E, K, N), dtype=e4, device=dev)
        self.W_s = torch.empty(E * (sb(N, K) + sb(K, N)), dtype=u8, device=dev)  # W[e] rows, then W[e]^T
        self.dYq, self.dYt = torch.empty((M, N), dtype=e5, device=dev), torch.empty((N, P), dtype=e5, device=dev)
        self.dY_s = torch.empty(sb(P, N) + sb(N, P), dtype=u8, device=dev)
        self.out = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        self.dX = torch.empty((M, K), dtype=torch.bfloat16, device=dev)
        self.dW = torch.empty((E, N, K), dtype=torch.bfloat16, device=dev)
        nws = max(fp8.fp8_workspace_size(fp8.OP_QUANTIZE, E, 0, granularity=fp8.GRAN_MX) // 4, 4)
        self.ws_a = torch.empty(nws, dtype=torch.int32, device=dev)
        self.ws_dy = torch.empty(nws, dtype=torch.int32, device=dev)
        self.nA, self.nW, self.ndY = sb(P, K), E * sb(N, K), sb(P, N)
        self.E, self.M, self.K, self.N = E, M, K, N
        f = 2.0 * M * N * K
        self.kernels = [("mx_quantize A e4m3 rows+cols jagged", "hbm", 4 * M * K + 2 * M * K // 32, "hbm"),
                        ("mx_quantize W[e] e4m3 rows+cols", "hbm", 4 * E * N * K + 2 * E * N * K // 32, "hbm"),
                        ("grouped_gemm_mx fwd jagged-M", "tensor", f, "fp8"),
                        ("mx_quantize dY e5m2 rows+cols jagged", "hbm", 4 * M * N + 2 * M * N // 32, "hbm"),
                        ("grouped_gemm_mx dX jagged-M", "tensor", f, "fp8"),
                        ("grouped_gemm_mx dW jagged-K", "tensor", f, "fp8")]

    @property
    def attainable_ms(self):
        pk = self.peak_of
        c, N, K = self.counts, self.N, self.K
        return {"grouped_gemm_mx fwd jagged-M": grouped_attainable_ms(c, N, K, 2, pk["fp8"], pk["hbm"]),
                "grouped_gemm_mx dX jagged-M": grouped_attainable_ms(c, K, N, 2, pk["fp8"], pk["hbm"]),
                "grouped_gemm_mx dW jagged-K": grouped_attainable_ms(c, N, K, 2, pk["fp8"], pk["hbm"], jagged_k=True)}

    def run(self, mark=lambda s: None):
        f = self.fp8
        mark(0)
        f.fp8_quantize(self.A, f.GRAN_MX, f.DT_E4M3, f.LAYOUT_BOTH, self.Aq, self.At, self.A_s, self.ends, self.ws_a)
        mark(1)
        f.fp8_quantize(self.Wt, f.GRAN_MX, f.DT_E4M3, f.LAYOUT_BOTH, self.Wq, self.Wtq, self.W_s)
        mark(2)
        f.fp8_grouped_mm(self.Aq, self.Wq, self.ends, self.A_s[:self.nA], self.W_s[:self.nW], self.out,
                         f.GROUPED_JAGGED_M)
        mark(3)
        f.fp8_quantize(self.dY, f.GRAN_MX, f.DT_E5M2, f.LAYOUT_BOTH, self.dYq, self.dYt, self.dY_s, self.ends,
                       self.ws_dy)
        mark(4)
        f.fp8_grouped_mm(self.dYq, self.Wtq, self.ends, self.dY_s[:self.ndY], self.W_s[self.nW:], self.dX,
                         f.GROUPED_JAGGED_M)
        mark(5)
        f.fp8_grouped_mm(self.dYt, self.At, self.ends, self.dY_s[self.ndY:], self.A_s[self.nA:], self.dW,
                         f.GROUPED_JAGGED_K)


class FusedAmaxStep(Step):
    """The grad-input GEMM of the Llama3-8B MLP-up Linear, dX = dY W (rowwise FP8 operands,
    quantized outside the timed region), with dX's column maxima as a side output of the GEMM's
    epilogue, then dX quantized column-wise (e5m2, column-major: the previous layer's dY^T for an
    FP8 weight gradient) from those maxima in one read. `alt_run` is the unfused chain timed in the
    same run: the plain GEMM, then the two-pass column-wise quantize (amax pass + cast pass)."""
    dtype = "fp8 e4m3/e5m2 (fp32 accumulate), bf16 dX"

    def __init__(self, fp8, seed=0, device="cuda"):
        self.fp8 = fp8
        self.name = "llama3-8b-dx-colquant-fused"
        d = W.WORKLOADS[self.name].dims
        M, K, N = d["M"], d["K"], d["N"]
        self.M, self.K, self.N = M, K, N
        x, w, dy = W.linear_inputs(M, K, N, seed=seed, device=device, outliers=True)
        self.dyq, _, self.dyi = fp8.quantize_alloc(dy, fp8.GRAN_ROW, fp8.DT_E5M2)
        _, self.wtq, self.wti = fp8.quantize_alloc(w, fp8.GRAN_COL, fp8.DT_E4M3)
        del x, w, dy
        self.dx = torch.empty((M, K), dtype=torch.bfloat16, device=device)
        self.amax = torch.empty(K, device=device)
        self.dxt = torch.empty((K, M), dtype=torch.float8_e5m2, device=device)
        self.dxti = torch.empty(K, device=device)
        self.ws = fp8.col_workspace(1, K, M, device)
        f = 2.0 * M * N * K
        self.kernels = [("gemm_fp8 dX + column amax side output", "tensor", f, "fp8"),
                        ("quantize_cols dX e5m2 from amax (one read)", "hbm", 3 * M * K + 4 * K, "hbm")]
        self.alt_kernels = [("gemm_fp8 dX", "tensor", f, "fp8"),
                            ("quantize_cols dX e5m2 (two passes)", "hbm", 3 * M * K + 4 * K, "hbm")]

    def total_units(self):
        return 2.0 * self.M * self.N * self.K

    def run(self, mark=lambda s: None):
        f = self.fp8
        mark(0)
        f.fp8_scaled_mm_amax(self.dyq, self.wtq, self.dyi, self.wti, self.dx, 0, col_amax=self.amax)
        mark(1)
        f.fp8_quantize_from_amax(self.dx, f.GRAN_COL, f.DT_E5M2, f.LAYOUT_COL_MAJOR, None, self.dxt, self.dxti,
                                 self.amax)

    def alt_run(self, mark=lambda s: None):
        f = self.fp8
        mark(0)
        f.fp8_scaled_mm(self.dyq, self.wtq, self.dyi, self.wti, self.dx, 0)
        mark(1)
        f.fp8_quantize(self.dx, f.GRAN_COL, f.DT_E5M2, f.LAYOUT_COL_MAJOR, None, self.dxt, self.dxti, None, self.ws)


class FusedQuantOutStep(Step):
    """The forward GEMM of the Llama3-8B MLP-up Linear, y = x W^T (rowwise FP8 operands, quantized
    outside the timed region), whose epilogue writes y already quantized for the next layer: e4m3
    codes with 1 x 128 block scales (the blockwise recipe's activation operand). `alt_run` is the
    unfused chain timed in the same run: the GEMM with a bf16 output, then the 1 x 128 quantize of
    it (the same codes and scales bit for bit)."""
    dtype = "fp8 e4m3 (fp32 accumulate), e4m3 1x128 output"

    def __init__(self, fp8, seed=0, device="cuda"):
        self.fp8 = fp8
        self.name = "llama3-8b-fwd-quant-fused"
        d = W.WORKLOADS[self.name].dims
        M, K, N = d["M"], d["K"], d["N"]
        self.M, self.K, self.N = M, K, N
        x, w, _ = W.linear_inputs(M, K, N, seed=seed, device=device, outliers=True)
        self.xq, _, self.xi = fp8.quantize_alloc(x, fp8.GRAN_ROW, fp8.DT_E4M3)
        self.wq, _, self.wi = fp8.quantize_alloc(w, fp8.GRAN_ROW, fp8.DT_E4M3)
        del x, w
        self.y = torch.empty((M, N), dtype=torch.bfloat16, device=device)
        self.yq = torch.empty((M, N), dtype=torch.float8_e4m3fn, device=device)
        self.yi = torch.empty((M, N // 128), device=device)
        f = 2.0 * M * N * K
        self.kernels = [("gemm_fp8 fwd, output quantized 1x128 in the epilogue", "tensor", f, "fp8")]
        self.alt_kernels = [("gemm_fp8 fwd (bf16 output)", "tensor", f, "fp8"),
                            ("blk_quantize y e4m3 1x128", "hbm", 3 * M * N + 4 * M * (N // 128), "hbm")]

    def total_units(self):
        return 2.0 * self.M * self.N * self.K

    def run(self, mark=lambda s: None):
        f = self.fp8
        mark(0)
        f.fp8_scaled_mm_quant(self.xq, self.wq, self.xi, self.wi, self.yq, self.yi, f.GRAN_BLOCK_1x128, f.MM_FAST_ACCUM)

    def alt_run(self, mark=lambda s: None):
        f = self.fp8
        mark(0)
        f.fp8_scaled_mm(self.xq, self.wq, self.xi, self.wi, self.y, f.MM_FAST_ACCUM)
        mark(1)
        f.fp8_quantize(self.y, f.GRAN_BLOCK_1x128, f.DT_E4M3, f.LAYOUT_ROW_MAJOR, self.yq, None, self.yi)


class DenseBlockwiseLinearStep(DenseLinearStep):
    """Linear fwd+bwd with blockwise scaling: x and dY in 1 x 128 tiles, W in 128 x 128 tiles
    (both layouts from one read); fwd and dX blockwise FP8 GEMMs, dW in bf16."""
    dtype = "fp8 e4m3/e5m2 blockwise (fp32 tile scales, fp32 accumulate), bf16 wgrad"

    def __init__(self, fp8, M, K, N, seed=0, device="cuda"):
        self.fp8, self.M, self.K, self.N = fp8, M, K, N
        self.name = "llama3-8b-mlp-up-blockwise"
        self.x, self.w, self.dy = W.linear_inputs(M, K, N, seed=seed, device=device, outliers=True)
        d = device
        e4, e5 = torch.float8_e4m3fn, torch.float8_e5m2
        self.saved, self.bufs = fp8.linear_saved_alloc(M, K, N, fp8.GRAN_BLOCK_1x128, keep_xt=False, device=d)
        (self.xq, self.xi, self.wq, self.wi, _, self.wtq, _, self.wti) = self.bufs
        self.wboth = torch.empty(2 * (N // 128) * (K // 128), device=d)
        self.dyq = torch.empty((M, N), dtype=e5, device=d)
        self.dyi = torch.empty((M, N // 128), device=d)
        self.y = torch.empty((M, N), dtype=torch.bfloat16, device=d)
        self.dx = torch.empty((M, K), dtype=torch.bfloat16, device=d)
        self.dw = torch.empty((N, K), dtype=torch.bfloat16, device=d)
        f = 2.0 * M * N * K
        self.kernels = [
            ("blk_quantize x e4m3 1x128", "hbm", 3 * M * K + 4 * M * K // 128, "hbm"),
            ("blk_quantize W e4m3 128x128 rows+cols", "hbm", 4 * N * K, "hbm"),
            ("gemm_blockwise fwd", "tensor", f, "fp8"),
            ("blk_quantize dY e5m2 1x128", "hbm", 3 * M * N + 4 * M * N // 128, "hbm"),
            ("gemm_blockwise dX", "tensor", f, "fp8"),
            ("gemm_bf16 dW", "tensor", f, "bf16"),
        ]

    def run(self, mark=lambda s: None):
        f = self.fp8
        nw = (self.N // 128) * (self.K // 128)
        mark(0)
        f.fp8_quantize(self.x, f.GRAN_BLOCK_1x128, f.DT_E4M3, f.LAYOUT_ROW_MAJOR, self.xq, None, self.xi)
        mark(1)
        f.fp8_quantize(self.w, f.GRAN_BLOCK_128x128, f.DT_E4M3, f.LAYOUT_BOTH, self.wq, self.wtq, self.wboth)
        mark(2)
        f.fp8_scaled_mm(self.xq, self.wq, self.xi, self.wboth[:nw], self.y, f.MM_FAST_ACCUM | f.MM_BLOCKWISE)
        mark(3)
        f.fp8_quantize(self.dy, f.GRAN_BLOCK_1x128, f.DT_E5M2, f.LAYOUT_ROW_MAJOR, self.dyq, None, self.dyi)
        mark(4)
        f.fp8_scaled_mm(self.dyq, self.wtq, self.dyi, self.wboth[nw:], self.dx, f.MM_BLOCKWISE)
        mark(5)
        f.fp8_scaled_mm(self.dy, self.x, None, None, self.dw, f.MM_A_MN_MAJOR | f.MM_B_MN_MAJOR)

    def e2e_buffers(self, dev):
        f = self.fp8
        self.e2e_gran, self.e2e_wgrad = f.GRAN_BLOCK_1x128, f.WGRAD_BF16
        self.saved, self.saved_bufs = f.linear_saved_alloc(self.M, self.K, self.N, f.GRAN_BLOCK_1x128, keep_xt=False,
                                                           device=dev)
        self.ws = torch.empty(max(f.fp8_workspace_size(f.OP_LINEAR_BWD, self.M, self.K, self.N, f.GRAN_BLOCK_1x128,
                                                       f.WGRAD_BF16), 256), dtype=torch.uint8, device=dev)

    def cpu_sample(self, rows):
        return blockwise_cpu_sample(self.x[:rows].cpu(), self.w.cpu(), self.dy[:rows].cpu(), self.M)


def blockwise_cpu_sample(x, w, dy, full_rows):
    """The oracle's blockwise Linear step on the first rows of x / dY and all of W: 1 x 128 tiles
    for x and dY, 128 x 128 tiles for W, blockwise fwd and dX GEMMs, bf16 dW."""
    import oracle
    rows, K = x.shape
    N = w.shape[0]
    xb, wb, db = W.bf16_bits(x), W.bf16_bits(w), W.bf16_bits(dy)

    def run():
        xq, xi = oracle.quantize_blocks(xb, oracle.E4M3, 1, 128)
        wq, wi = oracle.quantize_blocks(wb, oracle.E4M3, 128, 128)
        oracle.gemm_blockwise(xq, oracle.E4M3, wq, oracle.E4M3, xi, wi)
        dq, di = oracle.quantize_blocks(db, oracle.E5M2, 1, 128)
        oracle.gemm_blockwise(dq, oracle.E5M2, np.ascontiguousarray(wq.T), oracle.E4M3, di, np.ascontiguousarray(wi.T))
        oracle.gemm_bf16(db, xb, a_trans=True, b_trans=True)
    return run, 3 * 2.0 * rows * N * K, f"llama3-8b-mlp-up-blockwise step on the first {rows} of {full_rows} tokens"


def make_step(fp8, name):
    if name == "llama3-8b-mlp-up":
        return DenseLinearStep(fp8, 8192, 4096, 14336)
    if name == "linear-tensorwise-256x512":
        return TensorwiseLinearStep(fp8)
    if name == "colwise-8192x14336":
        return ColwiseStep(fp8)
    if name == "llama3-8b-tensorwise-quant":
        return TensorwiseQuantStep(fp8)
    if name in ("dsv3-moe-fwd", "dsv3-moe-fwd-32e"):
        return MoeFwdStep(fp8, name=name)
    if name == "llama4-moe-fwdbwd":
        return MoeFwdBwdStep(fp8)
    if name == "llama3-8b-mlp-up-mx":
        return DenseMxLinearStep(fp8, 8192, 4096, 14336)
    if name == "dsv3-moe-fwd-mx":
        return MoeFwdMxStep(fp8)
    if name == "llama4-moe-fwdbwd-mx":
        return MoeFwdBwdMxStep(fp8)
    if name == "llama3-8b-dx-colquant-fused":
        return FusedAmaxStep(fp8)
    if name == "llama3-8b-fwd-quant-fused":
        return FusedQuantOutStep(fp8)
    if name == "llama3-8b-mlp-up-blockwise":
        return DenseBlockwiseLinearStep(fp8, 8192, 4096, 14336)
    raise SystemExit(f"unknown workload {name}")


# ------------------------------------------------------------------------------------------
# clocks: nvidia-smi sampled every 20 ms from before the warm-up on (its start-up stays out of the
# timed region); the samples whose timestamps fall in the timed region are kept, or, when the
# region is shorter than the sampling interval, the samples nearest to it on either side. The GPU
# is named to nvidia-smi by its UUID (its index there need not be torch's when
# CUDA_VISIBLE_DEVICES remaps devices), or by the index when the UUID is not accepted.

CLOCK_FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
                "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
                "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


CLOCK_INTERVAL_MS = 20


def smi_gpu_id(gpu_index):
    """The id nvidia-smi knows this CUDA device by: "GPU-<uuid>" when nvidia-smi accepts it."""
    try:
        uid = "GPU-" + str(torch.cuda.get_device_properties(gpu_index).uuid)
        r = subprocess.run(["nvidia-smi", f"--id={uid}", "--query-gpu=index", "--format=csv,noheader"],
                           capture_output=True, text=True, timeout=20)
        if r.returncode == 0 and r.stdout.strip():
            return uid
    except Exception:  # no UUID in this torch, no nvidia-smi, or it refused the id
        pass
    return str(gpu_index)


class ClockSampler:
    def __init__(self, gpu_index):
        self.proc = None
        self.gpu = smi_gpu_id(gpu_index)
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={CLOCK_FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", str(CLOCK_INTERVAL_MS)],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self, t0, t1):
        """Clock summary of the samples taken between t0 and t1 (time.time() seconds)."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = []
        for line in out.strip().splitlines():
            f = [x.strip() for x in line.split(",")]
            if len(f) < 10:
                continue
            try:
                ts = datetime.datetime.strptime(f[0], "%Y/%m/%d %H:%M:%S.%f").timestamp()
                rows.append((ts, float(f[2]), float(f[3]), f[6:10]))
            except ValueError:
                continue
        inside = [r for r in rows if t0 <= r[0] <= t1]
        window = "timed region"
        if not inside:  # a region shorter than the interval: the nearest sample on either side
            before = [r for r in rows if r[0] < t0]
            after = [r for r in rows if r[0] > t1]
            inside = before[-1:] + after[:1]
            window = f"nearest samples (timed region shorter than the {CLOCK_INTERVAL_MS} ms interval)"
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in inside:
            for n, v in zip(names, r[3]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        sm = [r[1] for r in inside]
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(r[2] for r in inside) if inside else None,
                "reasons": sorted(reasons), "samples": len(inside), "window": window, "gpu": self.gpu}


# ------------------------------------------------------------------------------------------

def dist_setup():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if ws > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return ws, rank, local


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, ws: int) -> float:
    if ws == 1:
        return v
    import torch.distributed as dist
    dev = "cuda" if torch.cuda.is_available() else "cpu"
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_value(units_per_step: float, steps: int, world_size: int, max_total_ms: float, unit: str) -> float:
    """Throughput of the whole job: the work of every rank's steps over the slowest rank's time
    (weak scaling: every rank runs its own replica of the workload)."""
    scale = 1e9 if unit == "TFLOP/s" else 1e6  # flop/ms -> TFLOP/s, byte/ms -> GB/s
    return units_per_step * steps * world_size / max_total_ms / scale


def traffic_for(workload: str, label: str):
    """ncu DRAM bytes per launch for a kernel of a workload ("<workload>: <label>" in
    profiles/ncu_traffic.json); null when the kernel's source changed since the capture."""
    p = os.path.join(ROOT, "profiles", "ncu_traffic.json")
    if not os.path.exists(p):
        return None
    d = json.load(open(p))
    ent = d.get(f"{workload}: {label}")
    if not ent:
        return None
    src = os.path.join(ROOT, ent["source"])
    if not os.path.exists(src) or hashlib.sha256(open(src, "rb").read()).hexdigest() != ent["sha256"]:
        return None
    return ent["bytes_per_launch"]


def cpu_cores():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count()


def _bf16_bits_of(out64):
    """fp64 GEMM outputs as the bf16 bit patterns the GEMM stores (round to nearest even)."""
    return W.bf16_bits(torch.from_numpy(np.ascontiguousarray(out64)).to(torch.bfloat16))


def dx_colquant_cpu_sample(rows, seed=0):
    """The oracle on the first `rows` rows of the Llama3-8B grad-input GEMM dX = dY W (dY rowwise
    e5m2 and W per column e4m3, quantized before the sample as the step quantizes them outside its
    timed region), dX rounded to bf16, then dX quantized column-wise (e5m2) over those rows."""
    import oracle
    d = W.WORKLOADS["llama3-8b-dx-colquant-fused"].dims
    M, K, N = d["M"], d["K"], d["N"]
    _, w, dy = W.linear_inputs(rows, K, N, seed=seed, outliers=True)
    dq, di = oracle.quantize_rows(W.bf16_bits(dy), oracle.E5M2)
    wc, wi = oracle.quantize_cols(W.bf16_bits(w), oracle.E4M3)

    def run():
        out, _ = oracle.gemm_fp8(dq, oracle.E5M2, wc, oracle.E4M3, di, wi, b_trans=True)
        oracle.quantize_cols(_bf16_bits_of(out), oracle.E5M2)
    return run, 2.0 * rows * N * K, f"dX for the first {rows} of {M} rows, then its column-wise quantize over them"


def fwd_quant_cpu_sample(rows, seed=0):
    """The oracle on the first `rows` rows of the Llama3-8B forward GEMM y = x W^T (rowwise e4m3
    operands, quantized before the sample as the step quantizes them outside its timed region),
    y rounded to bf16, then its 1 x 128 e4m3 quantize."""
    import oracle
    d = W.WORKLOADS["llama3-8b-fwd-quant-fused"].dims
    M, K, N = d["M"], d["K"], d["N"]
    x, w, _ = W.linear_inputs(rows, K, N, seed=seed, outliers=True)
    xq, xi = oracle.quantize_rows(W.bf16_bits(x), oracle.E4M3)
    wq, wi = oracle.quantize_rows(W.bf16_bits(w), oracle.E4M3)

    def run():
        out, _ = oracle.gemm_fp8(xq, oracle.E4M3, wq, oracle.E4M3, xi, wi)
        oracle.quantize_blocks(_bf16_bits_of(out), oracle.E4M3, 1, 128)
    return run, 2.0 * rows * N * K, f"y for the first {rows} of {M} rows, then its 1 x 128 quantize"


# Size of each workload's host-drawn oracle sample: tokens or routed rows; for the column-wise
# workload the columns of G and the rows of X. Every sample takes a few seconds or less on 8-16
# host cores.
SAMPLE_ROWS = {"llama3-8b-mlp-up": 16, "llama3-8b-mlp-up-blockwise": 16, "llama3-8b-mlp-up-mx": 32,
               "llama3-8b-tensorwise-quant": 2048, "colwise-8192x14336": 1024, "dsv3-moe-fwd": 16,
               "dsv3-moe-fwd-32e": 16, "dsv3-moe-fwd-mx": 16, "llama4-moe-fwdbwd": 4, "llama4-moe-fwdbwd-mx": 4,
               "llama3-8b-dx-colquant-fused": 16, "llama3-8b-fwd-quant-fused": 16}


def host_cpu_sample(name, rows=None):
    """(run, work, sample) of the oracle on a sample of workload `name` drawn on the host (seeded,
    from the workload's distributions; no device memory): the reference arm's step, and the CPU
    baseline of the steps that keep no host-side inputs. `rows` defaults to SAMPLE_ROWS[name];
    the tensorwise Linear is always run whole."""
    r = rows if rows is not None else SAMPLE_ROWS.get(name)
    d = W.WORKLOADS[name].dims
    if name == "linear-tensorwise-256x512":
        return tensorwise_linear_cpu_sample(*W.linear_inputs(d["M"], d["K"], d["N"], seed=0))
    if name in ("llama3-8b-mlp-up", "llama3-8b-mlp-up-mx", "llama3-8b-mlp-up-blockwise"):
        x, w, dy = W.linear_inputs(r, d["K"], d["N"], seed=0, outliers=True)
        fn = {"llama3-8b-mlp-up": dense_cpu_sample, "llama3-8b-mlp-up-mx": dense_mx_cpu_sample,
              "llama3-8b-mlp-up-blockwise": blockwise_cpu_sample}[name]
        return fn(x, w, dy, d["M"])
    if name == "llama3-8b-tensorwise-quant":
        return tensorwise_quant_cpu_sample(W.outlier_channels_bf16((r, d["K"]), 1.0, 0.01, 50.0, 0))
    if name == "colwise-8192x14336":
        return colwise_cpu_sample(W.column_gain_bf16((d["R"], r), 1e-3, -2, 2, 0),
                                  W.normal_bf16((r, d["CX"]), 1.0, 1))
    if name in ("dsv3-moe-fwd", "dsv3-moe-fwd-32e", "dsv3-moe-fwd-mx"):
        return moe_fwd_cpu_sample(r, name="dsv3-moe-fwd" if name.endswith("-mx") else name,
                                  mx=name.endswith("-mx"))
    if name in ("llama4-moe-fwdbwd", "llama4-moe-fwdbwd-mx"):
        return moe_fwdbwd_cpu_sample(r, mx=name.endswith("-mx"))
    if name == "llama3-8b-dx-colquant-fused":
        return dx_colquant_cpu_sample(r)
    if name == "llama3-8b-fwd-quant-fused":
        return fwd_quant_cpu_sample(r)
    raise KeyError(name)


def workload_unit(name):
    return "GB/s" if name in ("colwise-8192x14336", "llama3-8b-tensorwise-quant") else "TFLOP/s"


def _host_bf16(shape, std, seed, outlier_cols=None, col_gain=None, chunk_rows=2048):
    """A full-size ~N(0, std^2) bf16 tensor drawn on the host in row chunks (bounded fp32 staging),
    optionally with outlier columns x50 or a per-column gain 10^U(lo, hi)."""
    R, C = shape
    g = torch.Generator().manual_seed(seed)
    out = torch.empty((R, C), dtype=torch.bfloat16)
    gain = None
    if outlier_cols is not None:
        gain = torch.ones(C)
        gain[torch.randperm(C, generator=torch.Generator().manual_seed(seed + 7919))[:max(1, round(outlier_cols * C))]] = 50.0
    elif col_gain is not None:
        lo, hi = col_gain
        u = torch.rand(C, generator=torch.Generator().manual_seed(seed + 104729), dtype=torch.float64)
        gain = torch.pow(10.0, lo + (hi - lo) * u).float()
    for r0 in range(0, R, chunk_rows):
        t = torch.randn(min(chunk_rows, R - r0), C, generator=g).mul_(std)
        if gain is not None:
            t.mul_(gain[None, :])
        out[r0:r0 + t.shape[0]] = t.to(torch.bfloat16)
    return out


def full_quantize_cpu(name):
    """The oracle's quantize steps of workload `name` on its full-size tensors (drawn on the host
    from the workload's distributions), each timed alone: [(label, elements, algorithmic bytes,
    seconds)]. Only the quantize call is timed, not the draw."""
    import oracle
    d = W.WORKLOADS[name].dims
    E4, E5 = oracle.E4M3, oracle.E5M2
    jobs = []  # (label, draw, quantize(bits), bytes)
    if name == "dsv3-moe-fwd":
        E, M, K, N = d["E"], d["M"], d["K"], d["N"]
        jobs = [("A e4m3 rows", lambda: _host_bf16((M, K), 1.0, 0), lambda b: oracle.quantize_rows(b, E4),
                 3 * M * K + 4 * M),
                ("W[e] e4m3 per expert column", lambda: _host_bf16((E * N, K), 0.02, 1),
                 lambda b: oracle.quantize_rows(b, E4), 3 * E * N * K + 4 * E * N)]
    elif name == "llama3-8b-mlp-up":
        M, K, N = d["M"], d["K"], d["N"]
        jobs = [("x e4m3 rows", lambda: _host_bf16((M, K), 1.0, 0, outlier_cols=0.01),
                 lambda b: oracle.quantize_rows(b, E4), 3 * M * K + 4 * M),
                ("W e4m3 rows", lambda: _host_bf16((N, K), 0.02, 1), lambda b: oracle.quantize_rows(b, E4),
                 3 * N * K + 4 * N),
                ("W e4m3 columns", lambda: _host_bf16((N, K), 0.02, 1), lambda b: oracle.quantize_cols(b, E4),
                 3 * N * K + 4 * K),
                ("dY e5m2 rows", lambda: _host_bf16((M, N), 1e-3, 2), lambda b: oracle.quantize_rows(b, E5),
                 3 * M * N + 4 * M)]
    elif name == "colwise-8192x14336":
        R, C, RX, CX = d["R"], d["C"], d["RX"], d["CX"]
        jobs = [("G e5m2 columns", lambda: _host_bf16((R, C), 1e-3, 0, col_gain=(-2, 2)),
                 lambda b: oracle.quantize_cols(b, E5), 3 * R * C + 4 * C),
                ("X e4m3 rows", lambda: _host_bf16((RX, CX), 1.0, 1), lambda b: oracle.quantize_rows(b, E4),
                 3 * RX * CX + 4 * RX)]
    elif name == "llama4-moe-fwdbwd":
        E, M, K, N = d["E"], d["M"], d["K"], d["N"]
        ends = W.ends_from_counts(W.llama4_counts(0))
        jobs = [("A e4m3 rows", lambda: _host_bf16((M, K), 1.0, 0), lambda b: oracle.quantize_rows(b, E4),
                 3 * M * K + 4 * M),
                ("W[e] e4m3 rows", lambda: _host_bf16((E * N, K), 0.02, 1), lambda b: oracle.quantize_rows(b, E4),
                 3 * E * N * K + 4 * E * N),
                ("W[e] e4m3 columns (per expert)", lambda: _host_bf16((E * N, K), 0.02, 1),
                 lambda b: [oracle.quantize_cols(b[e * N:(e + 1) * N], E4) for e in range(E)], 3 * E * N * K + 4 * E * K),
                ("dY e5m2 rows", lambda: _host_bf16((M, N), 1e-3, 2), lambda b: oracle.quantize_rows(b, E5),
                 3 * M * N + 4 * M),
                ("dY e5m2 segment columns", lambda: _host_bf16((M, N), 1e-3, 2),
                 lambda b: oracle.quantize_jagged_cols(b, ends, E5), 3 * M * N + 4 * E * N),
                ("A e4m3 segment columns", lambda: _host_bf16((M, K), 1.0, 0),
                 lambda b: oracle.quantize_jagged_cols(b, ends, E4), 3 * M * K + 4 * E * K)]
    elif name == "linear-tensorwise-256x512":
        M, K, N = d["M"], d["K"], d["N"]
        jobs = [(f"{t} tensorwise", (lambda r=r, c=c, sd=sd, sdn=sdn: _host_bf16((r, c), sd, sdn)),
                 (lambda b, f=f: oracle.quantize_tensor(b, f)), 3 * r * c + 4)
                for t, r, c, sd, sdn, f in (("x e4m3", M, K, 1.0, 0, E4), ("W e4m3", N, K, 0.02, 1, E4),
                                            ("dY e5m2", M, N, 1e-3, 2, E5))]
    else:
        raise KeyError(f"full-tensor quantize timing covers the five base workloads, not {name}")
    oracle.quantize_rows(np.zeros((64, 64), np.uint16), E4)  # the library's and threads' start-up, untimed
    out = []
    for label, draw, quant, nbytes in jobs:
        xb = W.bf16_bits(draw())
        t0 = time.perf_counter()
        quant(xb)
        dt = time.perf_counter() - t0
        out.append((label, int(xb.size), int(nbytes), dt))
        del xb
    return out


def run_cpu_full_quantize(args):
    """One JSON line: the oracle's quantize of every full-size tensor of the workload on the host
    cores (GB/s of algorithmic bytes: 2 read + 1 written per element, plus the scales)."""
    import oracle
    rows = full_quantize_cpu(args.workload)
    print(json.dumps({"impl": "reference", "kind": "oracle full-tensor quantize", "workload": args.workload,
                      "cores": oracle.num_threads(),
                      "tensors": [{"tensor": l, "elements": n, "GB/s": round(b / max(dt, 1e-9) / 1e9, 4), "seconds": round(dt, 3)}
                                  for l, n, b, dt in rows]}))


def run_reference(args, ws, rank):
    """The oracle as it stands, on the host cores, on a bounded sample of the workload drawn on
    the host: every step is the same sample."""
    if rank != 0:
        return
    import oracle
    run, work, sample = host_cpu_sample(args.workload)
    unit = workload_unit(args.workload)
    for _ in range(args.warmup):
        run()
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run()
    dt = time.perf_counter() - t0
    value = work * args.steps / dt / (1e12 if unit == "TFLOP/s" else 1e9)
    cores = oracle.num_threads()
    line = {"impl": "reference", "metric": METRIC, "value": value, "unit": unit, "n_gpus": ws,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt / args.steps * 1e3,
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": {"workload": args.workload, "sample": sample},
            "cpu_baseline": {"value": value, "unit": unit, "cores": cores, "kind": "oracle", "sample": sample},
            "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line))


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=30)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="fp8lin", choices=["fp8lin", "reference"])
    ap.add_argument("--workload", default="dsv3-moe-fwd", choices=list(W.WORKLOADS))
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-rows", type=int, default=64)
    ap.add_argument("--e2e-steps", type=int, default=30)
    ap.add_argument("--no-e2e", action="store_true", help="skip the host-buffer e2e measurement (profiling runs)")
    ap.add_argument("--cpu-full-quantize", action="store_true",
                    help="only time the oracle's quantize of the workload's full-size tensors on the host cores")
    args = ap.parse_args()
    assert args.warmup >= 3, "at least 3 warm-up steps"
    ws, rank, local = dist_setup()
    if args.cpu_full_quantize:
        run_cpu_full_quantize(args)
        return
    if args.impl == "reference":
        run_reference(args, ws, rank)
        return

    import moe_grouped_gemm_absmax_gb300 as fp8
    peaks = load_peaks()
    peak_of = {"hbm": peaks["hbm"], "fp8": 2.0 * peaks["bf16"], "bf16": peaks["bf16"]}
    step = make_step(fp8, args.workload)
    step.peak_of = peak_of
    stream = torch.cuda.current_stream()
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.int32, device="cuda")
    flush_rd = torch.ones(L2_FLUSH_BYTES // 4, dtype=torch.int32, device="cuda")
    nk = len(step.kernels)

    sampler = ClockSampler(torch.cuda.current_device()) if rank == 0 else None
    for _ in range(args.warmup):
        step.run()
    torch.cuda.synchronize()

    evs = [[torch.cuda.Event(enable_timing=True) for _ in range(nk + 1)] for _ in range(args.steps)]
    barrier(ws)
    torch.cuda.synchronize()
    t_start = time.time()
    wall0 = time.perf_counter()
    # a head start for the host (outside the events): the GPU spins ~1 ms per step while the
    # host queues the steps, so that no timed kernel waits for its own launch
    torch.cuda._sleep(2_000_000 * min(args.steps, 40))
    for i in range(args.steps):
        # evict L2 (outside the events): the write evicts the step's data, the read of another
        # buffer then evicts the write's dirty lines, so the first timed kernel does not pay
        # for writing the flush buffer back
        flush.zero_()
        torch.amax(flush_rd)
        # let the flush's write-backs drain (~50 us spin) so the first timed kernel does not pay
        # for them
        torch.cuda._sleep(100_000)
        ev = evs[i]
        step.run(lambda k: ev[k].record(stream))
        ev[nk].record(stream)
    torch.cuda.synchronize()
    barrier(ws)
    wall = time.perf_counter() - wall0
    clocks = sampler.stop(t_start, time.time()) if sampler else None

    per_kernel = np.zeros(nk)
    step_ms = []
    for ev in evs:
        t = [ev[k].elapsed_time(ev[k + 1]) for k in range(nk)]
        per_kernel += t
        step_ms.append(ev[0].elapsed_time(ev[nk]))
    per_kernel /= args.steps
    total_ms = float(np.sum(step_ms))
    total_ms_max = max_over_ranks(total_ms, ws)
    units = step.total_units()
    scale = 1e9 if step.unit == "TFLOP/s" else 1e6  # flop/ms -> TFLOP/s, byte/ms -> GB/s
    value = whole_job_value(units, args.steps, ws, total_ms_max, step.unit)

    kernels = []
    for (label, kind, amount, pk), ms in zip(step.kernels, per_kernel):
        if kind == "tensor":
            ach, unit = amount / ms / 1e9, "TFLOP/s"
        else:
            ach, unit = amount / ms / 1e6, "GB/s"
        entry = {"kernel": label, "ms": round(float(ms), 5), "achieved": round(ach, 1), "unit": unit,
                 "peak": peak_of[pk], "frac": round(ach / peak_of[pk], 4),
                 "frac_nominal": round(ach / NOMINAL_PEAK[pk], 4),
                 "algorithmic": amount, "share": round(float(ms / per_kernel.sum()), 4)}
        att = getattr(step, "attainable_ms", {}).get(label)
        if att is not None:  # grouped GEMMs: sum over experts of max(compute time, memory time)
            entry["attainable_ms"] = round(att, 5)
            entry["frac_attainable"] = round(att / ms, 4)
        kernels.append(entry)
    dom = max(range(nk), key=lambda k: per_kernel[k])
    dk = kernels[dom]
    roofline = {"kernel": dk["kernel"], "bound": "tensor" if step.kernels[dom][1] == "tensor" else "hbm",
                "achieved": dk["achieved"], "peak": dk["peak"], "unit": dk["unit"], "frac": dk["frac"],
                "traffic": traffic_for(step.name, dk["kernel"]),
                "peak_source": f"{peaks['src']} ({'2 x bf16 burst' if step.kernels[dom][3] == 'fp8' else step.kernels[dom][3]})"}

    # the unfused alternative of a fused step, timed the same way (per-kernel events, flushed L2)
    alt = None
    if hasattr(step, "alt_run"):
        for _ in range(args.warmup):
            step.alt_run()
        torch.cuda.synchronize()
        na = len(step.alt_kernels)
        aevs = [[torch.cuda.Event(enable_timing=True) for _ in range(na + 1)] for _ in range(args.steps)]
        torch.cuda._sleep(2_000_000 * min(args.steps, 40))  # host head start, as for the step
        for i in range(args.steps):
            flush.zero_()
            torch.amax(flush_rd)
            torch.cuda._sleep(100_000)  # the flush's write-backs drain, as for the step
            ev = aevs[i]
            step.alt_run(lambda k: ev[k].record(stream))
            ev[na].record(stream)
        torch.cuda.synchronize()
        aper = np.zeros(na)
        atot = 0.0
        for ev in aevs:
            aper += [ev[k].elapsed_time(ev[k + 1]) for k in range(na)]
            atot += ev[0].elapsed_time(ev[na])
        aper /= args.steps
        alt = {"ms_per_step": round(atot / args.steps, 5),
               "kernels": [{"kernel": lab, "ms": round(float(ms), 5)} for (lab, *_), ms in zip(step.alt_kernels, aper)],
               "value": round(whole_job_value(units, args.steps, 1, atot, step.unit), 2)}

    # e2e through the public entry points with host buffers
    e2e = None
    if hasattr(step, "e2e_setup") and not args.no_e2e:
        h2d, d2h = step.e2e_setup()
        step.e2e_run_steps(2)
        torch.cuda.synchronize()
        s0, s1 = step.e2e_run_steps(args.e2e_steps)
        torch.cuda.synchronize()
        ems = max_over_ranks(s0.elapsed_time(s1), ws)
        e2e = {"value": whole_job_value(units, args.e2e_steps, ws, ems, step.unit), "unit": step.unit,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "note": "inputs copied host->device and outputs device->host every step, overlapped with "
                       "the neighbouring steps' compute on separate streams"}

    cpu = None
    if rank == 0 and ws == 1 and not args.no_cpu_baseline:
        import oracle
        # steps that keep no host-side inputs take the host-drawn sample, scaled like --cpu-rows
        cpu_sample = getattr(step, "cpu_sample", None) or (
            lambda r: host_cpu_sample(step.name, max(1, SAMPLE_ROWS[step.name] * r // args.cpu_rows)))
        run, work, sample = cpu_sample(args.cpu_rows)
        t0 = time.perf_counter()
        run()
        dt = time.perf_counter() - t0
        scale = 1e12 if step.unit == "TFLOP/s" else 1e9
        cores = oracle.num_threads()
        cpu = {"value": work / dt / scale, "unit": step.unit,
               "cores": cores, "kind": "oracle", "sample": sample, "seconds": round(dt, 2)}
        # the same oracle on one core, on an eighth of the sample (skipped when that would take
        # more than ~40 s by the multi-core rate)
        run1, work1, sample1 = cpu_sample(max(1, args.cpu_rows // 8))
        est = dt * (work1 / work) * cores
        if est <= 40.0:
            oracle.set_num_threads(1)
            try:
                t0 = time.perf_counter()
                run1()
                dt1 = time.perf_counter() - t0
            finally:
                oracle.set_num_threads(cores)
            cpu.update({"value_1core": work1 / dt1 / scale, "sample_1core": sample1, "seconds_1core": round(dt1, 2)})
        else:
            cpu["value_1core"] = None
            cpu["note_1core"] = f"skipped: about {est:.0f} s on one core"

    launches = getattr(step, "launches_per_step", lambda: nk)() * args.steps
    if rank == 0:
        cfg = {"workload": step.name, "l2": "flushed between steps outside the timed events (256 MiB write, then 256 MiB read of another buffer)",
               "inputs": "seeded synthetic, resident in HBM"}
        for k in ("M", "K", "N", "E"):
            if hasattr(step, k):
                cfg[k] = getattr(step, k)
        line = {"metric": METRIC, "value": round(value, 2), "unit": step.unit, "n_gpus": ws, "steps": args.steps,
                "warmup": args.warmup, "ms_per_step": round(total_ms_max / args.steps, 5), "higher_is_better": True,
                "scaling": "weak", "vs_baseline": None,
                "dtype": getattr(step, "dtype", "fp8 e4m3/e5m2 (fp32 accumulate), bf16 wgrad"),
                "data": "synthetic", "config": cfg, "roofline": roofline, "kernels": kernels,
                "cpu_baseline": cpu, "e2e": e2e, "clocks": clocks, "gpu_launches": launches,
                **({"unfused": alt} if alt else {}),
                "wall_s": round(wall, 3), "impl": "fp8lin"}
        print(json.dumps(line))
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
