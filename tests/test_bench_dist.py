"""Host-side logic of the multi-process bench (CPU, gloo, two ranks): every rank runs its own
replica; timing is the max over ranks and the value counts the work of all ranks."""
import os
import socket

import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    s = socket.socket()
    s.bind(("127.0.0.1", 0))
    port = s.getsockname()[1]
    s.close()
    return port


def _worker(rank, world, port, out):
    import sys
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    import bench
    ws, r, _ = bench.dist_setup()
    assert (ws, r) == (world, rank)
    bench.barrier(ws)
    # each rank's own timing; the job is as slow as its slowest rank
    mine = 10.0 + 5.0 * rank
    m = bench.max_over_ranks(mine, ws)
    out[rank] = m
    dist.destroy_process_group()


def test_two_rank_gloo_aggregation():
    world, port = 2, _free_port()
    out = mp.Manager().dict()
    mp.start_processes(_worker, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
    assert out[0] == out[1] == 15.0


def test_whole_job_value_is_weak_scaling():
    import sys
    sys.path.insert(0, ROOT)
    import bench
    flop = 2.886e12
    one = bench.whole_job_value(flop, 10, 1, 12.7, "TFLOP/s")
    two = bench.whole_job_value(flop, 10, 2, 12.7, "TFLOP/s")
    assert abs(one - flop * 10 / 12.7 / 1e9) < 1e-9 * one and abs(two - 2 * one) < 1e-9 * two
    assert abs(bench.whole_job_value(3e8, 4, 1, 2.0, "GB/s") - 3e8 * 4 / 2.0 / 1e6) < 1e-6


class _FakeSmi:
    """Stands in for the nvidia-smi sampling process: fixed CSV output, no GPU."""

    def __init__(self, out):
        self.out = out

    def terminate(self):
        pass

    def communicate(self, timeout=None):
        return self.out, ""


def _smi_line(ts, sm, reasons=("Not Active",) * 4):
    stamp = ts.strftime("%Y/%m/%d %H:%M:%S.%f")[:-3]
    return f"{stamp}, 0, {sm}, 2070, 900.5, 0x0000000000000000, " + ", ".join(reasons)


def test_clock_sampler_keeps_the_timed_window():
    import datetime
    import sys
    sys.path.insert(0, ROOT)
    import bench
    t0 = datetime.datetime(2026, 1, 2, 3, 4, 5)
    lines = [_smi_line(t0, 1500),  # before the window (warm-up)
             _smi_line(t0 + datetime.timedelta(seconds=1), 2070),
             _smi_line(t0 + datetime.timedelta(seconds=1.05), 2055, ("Not Active", "Not Active", "Not Active", "Active")),
             _smi_line(t0 + datetime.timedelta(seconds=2), 1200, ("Active", "Not Active", "Not Active", "Not Active"))]
    s = object.__new__(bench.ClockSampler)
    s.proc = _FakeSmi("\n".join(lines) + "\n")
    s.gpu = "GPU-00000000-0000-0000-0000-000000000000"
    w0, w1 = (t0 + datetime.timedelta(seconds=0.9)).timestamp(), (t0 + datetime.timedelta(seconds=1.1)).timestamp()
    c = s.stop(w0, w1)
    assert c["samples"] == 2 and c["window"] == "timed region" and c["gpu"] == s.gpu
    assert c["sm_mhz"] == (2070 + 2055) / 2 and c["sm_max_mhz"] == 2070
    assert c["reasons"] == ["sw_power_cap"]  # the hw_slowdown sample lies outside the window


def test_clock_sampler_nearest_samples_for_a_short_window():
    import datetime
    import sys
    sys.path.insert(0, ROOT)
    import bench
    t0 = datetime.datetime(2026, 1, 2, 3, 4, 5)
    lines = [_smi_line(t0 + datetime.timedelta(seconds=x), sm) for x, sm in ((0.0, 1900), (0.05, 2000), (0.10, 2070))]
    s = object.__new__(bench.ClockSampler)
    s.proc = _FakeSmi("\n".join(lines) + "\n")
    s.gpu = "0"
    w0, w1 = (t0 + datetime.timedelta(seconds=0.06)).timestamp(), (t0 + datetime.timedelta(seconds=0.08)).timestamp()
    c = s.stop(w0, w1)
    assert c["samples"] == 2 and c["window"].startswith("nearest")
    assert c["sm_mhz"] == (2000 + 2070) / 2


def test_smi_gpu_id_falls_back_to_the_index(monkeypatch):
    """Without a usable UUID (no GPU here) or with nvidia-smi refusing it, the sampler names the
    GPU by its index."""
    import subprocess
    import sys
    sys.path.insert(0, ROOT)
    import bench

    class _Refused:
        returncode, stdout = 6, ""

    monkeypatch.setattr(subprocess, "run", lambda *a, **k: _Refused())
    assert bench.smi_gpu_id(3) == "3"
