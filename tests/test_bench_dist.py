"""Host-side logic of the multi-process bench (CPU, gloo, two ranks): every rank runs its own
replica; timing is the max over ranks and the value counts the work of all ranks."""
import os
import socket

import pytest
import torch
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
