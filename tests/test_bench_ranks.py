"""The multi-rank logic of bench.py on CPU: two gloo ranks (127.0.0.1) agree on the slowest rank's
time, scale the whole-job rate by the rank count, and only rank 0 runs the oracle arm."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, out):
    sys.path.insert(0, ROOT)
    import bench

    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        slowest = bench.max_over_ranks(1.5 + rank, world, "cpu")
        rate = bench.whole_job_rate(1000.0, world, slowest)

        class Args:
            steps, warmup, cpu_seconds = 1, 0, 1.0

        ref = bench.run_reference(Args, rank, world, rank) if rank != 0 else "skipped"
        dist.barrier()
        out[rank] = (slowest, rate, ref)
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_share_the_slowest_time():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    with ctx.Manager() as m:
        out = m.dict()
        mp.start_processes(_rank_main, args=(world, port, out), nprocs=world, join=True, start_method="spawn")
        res = dict(out)
    assert res[0][0] == res[1][0] == 2.5                      # the slowest rank's time on both
    assert res[0][1] == res[1][1] == pytest.approx(2 * 1000.0 / 2.5)
    assert res[1][2] is None                                   # the oracle arm runs on rank 0 only


def test_single_rank_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(3.25, 1) == 3.25
    assert bench.whole_job_rate(10.0, 1, 2.0) == 5.0
