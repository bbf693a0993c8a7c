"""The N > 1 host logic of bench.py on CPU, with two gloo ranks: every rank runs
its own replica, the timed region is the maximum over ranks, the rate counts
the units of all ranks, and the reference arm runs on rank 0 only."""
import os
import socket
import sys

import pytest
import torch
import torch.distributed as dist
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, out):
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world),
                      LOCAL_RANK=str(rank))
    sys.path.insert(0, ROOT)
    import bench

    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = [12.5, 20.0][rank]  # rank 1 is the slow replica
        ms = bench.max_over_ranks(local_ms, dist, device="cpu")
        rate = bench.whole_job_rate(world, 24576, 10, ms)
        dist.barrier()
        # the reference arm: every rank but 0 leaves before any work
        args = type("A", (), dict(steps=1, warmup=0, gpus=world))()
        if rank != 0:
            bench.run_reference(args)  # returns at once on rank != 0
        out.put((rank, ms, rate, bench.dist_env()))
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_max_time_and_whole_job_rate():
    world, port = 2, _free_port()
    ctx = mp.get_context("spawn")
    out = ctx.Queue()
    procs = [ctx.Process(target=_worker, args=(r, world, port, out)) for r in range(world)]
    for p in procs:
        p.start()
    res = sorted(out.get(timeout=120) for _ in range(world))
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    for rank, ms, rate, env in res:
        assert ms == 20.0                                    # the slowest rank's time, on every rank
        assert rate == pytest.approx(2 * 24576 * 10 / 0.020)  # units of both ranks per second
        assert env == (rank, world, rank)


def test_single_process_needs_no_process_group():
    sys.path.insert(0, ROOT)
    import bench

    assert bench.max_over_ranks(7.25, None) == 7.25
    assert bench.whole_job_rate(1, 100, 4, 2.0) == pytest.approx(100 * 4 / 0.002)
