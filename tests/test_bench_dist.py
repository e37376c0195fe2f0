"""Multi-rank bench logic on CPU: world_size 2 over gloo.

bench.py launches one process per GPU; every rank serves its own sequences
(no exchange on the data path), the timed region is bracketed by barriers,
the step time is the max over ranks, and the whole-job rate counts every
rank's units.  These tests run that host logic with two gloo ranks.
"""
from __future__ import annotations

import os
import socket
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank: int, world: int, port: int, queue) -> None:
    sys.path.insert(0, ROOT)
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank),
                      WORLD_SIZE=str(world), LOCAL_RANK=str(rank))
    import torch.distributed as dist
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        import bench
        # every rank times its own steps; rank 1 is the slow one
        local_ms = 2.0 + 3.0 * rank
        bench.barrier(world)
        ms = bench.max_over_ranks(local_ms, world)
        rate = bench.whole_job_rate(16, world, ms)
        # the reference arm: rank 0 alone runs it, the others return at once
        class A:
            workload, steps, warmup, gpus = "tiny", 1, 0, world
        ref_ran = None
        if rank != 0:
            bench.run_reference(A, world, rank)
            ref_ran = False
        queue.put((rank, ms, rate, ref_ran))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_and_whole_job_rate_gloo():
    import torch.multiprocessing as mp
    ctx = mp.get_context("spawn")
    queue = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank_main, args=(r, 2, port, queue)) for r in range(2)]
    for p in procs:
        p.start()
    out = [queue.get(timeout=120) for _ in procs]
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    out.sort()
    # both ranks see the slowest rank's time and the same whole-job rate
    for rank, ms, rate, _ in out:
        assert ms == pytest.approx(5.0)
        assert rate == pytest.approx(16 * 2 / 5e-3)
    assert out[1][3] is False


def test_whole_job_rate_single_rank():
    sys.path.insert(0, ROOT)
    import bench
    assert bench.whole_job_rate(16, 1, 2.0) == pytest.approx(8000.0)
    assert bench.max_over_ranks(3.5, 1) == 3.5
