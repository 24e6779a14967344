"""The multi-rank path of bench.py on CPU: two gloo ranks (one process each, as
torchrun launches them) agree on the job time = the slowest rank's, the
whole-job value counts every rank's units, and the reference arm runs on rank 0
only (the others exit without work)."""
import argparse
import os
import socket
import time

import pytest

import bench

torch = pytest.importorskip("torch")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    import torch.distributed as dist
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port), RANK=str(rank), WORLD_SIZE=str(world))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        dist.barrier()
        ms = bench.job_ms(1.5 + 2.5 * rank)  # rank 1 is the slow one
        t = time.perf_counter()
        if rank != 0:  # the reference arm: rank 0 alone runs it
            bench.run_reference(argparse.Namespace(warmup=3, steps=5))
        q.put((rank, ms, time.perf_counter() - t))
    finally:
        dist.destroy_process_group()


def test_job_time_is_the_slowest_rank_and_value_counts_all_ranks():
    ctx = torch.multiprocessing.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    got = sorted(q.get(timeout=5) for _ in range(2))
    assert [g[1] for g in got] == [4.0, 4.0]
    assert got[1][2] < 1.0  # rank 1's reference arm returns at once
    # weak scaling: 2 ranks x 1e9 units in 4 ms
    assert bench.job_value(1e9, 2, 4.0) == pytest.approx(5e11)


def test_single_process_keeps_its_own_time():
    assert bench.job_ms(2.25) == 2.25
    assert bench.job_value(10.0, 1, 1000.0) == pytest.approx(10.0)
