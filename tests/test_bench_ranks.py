"""The benchmark's multi-rank bookkeeping, on CPU ranks over gloo: each rank
times its own replica of the workload; the job's time is the slowest rank's,
and the value counts every rank's operations (weak scaling)."""
import os
import socket

import pytest

torch = pytest.importorskip("torch")
mp = pytest.importorskip("torch.multiprocessing")


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    import torch.distributed as dist

    import bench

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        local_ms = 10.0 + 5.0 * rank          # rank 1 is the slower one
        results[rank] = bench.job_time(local_ms, steps=100, pack=8, world=world, dist=dist, device="cpu")
    finally:
        dist.destroy_process_group()


def test_job_time_is_max_over_ranks_and_counts_all_operations():
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as manager:
        results = manager.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        for r in range(world):
            ms, us = results[r]
            assert ms == 15.0                              # the slowest rank's time, on every rank
            assert us == pytest.approx(15.0e3 / (100 * 8 * 2))


def test_job_time_single_rank():
    import bench

    assert bench.job_time(8.0, steps=100, pack=8, world=1) == (8.0, 8.0e3 / 800)
