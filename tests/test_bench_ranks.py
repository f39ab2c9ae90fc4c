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


def _run_bench(args, env_extra=None):
    import json
    import subprocess
    import sys

    root = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
    env = dict(os.environ)
    env.update(env_extra or {})
    r = subprocess.run([sys.executable, os.path.join(root, "bench.py")] + args, cwd=root, env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0, r.stderr[-2000:]
    lines = [l for l in r.stdout.splitlines() if l.strip()]
    return [json.loads(l) for l in lines]


def test_reference_arm_json_line():
    """`bench.py --impl reference` (the oracle on the host cores) prints one
    JSON line with the contract's keys; its cpu_baseline describes the run
    and its e2e is the line's own value with no device copies."""
    (line,) = _run_bench(["--impl", "reference", "--steps", "1", "--warmup", "1"])
    for key in ("impl", "metric", "value", "unit", "n_gpus", "steps", "warmup", "ms_per_step",
                "higher_is_better", "scaling", "vs_baseline", "dtype", "data", "config", "cpu_baseline", "e2e"):
        assert key in line, key
    assert line["impl"] == "reference" and line["higher_is_better"] is False and line["unit"] == "µs/op"
    assert line["steps"] == 1 and line["warmup"] >= 1 and line["value"] > 0
    cb = line["cpu_baseline"]
    assert cb["kind"] == "oracle" and cb["value"] == line["value"] and cb["cores"] >= 1 and cb["sample"]
    e2e = line["e2e"]
    assert e2e["value"] == line["value"] and e2e["unit"] == line["unit"]
    assert e2e["h2d_bytes_per_step"] == 0 and e2e["d2h_bytes_per_step"] == 0
    assert line["config"]["workload"] and line["config"]["M"] == 256


def test_reference_arm_other_ranks_print_nothing():
    assert _run_bench(["--impl", "reference", "--steps", "1", "--warmup", "1"], {"RANK": "1", "WORLD_SIZE": "2"}) == []
