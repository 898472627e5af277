"""bench.py's multi-rank logic on CPU: two gloo ranks (replicas, one per GPU
on a real box) agree on the slowest rank's times, the whole-job rate counts
every rank's units, and the reference arm prints only on rank 0."""
import json
import os
import socket
import subprocess
import sys

import pytest
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, ROOT)
import bench  # noqa: E402


def _free_port() -> int:
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank_main(rank, world, port, results):
    import torch
    import torch.distributed as dist

    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # rank r took 1 + r seconds for the prefill leg and 3 - r for decode
        mine = [1.0 + rank, 3.0 - rank, 4.0, 0.5 * (rank + 1)]
        dist.barrier()
        got = bench.max_over_ranks(mine, torch.device("cpu"))
        results[rank] = got
    finally:
        dist.destroy_process_group()


def test_two_gloo_ranks_take_the_slowest_rank_time():
    world = 2
    port = _free_port()
    ctx = mp.get_context("spawn")
    manager = ctx.Manager()
    results = manager.dict()
    procs = [ctx.Process(target=_rank_main, args=(r, world, port, results)) for r in range(world)]
    for p in procs:
        p.start()
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    expect = [2.0, 3.0, 4.0, 1.0]
    assert results[0] == expect and results[1] == expect


def test_single_process_keeps_its_own_times():
    import torch
    assert bench.max_over_ranks([1.5, 2.5], torch.device("cpu")) == [1.5, 2.5]


def test_job_rate_counts_all_ranks_units():
    # 2 ranks x 10 steps x 6.597 TFLOP in 0.1 s of the slowest rank
    assert bench.job_rate(6.597e12, 10, 2, 0.1) == pytest.approx(1.3194e15)
    assert bench.job_rate(6.597e12, 10, 1, 0.1) == pytest.approx(6.597e14)


def test_reference_arm_is_silent_on_other_ranks():
    env = dict(os.environ, RANK="1", WORLD_SIZE="2", LOCAL_RANK="1")
    out = subprocess.run([sys.executable, os.path.join(ROOT, "bench.py"), "--impl", "reference",
                          "--steps", "1", "--warmup", "0", "--ref-rows", "2", "--gpus", "2"],
                         capture_output=True, text=True, timeout=300, cwd=ROOT, env=env)
    assert out.returncode == 0, out.stderr
    assert [ln for ln in out.stdout.splitlines() if ln.startswith("{")] == []
