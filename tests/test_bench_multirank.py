"""The benchmark's multi-rank host logic on the CPU (gloo, world size 2): the job time
is the slowest rank's, throughput counts every rank's tokens, and the reference arm runs
on rank 0 only.  (The GPU path runs the same code under torchrun with NCCL.)"""

import argparse
import os
import socket

import pytest
import torch.multiprocessing as mp

import bench


def _free_port() -> int:
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        # each rank its own step time; every rank must end with the slowest one
        got = bench.max_over_ranks(1.25 + 0.5 * rank, world, "cpu")
        q.put((rank, got))
    finally:
        dist.destroy_process_group()


def test_max_over_ranks_gloo_world2():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    res = dict(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert res == {0: 1.75, 1: 1.75}


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.0, 1, "cpu") == 3.0


def test_job_throughput_counts_every_rank():
    # 4 ranks, 16 tokens each, 0.5 ms per step: 128k tokens/s for the job
    assert bench.job_tokens_per_s(4, 16, 0.5) == pytest.approx(128000.0)
    assert bench.job_tokens_per_s(1, 16, 0.5) == pytest.approx(32000.0)


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    args = argparse.Namespace(config="tiny_m4_h256_i128_e8_k2", steps=1, warmup=0)
    # a rank other than 0 returns at once, without touching inputs or the oracle
    monkeypatch.setattr(bench, "run_cpu_oracle", lambda *a, **k: (_ for _ in ()).throw(
        AssertionError("rank 1 ran the oracle")))
    assert bench.reference_arm(args, 1, 2) == 0


def test_dist_env(monkeypatch):
    monkeypatch.setenv("RANK", "3")
    monkeypatch.setenv("WORLD_SIZE", "4")
    monkeypatch.setenv("LOCAL_RANK", "1")
    assert bench.dist_env() == (3, 4, 1)
