"""The benchmark's multi-rank logic on CPU: two gloo ranks agree on the
slowest rank's time, the whole-job value counts every rank's work, and only
rank 0 runs the reference arm."""

from __future__ import annotations

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


def _rank_main(rank: int, world: int, port: int, times, out):
    import torch.distributed as dist
    os.environ["MASTER_ADDR"] = "127.0.0.1"
    os.environ["MASTER_PORT"] = str(port)
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        out[rank] = bench.max_over_ranks(times[rank], world, "cpu")
    finally:
        dist.destroy_process_group()


@pytest.mark.parametrize("times", [[1.5, 4.25], [9.0, 2.0]])
def test_max_over_two_gloo_ranks(times):
    world = 2
    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        out = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_rank_main, args=(r, world, port, times, out)) for r in range(world)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        assert [out[r] for r in range(world)] == [max(times)] * world


def test_single_rank_needs_no_process_group():
    assert bench.max_over_ranks(3.0, 1, "cpu") == 3.0


def test_whole_job_value_counts_every_rank():
    ops = 2.0 * 4096 ** 3
    one = bench.whole_job_value(1, ops, 0.1)
    assert abs(one - ops / 1e-4 / 1e12) < 1e-9
    assert abs(bench.whole_job_value(8, ops, 0.1) - 8 * one) < 1e-9


def test_reference_arm_runs_on_rank_zero_only(monkeypatch):
    # a rank other than 0 exits at once, without touching the oracle
    monkeypatch.setenv("RANK", "1")
    monkeypatch.setenv("WORLD_SIZE", "2")
    monkeypatch.setattr(bench, "OracleRunner", lambda *a, **k: pytest.fail("oracle ran on rank 1"))
    args = argparse.Namespace(workload="i8_256", steps=3, warmup=3, gpus=2)
    assert bench.run_reference(args) == 0
