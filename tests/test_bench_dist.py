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


def test_bench_covers_every_configuration_and_defaults_to_8192():
    # the configuration list: 256^3, 4096^3, the skinny sweep, the three
    # ragged shapes and bf16 8192^3, each once; INT8 8192^3 is the headline
    shapes = {k: v[1] for k, v in bench.BENCH_WORKLOADS.items()}
    want = [(256, 256, 256), (4096, 4096, 4096)] + [(m, 8192, 8192) for m in (1, 8, 16, 32, 64, 128)] + \
        [(1000, 777, 3000), (4097, 16384, 255), (8192, 8192, 8192), (8192, 8192, 8192)]
    assert sorted(shapes.values()) == sorted(want)
    assert bench.parse([]).workload == "i8_8192" and bench.DEFAULT_WORKLOAD == "i8_8192"
    assert bench.BENCH_WORKLOADS["bf16_8192"][0] == "bf16_8192"


def test_reference_arm_prints_this_arms_config(monkeypatch, capsys):
    # the reference arm's JSON line carries exactly the config dict that the
    # GPU arm prints for the same workload (a fake oracle runner stands in)
    import json

    class FakeRunner:
        threads = 4

        def __init__(self, workload, shape, A=None, Bt=None):
            self.m, self.k, self.n = shape

        def rows_for(self, seconds):
            return 1

        def run(self, rows):
            return 0.01

        def ops(self, rows):
            return 2.0 * rows * self.n * self.k

        def sample_text(self, rows):
            return "first %d rows" % rows

    monkeypatch.setenv("RANK", "0")
    monkeypatch.setenv("WORLD_SIZE", "1")
    monkeypatch.setattr(bench, "OracleRunner", FakeRunner)
    for key in ("i8_8192", "bf16_8192", "i8_skinny_m64"):
        args = argparse.Namespace(workload=key, steps=3, warmup=3, gpus=1)
        assert bench.run_reference(args) == 0
        line = json.loads(capsys.readouterr().out.strip().splitlines()[-1])
        assert line["impl"] == "reference" and line["config"] == bench.config_of(key, 1)
        assert set(line["config"]) == {"workload", "m", "k", "n", "parallelism"}


def test_clock_summary_reasons_and_median():
    s = bench.ClockSampler(0)
    s.rows = [{"sm": 2070.0, "max": 2070.0, "power": 900.0, "reasons": []},
              {"sm": 1900.0, "max": 2070.0, "power": 1400.0, "reasons": ["sw_power_cap"]},
              {"sm": 2000.0, "max": 2070.0, "power": 1300.0, "reasons": []}]
    out = s.summary()
    assert out["sm_mhz"] == 2000.0 and out["sm_max_mhz"] == 2070.0
    assert out["reasons"] == ["sw_power_cap"] and out["samples"] == 3
    empty = bench.ClockSampler(0).summary()
    assert empty["samples"] == 0 and empty["sm_mhz"] is None


def test_traffic_records_match_the_kernel_sources():
    # the headline's DRAM traffic and the skinny one are reported only while
    # the kernel sources still match the digest recorded with the ncu capture:
    # a kernel change must come with a new capture
    rec = bench.load_traffic()
    assert rec["i8_8192"][1] == bench.kernel_source_digest("tc")
    assert rec["i8_skinny_m64"][1] == bench.kernel_source_digest("skinny")
    # DRAM bytes of one launch: at least the algorithmic bytes each kernel moves
    k = n = 8192
    assert rec["i8_8192"][0] >= 2 * 8192 * 8192 * 2 + 4 * 8192 * 8192   # f16 A and Bt once, int32 C
    assert rec["i8_skinny_m64"][0] >= n * k                           # Bt once
