"""Benchmark of the dense GEMM hot path on GB300.

Default workload: INT8 GEMM m = k = n = 4096 (A row-major, B K-major, int8
uniform in [-128, 127], seed 1), int32 output; metric TOPS = 2*m*n*k / t.
A step is one gemm_i8_run through the C ABI: plan lookup, int8 -> f16
operand staging, tcgen05 tensor-core GEMM.  Inputs are resident in HBM and
rotated through enough distinct input sets that they are never L2 hits.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   (the CPU oracle, timed alone)

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the path has no exchange step); rank 0 prints one JSON line.
"""

from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "INT8 GEMM TOPS (2mnk/s) and % of GB300 dense INT8 peak / HBM roofline"
TRACE_EVERY = 16   # one step in TRACE_EVERY is timed kernel by kernel

# name -> (workload, shape)
BENCH_WORKLOADS = {
    "i8_4096": ("i8_4096", (4096, 4096, 4096)),
    "i8_256": ("i8_256", (256, 256, 256)),
    "i8_8192": ("i8_ragged", (8192, 8192, 8192)),
    "i8_4097x16384x255": ("i8_ragged", (4097, 16384, 255)),
    "i8_1000x777x3000": ("i8_ragged", (1000, 777, 3000)),
    "bf16_8192": ("bf16_8192", (8192, 8192, 8192)),
    **{"i8_skinny_m%d" % m: ("i8_skinny", (m, 8192, 8192)) for m in (1, 8, 16, 32, 64, 128)},
}

DESCRIPTIONS = {
    "i8_4096": "INT8 GEMM m=k=n=4096, A row-major, B K-major, int8 uniform [-128,127] seed 1, int32 out",
    "i8_256": "INT8 GEMM m=k=n=256, int8 uniform [-128,127] seed 0, int32 out",
    "i8_8192": "INT8 GEMM m=k=n=8192, int8 uniform [-128,127] seed 3, int32 out",
    "i8_4097x16384x255": "INT8 GEMM (4097,16384,255), int8 uniform [-128,127] seed 3, int32 out",
    "i8_1000x777x3000": "INT8 GEMM (1000,777,3000), int8 uniform [-128,127] seed 3, int32 out",
    "bf16_8192": "BF16 GEMM m=k=n=8192, N(0,1) rounded to bf16 seed 4, fp32 accumulate and out",
}
for _m in (1, 8, 16, 32, 64, 128):
    DESCRIPTIONS["i8_skinny_m%d" % _m] = ("INT8 skinny GEMM m=%d, k=n=8192, A U[-64,63], B round(32 N(0,1)) "
                                          "clipped, seed 2, int32 out" % _m)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=sorted(BENCH_WORKLOADS), default="i8_4096")
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target CPU time of the oracle baseline sample")
    return ap.parse_args()


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def max_over_ranks(ms: float, world: int, device: str) -> float:
    """The slowest rank's time: every rank runs an independent replica, so
    the job takes as long as its slowest one.  All ranks must call it."""
    if world <= 1:
        return ms
    import torch
    import torch.distributed as dist
    t = torch.tensor([ms], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    dist.barrier()
    return float(t.item())


def whole_job_value(world: int, ops_per_step: float, ms_per_step: float) -> float:
    """Tera-operations per second of all ranks together (weak scaling: each
    rank does one step's work per step)."""
    return world * ops_per_step / (ms_per_step / 1000.0) / 1e12


def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return d, "measured"
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}, "fallback"


def load_traffic():
    """Per-launch DRAM bytes of the dominant kernels from the committed ncu
    summary, keyed by workload, valid only for the kernel sources they were
    measured on."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    out = {}
    if not os.path.exists(path):
        return out
    for line in open(path):
        line = line.strip()
        if not line or line.startswith("#"):
            continue
        parts = line.split()
        if len(parts) >= 3:
            out[parts[0]] = (float(parts[1]), parts[2])
    return out


# the sources each recorded kernel is compiled from (its own file, the PTX
# helpers and the shared constants)
KERNEL_SOURCES = {
    "tc": ("gemm_tc2.cu", "gemm_tc.cu", "ptx.cuh", "internal.h"),
    "skinny": ("gemm_skinny_tc.cu", "ptx.cuh", "internal.h"),
}


def kernel_source_digest(kind: str) -> str:
    """Digest of the code (comments and blank lines removed) of the sources
    a recorded kernel is compiled from: an edited comment keeps the record."""
    import hashlib
    import re
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "dense_int8_matrix_gb300", "csrc")
    for name in sorted(KERNEL_SOURCES[kind]):
        text = open(os.path.join(csrc, name), encoding="utf-8").read()
        text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
        text = re.sub(r"//[^\n]*", "", text)
        code = "\n".join(line.rstrip() for line in text.splitlines() if line.strip())
        h.update(name.encode())
        h.update(code.encode())
    return h.hexdigest()[:16]


class ClockSampler:
    """nvidia-smi clock / throttle-reason samples while the timed region runs."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int):
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None
        time.sleep(0.3)
        return self

    def __exit__(self, *exc):
        if self.proc is None:
            self.out = ""
            return False
        time.sleep(0.2)
        self.proc.terminate()
        try:
            self.out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            self.out, _ = self.proc.communicate()
        return False

    def summary(self):
        rows = []
        for line in (getattr(self, "out", "") or "").splitlines():
            parts = [p.strip() for p in line.split(",")]
            if len(parts) < 9:
                continue
            try:
                rows.append({"sm": float(parts[1]), "max": float(parts[2]), "power": float(parts[3]),
                             "hw": parts[5], "hw_thermal": parts[6], "sw_thermal": parts[7],
                             "sw_power": parts[8]})
            except ValueError:
                continue
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no nvidia-smi samples"], "samples": 0}
        loaded = [r for r in rows if r["power"] > 200.0] or rows
        reasons = set()
        for r in rows:
            if r["hw"].lower().startswith("active"):
                reasons.add("hw_slowdown")
            if r["hw_thermal"].lower().startswith("active"):
                reasons.add("hw_thermal_slowdown")
            if r["sw_thermal"].lower().startswith("active"):
                reasons.add("sw_thermal_slowdown")
            if r["sw_power"].lower().startswith("active"):
                reasons.add("sw_power_cap")
        return {"sm_mhz": statistics.median(r["sm"] for r in loaded),
                "sm_max_mhz": max(r["max"] for r in rows), "reasons": sorted(reasons),
                "samples": len(rows), "samples_under_load": len([r for r in rows if r["power"] > 200.0])}


# ------------------------------------------------------------ CPU oracle --

class OracleRunner:
    """The CPU oracle on a bounded sample of a workload: the first R rows of C
    (all n columns, full k).  Only this benchmark leg touches the oracle."""

    def __init__(self, workload: str, shape):
        import numpy as np

        import oracle
        from dense_int8_matrix_gb300 import workloads

        oracle.build()
        self.m, self.k, self.n = shape
        A, Bt = workloads.make_inputs(workload, shape)
        self.threads = host_cores()
        if workloads.WORKLOADS[workload]["dtype"] == "i8":
            An, Bn = A.numpy(), Bt.numpy()
            self._run = lambda r: oracle.gemm_i8(An[:r], Bn, nthreads=self.threads)
        else:
            import torch
            bits = lambda t: t.contiguous().view(torch.int16).numpy().view(np.uint16)  # noqa: E731
            An, Bn = bits(A), bits(Bt)
            self._run = lambda r: oracle.gemm_bf16(An[:r], Bn, nthreads=self.threads, with_abs=False)

    def run(self, rows: int) -> float:
        t0 = time.perf_counter()
        self._run(rows)
        return time.perf_counter() - t0

    def rows_for(self, seconds: float) -> int:
        cal = min(self.m, self.threads)
        per_row = max(self.run(cal), 1e-6) / cal
        rows = int(max(1, min(self.m, seconds / per_row)))
        if rows >= self.threads:
            rows = rows // self.threads * self.threads
        return rows

    def ops(self, rows: int) -> float:
        return 2.0 * rows * self.n * self.k

    def sample_text(self, rows: int) -> str:
        return "first %d of %d rows of C (all %d columns, k=%d)" % (rows, self.m, self.n, self.k)


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    workload, shape = BENCH_WORKLOADS[args.workload]
    m, k, n = shape
    runner = OracleRunner(workload, shape)
    budget = 120.0  # seconds for the whole reference run
    rows = runner.rows_for(max(0.02, budget / max(1, args.steps + args.warmup)))
    times = []
    for i in range(args.warmup + args.steps):
        dt = runner.run(rows)
        if i >= args.warmup:
            times.append(dt)
    ms = 1000.0 * statistics.mean(times)
    value = runner.ops(rows) / (ms / 1000.0) / 1e12
    is_i8 = workload != "bf16_8192"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TOPS" if is_i8 else "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "i8->i64 exact" if is_i8 else "f64", "data": "synthetic",
        "config": {"workload": DESCRIPTIONS[args.workload], "m": m, "k": k, "n": n,
                   "oracle": "plain C triple loop, rows split over POSIX threads"},
        "cpu_baseline": {"value": value, "unit": "TOPS" if is_i8 else "TFLOP/s", "cores": runner.threads,
                         "kind": "oracle", "sample": runner.sample_text(rows) + " per step"},
        "e2e": {"value": value, "unit": "TOPS" if is_i8 else "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------ GPU path ----

def graph_throughput(run, plan, sets, C, nsets, steps, world, ops):
    """Steps captured once into a CUDA graph (every input set a few times)
    and the graph replayed until about `steps` steps have run; the device time
    per step over the replays, max over ranks."""
    import torch
    try:
        per_graph = nsets * max(1, 32 // nsets)
        replays = max(3, steps // per_graph)
        gs = torch.cuda.Stream()
        gs.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=gs):
            cur = torch.cuda.current_stream()
            for i in range(per_graph):
                A, Bt = sets[i % nsets]
                run(plan, A, Bt, C, cur)
        for _ in range(2):
            g.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(gs):
            e0.record(gs)
            for _ in range(replays):
                g.replay()
            e1.record(gs)
        torch.cuda.synchronize()
        ms = max_over_ranks(e0.elapsed_time(e1), world, "cuda") / (replays * per_graph)
        return {"value": whole_job_value(world, ops, ms), "ms_per_step": ms, "steps_per_replay": per_graph,
                "replays": replays}
    except Exception as exc:   # noqa: BLE001 - reported, not fatal
        return {"unavailable": "%s: %s" % (type(exc).__name__, str(exc)[:200])}


def run_ours(args):
    import torch

    from dense_int8_matrix_gb300 import binding as B
    from dense_int8_matrix_gb300 import build as lib_build
    from dense_int8_matrix_gb300 import workloads

    world, rank, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.cuda.current_device()
    lib_build.build()
    B.load()

    workload, shape = BENCH_WORKLOADS[args.workload]
    m, k, n = shape
    is_i8 = workloads.WORKLOADS[workload]["dtype"] == "i8"
    plan = B.gemm_i8_plan(m, k, n) if is_i8 else B.gemm_bf16_plan(m, k, n)
    run = B.gemm_i8_run if is_i8 else B.gemm_bf16_run
    run_host = B.gemm_i8_run_host if is_i8 else B.gemm_bf16_run_host
    out_dtype = torch.int32 if is_i8 else torch.float32
    esize = 1 if is_i8 else 2

    # distinct input sets, together larger than 2x L2, so no step hits in L2
    l2 = torch.cuda.get_device_properties(dev).L2_cache_size
    set_bytes = (m * k + n * k) * esize
    nsets = max(2, min(64, -(-(2 * l2) // set_bytes)))
    base_A, base_B = workloads.make_inputs(workload, shape)
    sets = []
    for s in range(nsets):
        if s == 0:
            A, Bt = base_A, base_B
        else:
            # cheap distinct copies: a per-set rotation of the rows
            A = torch.roll(base_A, shifts=s, dims=0)
            Bt = torch.roll(base_B, shifts=3 * s, dims=0)
        sets.append((A.cuda(), Bt.cuda()))
    C = torch.empty((m, n), dtype=out_dtype, device="cuda")
    stream = torch.cuda.current_stream()

    for i in range(args.warmup):
        A, Bt = sets[i % nsets]
        run(plan, A, Bt, C, stream)
    torch.cuda.synchronize()

    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    # sampled trace: every TRACE_EVERY-th step times its launches with events,
    # the other steps run undisturbed.  On the skinny path consecutive calls
    # overlap (each call's kernels may start before the previous call's end,
    # through programmatic dependent launch) and an event between two calls
    # would serialise them, so there the launches are only counted and the
    # timed region itself gives the duration of a launch unit.
    skinny = plan.path == B.GEMM_PATH_SKINNY
    B.gemm_trace_begin(0 if skinny else 2 * (args.steps // TRACE_EVERY) + 8, TRACE_EVERY)
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev) as clk:
        ev0.record(stream)
        for i in range(args.steps):
            A, Bt = sets[i % nsets]
            run(plan, A, Bt, C, stream)
        ev1.record(stream)
        torch.cuda.synchronize()
    elapsed_ms = ev0.elapsed_time(ev1)
    clk_summary = clk.summary()
    kernel_ms, timed, launches = B.gemm_trace_collect()
    st, code = B.gemm_device_error()
    if st != B.GEMM_OK:
        raise RuntimeError("device error during bench: code %d" % code)
    max_ms = max_over_ranks(elapsed_ms, world, "cuda")

    ops = 2.0 * m * n * k
    ms_per_step = max_ms / args.steps
    value = whole_job_value(world, ops, ms_per_step)

    # the same steps captured into a CUDA graph and replayed: the loop a
    # serving process would replay (a user may capture gemm_*_run calls);
    # reported beside the stream-launched value, which stays the headline
    graph_line = graph_throughput(run, plan, sets, C, nsets, args.steps, world, ops)

    # end to end through the host-buffer entry point: H2D of A and Bt,
    # the GEMM, D2H of C, inside the timed region
    hA = base_A.pin_memory()
    hB = base_B.pin_memory()
    hC = torch.empty((m, n), dtype=out_dtype).pin_memory()
    run_host(plan, hA, hB, hC, stream)
    e2e_times = []
    for _ in range(args.e2e_steps):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        run_host(plan, hA, hB, hC, stream)
        e2e_times.append(time.perf_counter() - t0)
    e2e_s = statistics.median(e2e_times)
    e2e_value = ops / e2e_s / 1e12

    # roofline of the dominant kernel
    peaks, peak_src = load_peaks()
    if skinny:
        # one launch unit (prologue + skinny kernel) per step; units overlap
        # their neighbours, so a unit lasts the timed region over the steps
        per_launch_ms = ms_per_step
        alg_bytes = m * k + n * k + 4 * m * n
        achieved = alg_bytes / (per_launch_ms / 1000.0) / 1e9
        roof = {"kernel": "skinny_prologue + skinny_tc, one unit per step (CUDA events around the timed "
                          "region: consecutive units overlap through programmatic dependent launch)",
                "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"],
                "unit": "GB/s", "frac": achieved / peaks["hbm_gbs"],
                "peak_source": "%s hbm_gbs (STREAM-style copy)" % peak_src,
                "algorithmic_bytes_per_launch": alg_bytes}
        traffic_key = args.workload
    else:
        kind = B.GEMM_KERNEL_TC
        per_launch_ms = kernel_ms[kind] / max(1, timed[kind])
        achieved = ops / (per_launch_ms / 1000.0) / 1e12
        # the burst peak for a kernel the power cap did not touch, the
        # sustained one when the clocks sampled in the timed region show the
        # power cap (the kernel then runs like one inside a long step)
        capped = "sw_power_cap" in (clk_summary.get("reasons") or [])
        peak_key = "bf16_tflops_sustained" if capped and "bf16_tflops_sustained" in peaks else "bf16_tflops"
        peak = peaks[peak_key]
        roof = {"kernel": "gemm_tc2 / gemm_tc (tcgen05 kind::f16)", "bound": "tensor", "achieved": achieved,
                "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
                "peak_source": ("%s %s (%s cuBLAS bf16 GEMM%s); the int8 path runs on f16 tensor-core MMAs, "
                                "whose nominal dense rate equals bf16's"
                                % (peak_src, peak_key, "sustained" if capped else "burst",
                                   ", clocks under sw_power_cap" if capped else "")),
                "algorithmic_flops_per_launch": ops}
        traffic_key = args.workload
    traffic = load_traffic().get(traffic_key)
    digest = kernel_source_digest("skinny" if skinny else "tc")
    roof["traffic"] = traffic[0] if traffic and traffic[1] == digest else None
    roof["kernel_ms_per_launch"] = per_launch_ms

    line = {
        "metric": METRIC, "value": value, "unit": "TOPS" if is_i8 else "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "i8->i32 exact (f16 tensor-core MMA, fp32 chunks <= 2^24, int32 sum)" if is_i8
        else "bf16->f32 (fp32 accumulate)",
        "data": "synthetic",
        "config": {"workload": DESCRIPTIONS[args.workload], "m": m, "k": k, "n": n,
                   "l2": "inputs rotated over %d distinct sets (%d MiB) > 2x L2 (%d MiB)"
                         % (nsets, nsets * set_bytes >> 20, l2 >> 20),
                   "plan": {"path": "tensor" if plan.path == 0 else "skinny", "bm": plan.bm,
                            "bn": plan.bn, "grid": plan.grid, "tiles": plan.tiles, "waves": plan.waves,
                            "num_sms": plan.num_sms},
                   "parallelism": "replicas" if world > 1 else "single-gpu"},
        "gpu_launches": int(sum(launches)),
        "gpu_launches_by_kind": {"stage": launches[0], "tc": launches[1], "skinny": launches[2]},
        "kernel_ms_per_timed_unit": {name: kernel_ms[i] / timed[i] if timed[i] else None
                                     for i, name in enumerate(("stage", "tc", "skinny"))},
        "timed_units": {"every": TRACE_EVERY, "stage": timed[0], "tc": timed[1], "skinny": timed[2]},
        "roofline": roof,
        "graph": graph_line,
        "clocks": clk_summary,
        "e2e": {"value": e2e_value, "unit": "TOPS" if is_i8 else "TFLOP/s",
                "h2d_bytes_per_step": (m * k + n * k) * esize, "d2h_bytes_per_step": m * n * 4,
                "ms_per_step": e2e_s * 1000.0},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        runner = OracleRunner(workload, shape)
        rows = runner.rows_for(args.cpu_seconds)
        dt = runner.run(rows)
        line["cpu_baseline"] = {"value": runner.ops(rows) / dt / 1e12, "unit": line["unit"],
                                "cores": runner.threads, "kind": "oracle",
                                "sample": runner.sample_text(rows) + ": %.1f s" % dt}
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


def main():
    args = parse()
    if args.warmup < 3:
        args.warmup = 3
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
