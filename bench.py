"""Benchmark of the dense GEMM hot path on GB300.

Headline workload: INT8 GEMM m = k = n = 8192 (A row-major, B K-major, int8
uniform in [-128, 127], seed 3), int32 output; metric TOPS = 2*m*n*k / t.
A step is one gemm_i8_run through the C ABI: plan lookup, int8 -> f16
operand staging, tcgen05 tensor-core GEMM.  Inputs are resident in HBM and
rotated through enough distinct input sets that they are never L2 hits.

The same JSON line carries, besides the headline:
  roofline    the dominant kernel's work per launch over its average launch
              duration, from a separate pass of 200 launches timed with CUDA
              events on the launching stream after the timed region;
  per_config  every configuration of the benchmark list (256^3, 4096^3, the
              skinny sweep m in {1..128} x 8192^2, the three ragged shapes,
              bf16 8192^3), then int8 8192^3 requantised to bfloat16 and to
              int8: throughput, roofline fraction of its dominant kernel and
              the CPU oracle on a bounded sample (N = 1 only);
  e2e         the headline through the host-buffer entry point (H2D and D2H
              inside the timed region);
  clocks      SM clocks and throttle reasons sampled during the timed region.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
    python bench.py --impl reference ...   (the CPU oracle, timed alone)

Under torchrun (N > 1) every rank runs an independent replica on its own GPU
(the path has no exchange step); rank 0 prints one JSON line.
"""

from __future__ import annotations

import argparse
import ctypes
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "INT8 GEMM TOPS (2mnk/s) and % of GB300 dense INT8 peak / HBM roofline"
TRACE_EVERY = 16          # in the timed region one step in TRACE_EVERY is timed kernel by kernel
KERNEL_PASS_LAUNCHES = 200
DEFAULT_WORKLOAD = "i8_8192"

# name -> (workload, shape), in the order of the benchmark's configuration list
BENCH_WORKLOADS = {
    "i8_256": ("i8_256", (256, 256, 256)),
    "i8_4096": ("i8_4096", (4096, 4096, 4096)),
    **{"i8_skinny_m%d" % m: ("i8_skinny", (m, 8192, 8192)) for m in (1, 8, 16, 32, 64, 128)},
    "i8_1000x777x3000": ("i8_ragged", (1000, 777, 3000)),
    "i8_4097x16384x255": ("i8_ragged", (4097, 16384, 255)),
    "i8_8192": ("i8_ragged", (8192, 8192, 8192)),
    "bf16_8192": ("bf16_8192", (8192, 8192, 8192)),
}
# the requantising epilogue (int8 8192^3 to bfloat16 and to int8 through
# gemm_i8_run_requant): per_config entries beyond the configuration list
REQUANT_WORKLOADS = {
    "i8_8192_requant_bf16": ("i8_ragged", (8192, 8192, 8192), "bf16"),
    "i8_8192_requant_i8": ("i8_ragged", (8192, 8192, 8192), "i8"),
}

DESCRIPTIONS = {
    "i8_4096": "INT8 GEMM m=k=n=4096, A row-major, B K-major, int8 uniform [-128,127] seed 1, int32 out",
    "i8_256": "INT8 GEMM m=k=n=256, int8 uniform [-128,127] seed 0, int32 out",
    "i8_8192": "INT8 GEMM m=k=n=8192, A row-major, B K-major, int8 uniform [-128,127] seed 3, int32 out",
    "i8_4097x16384x255": "INT8 GEMM (4097,16384,255), int8 uniform [-128,127] seed 3, int32 out",
    "i8_1000x777x3000": "INT8 GEMM (1000,777,3000), int8 uniform [-128,127] seed 3, int32 out",
    "bf16_8192": "BF16 GEMM m=k=n=8192, N(0,1) rounded to bf16 seed 4, fp32 accumulate and out",
}
DESCRIPTIONS["i8_8192_requant_bf16"] = ("INT8 GEMM m=k=n=8192 (seed 3) requantised to bfloat16: "
                                        "D = bf16((float(C) * row_scale) * col_scale), scales seed 7")
DESCRIPTIONS["i8_8192_requant_i8"] = ("INT8 GEMM m=k=n=8192 (seed 3) requantised to int8 (ties to even, "
                                      "saturated), scales seed 7")
for _m in (1, 8, 16, 32, 64, 128):
    DESCRIPTIONS["i8_skinny_m%d" % _m] = ("INT8 skinny GEMM m=%d, k=n=8192, A U[-64,63], B round(32 N(0,1)) "
                                          "clipped, seed 2, int32 out" % _m)


def parse(argv=None):
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=list(BENCH_WORKLOADS), default=DEFAULT_WORKLOAD)
    ap.add_argument("--e2e-steps", type=int, default=10)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-per-config", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0,
                    help="target CPU time of the headline's oracle baseline sample")
    ap.add_argument("--config-cpu-seconds", type=float, default=1.5,
                    help="target CPU time of each per_config oracle baseline sample")
    ap.add_argument("--config-steps", type=int, default=200,
                    help="timed steps of each per_config entry (at least --steps)")
    return ap.parse_args(argv)


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


def config_of(key: str, world: int) -> dict:
    """The workload label both arms print (the same dict, so the two lines
    can be matched)."""
    m, k, n = BENCH_WORKLOADS[key][1]
    return {"workload": DESCRIPTIONS[key], "m": m, "k": k, "n": n,
            "parallelism": "replicas" if world > 1 else "single-gpu"}


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
    "tc": ("gemm_tc2.cu", "gemm_tc.cu", "ptx.cuh", "internal.h", "requant.cuh"),
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


# ------------------------------------------------------------ clock samples --

# clock-event reason bits of NVML's nvmlDeviceGetCurrentClocksEventReasons
_NVML_REASONS = {0x4: "sw_power_cap", 0x8: "hw_slowdown", 0x20: "sw_thermal_slowdown",
                 0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown"}


class _Nvml:
    """Read-only NVML queries through ctypes (clocks, power, clock-event
    reasons of one device); nothing is set."""

    NVML_CLOCK_SM = 1

    def __init__(self, torch_device: int):
        self.lib = ctypes.CDLL("libnvidia-ml.so.1")
        if self.lib.nvmlInit_v2() != 0:
            raise OSError("nvmlInit_v2 failed")
        self.handle = ctypes.c_void_p()
        if not self._handle_for(torch_device):
            raise OSError("no NVML handle for CUDA device %d" % torch_device)
        fn = getattr(self.lib, "nvmlDeviceGetCurrentClocksEventReasons", None)
        self._reasons_fn = fn or self.lib.nvmlDeviceGetCurrentClocksThrottleReasons

    def _handle_for(self, dev: int) -> bool:
        import torch
        props = torch.cuda.get_device_properties(dev)
        uuid = str(getattr(props, "uuid", "") or "")
        if uuid:
            tag = uuid if uuid.startswith("GPU-") else "GPU-" + uuid
            if self.lib.nvmlDeviceGetHandleByUUID(tag.encode(), ctypes.byref(self.handle)) == 0:
                return True
        bus = getattr(props, "pci_bus_id", None)
        if bus is not None:
            pci = "%08X:%02X:%02X.0" % (getattr(props, "pci_domain_id", 0), bus, getattr(props, "pci_device_id", 0))
            if self.lib.nvmlDeviceGetHandleByPciBusId_v2(pci.encode(), ctypes.byref(self.handle)) == 0:
                return True
        if not os.environ.get("CUDA_VISIBLE_DEVICES"):
            return self.lib.nvmlDeviceGetHandleByIndex_v2(ctypes.c_uint(dev), ctypes.byref(self.handle)) == 0
        return False

    def sample(self):
        sm, mx, pw = ctypes.c_uint(0), ctypes.c_uint(0), ctypes.c_uint(0)
        rs = ctypes.c_ulonglong(0)
        if (self.lib.nvmlDeviceGetClockInfo(self.handle, self.NVML_CLOCK_SM, ctypes.byref(sm)) != 0
                or self.lib.nvmlDeviceGetMaxClockInfo(self.handle, self.NVML_CLOCK_SM, ctypes.byref(mx)) != 0):
            return None
        self.lib.nvmlDeviceGetPowerUsage(self.handle, ctypes.byref(pw))
        self._reasons_fn(self.handle, ctypes.byref(rs))
        reasons = [name for bit, name in _NVML_REASONS.items() if rs.value & bit]
        return {"sm": float(sm.value), "max": float(mx.value), "power": pw.value / 1000.0, "reasons": reasons}


class ClockSampler:
    """SM clock, power and throttle-reason samples taken while a timed region
    runs: NVML every 2 ms from a thread (read-only queries), else nvidia-smi
    at its 100 ms period.  Every sample taken inside the `with` block, which
    wraps only GPU work and its synchronisation, counts as under load."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, torch_device: int, period_s: float = 0.002):
        self.dev = torch_device
        self.period = period_s
        self.rows = []
        self.source = None
        self._stop = threading.Event()
        self._thread = None
        self._proc = None
        self._nvml = None

    def __enter__(self):
        try:
            self._nvml = _Nvml(self.dev)
            self.source = "nvml"
            self._thread = threading.Thread(target=self._poll, daemon=True)
            self._thread.start()
        except (OSError, AttributeError):
            self._nvml = None
            self._start_smi()
        return self

    def _poll(self):
        while not self._stop.is_set():
            s = self._nvml.sample()
            if s is not None:
                self.rows.append(s)
            self._stop.wait(self.period)

    def _start_smi(self):
        import torch
        uuid = str(getattr(torch.cuda.get_device_properties(self.dev), "uuid", "") or "")
        target = (uuid if uuid.startswith("GPU-") else "GPU-" + uuid) if uuid else str(self.dev)
        try:
            self._proc = subprocess.Popen(
                ["nvidia-smi", "-i", target, "--query-gpu=" + self.FIELDS,
                 "--format=csv,noheader,nounits", "-lms", "100"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.source = "nvidia-smi"
            time.sleep(0.3)
        except (OSError, FileNotFoundError):
            self._proc = None

    def __exit__(self, *exc):
        if self._thread is not None:
            s = self._nvml.sample()   # one sample at the end of the region
            if s is not None:
                self.rows.append(s)
            self._stop.set()
            self._thread.join(timeout=5)
        if self._proc is not None:
            time.sleep(0.2)
            self._proc.terminate()
            try:
                out, _ = self._proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self._proc.kill()
                out, _ = self._proc.communicate()
            for line in (out or "").splitlines():
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    names = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")
                    reasons = [nm for nm, v in zip(names, parts[5:9]) if v.lower().startswith("active")]
                    self.rows.append({"sm": float(parts[1]), "max": float(parts[2]), "power": float(parts[3]),
                                      "reasons": reasons})
                except ValueError:
                    continue
        return False

    def summary(self):
        rows = self.rows
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no clock samples"], "samples": 0,
                    "samples_under_load": 0, "source": self.source}
        reasons = sorted({r for row in rows for r in row["reasons"]})
        return {"sm_mhz": statistics.median(r["sm"] for r in rows),
                "sm_max_mhz": max(r["max"] for r in rows), "reasons": reasons,
                "samples": len(rows), "samples_under_load": len(rows),
                "power_w_max": max(r["power"] for r in rows), "source": self.source}


# ------------------------------------------------------------ CPU oracle --

class OracleRunner:
    """The CPU oracle on a bounded sample of a workload: the first R rows of C
    (all n columns, full k).  Only this benchmark leg touches the oracle."""

    def __init__(self, workload: str, shape, A=None, Bt=None):
        import numpy as np

        import oracle
        from dense_int8_matrix_gb300 import workloads

        oracle.build()
        self.m, self.k, self.n = shape
        if A is None or Bt is None:
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


def cpu_baseline(workload: str, shape, seconds: float, unit: str, A=None, Bt=None) -> dict:
    runner = OracleRunner(workload, shape, A, Bt)
    rows = runner.rows_for(seconds)
    dt = runner.run(rows)
    return {"value": runner.ops(rows) / dt / 1e12, "unit": unit, "cores": runner.threads, "kind": "oracle",
            "sample": runner.sample_text(rows) + ": %.2f s" % dt}


def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return 0
    workload, shape = BENCH_WORKLOADS[args.workload]
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
    unit = "TOPS" if is_i8 else "TFLOP/s"
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": unit,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "i8->i64 exact" if is_i8 else "f64", "data": "synthetic",
        "config": config_of(args.workload, world),
        "cpu_baseline": {"value": value, "unit": unit, "cores": runner.threads, "kind": "oracle",
                         "sample": runner.sample_text(rows) + " per step (plain C triple loop, rows split "
                                                              "over POSIX threads)"},
        "e2e": {"value": value, "unit": unit, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


# ------------------------------------------------------------ GPU path ----

class Problem:
    """One workload resident on the GPU: its plan, rotated input sets (more
    bytes than 2x L2 together, so no step reads its inputs from L2) and C."""

    def __init__(self, key: str, dev: int, base=None):
        import torch

        from dense_int8_matrix_gb300 import binding as B
        from dense_int8_matrix_gb300 import workloads

        self.key = key
        if key in REQUANT_WORKLOADS:
            self.workload, self.shape, self.requant = REQUANT_WORKLOADS[key]
        else:
            (self.workload, self.shape), self.requant = BENCH_WORKLOADS[key], None
        m, k, n = self.shape
        self.is_i8 = workloads.WORKLOADS[self.workload]["dtype"] == "i8"
        self.plan = B.gemm_i8_plan(m, k, n) if self.is_i8 else B.gemm_bf16_plan(m, k, n)
        self.run = B.gemm_i8_run if self.is_i8 else B.gemm_bf16_run
        if self.requant is not None:
            rs, cs = workloads.requant_scales(m, n, k, 7)
            self.rs, self.cs = rs.cuda(), cs.cuda()
            out = B.GEMM_OUT_BF16 if self.requant == "bf16" else B.GEMM_OUT_I8
            self.run = (lambda plan, A, Bt, D, stream:
                        B.gemm_i8_run_requant(plan, A, Bt, self.rs, self.cs, D, out_type=out, stream=stream))
        self.run_host = B.gemm_i8_run_host if self.is_i8 else B.gemm_bf16_run_host
        self.out_dtype = torch.int32 if self.is_i8 else torch.float32
        self.esize = 1 if self.is_i8 else 2
        self.skinny = self.plan.path == B.GEMM_PATH_SKINNY
        self.ops = 2.0 * m * n * k
        self.unit = "TOPS" if self.is_i8 else "TFLOP/s"
        self.l2 = torch.cuda.get_device_properties(dev).L2_cache_size
        self.set_bytes = (m * k + n * k) * self.esize
        self.nsets = max(2, min(64, -(-(2 * self.l2) // self.set_bytes)))
        self.base_A, self.base_B = base if base is not None else workloads.make_inputs(self.workload, self.shape)
        self.sets = []
        for s in range(self.nsets):
            if s == 0:
                A, Bt = self.base_A, self.base_B
            else:
                # cheap distinct copies: a per-set rotation of the rows
                A = torch.roll(self.base_A, shifts=s, dims=0)
                Bt = torch.roll(self.base_B, shifts=3 * s, dims=0)
            self.sets.append((A.cuda(), Bt.cuda()))
        if self.requant is not None:
            self.out_dtype = torch.bfloat16 if self.requant == "bf16" else torch.int8
        self.C = torch.empty((m, n), dtype=self.out_dtype, device="cuda")

    def step(self, i: int, stream):
        A, Bt = self.sets[i % self.nsets]
        self.run(self.plan, A, Bt, self.C, stream)

    def alg_bytes(self) -> int:
        m, k, n = self.shape
        return (m * k + n * k) * self.esize + self.C.element_size() * m * n

    def plan_dict(self) -> dict:
        p = self.plan
        return {"path": "tensor" if p.path == 0 else "skinny", "bm": p.bm, "bn": p.bn, "grid": p.grid,
                "tiles": p.tiles, "waves": p.waves, "split_k": p.split_k, "num_sms": p.num_sms}

    def inputs_text(self) -> str:
        return "inputs rotated over %d distinct sets (%d MiB) > 2x L2 (%d MiB)" % (
            self.nsets, self.nsets * self.set_bytes >> 20, self.l2 >> 20)


def timed_region(prob: Problem, steps: int, start: int, stream):
    """Device time in ms of `steps` consecutive steps, CUDA events on the
    launching stream around the whole region."""
    import torch
    ev0 = torch.cuda.Event(enable_timing=True)
    ev1 = torch.cuda.Event(enable_timing=True)
    ev0.record(stream)
    for i in range(steps):
        prob.step(start + i, stream)
    ev1.record(stream)
    torch.cuda.synchronize()
    return ev0.elapsed_time(ev1)


def kernel_pass(prob: Problem, launches: int, stream) -> dict:
    """Average launch duration of the dominant kernel over `launches` calls
    after the timed region.  Tensor path: every call records CUDA events on
    its stream around its staging launch and its GEMM launch (the library's
    trace with every = 1).  Skinny path: consecutive calls overlap (each
    call's kernels start before the previous call's end), so the launch unit
    (prologue + skinny kernel) is timed as the region over the calls."""
    from dense_int8_matrix_gb300 import binding as B
    if prob.skinny:
        B.gemm_trace_begin(0, 1)   # launches counted, no events recorded
        ms = timed_region(prob, launches, 0, stream)
        _, _, counted = B.gemm_trace_collect()
        return {"unit_ms": ms / launches, "launches": launches, "counted": counted}
    B.gemm_trace_begin(2 * launches + 8, 1)
    timed_region(prob, launches, 0, stream)
    ms, timed, counted = B.gemm_trace_collect()
    tc = ms[B.GEMM_KERNEL_TC] / max(1, timed[B.GEMM_KERNEL_TC])
    st = ms[B.GEMM_KERNEL_STAGE] / timed[B.GEMM_KERNEL_STAGE] if timed[B.GEMM_KERNEL_STAGE] else None
    return {"unit_ms": tc, "stage_ms": st, "launches": timed[B.GEMM_KERNEL_TC], "counted": counted}


def roofline_of(prob: Problem, kp: dict, peaks: dict, peak_src: str) -> dict:
    """Roofline of the dominant kernel: tensor-bound GEMM kernels against the
    measured burst bf16 tensor peak (f16 and bf16 MMAs share the dense rate;
    int8 runs on f16 MMAs; the kernel pass times each launch alone, so the
    burst figure applies), the skinny unit against the measured copy
    bandwidth."""
    ms = kp["unit_ms"]
    if prob.skinny:
        alg = prob.alg_bytes()
        achieved = alg / (ms / 1000.0) / 1e9
        return {"kernel": "skinny_prologue + skinny_tc, one unit per call (CUDA events around %d consecutive "
                          "calls: units overlap through programmatic dependent launch)" % kp["launches"],
                "bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": achieved / peaks["hbm_gbs"],
                "peak_source": "%s hbm_gbs (STREAM-style copy)" % peak_src,
                "algorithmic_bytes_per_launch": alg, "kernel_ms_per_launch": ms, "launches_timed": kp["launches"]}
    peak = peaks["bf16_tflops"]
    achieved = prob.ops / (ms / 1000.0) / 1e12
    name = "gemm_tc2 (two-SM 256x256 tile)" if prob.plan.bm == 256 else "gemm_tc (%dx%d tile)" % (
        prob.plan.bm, prob.plan.bn)
    out = {"kernel": name + ", tcgen05 kind::f16; mean of %d launches, CUDA events around each launch"
           % kp["launches"],
           "bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s", "frac": achieved / peak,
           "peak_source": ("%s bf16_tflops (burst cuBLAS bf16 GEMM); the int8 path runs on f16 tensor-core MMAs, "
                           "whose nominal dense rate equals bf16's" % peak_src),
           "algorithmic_flops_per_launch": prob.ops, "kernel_ms_per_launch": ms,
           "staging_ms_per_launch": kp.get("stage_ms"), "launches_timed": kp["launches"]}
    if "bf16_tflops_sustained" in peaks:
        out["frac_of_sustained"] = achieved / peaks["bf16_tflops_sustained"]
    return out


def graph_throughput(prob: Problem, steps, world):
    """Steps captured once into a CUDA graph (every input set a few times)
    and the graph replayed until about `steps` steps have run; the device time
    per step over the replays, max over ranks."""
    import torch
    try:
        nsets = prob.nsets
        per_graph = nsets * max(1, 32 // nsets)
        replays = max(3, steps // per_graph)
        gs = torch.cuda.Stream()
        gs.wait_stream(torch.cuda.current_stream())
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g, stream=gs):
            cur = torch.cuda.current_stream()
            for i in range(per_graph):
                prob.step(i, cur)
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
        return {"value": whole_job_value(world, prob.ops, ms), "ms_per_step": ms, "steps_per_replay": per_graph,
                "replays": replays}
    except Exception as exc:   # noqa: BLE001 - reported, not fatal
        return {"unavailable": "%s: %s" % (type(exc).__name__, str(exc)[:200])}


def per_config_entry(key: str, dev: int, args, peaks, peak_src, base=None) -> dict:
    """One configuration of the benchmark list at N = 1: throughput over
    max(--steps, --config-steps) steps, the dominant kernel's roofline from a
    separate pass of KERNEL_PASS_LAUNCHES launches, the oracle's throughput
    on a bounded sample."""
    import torch

    from dense_int8_matrix_gb300 import binding as B
    prob = Problem(key, dev, base)
    stream = torch.cuda.current_stream()
    for i in range(args.warmup):
        prob.step(i, stream)
    torch.cuda.synchronize()
    steps = max(args.steps, args.config_steps)
    ms = timed_region(prob, steps, 0, stream) / steps
    kp = kernel_pass(prob, KERNEL_PASS_LAUNCHES, stream)
    st, code = B.gemm_device_error()
    if st != B.GEMM_OK:
        raise RuntimeError("device error in %s: code %d" % (key, code))
    roof = roofline_of(prob, kp, peaks, peak_src)
    value = prob.ops / (ms / 1000.0) / 1e12
    entry = {"workload": DESCRIPTIONS[key], "m": prob.shape[0], "k": prob.shape[1], "n": prob.shape[2],
             "in_configuration_list": key in BENCH_WORKLOADS,
             "value": value, "unit": prob.unit, "ms_per_step": ms, "steps": steps,
             "plan": prob.plan_dict(), "inputs": prob.inputs_text(),
             "roofline": {"bound": roof["bound"], "achieved": roof["achieved"], "peak": roof["peak"],
                          "unit": roof["unit"], "frac": roof["frac"],
                          "kernel_ms_per_launch": roof["kernel_ms_per_launch"],
                          "launches_timed": roof["launches_timed"]}}
    if roof["bound"] == "tensor":
        entry["roofline"]["step_frac"] = value / roof["peak"]
        if roof.get("staging_ms_per_launch") is not None:
            entry["roofline"]["staging_ms_per_launch"] = roof["staging_ms_per_launch"]
    if not args.no_cpu_baseline and prob.requant is None:
        entry["cpu_baseline"] = cpu_baseline(prob.workload, prob.shape, args.config_cpu_seconds, prob.unit,
                                             prob.base_A, prob.base_B)
    del prob
    torch.cuda.empty_cache()
    return entry


def run_ours(args):
    import torch

    from dense_int8_matrix_gb300 import binding as B
    from dense_int8_matrix_gb300 import build as lib_build

    world, rank, local = dist_env()
    if world > 1:
        torch.cuda.set_device(local)
        import torch.distributed as dist
        dist.init_process_group("nccl")
    dev = torch.cuda.current_device()
    lib_build.build()
    B.load()

    prob = Problem(args.workload, dev)
    m, k, n = prob.shape
    stream = torch.cuda.current_stream()
    for i in range(args.warmup):
        prob.step(i, stream)
    torch.cuda.synchronize()

    if world > 1:
        import torch.distributed as dist
        dist.barrier()
    torch.cuda.synchronize()
    # sampled trace: every TRACE_EVERY-th step times its launches with events,
    # the other steps run undisturbed.  On the skinny path consecutive calls
    # overlap and an event between two calls would serialise them, so there
    # the launches are only counted.
    B.gemm_trace_begin(0 if prob.skinny else 2 * (args.steps // TRACE_EVERY) + 8, TRACE_EVERY)
    with ClockSampler(dev) as clk:
        elapsed_ms = timed_region(prob, args.steps, 0, stream)
        sampled_ms, sampled_timed, launches = B.gemm_trace_collect()
        # the dominant kernel, alone, over a separate pass of launches
        kp = kernel_pass(prob, KERNEL_PASS_LAUNCHES, stream)
    clk_summary = clk.summary()
    st, code = B.gemm_device_error()
    if st != B.GEMM_OK:
        raise RuntimeError("device error during bench: code %d" % code)
    max_ms = max_over_ranks(elapsed_ms, world, "cuda")
    ms_per_step = max_ms / args.steps
    value = whole_job_value(world, prob.ops, ms_per_step)

    # the same steps captured into a CUDA graph and replayed: the loop a
    # serving process would replay (a user may capture gemm_*_run calls);
    # reported beside the stream-launched value, which stays the headline
    graph_line = graph_throughput(prob, args.steps, world)

    # end to end through the host-buffer entry point: H2D of A and Bt,
    # the GEMM, D2H of C, inside the timed region
    hA = prob.base_A.pin_memory()
    hB = prob.base_B.pin_memory()
    hC = torch.empty((m, n), dtype=prob.out_dtype).pin_memory()
    prob.run_host(prob.plan, hA, hB, hC, stream)
    e2e_times = []
    for _ in range(args.e2e_steps):
        torch.cuda.synchronize()
        t0 = time.perf_counter()
        prob.run_host(prob.plan, hA, hB, hC, stream)
        e2e_times.append(time.perf_counter() - t0)
    e2e_s = statistics.median(e2e_times)
    e2e_value = prob.ops / e2e_s / 1e12
    del hA, hB, hC

    peaks, peak_src = load_peaks()
    roof = roofline_of(prob, kp, peaks, peak_src)
    traffic = load_traffic().get(args.workload)
    digest = kernel_source_digest("skinny" if prob.skinny else "tc")
    roof["traffic"] = traffic[0] if traffic and traffic[1] == digest else None
    if not prob.skinny:
        # the sampled launches inside the timed region, as a cross-check
        kind = B.GEMM_KERNEL_TC
        roof["kernel_ms_sampled_in_timed_region"] = (sampled_ms[kind] / sampled_timed[kind]
                                                     if sampled_timed[kind] else None)

    line = {
        "metric": METRIC, "value": value, "unit": prob.unit, "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None,
        "dtype": "i8->i32 exact (f16 tensor-core MMA, fp32 chunks <= 2^24, int32 sum)" if prob.is_i8
        else "bf16->f32 (fp32 accumulate)",
        "data": "synthetic",
        "config": config_of(args.workload, world),
        "inputs": prob.inputs_text(),
        "plan": prob.plan_dict(),
        "gpu_launches": int(sum(launches)),
        "gpu_launches_by_kind": {"stage": launches[0], "tc": launches[1], "skinny": launches[2],
                                 "requant": launches[3]},
        "roofline": roof,
        "graph": graph_line,
        "clocks": clk_summary,
        "e2e": {"value": e2e_value, "unit": prob.unit,
                "h2d_bytes_per_step": (m * k + n * k) * prob.esize, "d2h_bytes_per_step": m * n * 4,
                "ms_per_step": e2e_s * 1000.0},
    }
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        line["cpu_baseline"] = cpu_baseline(prob.workload, prob.shape, args.cpu_seconds, prob.unit,
                                            prob.base_A, prob.base_B)
    base = (prob.base_A, prob.base_B)
    del prob
    torch.cuda.empty_cache()
    if world == 1 and not args.no_per_config:
        entries = {}
        for key in list(BENCH_WORKLOADS) + list(REQUANT_WORKLOADS):
            same_inputs = BENCH_WORKLOADS.get(key) == BENCH_WORKLOADS[args.workload] or (
                key in REQUANT_WORKLOADS and REQUANT_WORKLOADS[key][:2] == BENCH_WORKLOADS[args.workload])
            entries[key] = per_config_entry(key, dev, args, peaks, peak_src, base if same_inputs else None)
        line["per_config"] = entries
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
