"""Benchmark of the fused cascaded GEMM on GB300.

One JSON line on stdout (rank 0).  The headline workload is the batched fp16
chain (batch 64, A 4096x128, B and C 128x128 per batch, fp16 out); a step is
one fused call over the whole batch with inputs already resident in HBM.
``per_config`` adds every workload (fp16 tiny, fp16 batched, tf32, fp64,
three-stage bf16) with its roofline fraction and the two unfused baselines
(torch/cuBLAS per GEMM, and this library's own single-GEMM kernel per
stage, the intermediate going through HBM).

``--impl reference`` times the CPU oracle instead (the only reference this
method has), on a bounded sample of the same workload.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads as wl  # noqa: E402

L2_BYTES = 129 * 1024 * 1024
ROTATE_TARGET = 3 * L2_BYTES     # rotate input copies until the set is > 3x L2


# ----------------------------------------------------------------- helpers --

def dist_env():
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return rank, world, local


def max_over_ranks(value: float, device=None) -> float:
    """Largest value over all ranks (the job is as slow as its slowest rank)."""
    import torch
    import torch.distributed as dist
    if not dist.is_available() or not dist.is_initialized() or dist.get_world_size() == 1:
        return value
    t = torch.tensor([float(value)], dtype=torch.float64, device=device if device is not None else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_tflops(world: int, flops_per_rank: int, ms_per_step: float) -> float:
    """Throughput of the whole job: every rank runs its own replica of the workload."""
    return world * flops_per_rank / (ms_per_step * 1e-3) / 1e12


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return {"hbm_gbs": d.get("hbm_gbs", 6800.0), "bf16_tflops": d.get("bf16_tflops", 1900.0),
                "bf16_tflops_sustained": d.get("bf16_tflops_sustained", 1700.0), "source": "measured"}
    return {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}


class ClockSampler:
    """nvidia-smi clocks and throttle reasons, sampled while the GPU works."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index: int, period_ms: int = 50):
        self.gpu, self.period = gpu_index, period_ms
        self.proc = None
        self.lines = []
        self.t = None

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", str(self.period)], stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except OSError:
            self.proc = None
            return
        self.t = threading.Thread(target=self._read, daemon=True)
        self.t.start()

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.t:
            self.t.join(timeout=2)
        sm, smax, power, reasons = [], [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for ln in self.lines:
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                power.append(float(parts[3]))
            except ValueError:
                continue
            for name, val in zip(names, parts[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(smax), "reasons": sorted(reasons),
                "samples": len(sm), "power_w_max": max(power)}


def event_time_ms(fn, steps, stream):
    """Time `steps` calls of fn() on `stream`; per-call and total event times."""
    import torch
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    torch.cuda.synchronize()
    with torch.cuda.stream(stream):
        for i in range(steps):
            starts[i].record(stream)
            fn(i)
            ends[i].record(stream)
    torch.cuda.synchronize()
    per = [s.elapsed_time(e) for s, e in zip(starts, ends)]
    total = starts[0].elapsed_time(ends[-1])
    return per, total


def graph_of(fn, steps, stream):
    """Capture `steps` calls of fn(i) into one CUDA graph (launch overhead off the timed path)."""
    import torch
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(steps):
            fn(i)
    torch.cuda.synchronize()
    return g


def graph_time_ms(g, stream, reps=1):
    """Device time of `reps` replays of graph g, events on the replay stream."""
    import torch
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    s.record(stream)
    for _ in range(reps):
        g.replay()
    e.record(stream)
    torch.cuda.synchronize()
    return s.elapsed_time(e)


def oracle_kinds(dtype):
    import oracle
    return {"f16_f32out": (oracle.F32, oracle.F16, oracle.F32), "f16": (oracle.F32, oracle.F16, oracle.F16),
            "bf16": (oracle.F32, oracle.BF16, oracle.BF16), "bf16_f32out": (oracle.F32, oracle.BF16, oracle.F32),
            "tf32": (oracle.F32, oracle.TF32, oracle.F32), "f64": (oracle.NONE, oracle.NONE, oracle.NONE),
            "tf32_f16": (oracle.F32, oracle.F16, oracle.F32), "tf32_bf16": (oracle.F32, oracle.BF16, oracle.F32)}[dtype]


def oracle_sample(w: wl.Workload, rows: int, batches: int = 1, threads: int = 0):
    """Run the oracle on a sample (first `batches` batches, first `rows` rows)."""
    import oracle
    sw = w.with_(batch=min(batches, w.batch), M=min(rows, w.M))
    host = wl.make_inputs(sw)
    acc, mid, fin = oracle_kinds(w.dtype)
    A = oracle.widen(host[0])
    Ws = [oracle.widen(t) for t in host[1:]]
    t0 = time.perf_counter()
    oracle.chain(A, Ws, acc, mid, fin, n_threads=threads)
    dt = time.perf_counter() - t0
    return sw, dt


_ALL_CORES = []


def all_cores() -> int:
    """The oracle's thread count before any run has set one (a run with an
    explicit count leaves it set for the process)."""
    import oracle
    if not _ALL_CORES:
        _ALL_CORES.append(oracle.max_threads())
    return _ALL_CORES[0]


def cpu_baseline(w: wl.Workload, target_s: float = 10.0, threads: int = 0):
    """Oracle throughput on a bounded sample sized for about `target_s` of CPU
    work, on all host cores (threads = 0) or on `threads` of them."""
    import oracle
    cores = all_cores()  # (taken before this call may set a count)
    threads = threads if threads > 0 else cores
    rows = 256
    sw, dt = oracle_sample(w, rows, threads=threads)
    per_row = dt / (sw.batch * sw.M)
    want_rows = int(max(256, min(w.batch * w.M, target_s / max(per_row, 1e-9))))
    batches = max(1, min(w.batch, want_rows // w.M))
    rows = want_rows if batches == 1 else w.M
    sw, dt = oracle_sample(w, rows, batches, threads=threads)
    return {"value": sw.flops() / dt / 1e12, "unit": "TFLOP/s", "cores": threads, "kind": "oracle",
            "sample": f"{sw.batch} batch x {sw.M} rows of {w.name} ({sw.flops() / 1e9:.2f} GFLOP, {dt:.2f} s)"}


# ------------------------------------------------------------ GPU workloads --

def rotated_copies(w: wl.Workload) -> int:
    """Input/output copies rotated between timed calls so that their set exceeds L2."""
    return max(1, min(8, -(-ROTATE_TARGET // w.unique_bytes())))


def workload_config(w: wl.Workload, world: int) -> dict:
    """The `config` object of the JSON line (the same for both arms)."""
    copies = rotated_copies(w)
    return {"workload": w.name, "batch": w.batch, "M": w.M, "K": w.K, "N": list(w.N), "io": w.dtype,
            "l2": f"rotating {copies} input/output copies ({copies * w.unique_bytes() / 2**20:.0f} MiB > L2)",
            "parallelism": f"replica x{world}" if world > 1 else "single GPU"}


class Case:
    """Device buffers (rotated copies), the fused plan and the unfused paths of one workload."""

    def __init__(self, w: wl.Workload, device):
        import torch
        import fusion_b2b_gemm_gb300 as b2b
        self.w = w
        self.plan = b2b.ChainPlan(w.dtype, w.batch, w.M, w.K, w.N)
        host = wl.make_inputs(w)
        self.host = host
        self.copies = rotated_copies(w)
        self.inputs = [[t.to(device) for t in host] for _ in range(self.copies)]
        _, out_dt = wl.io_dtypes(w.dtype)
        self.outs = [torch.empty(w.out_shape(), dtype=out_dt, device=device) for _ in range(self.copies)]
        self.info = self.plan.info()

    def fused(self, i):
        k = i % self.copies
        self.plan.run(self.inputs[k][0], self.inputs[k][1:], D=self.outs[k])

    # -- unfused: torch / cuBLAS per GEMM, intermediate in HBM in the operand type
    def make_unfused_torch(self):
        import torch
        w = self.w
        in_dt, out_dt = wl.io_dtypes(w.dtype)

        def run(i):
            k = i % self.copies
            x = self.inputs[k][0]
            for s, W in enumerate(self.inputs[k][1:]):
                if x.dtype != W.dtype:  # mixed types: the intermediate takes the next weight's type
                    x = x.to(W.dtype)
                x = torch.bmm(x, W)
                if s == w.stages - 1 and x.dtype != out_dt:
                    x = x.to(out_dt)
            return x
        return run

    # -- unfused: this library's single-GEMM kernel per stage
    def make_unfused_own(self):
        import torch
        import fusion_b2b_gemm_gb300 as b2b
        w = self.w
        in_dt, out_dt = wl.io_dtypes(w.dtype)
        single_dt = {"f16_f32out": "f16", "f16": "f16", "bf16": "bf16", "bf16_f32out": "bf16",
                     "tf32": "tf32", "f64": "f64", "tf32_f16": "f16", "tf32_bf16": "bf16"}[w.dtype]
        last_dt = {"tf32_f16": "f16_f32out", "tf32_bf16": "bf16_f32out"}.get(w.dtype, w.dtype)
        mixed = w.dtype in ("tf32_f16", "tf32_bf16")
        mid_dt = wl.input_dtypes(w.dtype, w.stages)[-1]
        plans, mids = [], []
        kin = w.K
        for s, n in enumerate(w.N):
            dt = "tf32" if (mixed and s == 0) else (last_dt if s == w.stages - 1 else single_dt)
            plans.append(b2b.GemmPlan(dt, w.batch, w.M, kin, n))
            if s < w.stages - 1:
                # (mixed: the tf32 GEMM writes fp32, cast to the 16-bit type below)
                mids.append(torch.empty((w.batch, w.M, n), dtype=torch.float32 if (mixed and s == 0) else mid_dt,
                                        device=self.outs[0].device))
            kin = n
        self._own = (plans, mids)

        def run(i):
            k = i % self.copies
            x = self.inputs[k][0]
            for s, W in enumerate(self.inputs[k][1:]):
                if x.dtype != W.dtype:
                    x = x.to(W.dtype)
                dst = mids[s] if s < w.stages - 1 else self.outs[k]
                plans[s].run(x, W, D=dst)
                x = dst
        launches = sum(p.info()["launches_per_run"] for p in plans) + (1 if mixed else 0)
        return run, launches


def measure_peak_matmul(dtype_name: str, n: int, reps: int = 5):
    """torch.matmul n^3 throughput (best of reps) in TFLOP/s, as the driver measures bf16."""
    import torch
    dt = getattr(torch, dtype_name)
    old = torch.backends.cuda.matmul.allow_tf32
    torch.backends.cuda.matmul.allow_tf32 = dtype_name == "float32"
    a = torch.randn(n, n, device="cuda").to(dt)
    b = torch.randn(n, n, device="cuda").to(dt)
    for _ in range(2):
        torch.matmul(a, b)
    best = 1e30
    for _ in range(reps):
        s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        s.record()
        torch.matmul(a, b)
        e.record()
        torch.cuda.synchronize()
        best = min(best, s.elapsed_time(e))
    torch.backends.cuda.matmul.allow_tf32 = old
    return 2.0 * n ** 3 / (best * 1e-3) / 1e12


def roofline_for(w: wl.Workload, kernel_ms: float, peaks: dict, traffic=None):
    """Bound, achieved and peak for the fused kernel of workload w."""
    flops = w.flops()
    byts = w.unique_bytes()
    if w.dtype in ("tf32_f16", "tf32_bf16"):
        # mixed types: the first GEMM at the tf32 rate, the rest at the 16-bit
        # rate; the peak is the blend for this workload's split of the work
        f0 = 2 * w.batch * w.M * w.K * w.N[0]
        tflops_peak = flops / (f0 / peaks["tensor"]["tf32"] + (flops - f0) / peaks["tensor"]["bf16"])
    else:
        tflops_peak = peaks["tensor"][w.dtype]
    t_compute = flops / (tflops_peak * 1e12)
    t_mem = byts / (peaks["hbm_gbs"] * 1e9)
    if t_mem >= t_compute:
        achieved = byts / (kernel_ms * 1e-3) / 1e9
        r = {"bound": "hbm", "achieved": achieved, "peak": peaks["hbm_gbs"], "unit": "GB/s"}
    else:
        achieved = flops / (kernel_ms * 1e-3) / 1e12
        r = {"bound": "tensor", "achieved": achieved, "peak": tflops_peak, "unit": "TFLOP/s"}
    r["frac"] = r["achieved"] / r["peak"]
    r["traffic"] = traffic
    r["algorithmic_bytes"] = byts
    r["algorithmic_flops"] = flops
    r["roofline_ms"] = max(t_mem, t_compute) * 1e3
    return r


PROFILE_TRAFFIC = os.path.join(ROOT, "profiles", "traffic.json")

# the arithmetic type of a workload's GEMMs (operands; accumulation is fp32,
# fp64 for f64)
COMPUTE_DTYPE = {"f16_f32out": "f16", "f16": "f16", "bf16": "bf16", "bf16_f32out": "bf16", "tf32": "tf32",
                 "f64": "f64", "tf32_f16": "tf32+f16", "tf32_bf16": "tf32+bf16"}


def kernel_source_digest() -> str:
    import hashlib
    root = os.path.join(ROOT, "fusion_b2b_gemm_gb300", "csrc")
    h = hashlib.sha256()
    for f in sorted(os.listdir(root)):
        if f.endswith((".cu", ".cuh", ".h", ".cpp")):
            h.update(f.encode())
            with open(os.path.join(root, f), "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_traffic(name: str):
    """DRAM bytes per launch from the committed ncu summary, or None when the
    kernel sources changed since those counters were taken."""
    try:
        with open(PROFILE_TRAFFIC) as f:
            d = json.load(f)
    except (OSError, ValueError):
        return None
    if d.get("source_digest") != kernel_source_digest():
        return None
    return d.get(name)


# --------------------------------------------------------------------- arms --

def run_reference(args):
    """The CPU oracle, timed on this host's cores, on bounded samples."""
    rank, world, _ = dist_env()
    if rank != 0:
        return 0
    import oracle
    w = wl.ALL_WORKLOADS[args.workload]
    rows = args.ref_rows
    sw = w.with_(batch=1, M=min(rows, w.M))
    host = wl.make_inputs(sw)
    acc, mid, fin = oracle_kinds(w.dtype)
    A = oracle.widen(host[0])
    Ws = [oracle.widen(t) for t in host[1:]]
    for _ in range(args.warmup):
        oracle.chain(A, Ws, acc, mid, fin)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        oracle.chain(A, Ws, acc, mid, fin)
    dt = (time.perf_counter() - t0) / args.steps
    value = sw.flops() / dt / 1e12
    line = {
        "impl": "reference", "metric": "fused B2B GEMM TFLOPS", "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": dt * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64",
        "data": "synthetic", "config": workload_config(w, world),
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.max_threads(), "kind": "oracle",
                         "sample": f"1 batch x {sw.M} rows of {w.name} per step ({sw.flops() / 1e9:.3f} GFLOP)"},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)
    return 0


def run_ours(args):
    import torch
    rank, world, local = dist_env()
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl" if torch.cuda.is_available() else "gloo")
    torch.cuda.set_device(local)
    device = torch.device("cuda", local)
    import fusion_b2b_gemm_gb300  # noqa: F401  (fails loudly if the library is missing)

    peaks = load_peaks()
    w = wl.ALL_WORKLOADS[args.workload]
    case = Case(w, device)
    stream = torch.cuda.current_stream()

    # warm-up (eager calls), then the K timed steps captured as one CUDA graph
    for i in range(args.warmup):
        case.fused(i)
    torch.cuda.synchronize()
    graph = graph_of(case.fused, args.steps, stream)
    graph.replay()
    torch.cuda.synchronize()

    # soak so that the clock samples see the GPU under load, then the timed region
    sampler = ClockSampler(local)
    sampler.start()
    t_end = time.perf_counter() + args.soak_s
    while time.perf_counter() < t_end:
        graph.replay()
        torch.cuda.synchronize()

    def barrier():
        if world > 1:
            torch.distributed.barrier()
        torch.cuda.synchronize()

    barrier()
    total_ms = graph_time_ms(graph, torch.cuda.current_stream())
    barrier()
    clocks = sampler.stop()
    total_ms = max_over_ranks(total_ms, device)
    if case.plan.status() != 0:
        raise RuntimeError("a bounded wait of the fused kernel gave up during the timed region")

    ms_per_step = total_ms / args.steps
    kernel_ms = ms_per_step      # one kernel launch per step, back to back in the graph
    value = whole_job_tflops(world, w.flops(), ms_per_step)
    # eager calls (host launch path included), for reference
    per_eager, _ = event_time_ms(case.fused, min(args.steps, 50), stream)

    # end to end: pinned host buffers in, host result out, through the public API
    h_in = [t.pin_memory() for t in case.host]
    _, out_dt = wl.io_dtypes(w.dtype)
    h_out = torch.empty(w.out_shape(), dtype=out_dt).pin_memory()
    h2d = d2h = 0

    def e2e_step(i):
        nonlocal h2d, d2h
        h2d, d2h = case.plan.run_from_host(h_in, h_out, case.inputs[0], case.outs[0], stream=stream)

    for i in range(2):
        e2e_step(i)
    barrier()
    e_steps = max(3, min(args.steps, 20))
    _, e_total = event_time_ms(e2e_step, e_steps, stream)
    e_total = max_over_ranks(e_total, device)
    e2e_value = whole_job_tflops(world, w.flops(), e_total / e_steps)

    tensor_peaks = {"f16": peaks["bf16_tflops"], "f16_f32out": peaks["bf16_tflops"], "bf16": peaks["bf16_tflops"],
                    "bf16_f32out": peaks["bf16_tflops"]}
    extra_peaks = {}
    if not args.quick:
        extra_peaks["tf32_tflops"] = measure_peak_matmul("float32", 8192)
        extra_peaks["f64_tflops"] = measure_peak_matmul("float64", 4096, reps=3)
    tensor_peaks["tf32"] = extra_peaks.get("tf32_tflops", peaks["bf16_tflops"] / 2)
    tensor_peaks["f64"] = extra_peaks.get("f64_tflops", 1.25)
    peaks_all = dict(peaks, tensor=tensor_peaks)

    line = {
        "metric": "fused B2B GEMM TFLOPS", "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": ms_per_step, "higher_is_better": True,
        "scaling": "weak", "vs_baseline": None, "dtype": COMPUTE_DTYPE[w.dtype], "data": "synthetic",
        "config": workload_config(w, world),
        "kernel_ms": kernel_ms,
        "eager_ms_per_call": float(np.median(per_eager)),
        "eager_ms_p10_p90": [float(np.percentile(per_eager, 10)), float(np.percentile(per_eager, 90))],
        "timing": "K steps captured in one CUDA graph, CUDA events around one replay",
        "roofline": roofline_for(w, kernel_ms, peaks_all, recorded_traffic(w.name)),
        "clocks": clocks,
        "gpu_launches": args.steps * case.info["launches_per_run"],
        "e2e": {"value": e2e_value, "unit": "TFLOP/s", "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h},
        "peaks": {"hbm_gbs": peaks["hbm_gbs"], "bf16_tflops": peaks["bf16_tflops"], "source": peaks["source"],
                  **{k: round(v, 2) for k, v in extra_peaks.items()}},
    }
    if rank == 0 and not args.quick:
        line["cpu_baseline"] = cpu_baseline(w, target_s=args.cpu_s)
        detail = per_config(args, peaks_all, device, stream)
        # the full record of every workload first, one line each; the
        # headline line ends with the short form of each, so that a reader
        # who keeps only the end of the output still sees every workload
        for entry in detail:
            print(json.dumps({"per_config_detail": entry}), flush=True)
        line["per_config"] = [compact_config(e) for e in detail]
    if rank == 0:
        print(json.dumps(line), flush=True)
    if world > 1:
        torch.distributed.destroy_process_group()
    return 0


def _sig(x, digits=3):
    """x rounded to `digits` significant digits (None stays None)."""
    if x is None:
        return None
    return float(f"{x:.{digits}g}")


def compact_config(e: dict) -> dict:
    """The short record of one workload for the headline line: device times
    per call in microseconds, the speed-up over the faster unfused path, the
    roofline side and fraction, and the CPU oracle's rate."""
    r = e["roofline"]
    out = {"w": e["workload"], "fused_us": _sig(e["fused_ms"] * 1e3), "torch_us": _sig(e["unfused_torch_ms"] * 1e3),
           "own_us": _sig(e["unfused_own_ms"] * 1e3) if e["unfused_own_ms"] is not None else None,
           "speedup": _sig(e["speedup_vs_best_unfused"]),
           "bound": r["bound"], "frac": _sig(r["frac"])}
    if "cpu_oracle" in e:
        out["cpu_tflops"] = _sig(e["cpu_oracle"]["value"])
    return out


def per_config(args, peaks_all, device, stream):
    import torch
    out = []
    steps = args.cfg_steps
    for name, w in wl.ALL_WORKLOADS.items():
        case = Case(w, device)
        for i in range(3):
            case.fused(i)
        g = graph_of(case.fused, steps, stream)
        g.replay()
        fused_ms = graph_time_ms(g, torch.cuda.current_stream(), reps=3) / (3 * steps)
        if case.plan.status() != 0:
            raise RuntimeError(f"{name}: a bounded wait of the fused kernel gave up")
        per, _ = event_time_ms(case.fused, steps, stream)
        torch_fn = case.make_unfused_torch()
        old = torch.backends.cuda.matmul.allow_tf32
        torch.backends.cuda.matmul.allow_tf32 = True
        for i in range(3):
            torch_fn(i)
        gt = graph_of(torch_fn, steps, stream)
        gt.replay()
        t_ms = graph_time_ms(gt, torch.cuda.current_stream(), reps=3) / (3 * steps)
        torch.backends.cuda.matmul.allow_tf32 = old
        own_fn, own_launches = case.make_unfused_own()
        for i in range(3):
            own_fn(i)
        go = graph_of(own_fn, steps, stream)
        go.replay()
        o_ms = graph_time_ms(go, torch.cuda.current_stream(), reps=3) / (3 * steps)
        if any(p.status() != 0 for p in case._own[0]):
            o_ms = None  # a single-GEMM kernel gave up a wait: no valid time
        entry = {
            "workload": name, "extra": name in wl.EXTRA_WORKLOADS, "dtype": w.dtype, "gflop": w.flops() / 1e9, "unique_mb": w.unique_bytes() / 2**20,
            "fused_ms": fused_ms, "fused_tflops": w.flops() / (fused_ms * 1e-3) / 1e12,
            "fused_eager_median_ms": float(np.median(per)),
            "fused_eager_p10_p90_ms": [float(np.percentile(per, 10)), float(np.percentile(per, 90))],
            "roofline": roofline_for(w, fused_ms, peaks_all, recorded_traffic(name)),
            "unfused_torch_ms": t_ms, "unfused_own_ms": o_ms, "unfused_own_launches": own_launches,
            "speedup_vs_best_unfused": min(t_ms, o_ms if o_ms is not None else t_ms) / fused_ms,
            "launches_per_run": case.info["launches_per_run"], "plan": case.info,
            "timing": f"{steps} calls per CUDA graph, 3 replays",
        }
        if not args.no_cpu_configs:
            entry["cpu_oracle"] = cpu_baseline(w, target_s=args.cpu_cfg_s)
            if name in ("tiny_f16", "tf32"):
                entry["cpu_oracle_1_thread"] = cpu_baseline(w, target_s=args.cpu_cfg_s, threads=1)
        out.append(entry)
        del case, g, gt, go
        torch.cuda.empty_cache()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=wl.BENCH_WORKLOAD, choices=list(wl.ALL_WORKLOADS))
    ap.add_argument("--soak-s", type=float, default=1.5, dest="soak_s")
    ap.add_argument("--cfg-steps", type=int, default=50, dest="cfg_steps")
    ap.add_argument("--cpu-s", type=float, default=10.0, dest="cpu_s")
    ap.add_argument("--cpu-cfg-s", type=float, default=3.0, dest="cpu_cfg_s")
    ap.add_argument("--ref-rows", type=int, default=2048, dest="ref_rows")
    ap.add_argument("--no-cpu-configs", action="store_true", dest="no_cpu_configs")
    ap.add_argument("--quick", action="store_true", help="headline line only")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)   # at least three untimed warm-up steps
    if args.impl == "reference":
        return run_reference(args)
    return run_ours(args)


if __name__ == "__main__":
    sys.exit(main())
