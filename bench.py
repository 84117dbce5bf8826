#!/usr/bin/env python
"""Benchmark of the fused GEMM + bias/activation epilogue on GB300.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

One step is one fused call D = RELU(A.B + bias) on the largest RELU_BIAS workload
(A[65536,8192] . B[8192,16384], bf16 in and out, fp32 accumulate), inputs resident in
device memory.  Every input is larger than L2, so no flush is needed between steps.
Rank 0 prints one JSON line: whole-job TFLOP/s, the roofline of the fused kernel, the
end-to-end figure through the same API with host buffers (copies inside the timed region),
the CPU oracle timed on a bounded sample, SM clocks sampled during the timed region, and
extras: the unfused baseline on the same workload, the other workloads, and small-m
microseconds per call.

With N > 1 each rank runs its own replica of the workload on its own GPU (the problem is
independent per GPU; no collective is on the data path); the JSON value is the sum of all
ranks' work divided by the slowest rank's time.  The ranks come from torchrun, or, when no
launcher set WORLD_SIZE, the script starts N replica processes itself (one per GPU, a local
rendezvous); n_gpus is the rank count either way.

--impl reference times the reference arm: the CPU oracle as it stands, on this host's
cores, on a bounded sample of the same workload per step (rank 0 only).
"""
from __future__ import annotations

import argparse
import json
import math
import os
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "fused GEMM+epilogue TFLOP/s and % of GB300 bf16 peak; µs/call at small M"
HEADLINE = "relu_bias_bf16_65536x16384x8192"
FALLBACK_PEAKS = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0}


def log(*a):
    print(*a, file=sys.stderr, flush=True)


def load_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as fh:
            d = json.load(fh)
        return {k: float(d[k]) for k in FALLBACK_PEAKS}, "measured"
    except Exception:
        return dict(FALLBACK_PEAKS), "fallback"


# ---- clocks during the timed region ---------------------------------------------------------

class ClockSampler:
    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        self.proc = None
        self.path = None
        self.dev = device_index

    def start(self):
        try:
            import torch
            uuid = str(torch.cuda.get_device_properties(self.dev).uuid)
            sel = ["-i", uuid if uuid.startswith("GPU-") else f"GPU-{uuid}"]
        except Exception:
            sel = []
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", *sel, f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
                 "-lms", "200", "-f", self.path], stdout=subprocess.DEVNULL,
                stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None
        time.sleep(0.3)

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        rows = []
        with open(self.path) as fh:
            for line in fh:
                parts = [x.strip() for x in line.split(",")]
                if len(parts) >= 8:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}

        def num(x):
            try:
                return float(x)
            except ValueError:
                return None
        sm = [num(r[0]) for r in rows if num(r[0]) is not None]
        mx = [num(r[1]) for r in rows if num(r[1]) is not None]
        pw = [num(r[2]) for r in rows if num(r[2]) is not None]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i] == "Active"})
        return {"sm_mhz": statistics.median(sm) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "power_w_max": max(pw) if pw else None,
                "samples": len(rows), "reasons": reasons}


# ---- timing helpers -------------------------------------------------------------------------

def time_steps(fn, steps: int, warmup: int, stream, dist_barrier=None) -> float:
    """Seconds for `steps` calls of fn() on `stream`, CUDA events, synchronised both sides."""
    import torch
    for _ in range(warmup):
        fn()
    torch.cuda.synchronize()
    if dist_barrier:
        dist_barrier()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(steps):
        fn()
    e1.record(stream)
    torch.cuda.synchronize()
    if dist_barrier:
        dist_barrier()
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3


def time_cold(fn, iters: int, stream, flush) -> float:
    """Seconds of fn() with L2 flushed before every call (events around the call): the mean
    of 2 x iters samples without the top and bottom tenth.  The event clock of the GB300
    boxes advances in steps of about 2 us, so a median of single calls lands on those steps;
    a trimmed mean over many calls resolves fractions of a step."""
    import torch
    iters *= 2
    ts = []
    for i in range(iters + 2):
        flush()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        fn()
        e1.record(stream)
        torch.cuda.synchronize()
        if i >= 2:
            ts.append(e0.elapsed_time(e1) / 1e3)
    ts.sort()
    cut = len(ts) // 10
    return statistics.mean(ts[cut:len(ts) - cut])


def time_graph(fn, calls: int, replays: int, stream) -> float:
    """Seconds per call from a CUDA graph of `calls` back-to-back calls (hot L2)."""
    import torch
    fn()
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    capture = torch.cuda.Stream()          # capture needs a non-default stream
    with torch.cuda.graph(g, stream=capture):
        for _ in range(calls):
            fn()
    g.replay()
    torch.cuda.synchronize()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for _ in range(replays):
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3 / (calls * replays)


def time_cold_graph(fn, flush, calls: int, replays: int, stream) -> float:
    """Seconds per call with L2 flushed before every call, resolved below the event clock's
    step: a CUDA graph of `calls` (flush, call) pairs and one of `calls` flushes alone, each
    replayed `replays` times; the difference per call.  (A programmatic dependent launch may
    start its set-up while the flush ends, as it would behind any other kernel.)"""
    import torch

    def graph_time(body):
        body()
        torch.cuda.synchronize()
        g = torch.cuda.CUDAGraph()
        capture = torch.cuda.Stream()
        with torch.cuda.graph(g, stream=capture):
            for _ in range(calls):
                body()
        g.replay()
        torch.cuda.synchronize()
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        for _ in range(replays):
            g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        return e0.elapsed_time(e1) / 1e3

    def pair():
        flush()
        fn()

    with_call = graph_time(pair)
    alone = graph_time(flush)
    return max(with_call - alone, 0.0) / (calls * replays)


# ---- the CPU oracle on a sample -------------------------------------------------------------

def oracle_sample_rate(A_rows_host, B_host, bias_host, w, target_s: float):
    """(TFLOP/s, rows, seconds) of the oracle on `rows` full rows of the workload, sized so
    one call takes about target_s seconds."""
    import numpy as np

    import oracle
    rows = min(8, A_rows_host.shape[0])
    while True:
        t0 = time.perf_counter()
        oracle.gemm_epi(A_rows_host[:rows], B_host, bias_host, dtype=w.dtype, epilog=w.epilog,
                        bias_layout=w.bias_layout)
        dt = time.perf_counter() - t0
        if dt >= target_s * 0.5 or rows >= A_rows_host.shape[0]:
            break
        rows = int(min(A_rows_host.shape[0], max(rows * 2, rows * target_s / max(dt, 1e-3))))
    flops = 2.0 * rows * w.n * w.k
    return flops / dt / 1e12, rows, dt


def cpu_inputs_for(w, rows_needed: int, dev):
    """Host copies of the first rows of A, all of B and the bias (drawn on the device)."""
    from activation_epilogue_gb300 import workloads
    inp = workloads.gemm_inputs(w, device=dev)
    A = inp["A"][:rows_needed].cpu()
    B = inp["B"].cpu()
    b = inp["bias"].cpu()
    del inp
    return A, B, b


def run_reference(args, world: int):
    """The reference arm: the CPU oracle, as it stands, on a bounded sample per step (rank 0
    of `world` ranks runs it; the line reports the job's rank count)."""
    import torch

    import oracle
    from activation_epilogue_gb300 import workloads
    w = workloads.GEMMS[HEADLINE]
    oracle.build()
    dev = torch.device("cuda", 0) if torch.cuda.is_available() else torch.device("cpu")
    A, B, b = cpu_inputs_for(w, 4096, dev)
    rate, rows, dt = oracle_sample_rate(A, B, b, w, target_s=2.0)
    ts = []
    for i in range(args.warmup + args.steps):
        t0 = time.perf_counter()
        oracle.gemm_epi(A[:rows], B, b, dtype=w.dtype, epilog=w.epilog, bias_layout=w.bias_layout)
        if i >= args.warmup:
            ts.append(time.perf_counter() - t0)
    total = sum(ts)
    flops = 2.0 * rows * w.n * w.k
    value = flops * len(ts) / total / 1e12
    sample = (f"{rows} full rows (all {w.n} columns, k={w.k}) of the {w.m}x{w.n}x{w.k} "
              f"{w.epilog} problem per step, fp64 oracle")
    line = {
        "impl": "reference", "metric": METRIC, "value": value, "unit": "TFLOP/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": total / len(ts) * 1e3, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {"workload": HEADLINE, "m": w.m, "n": w.n, "k": w.k, "epilog": w.epilog,
                   "sample_rows_per_step": rows},
        "cpu_baseline": {"value": value, "unit": "TFLOP/s", "cores": oracle.num_threads(),
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": value, "unit": "TFLOP/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
        "gpu_launches": 0,
    }
    print(json.dumps(line), flush=True)


# ---- our arm ----------------------------------------------------------------------------------

def run_ours(args, rank, world, local_rank, dist):
    import torch

    from activation_epilogue_gb300 import build as libbuild
    from activation_epilogue_gb300 import gemm_epi, workloads

    libbuild.build()
    dev = torch.device("cuda", local_rank)
    torch.cuda.set_device(dev)
    stream = torch.cuda.current_stream(dev)
    peaks, peaks_src = load_peaks()
    barrier = (lambda: dist.barrier()) if dist is not None else None

    w = workloads.GEMMS[args.workload]
    if args.rows:
        # a row slice of the same workload (same shapes of B and bias, same distributions)
        import dataclasses
        w = dataclasses.replace(w, m=args.rows, name=f"{w.name}_rows{args.rows}")
    td = workloads.TORCH_DTYPES[w.dtype]
    inp = workloads.gemm_inputs(w, device=dev)
    A, B, bias = inp["A"], inp["B"], inp["bias"]
    D = torch.empty((w.m, w.n), dtype=td, device=dev)
    aux = None
    if w.epilog == "RELU_AUX_BIAS":
        aux = torch.empty((w.m, (w.n + 31) // 32), dtype=torch.int32, device=dev)
    opts = dict(kv.split("=") for kv in args.opt)
    plan = gemm_epi.Plan(w.m, w.n, w.k, w.dtype, w.epilog, w.bias_layout,
                         **{k: int(v) for k, v in opts.items()})
    log(f"[bench] rank {rank}: {plan.describe()}")

    def step():
        plan.execute(A, B, bias, D, aux=aux)

    sampler = ClockSampler(local_rank) if rank == 0 else None
    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize()
    if sampler:
        sampler.start()
    secs = time_steps(step, args.steps, 0, stream, barrier)
    clocks = sampler.stop() if sampler else None
    st = plan.sync_status()
    if st != 0:
        raise RuntimeError(f"device status {gemm_epi.status_string(st)}")

    flops_step = float(w.flops)
    secs, value = whole_job(secs, flops_step, args.steps, world, dist, dev)
    kernel_s = secs / args.steps
    if rank != 0:
        plan.free()
        return

    achieved = flops_step / kernel_s / 1e12
    sustained = secs >= 1.0
    peak = peaks["bf16_tflops_sustained" if sustained else "bf16_tflops"]
    traffic = load_traffic(w.name)
    line = {
        "metric": METRIC, "value": value, "unit": "TFLOP/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": kernel_s * 1e3,
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16",
        "data": "synthetic",
        "config": {"workload": w.name, "m": w.m, "n": w.n, "k": w.k, "epilog": w.epilog,
                   "bias_layout": "(1,n)" if w.bias_layout == "1N" else "(m,1)",
                   "l2": "inputs larger than L2 (no flush needed)",
                   "parallelism": f"replicas x{world}", "plan": plan.describe()},
        "roofline": {"bound": "tensor", "achieved": achieved, "peak": peak, "unit": "TFLOP/s",
                     "frac": achieved / peak, "traffic": traffic,
                     "peak_source": f"{peaks_src} {'sustained' if sustained else 'burst'} bf16"},
        "gpu_launches": args.steps,
        "clocks": clocks,
    }
    plan_ms = kernel_s * 1e3
    log(f"[bench] fused: {plan_ms:.3f} ms/step, {achieved:.1f} TFLOP/s "
        f"({100 * achieved / peak:.1f}% of {peaks_src} peak {peak:.0f})")

    # e2e through the same API with host buffers: H2D of the inputs, D2H of the result
    if not args.no_e2e:
        line["e2e"] = measure_e2e(plan, w, A, B, bias, D, aux, stream, args)
    # extras before the CPU work, while the device buffers are still held
    if not args.no_extras:
        del inp
        line["extras"] = measure_extras(plan, w, A, B, bias, D, aux, stream, peaks)
    plan.free()
    del A, B, D, aux
    torch.cuda.empty_cache()
    if not args.no_cpu_baseline and world == 1:
        Ah, Bh, bh = cpu_inputs_for(w, 4096, dev)
        rate, rows, dt = oracle_sample_rate(Ah, Bh, bh, w, target_s=args.cpu_seconds)
        import oracle
        line["cpu_baseline"] = {
            "value": rate, "unit": "TFLOP/s", "cores": oracle.num_threads(), "kind": "oracle",
            "sample": f"{rows} full rows (all {w.n} columns, k={w.k}) of the "
                      f"{w.m}x{w.n}x{w.k} {w.epilog} problem, fp64 oracle, {dt:.1f} s"}
        if not args.no_extras:
            line["cpu_baseline"]["full_problems"] = oracle_full_problems(dev)
    print(json.dumps(line), flush=True)


def oracle_full_problems(dev) -> dict:
    """The oracle, as it stands, on each of the smaller workloads in full (one call each,
    inputs drawn on the device as for the fused runs, then copied to the host): seconds and
    TFLOP/s, the CPU time beside each GPU row."""
    import oracle
    from activation_epilogue_gb300 import workloads
    out = {}
    for name, g in workloads.GEMMS.items():
        if g.flops > 3e11:
            continue  # the headline problem: sampled above
        inp = {k: v.cpu() for k, v in workloads.gemm_inputs(g, device=dev).items()}
        t0 = time.perf_counter()
        oracle.gemm_epi(inp["A"], inp["B"], inp["bias"], dtype=g.dtype, epilog=g.epilog,
                        bias_layout=g.bias_layout)
        dt = time.perf_counter() - t0
        out[name] = {"seconds": dt, "tflops": g.flops / dt / 1e12}
    for name, f in workloads.FFNS.items():
        fi = {k: v.cpu() for k, v in workloads.ffn_inputs(f, device=dev).items()}
        t0 = time.perf_counter()
        oracle.ffn(fi["X"], fi["W1"], fi["b1"], fi["W2"], fi["b2"], fi["R"], dtype=f.dtype)
        dt = time.perf_counter() - t0
        out[name] = {"seconds": dt, "tflops": f.flops / dt / 1e12}
    return out


def whole_job(secs: float, flops_per_step: float, steps: int, world: int, dist, device):
    """(slowest rank's seconds, whole-job TFLOP/s): every rank ran `steps` steps of its own
    replica; the job's throughput is all ranks' work over the slowest rank's time."""
    import torch
    if dist is not None and world > 1:
        t = torch.tensor([secs], dtype=torch.float64, device=device)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        secs = float(t.item())
    return secs, flops_per_step * steps * world / secs / 1e12


def load_small_ncu():
    """Per workload, the ncu kernel duration (cold caches) and DRAM bytes of the committed
    summary of `bench.py --only small`, with the plan it was taken on."""
    path = os.path.join(ROOT, "profiles", "small_shapes_ncu.json")
    try:
        with open(path) as fh:
            return json.load(fh)
    except Exception:
        return {}


def run_small_for_ncu(dev):
    """Every workload but the headline, three calls each with L2 flushed before each: the
    command an ncu capture of the small shapes' kernel durations runs."""
    import torch

    from activation_epilogue_gb300 import gemm_epi, workloads
    flush_buf = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)
    plans = {}
    for name, g in workloads.GEMMS.items():
        if name == HEADLINE:
            continue
        td = workloads.TORCH_DTYPES[g.dtype]
        inp = workloads.gemm_inputs(g, device=dev)
        Dg = torch.empty((g.m, g.n), dtype=td, device=dev)
        auxg = (torch.empty((g.m, (g.n + 31) // 32), dtype=torch.int32, device=dev)
                if g.epilog == "RELU_AUX_BIAS" else None)
        with gemm_epi.Plan(g.m, g.n, g.k, g.dtype, g.epilog, g.bias_layout) as pg:
            for _ in range(3):
                flush_buf.zero_()
                pg.execute(inp["A"], inp["B"], inp["bias"], Dg, aux=auxg)
            torch.cuda.synchronize()
            if pg.sync_status() != 0:
                raise RuntimeError(f"{name}: device status {pg.sync_status()}")
            plans[name] = pg.describe()
    return plans


def load_traffic(workload: str):
    """DRAM bytes per launch of the fused kernel from the committed ncu summary, if any."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as fh:
            return json.load(fh).get(workload)
    except Exception:
        return None


def measure_e2e(plan, w, A, B, bias, D, aux, stream, args):
    import torch
    Ah = torch.empty(A.shape, dtype=A.dtype, pin_memory=True)
    Bh = torch.empty(B.shape, dtype=B.dtype, pin_memory=True)
    bh = torch.empty(bias.shape, dtype=bias.dtype, pin_memory=True)
    Ah.copy_(A)
    Bh.copy_(B)
    bh.copy_(bias)
    Dh = torch.empty(D.shape, dtype=D.dtype, pin_memory=True)
    auxh = None if aux is None else torch.empty(aux.shape, dtype=aux.dtype, pin_memory=True)

    # through the library's host-buffer call: A, B and bias copied in, D (and aux) copied out
    # every step, in row chunks pipelined against the GEMMs on the plan's own streams
    def e2e_step():
        plan.execute_host(Ah, Bh, bh, Dh, aux=auxh)

    # The host link and host memory are shared with the machine's other GPUs: a single call
    # now and then takes 18-130 ms instead of 13.5 (seen with every build), so the figure is
    # the median of three timed runs of `steps` calls each (every run reported).
    steps = max(2, min(args.steps, 5))
    runs = [time_steps(e2e_step, steps, 1 if r == 0 else 0, stream) for r in range(3)]
    secs = sorted(runs)[1]
    h2d = (A.numel() + B.numel() + bias.numel()) * A.element_size()
    d2h = D.numel() * D.element_size() + (0 if aux is None else aux.numel() * 4)
    return {"value": float(w.flops) * steps / secs / 1e12, "unit": "TFLOP/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
            "ms_per_step": secs / steps * 1e3, "steps": steps, "stat": "median of 3 runs",
            "runs_ms_per_step": [round(r / steps * 1e3, 3) for r in runs]}


def measure_extras(plan, w, A, B, bias, D, aux, stream, peaks):
    """Unfused baseline on the headline workload; the other workloads; small-m us/call."""
    import torch

    from activation_epilogue_gb300 import gemm_epi, workloads
    out = {}
    # unfused on the same workload: GEMM writes pre (bf16), elementwise pass reads it back
    pre = torch.empty_like(D)
    t_unf = time_steps(lambda: plan.execute_unfused(A, B, bias, pre, D, aux=aux), 5, 2, stream)
    out["unfused_same_workload"] = {"ms_per_step": t_unf / 5 * 1e3,
                                    "tflops": float(w.flops) * 5 / t_unf / 1e12,
                                    "launches_per_step": 2,
                                    "extra_bytes": 2 * w.m * w.n * 2}
    del pre
    torch.cuda.empty_cache()

    flush_buf = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.int32, device=A.device)

    def flush():
        flush_buf.zero_()

    per = {}
    # ncu durations (cold caches) from the committed summary, used only when it was taken on
    # the plan this run picks
    small_ncu = load_small_ncu()
    for name, g in workloads.GEMMS.items():
        if name == w.name:
            continue
        td = workloads.TORCH_DTYPES[g.dtype]
        inp = workloads.gemm_inputs(g, device=A.device)
        Dg = torch.empty((g.m, g.n), dtype=td, device=A.device)
        auxg = (torch.empty((g.m, (g.n + 31) // 32), dtype=torch.int32, device=A.device)
                if g.epilog == "RELU_AUX_BIAS" else None)
        with gemm_epi.Plan(g.m, g.n, g.k, g.dtype, g.epilog, g.bias_layout) as pg:
            fn = lambda: pg.execute(inp["A"], inp["B"], inp["bias"], Dg, aux=auxg)  # noqa: E731
            cold = time_cold(fn, 20, stream, flush)
            # (the difference of two graph timings: the best of three, as the flush's own
            # time varies from graph to graph)
            cold_graph = min(time_cold_graph(fn, flush, 20, 5, stream) for _ in range(3))
            hot = time_graph(fn, 20, 10, stream)
            pre = torch.empty_like(Dg)
            fu = lambda: pg.execute_unfused(inp["A"], inp["B"], inp["bias"], pre, Dg, aux=auxg)  # noqa: E731
            cold_unf = time_cold(fu, 20, stream, flush)
            st = pg.sync_status()
            desc = pg.describe()
        e = 2
        unavoidable = (g.m * g.k + g.k * g.n + (g.m if g.bias_layout == "M1" else g.n)
                       + g.m * g.n) * e + (0 if auxg is None else auxg.numel() * 4)
        rec = small_ncu.get(name, {})
        ncu_us = rec.get("us") if rec.get("plan") == desc else None
        per[name] = {
            "us_per_call_cold_l2": cold * 1e6, "us_per_call_cold_l2_graph": cold_graph * 1e6,
            "us_ncu_cold": ncu_us,
            "hbm_frac_ncu": (unavoidable / (ncu_us * 1e-6) / 1e9 / peaks["hbm_gbs"]
                             if ncu_us else None),
            "us_per_call_graph_hot_l2": hot * 1e6,
            "tflops_cold": g.flops / cold / 1e12,
            "hbm_gbs_cold": unavoidable / cold / 1e9,
            "hbm_frac_cold": unavoidable / cold / 1e9 / peaks["hbm_gbs"],
            "tensor_frac_cold": g.flops / cold / 1e12 / peaks["bf16_tflops"],
            "unfused_us_cold_l2": cold_unf * 1e6, "unavoidable_bytes": unavoidable,
            "status": st, "plan": desc}
        del inp, Dg, auxg, pre
    per.update(measure_ffn(A.device, stream, flush, peaks))
    out["workloads"] = per
    out["backward"] = measure_backward(A.device, stream, flush, peaks)
    out["fp8"] = measure_fp8(A.device, stream, peaks)
    out["layer_stack"] = measure_layer_stack(A.device, stream, peaks)
    return out


def measure_layer_stack(device, stream, peaks):
    """Small-batch FFN layers back to back, as a decoder runs them (T = 16, 64, 256):
    X[T,768] -> GELU_BIAS up to 3072 -> BIAS_RESIDUAL down to 768 (in place: X += H.W2 +
    b2), 24 layers with weights
    of their own (226 MB, more than L2, so each replay reads them from HBM again), captured
    in a CUDA graph and replayed.  Microseconds per GEMM call with plain launches, with
    programmatic dependent launch (the default), and with the weights promised ready
    (B_READY: each call copies its weight while the previous call still runs)."""
    import torch

    from activation_epilogue_gb300 import gemm_epi, workloads
    d, f, layers = 768, 3072, 24
    out = {}
    for t in (16, 64, 256):
        inp = workloads.layer_stack_inputs(t, d, f, layers, seed=4000 + t, device=device)
        X = inp["X"].clone()
        H = torch.empty((t, f), dtype=torch.bfloat16, device=device)
        # bytes a call must move: weight, bias, input, output (and the residual)
        up_bytes = (d * f + f + t * d + t * f) * 2
        down_bytes = (f * d + d + t * f + t * d + t * d) * 2
        call_bytes = (up_bytes + down_bytes) / 2
        rec = {"bytes_per_call": call_bytes, "layers": layers}
        for mode, opts in (("plain", {"PDL": 0}), ("pdl", {}), ("pdl_b_ready", {"B_READY": 1})):
            with gemm_epi.Plan(t, f, d, "bf16", "GELU_BIAS", "1N", **opts) as up, \
                    gemm_epi.Plan(t, d, f, "bf16", "BIAS_RESIDUAL", "1N", **opts) as down:
                def stack():
                    for W1, b1, W2, b2 in inp["layers"]:
                        up.execute(X, W1, b1, H)
                        down.execute(H, W2, b2, X, residual=X)
                secs = min(time_graph(stack, 1, 20, stream) for _ in range(3))
                us = secs / (2 * layers) * 1e6
                rec[mode] = {"us_per_call": us,
                             "hbm_gbs": call_bytes / (us * 1e-6) / 1e9,
                             "hbm_frac": call_bytes / (us * 1e-6) / 1e9 / peaks["hbm_gbs"],
                             "status": up.sync_status() | down.sync_status(),
                             "plans": [up.describe(), down.describe()]}
        out[f"t{t}_d{d}_f{f}"] = rec
        del inp, X, H
        torch.cuda.empty_cache()
    return out


def measure_fp8(device, stream, peaks):
    """RELU_BIAS on E4M3 inputs (per-tensor scales, bf16 bias and output) at 4096^3 and at the
    headline shape: TFLOP/s against the FP8 peak taken as the measured bf16 peak x 2 (the
    nominal dense ratio, 4.5 / 2.25 PFLOP/s).  Inputs larger than L2 at the headline shape;
    4096^3 reported hot (back-to-back calls)."""
    import torch

    from activation_epilogue_gb300 import gemm_epi, workloads
    peak8 = 2.0 * peaks["bf16_tflops"]
    res = {}
    for m, n, k in [(4096, 4096, 4096), (65536, 16384, 8192)]:
        p = workloads.random_fp8_problem(m, n, k, seed=1008, device=device)
        sa = torch.tensor([p["scale_a"]], dtype=torch.float32, device=device)
        sb = torch.tensor([p["scale_b"]], dtype=torch.float32, device=device)
        D = torch.empty((m, n), dtype=torch.bfloat16, device=device)
        with gemm_epi.Plan(m, n, k, "e4m3", "RELU_BIAS", "1N") as pl:
            fn = lambda: pl.execute(p["A"], p["Bt"], p["bias"], D, scales=(sa, sb))  # noqa: E731
            steps = 5 if m > 8192 else 50
            secs = time_steps(fn, steps, 3, stream) / steps
            tf = 2.0 * m * n * k / secs / 1e12
            res[f"relu_bias_e4m3_{m}x{n}x{k}"] = {
                "us_per_call": secs * 1e6, "tflops": tf, "peak_tflops": peak8,
                "frac_of_fp8_peak": tf / peak8, "status": pl.sync_status(), "plan": pl.describe()}
        del p, D
        torch.cuda.empty_cache()
    return res


def measure_ffn(device, stream, flush, peaks):
    """The FFN block through its plan (automatic mode; one launch, two launches and one launch
    with GEMM 2 in K slices forced) and
    the unfused chain (GEMM, bias+GELU pass, GEMM, bias+residual pass: four launches, two
    extra round trips of pre-activations), cold L2 and CUDA Graph replay."""
    import torch

    from activation_epilogue_gb300 import gemm_epi, workloads
    f = workloads.FFNS["ffn_bf16_4096x1024x4096"]
    fi = workloads.ffn_inputs(f, device=device)
    Y = torch.empty((f.t, f.d), dtype=torch.bfloat16, device=device)
    H = torch.empty((f.t, f.f), dtype=torch.bfloat16, device=device)
    pre1 = torch.empty((f.t, f.f), dtype=torch.bfloat16, device=device)
    pre2 = torch.empty((f.t, f.d), dtype=torch.bfloat16, device=device)
    out = {}
    with gemm_epi.Plan(f.t, f.f, f.d, "bf16", "GELU_BIAS", "1N") as p1, \
            gemm_epi.Plan(f.t, f.d, f.f, "bf16", "BIAS_RESIDUAL", "1N") as p2:
        def ffn_unfused():
            p1.execute_unfused(fi["X"], fi["W1"], fi["b1"], pre1, H)
            p2.execute_unfused(H, fi["W2"], fi["b2"], pre2, Y, residual=fi["R"])
        cold_unf = time_cold(ffn_unfused, 20, stream, flush)
        # (one launch with GEMM 2 in 4 K slices, and one launch with H kept on chip: the
        # layouts that cost more than they gain, measured every run)
        for mode, opts in [("", {}), ("_one_launch", {"launches": 1}),
                           ("_two_launches", {"launches": 2}),
                           ("_one_launch_split4", {"launches": 1, "split2": 4}),
                           ("_onchip", {"launches": 3})]:
            with gemm_epi.FfnPlan(f.t, f.d, f.f, "bf16", **opts) as fp:
                def ffn():
                    fp.execute(fi["X"], fi["W1"], fi["b1"], fi["W2"], fi["b2"], fi["R"], Y)
                cold = time_cold(ffn, 20, stream, flush)
                hot = time_graph(ffn, 10, 10, stream)
                out[f.name + mode] = {
                    "us_per_call_cold_l2": cold * 1e6, "us_per_call_graph_hot_l2": hot * 1e6,
                    "tflops_cold": f.flops / cold / 1e12,
                    "tensor_frac_cold": f.flops / cold / 1e12 / peaks["bf16_tflops"],
                    "unfused_us_cold_l2": cold_unf * 1e6, "unfused_launches": 4,
                    "status": fp.sync_status(), "plan": fp.describe()}
    # the pre-LayerNorm block Y = X + FFN(LayerNorm(X)) (LayerNorm gamma ~ 1 + N(0, 0.1^2),
    # beta ~ N(0, 0.1^2)): row statistics + GEMM 1 with the LayerNorm folded into its
    # epilogue + GEMM 2, against the fused LayerNorm kernel writing LN(X) followed by the FFN
    g = torch.Generator(device=device)
    g.manual_seed(1006)
    gamma = (1.0 + 0.1 * torch.randn(f.d, generator=g, device=device)).to(torch.bfloat16)
    beta = (0.1 * torch.randn(f.d, generator=g, device=device)).to(torch.bfloat16)
    W1f = torch.empty_like(fi["W1"])
    cs = torch.empty(f.f, dtype=torch.float32, device=device)
    b1f = torch.empty(f.f, dtype=torch.float32, device=device)
    gemm_epi.gemm_epi_layernorm_fold(f.d, f.f, "bf16", gamma, beta, fi["W1"], fi["b1"], W1f, cs,
                                     b1f)
    Xn = torch.empty_like(fi["X"])
    with gemm_epi.FfnPlan(f.t, f.d, f.f, "bf16", layernorm=True) as lp, \
            gemm_epi.FfnPlan(f.t, f.d, f.f, "bf16") as fp:
        def ln_ffn():
            lp.execute_layernorm(fi["X"], 1e-5, W1f, cs, b1f, fi["W2"], fi["b2"], fi["X"], Y)

        def ln_then_ffn():
            gemm_epi.gemm_epi_layernorm(f.t, f.d, "bf16", fi["X"], None, gamma, beta, 1e-5, Xn)
            fp.execute(Xn, fi["W1"], fi["b1"], fi["W2"], fi["b2"], fi["X"], Y)
        cold = time_cold(ln_ffn, 20, stream, flush)
        hot = time_graph(ln_ffn, 10, 10, stream)
        cold_sep = time_cold(ln_then_ffn, 20, stream, flush)
        hot_sep = time_graph(ln_then_ffn, 10, 10, stream)
        out[f.name + "_layernorm"] = {
            "us_per_call_cold_l2": cold * 1e6, "us_per_call_graph_hot_l2": hot * 1e6,
            "tflops_cold": f.flops / cold / 1e12,
            "separate_layernorm_us_cold_l2": cold_sep * 1e6,
            "separate_layernorm_us_graph_hot_l2": hot_sep * 1e6,
            "status": lp.sync_status(), "plan": lp.describe()}
    return out


def measure_backward(device, stream, flush, peaks):
    """GELU_AUX_BIAS (forward keeping pre) and the backward epilogues DRELU_BGRAD and
    DGELU_BGRAD on a 4096 x 4096 x 4096 bf16 layer, bias (1,n): fused against unfused
    (GEMM writing bf16(A.B), then the elementwise pass with the mask or GELU' factor and the
    bias-gradient sums), cold L2."""
    import numpy as np
    import torch

    from activation_epilogue_gb300 import gemm_epi, workloads
    m = n = k = 4096
    inp = workloads.random_backward_problem(m, n, k, dtype="bf16", seed=2024, device=device)
    fw = workloads.random_problem(m, n, k, dtype="bf16", seed=2025, device=device)
    mask = torch.from_numpy(inp["mask"].view(np.int32)).to(device)
    D = torch.empty((m, n), dtype=torch.bfloat16, device=device)
    pre = torch.empty_like(D)
    aux16 = torch.empty_like(D)
    dbias = torch.empty((n,), dtype=torch.float32, device=device)
    flops = 2.0 * m * n * k
    res = {}
    for epilog in ["GELU_AUX_BIAS", "DRELU_BGRAD", "DGELU_BGRAD"]:
        if epilog == "GELU_AUX_BIAS":
            kw = dict(aux=aux16)
            bias = fw["bias"]
            extra = m * n * 2                                  # the stored pre-activation
        else:
            kw = dict(aux_in=mask if epilog == "DRELU_BGRAD" else inp["pre"], dbias=dbias)
            bias = None
            extra = mask.numel() * 4 if epilog == "DRELU_BGRAD" else m * n * 2
        with gemm_epi.Plan(m, n, k, "bf16", epilog, "1N") as pl:
            fn = lambda: pl.execute(inp["A"], inp["B"], bias, D, **kw)  # noqa: E731
            fu = lambda: pl.execute_unfused(inp["A"], inp["B"], bias, pre, D, **kw)  # noqa: E731
            cold = time_cold(fn, 20, stream, flush)
            cold_unf = time_cold(fu, 20, stream, flush)
            res[epilog] = {"shape": [m, n, k], "us_per_call_cold_l2": cold * 1e6,
                           "tflops_cold": flops / cold / 1e12,
                           "tensor_frac_cold": flops / cold / 1e12 / peaks["bf16_tflops"],
                           "unfused_us_cold_l2": cold_unf * 1e6,
                           "extra_aux_bytes": extra, "status": pl.sync_status(),
                           "plan": pl.describe()}
    return res


def parse_args(argv=None):
    ap = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default=HEADLINE)
    ap.add_argument("--opt", action="append", default=[], metavar="KEY=VALUE",
                    help="plan option for the timed workload, e.g. SPLIT_K=1 (repeatable)")
    ap.add_argument("--rows", type=int, default=0,
                    help="time only this many rows of the workload (for profiler captures)")
    ap.add_argument("--no-extras", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--only", choices=["backward", "ffn", "fp8", "small", "stack"],
                    help="print only these measurements (one JSON object), for profiling")
    args = ap.parse_args(argv)
    if args.gpus < 1:
        ap.error("--gpus must be >= 1")
    if args.warmup < 3:
        log("[bench] warm-up raised to 3 steps")
        args.warmup = 3
    return args


# ---- replicas without a launcher --------------------------------------------------------------

def _replica_main(local_rank: int, argv, world: int, port: int):
    """Entry point of one replica process started by launch_replicas: the rank variables a
    launcher would set, then the same code path as under torchrun."""
    os.environ.update(RANK=str(local_rank), LOCAL_RANK=str(local_rank), WORLD_SIZE=str(world),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    rank_main(parse_args(argv))


def launch_replicas(argv, world: int, target=_replica_main):
    """`--gpus N` with no launcher around the process: start N replica processes (spawn, one
    per GPU, a local rendezvous on 127.0.0.1), wait for all of them; raises if one fails."""
    import socket

    import torch.multiprocessing as mp
    with socket.socket() as sk:
        sk.bind(("127.0.0.1", 0))
        port = sk.getsockname()[1]
    mp.start_processes(target, args=(list(argv), world, port), nprocs=world, join=True,
                       start_method="spawn")


def rank_main(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            run_reference(args, world)
        return

    if args.only:
        import torch
        dev = torch.device("cuda", local_rank)
        torch.cuda.set_device(dev)
        stream = torch.cuda.current_stream()
        flush_buf = torch.empty(512 * 1024 * 1024 // 4, dtype=torch.int32, device=dev)
        if args.only == "fp8":
            res = measure_fp8(dev, stream, load_peaks()[0])
        elif args.only == "small":
            res = run_small_for_ncu(dev)
        elif args.only == "stack":
            res = measure_layer_stack(dev, stream, load_peaks()[0])
        else:
            measure = measure_backward if args.only == "backward" else measure_ffn
            res = measure(dev, stream, flush_buf.zero_, load_peaks()[0])
        if rank == 0:
            print(json.dumps({args.only: res}))
        return

    dist = None
    if world > 1:
        import torch
        import torch.distributed as tdist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local_rank)
        tdist.init_process_group(backend)
        dist = tdist
    try:
        run_ours(args, rank, world, local_rank, dist)
    finally:
        if dist is not None:
            dist.destroy_process_group()


def main(argv=None):
    argv = sys.argv[1:] if argv is None else list(argv)
    args = parse_args(argv)
    if "WORLD_SIZE" not in os.environ and args.gpus > 1:
        launch_replicas(argv, args.gpus)
        return
    if int(os.environ.get("WORLD_SIZE", "1")) != args.gpus:
        log(f"[bench] --gpus {args.gpus} but WORLD_SIZE={os.environ.get('WORLD_SIZE', '1')}: "
            "reporting the launcher's rank count")
    rank_main(args)


if __name__ == "__main__":
    main()
