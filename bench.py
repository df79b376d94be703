#!/usr/bin/env python3
"""Benchmark: achieved HBM GB/s (fraction of the GB300 roofline) and us/call of
the quantized reduce + RMSNorm hot path.

One step = one pass of the whole hot path over one batch of synthetic
activations (inputs resident in HBM): sender-side group quantization of the
P partial-sum slabs, then the fused two-step reduce (dequantize, fixed-order
sum, requantize the all-gather payload, dequantize) + residual add + RMSNorm.
Default workload: prefill, P=4 slabs of 8192 x 8192 bf16, INT4 asymmetric
g32.  value = algorithmic bytes per step / device time per step.

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
  python bench.py --impl reference ...   # the CPU oracle, timed on host cores
  torchrun --nproc-per-node N bench.py --gpus N ...   # N independent replicas

Prints one JSON line on rank 0.
"""
from __future__ import annotations

import argparse
import contextlib
import ctypes
import hashlib
import json
import os
import statistics
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "achieved HBM GB/s (% of GB300 roofline) and us/call for quantized reduce+RMSNorm"
UNIT = "GB/s"
L2_BYTES = 129 * 2 ** 20


# Before a timed call the stream is held by a spinning kernel for about
# 100 us (at 2 GHz), so the call's launches are already queued when the
# start event fires: event intervals are device time, not the host's cost of
# issuing the call (which is reported on its own).
HOLD_CYCLES = 200_000
NOMINAL_HBM_GBS = 8000.0  # GB300 HBM3e, nominal


@contextlib.contextmanager
def nvtx(name):
    """An NVTX range around a timed region (visible in nsys/ncu timelines;
    a host-side marker only, nothing is added to the device work)."""
    import torch
    torch.cuda.nvtx.range_push(name)
    try:
        yield
    finally:
        torch.cuda.nvtx.range_pop()


def scrub_l2(buf):
    """Evicts the inputs of the next call from L2 by reading `buf` (larger
    than L2) into one scalar.  Only a read: L2 is left holding clean lines,
    so the timed call pays no write-back of the scrub's own data."""
    buf.sum(dtype=buf.dtype)


def spread(xs):
    """(median, p10, p90) of a list of numbers."""
    a = np.sort(np.asarray(xs, dtype=np.float64))
    return (float(np.median(a)), float(np.percentile(a, 10)), float(np.percentile(a, 90)))


def device_timed(fn, reps, warm=2, scrub=None):
    """(median device us, median host us, (p10, p90) device us) of fn() over
    `reps` repetitions after `warm` untimed ones; `scrub` (a tensor larger
    than L2) is read before every repetition, outside the events.  One call
    per event pair: the event clock's tick (about 2 us on GB300) bounds the
    resolution, so short calls are timed by stream_timed as well."""
    import torch
    dev_us, host_us = [], []
    for i in range(reps + warm):
        torch.cuda._sleep(HOLD_CYCLES)
        if scrub is not None:
            scrub_l2(scrub)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        t0 = time.perf_counter()
        fn()
        t1 = time.perf_counter()
        b.record()
        b.synchronize()
        if i >= warm:
            dev_us.append(a.elapsed_time(b) * 1e3)
            host_us.append((t1 - t0) * 1e6)
    med, p10, p90 = spread(dev_us)
    return med, statistics.median(host_us), (p10, p90)


def stream_timed(calls, per_rep, reps):
    """Device us per call: `per_rep` calls launched back to back between one
    pair of events, cycling through `calls` (one call per buffer set), the
    stream held while the host queues them; `reps` such repetitions after an
    untimed one.  Returns (median, p10, p90) over the repetitions."""
    import torch
    out = []
    for r in range(reps + 1):
        torch.cuda._sleep(HOLD_CYCLES + 40_000 * per_rep)  # ~20 us of queueing time per call
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for i in range(per_rep):
            calls[i % len(calls)]()
        b.record()
        b.synchronize()
        if r:
            out.append(a.elapsed_time(b) * 1e3 / per_rep)
    return spread(out)


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=200)
    ap.add_argument("--warmup", type=int, default=10)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", default="prefill")
    ap.add_argument("--rows", type=int, default=0,
                    help="override the workload's token count (profiling runs)")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--graph", action="store_true",
                    help="issue every timed step as one CUDA graph replay (untagged workloads)")
    ap.add_argument("--cpu-seconds", type=float, default=12.0,
                    help="target CPU time of the oracle sample")
    ap.add_argument("--split", choices=["even", "wave"], default="even",
                    help="token-subset boundary for workloads that split rows")
    ap.add_argument("--overlap", action="store_true",
                    help="SM-capped fused kernel beside a GEMM on another stream (one JSON line per cap)")
    ap.add_argument("--gather", action="store_true",
                    help="standalone quantized all-gather (shards -> whole dequantized tensor): one JSON line per case")
    ap.add_argument("--sweep", choices=["quick", "full"], default=None,
                    help="message-size sweep (16 KB..256 MB x P x format): one JSON line per point")
    ap.add_argument("--sizes", default="",
                    help="sweep: only these message sizes (e.g. 16M,32M)")
    ap.add_argument("--only", default="",
                    help="sweep: only these points, MSG:H:P:FMT[,...] (FMT bf16, int8 or int4)")
    ap.add_argument("--formats", default="",
                    help="sweep: these formats (bf16, int8, int4 and the tagged bf16t, int8t, int4t; "
                         "comma-separated; default the untagged three)")
    ap.add_argument("--calls", type=int, default=50,
                    help="sweep: calls per pair of events in the steady measurement (>= 50)")
    ap.add_argument("--split-table", action="store_true",
                    help="even vs wave-aware token split on row counts around wave multiples")
    ap.add_argument("--selector", action="store_true",
                    help="the protocol selector's estimates and picks against measured steps")
    ap.add_argument("--report-sweep", default="",
                    help="print the markdown table of a file of sweep JSON lines and exit")
    return ap.parse_args()


# ------------------------------------------------------------- clocks -----
class ClockSampler:
    """Samples SM clock and throttle reasons through NVML (ctypes) while active."""

    REASONS = {0x1: "gpu_idle", 0x2: "applications_clocks_setting", 0x4: "sw_power_cap",
               0x8: "hw_slowdown", 0x10: "sync_boost", 0x20: "sw_thermal_slowdown",
               0x40: "hw_thermal_slowdown", 0x80: "hw_power_brake_slowdown",
               0x100: "display_clock_setting"}

    def __init__(self, index: int, period_s: float = 0.005):
        self.samples, self.reasons, self.ok = [], 0, False
        self.period = period_s
        try:
            self.nv = ctypes.CDLL("libnvidia-ml.so.1")
            if self.nv.nvmlInit_v2() != 0:
                return
            self.h = ctypes.c_void_p()
            if self.nv.nvmlDeviceGetHandleByIndex_v2(index, ctypes.byref(self.h)) != 0:
                return
            mx = ctypes.c_uint()
            self.nv.nvmlDeviceGetMaxClockInfo(self.h, 1, ctypes.byref(mx))  # 1 = SM
            self.max_mhz = mx.value
            self.ok = True
        except OSError:
            pass

    def _run(self):
        clk, rs = ctypes.c_uint(), ctypes.c_ulonglong()
        while not self._stop.is_set():
            if self.nv.nvmlDeviceGetClockInfo(self.h, 1, ctypes.byref(clk)) == 0:
                self.samples.append(clk.value)
            if self.nv.nvmlDeviceGetCurrentClocksEventReasons(self.h, ctypes.byref(rs)) == 0:
                self.reasons |= rs.value
            time.sleep(self.period)

    def __enter__(self):
        if self.ok:
            self._stop = threading.Event()
            self._t = threading.Thread(target=self._run, daemon=True)
            self._t.start()
        return self

    def __exit__(self, *a):
        if self.ok:
            self._stop.set()
            self._t.join()

    def report(self):
        if not self.ok or not self.samples:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvml unavailable"]}
        names = [n for b, n in self.REASONS.items() if self.reasons & b and n != "gpu_idle"]
        return {"sm_mhz": statistics.median(self.samples), "sm_max_mhz": self.max_mhz,
                "samples": len(self.samples), "reasons": names}


# ------------------------------------------------------------- helpers ----
def dist_env():
    ws = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return ws, rank, local


def code_only(text: str) -> str:
    """C/C++/CUDA source without its comments and blank-line or trailing-space
    differences (string literals in these sources hold no comment markers)."""
    import re
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(l.rstrip() for l in text.splitlines() if l.strip())


def source_hash():
    """Hash of the kernel and launch code (comments excluded): ncu counters
    are reported only for the code they were taken on.  api.cu is left out:
    it holds the C entry points' argument checks and the host-only queries,
    and defines no kernel and no launch shape; so is rates.inc, the measured
    table the host-only protocol selector reads."""
    h = hashlib.sha256()
    d = os.path.join(ROOT, "quantized_reduce_rmsnorm_gb300", "csrc")
    for f in sorted(os.listdir(d)):
        if f in ("api.cu", "rates.inc"):
            continue
        h.update(f.encode())
        with open(os.path.join(d, f), encoding="utf-8") as fh:
            h.update(code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def measured_traffic(kernel: str, workload: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel sources; else None."""
    p = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(p) as f:
            tab = json.load(f)
    except (OSError, ValueError):
        return None
    e = tab.get(f"{workload}/{kernel}")
    if not e or e.get("source_hash") != source_hash():
        return None
    return e.get("dram_bytes_per_launch")


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    except (OSError, ValueError, KeyError):
        return 6800.0, "fallback"


# ------------------------------------------------------------- CPU arm ----
def host_cores() -> int:
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def oracle_sample(w, inputs, target_s: float, threads: int = 1):
    """Time the oracle on a bounded row sample of the workload's own inputs.
    With threads > 1 the sample's rows are cut into that many contiguous
    ranges, each run by the unmodified oracle on its own host thread (rows
    are independent; the C calls release the interpreter lock).

    When every row of the inputs takes less than target_s, the whole
    workload is run repeatedly (passes) until about target_s has elapsed.

    Returns (GB/s of algorithmic bytes, seconds, rows, passes)."""
    import concurrent.futures as cf
    import oracle
    from quantized_reduce_rmsnorm_gb300.pipeline import qs_bytes
    from quantized_reduce_rmsnorm_gb300.synth import (FMT_BF16, FMT_BF16_TAGGED, FMT_INT4_ASYM,
                                                      FMT_INT8_SYM, Workload)
    from quantized_reduce_rmsnorm_gb300.synth import base_format
    orc = oracle.default()
    fmt = FMT_BF16 if w.fmt == FMT_BF16_TAGGED else base_format(w.fmt)

    pool = cf.ThreadPoolExecutor(threads) if threads > 1 else None

    def run(rows):
        def part(k):
            r0, r1 = rows * k // threads, rows * (k + 1) // threads
            if r1 > r0:
                orc.allreduce_residual_rmsnorm(fmt, [s[r0:r1] for s in inputs["slabs"]],
                                               inputs["residual"][r0:r1], inputs["gamma"],
                                               r1 - r0, w.H, w.group, w.eps)
        t0 = time.perf_counter()
        if pool is None:
            part(0)
        else:
            list(pool.map(part, range(threads)))
        return time.perf_counter() - t0

    avail = int(inputs["residual"].shape[0])  # rows actually present in `inputs`
    probe = min(avail, 8 * threads)
    dt = run(probe)
    rows = int(min(avail, max(probe, probe * target_s / max(dt, 1e-6))))
    dt = run(rows)
    passes = 1
    if rows == avail and dt < target_s:
        passes = max(1, int(round(target_s / max(dt, 1e-6))))
        t0 = time.perf_counter()
        for _ in range(passes):
            run(rows)
        dt = time.perf_counter() - t0
    if pool is not None:
        pool.shutdown()
    sub = Workload(**{**w.__dict__, "T": rows})
    E = rows * w.H
    if fmt in (FMT_INT8_SYM, FMT_INT4_ASYM):
        qs = qs_bytes(sub, E)
        alg = (w.P * 2 * E + w.P * qs) + (w.P * qs + 2 * E + 2 * w.H + qs + 4 * E)
    else:
        alg = w.P * 2 * E + 2 * E + 2 * w.H + 4 * E
    return passes * alg / dt / 1e9, dt, rows, passes


def run_reference(args):
    ws, rank, _ = dist_env()
    if rank != 0:
        return
    from quantized_reduce_rmsnorm_gb300 import synth
    w = get_workload(args)
    # each step is a bounded sample of rows, sized so the whole run stays
    # within about two minutes of CPU time
    per_step = min(10.0, max(0.2, 120.0 / max(1, args.steps + args.warmup)))
    rows = min(w.T, 4096)
    inputs = synth.make_inputs(w, seed=0, rows=np.arange(rows))
    n = host_cores()
    vals = []
    for i in range(args.warmup + args.steps):
        gbs, dt, r, passes = oracle_sample(w, inputs, per_step, threads=n)
        if i >= args.warmup:
            vals.append((gbs, dt, r, passes))
    v = statistics.median(x[0] for x in vals)
    ms = statistics.median(x[1] for x in vals) * 1e3
    r, passes = vals[-1][2], vals[-1][3]
    reps = f" ({passes} passes over them)" if passes > 1 else ""
    line = {
        "impl": "reference", "metric": METRIC, "value": round(v, 4), "unit": UNIT,
        "n_gpus": args.gpus, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms, 3), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32", "data": "synthetic",
        "config": workload_config(w, note=f"oracle on {r} of {w.T} rows per step{reps}, {n} host threads"),
        "cpu_baseline": {"value": round(v, 4), "unit": UNIT, "cores": n, "kind": "oracle",
                         "sample": f"{r} of {w.T} rows of the {w.name} workload per step{reps}, in {n} "
                                   f"contiguous row ranges on {n} host threads"},
        "e2e": {"value": round(v, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def get_workload(args):
    from quantized_reduce_rmsnorm_gb300 import synth
    w = synth.WORKLOADS[args.workload]
    if args.rows:
        w = synth.Workload(**{**w.__dict__, "T": args.rows})
    return w


def workload_config(w, note=None):
    from quantized_reduce_rmsnorm_gb300.synth import FMT_NAMES
    c = {"workload": f"{w.name}: P={w.P} slabs of {w.T}x{w.H} bf16, {FMT_NAMES[w.fmt]}"
                     + (f", {w.splits} token subsets on {w.splits} streams" if w.splits > 1
                        else ""),
         "P": w.P, "tokens": w.T, "hidden": w.H, "format": FMT_NAMES[w.fmt], "group": w.group,
         "dist": w.dist, "outlier_frac": w.outlier_frac, "outlier_scale": w.outlier_scale,
         "eps": w.eps, "parallelism": "replicas"}
    if note:
        c["note"] = note
    return c


# ------------------------------------------------------------- GPU arm ----
def run_ours(args):
    import torch
    ws, rank, local = dist_env()
    if ws > 1:
        import torch.distributed as dist
        torch.cuda.set_device(local)
        dist.init_process_group("nccl")
    dev = torch.device("cuda", local if ws > 1 else 0)
    torch.cuda.set_device(dev)

    from quantized_reduce_rmsnorm_gb300 import fcomm, synth
    from quantized_reduce_rmsnorm_gb300.pipeline import Pipeline
    fcomm.load()
    w = get_workload(args)
    inputs = synth.make_inputs(w, seed=rank)
    pipe = Pipeline(w, inputs, device=dev, split=args.split)
    alg = pipe.alg_bytes()
    step_bytes = alg["sender"] + alg["fused"]
    in_bytes = w.P * 2 * w.T * w.H  # bf16 slabs read by the first stage
    step_in = in_bytes + 2 * w.T * w.H  # + the residual
    # Workloads whose inputs fit in L2: k pipelines over copies of the inputs,
    # used in turn, so that every timed step reads cold inputs (together they
    # exceed twice L2; at most 64 copies, beyond which the inputs stay warm).
    sets_needed = 1 if step_in >= 2 * L2_BYTES else -(-2 * L2_BYTES // step_in) + 1
    n_sets = min(sets_needed, 64)
    pipes = [pipe] + [Pipeline(w, inputs, device=dev, split=args.split) for _ in range(n_sets - 1)]

    st = torch.cuda.current_stream(dev)
    if args.graph:
        for p in pipes:
            p.capture()
    runs = [(p.replay if args.graph else p.step) for p in pipes]
    for i in range(max(args.warmup, n_sets)):
        runs[i % n_sets](st)
    torch.cuda.synchronize(dev)

    # timed region 1, the step: one pair of events around all K steps
    # (consecutive kernels may overlap their launch with the previous
    # kernel's tail, as in a stream of layers); then one pair per step for
    # the spread; then, region 2, events around each stage of each step.
    n = args.steps
    hold = HOLD_CYCLES + 40_000 * min(n, 200)  # covers the host's issue time of the steps
    barrier(ws)
    torch.cuda.synchronize(dev)
    sampler = ClockSampler(dev.index)
    with sampler:
        t_wall = time.perf_counter()
        torch.cuda._sleep(hold)  # the host queues ahead of the first timed step
        host_s = 0.0  # host time spent issuing the steps
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with nvtx(f"{w.name}: {n} timed steps"):
            e0.record(st)
            for i in range(n):
                t0 = time.perf_counter()
                runs[i % n_sets](st)
                host_s += time.perf_counter() - t0
            e1.record(st)
            torch.cuda.synchronize(dev)
        step_ms = e0.elapsed_time(e1) / n
        t_wall = time.perf_counter() - t_wall
        evs = [[torch.cuda.Event(enable_timing=True) for _ in range(2)] for _ in range(n)]
        torch.cuda._sleep(hold)
        with nvtx(f"{w.name}: per-step events"):
            for i in range(n):
                evs[i][0].record(st)
                runs[i % n_sets](st)
                evs[i][1].record(st)
            torch.cuda.synchronize(dev)
        per_step = [a.elapsed_time(b) for a, b in evs]
        ev = [[torch.cuda.Event(enable_timing=True) for _ in range(3)] for _ in range(n)]
        torch.cuda._sleep(hold)
        with nvtx(f"{w.name}: stage pass"):
            for i in range(n):
                pipes[i % n_sets].step_marked(st, ev[i])
            torch.cuda.synchronize(dev)
    barrier(ws)
    sender_ms = [e[0].elapsed_time(e[1]) for e in ev]
    fused_ms = [e[1].elapsed_time(e[2]) for e in ev]
    step_ms = allreduce_max(step_ms, ws, dev)

    value = whole_job_gbs(step_bytes, ws, step_ms)
    peak, peak_kind = peaks()
    kern = [("sender", "k_quantize" if w.fmt in synth.QUANTIZED else "k_pack_tagged", alg["sender"],
             statistics.mean(sender_ms), spread(sender_ms)),
            ("fused", "k_fused_tagged" if w.fmt == 3 else "k_fused", alg["fused"],
             statistics.mean(fused_ms), spread(fused_ms))]
    dom = max(kern, key=lambda k: k[3])
    achieved = dom[2] / (dom[3] * 1e-3) / 1e9
    out = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": ws,
        "steps": n, "warmup": args.warmup, "ms_per_step": round(step_ms, 5),
        "step_ms_spread": dict(zip(("median", "p10", "p90"), (round(v, 5) for v in spread(per_step))),
                               timing="one pair of CUDA events per step, back to back"),
        "us_per_call": round(statistics.mean(fused_ms) * 1e3, 2),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32", "data": "synthetic",
        "config": {**workload_config(w),
                   **({"split": args.split, "split_rows": pipe.bounds, "wave_rows": pipe.wave_rows}
                      if w.splits > 1 else {}),
                   "l2": (f"inputs larger than L2 ({in_bytes / 2**20:.0f} MB of bf16 slabs "
                          f"read per step vs 129 MB L2)" if n_sets == 1 else
                          f"{n_sets} copies of the inputs used in turn ({n_sets * step_in / 2**20:.0f} MB"
                          + (" > twice L2: every step reads cold inputs)" if n_sets == sets_needed else
                             ", which stay in L2: warm inputs)")),
                   "alg_bytes_per_step": step_bytes},
        "roofline": {"bound": "hbm", "kernel": dom[1], "achieved": round(achieved, 1),
                     "peak": peak, "peak_kind": peak_kind, "unit": "GB/s",
                     "frac": round(achieved / peak, 4),
                     "frac_of_nominal": round(achieved / NOMINAL_HBM_GBS, 4),
                     "nominal_peak": NOMINAL_HBM_GBS,
                     "traffic": measured_traffic(dom[1], w.name),
                     "alg_bytes_per_launch": dom[2]},
        "stages": {k[0]: {"kernel": k[1], "alg_bytes": k[2], "us": round(k[3] * 1e3, 2),
                          "us_median_p10_p90": [round(v * 1e3, 2) for v in k[4]],
                          "GB/s": round(k[2] / (k[3] * 1e-3) / 1e9, 1),
                          "frac": round(k[2] / (k[3] * 1e-3) / 1e9 / peak, 4)} for k in kern},
        "host_us_per_step": round(host_s / n * 1e6, 2),
        "issue": "one CUDA graph replay per step" if args.graph else "launches per step through bound calls",
        "gpu_launches": n * pipe.launches_per_step,
        "stage_pass": {"steps": n, "gpu_launches": n * pipe.launches_per_step,
                       "timing": "second timed pass of the same steps with CUDA events around each "
                                 "stage; gives stages and roofline"},
        "clocks": sampler.report(),
        "timed_wall_s": round(t_wall, 4),
    }
    if not args.no_e2e:
        out["e2e"] = run_e2e(pipe, inputs, step_bytes, args, ws, dev)
    if ws == 1 and rank == 0 and not args.no_cpu_baseline:
        n = host_cores()
        gbs, dt, rows, passes = oracle_sample(w, inputs, args.cpu_seconds / 2, threads=n)
        gbs1, dt1, rows1, passes1 = oracle_sample(w, inputs, args.cpu_seconds / 2)
        out["cpu_baseline"] = {"value": round(gbs, 4), "unit": UNIT, "cores": n,
                               "kind": "oracle",
                               "sample": f"first {rows} of {w.T} rows of the same inputs"
                                         + (f" ({passes} passes over them)" if passes > 1 else "")
                                         + f" in {n} contiguous row ranges on {n} host threads, "
                                           f"{dt:.1f} s",
                               "single_core": {"value": round(gbs1, 4), "cores": 1,
                                               "sample": f"first {rows1} rows"
                                                         + (f", {passes1} passes" if passes1 > 1 else "")
                                                         + f", {dt1:.1f} s"}}
    if rank == 0:
        print(json.dumps(out), flush=True)
    if ws > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


def run_e2e(pipe, inputs, step_bytes, args, ws, dev):
    """The same metric through the public API with host buffers: every step
    copies its inputs from pinned host memory and reads y and residual_out
    back, all inside the timed region.  Steps are pipelined as a serving loop
    would run them: two device buffer sets, the uploads on one stream, the
    step on a second and the downloads on a third, so step i+1's upload
    overlaps step i's compute and download (measured on GB300: the upload,
    at ~190 GB/s from pinned memory, bounds the step; a second upload stream
    gains nothing)."""
    import torch
    from quantized_reduce_rmsnorm_gb300.pipeline import Pipeline
    w = pipe.w
    pin = lambda a: torch.from_numpy(np.ascontiguousarray(a).view(np.int16)).view(
        torch.bfloat16).reshape(a.shape).pin_memory()
    h_slabs = [pin(s) for s in inputs["slabs"]]
    h_res, h_gam = pin(inputs["residual"]), pin(inputs["gamma"])
    h_y = torch.empty(pipe.y.shape, dtype=torch.bfloat16).pin_memory()
    h_h = torch.empty(pipe.y.shape, dtype=torch.bfloat16).pin_memory()
    h2d = sum(t.numel() * 2 for t in h_slabs) + h_res.numel() * 2 + h_gam.numel() * 2
    d2h = 2 * h_y.numel() * 2
    sets = [pipe, Pipeline(w, inputs, device=dev, split=args.split)]
    s_up, s_cp, s_dn = (torch.cuda.Stream(dev) for _ in range(3))
    up_done, comp_done, down_done = ([torch.cuda.Event() for _ in range(2)] for _ in range(3))
    for ev in comp_done + down_done:
        ev.record(torch.cuda.current_stream(dev))

    def one(i):
        k = i & 1
        p = sets[k]
        s_up.wait_event(comp_done[k])  # the set's previous step has read its inputs
        with torch.cuda.stream(s_up):
            for d, h in zip(p.x, h_slabs):
                d.copy_(h, non_blocking=True)
            p.residual.copy_(h_res, non_blocking=True)
            p.gamma.copy_(h_gam, non_blocking=True)
        up_done[k].record(s_up)
        s_cp.wait_event(up_done[k])
        s_cp.wait_event(down_done[k])  # the set's previous outputs are read back
        p.step(s_cp)
        comp_done[k].record(s_cp)
        s_dn.wait_event(comp_done[k])
        with torch.cuda.stream(s_dn):
            h_y.copy_(p.y, non_blocking=True)
            h_h.copy_(p.residual_out, non_blocking=True)
        down_done[k].record(s_dn)

    steps = max(3, min(args.steps, 20))
    warm = max(2, min(3, args.warmup))
    for i in range(warm):
        one(i)
    torch.cuda.synchronize(dev)
    barrier(ws)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with nvtx("e2e: timed steps with host copies"):
        e0.record(s_up)
        for i in range(steps):
            one(warm + i)
        e1.record(s_dn)
        torch.cuda.synchronize(dev)
    ms = allreduce_max(e0.elapsed_time(e1) / steps, ws, dev)
    return {"value": round(whole_job_gbs(step_bytes, ws, ms), 2), "unit": UNIT,
            "ms_per_step": round(ms, 4), "steps": steps, "h2d_bytes_per_step": h2d,
            "d2h_bytes_per_step": d2h,
            "pipelining": "two device buffer sets; upload, step and download on three streams"}


def whole_job_gbs(bytes_per_rank_step: int, ws: int, max_step_ms: float) -> float:
    """Weak scaling: every rank moves bytes_per_rank_step per step; the job's
    throughput is all ranks' bytes over the slowest rank's step time."""
    return ws * bytes_per_rank_step / (max_step_ms * 1e-3) / 1e9


def barrier(ws):
    if ws > 1:
        import torch.distributed as dist
        dist.barrier()


def allreduce_max(v, ws, dev):
    if ws == 1:
        return v
    import torch
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device=dev)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def parse_size(t: str) -> int:
    t = t.strip().upper()
    mult = {"K": 1 << 10, "M": 1 << 20, "G": 1 << 30}
    return int(t[:-1]) * mult[t[-1]] if t[-1] in mult else int(t)


def sweep_selection(args):
    """The sweep points to run: every point, the quick subset, or those
    matching --sizes / --only (MSG:H:P:FMT, FMT one of bf16, int8, int4)."""
    from quantized_reduce_rmsnorm_gb300 import synth
    pts = synth.sweep_points(synth.SWEEP_FORMATS + synth.SWEEP_TAGGED_FORMATS)
    if args.sweep == "quick":
        pts = [p for p in pts if p[0] in (16 << 10, 1 << 20, 16 << 20, 64 << 20, 256 << 20)]
    if args.sizes:
        keep = {parse_size(t) for t in args.sizes.split(",")}
        pts = [p for p in pts if p[0] in keep]
    names = {"bf16": synth.FMT_BF16, "int8": synth.FMT_INT8_SYM, "int4": synth.FMT_INT4_ASYM,
             "bf16t": synth.FMT_BF16_TAGGED, "int8t": synth.FMT_INT8_TAGGED,
             "int4t": synth.FMT_INT4_TAGGED}
    keep = {names[f] for f in (args.formats or "bf16,int8,int4").split(",")}
    pts = [p for p in pts if p[4] in keep]
    if args.only:
        want = set()
        for item in args.only.split(","):
            m, h, p, f = item.split(":")
            want.add((parse_size(m), int(h), int(p), names[f]))
        pts = [p for p in pts if (p[0], p[1], p[3], p[4]) in want]
    return pts


def measure_point(msg, H, T, P, fmt, G, calls=50, reps=7, flush=None, gen=None, held=True):
    """Steady (and held) device time of the fused call and the sender call of
    one sweep shape on seeded N(0,1) inputs generated on the device: see
    run_sweep.  Returns a dict of the sweep's JSON fields."""
    import torch
    from quantized_reduce_rmsnorm_gb300 import fcomm, synth
    from quantized_reduce_rmsnorm_gb300.pipeline import qs_bytes
    dev = torch.device("cuda", torch.cuda.current_device())
    peak, kind = peaks()
    if gen is None:
        gen = torch.Generator(device=dev)
    gen.manual_seed(msg ^ (H << 8) ^ (P << 4) ^ fmt)
    w = synth.sweep_workload(H, T, P, fmt, G)
    spec = fcomm.QSpec(fmt, G)
    xs = [torch.randn(T, H, generator=gen, device=dev).to(torch.bfloat16) for _ in range(P)]
    res = torch.randn(T, H, generator=gen, device=dev).to(torch.bfloat16)
    gam = (1 + 0.1 * torch.randn(H, generator=gen, device=dev)).to(torch.bfloat16)
    E = T * H
    quant = fmt in (synth.FMT_INT8_SYM, synth.FMT_INT4_ASYM)
    qtag = fmt in synth.QTAGGED
    btag = fmt == synth.FMT_BF16_TAGGED
    if quant or qtag:
        qs = qs_bytes(w, E)
        wire = fcomm.codes_bytes(spec, T, H) if qtag else qs  # one slab's payload
        sender_bytes = P * 2 * E + P * wire
        fused_bytes = P * wire + 2 * E + 2 * H + qs + 4 * E
        fused_in = P * wire + 2 * E
    elif btag:
        wire = fcomm.tagged_bytes(T, H)
        sender_bytes = P * 2 * E + P * wire
        fused_bytes = P * wire + 2 * E + 2 * H + 4 * E
        fused_in = P * wire + 2 * E
    else:
        sender_bytes = 0
        fused_bytes = P * 2 * E + 2 * E + 2 * H + 4 * E
        fused_in = P * 2 * E + 2 * E
    epoch = 1  # every call packs and expects the same epoch (timing only)

    def make_set(xset):
        """One set of buffers for a sender call and a fused call."""
        r_out, y = torch.empty_like(res), torch.empty_like(res)
        if quant:
            codes = [fcomm.alloc_qtensor(spec, T, H, dev) for _ in range(P)]
            payload = fcomm.alloc_qtensor(spec, T, H, dev)
            send = fcomm.bind_group_quantize_multi(xset, spec, codes)
            send()
            fuse = fcomm.bind_allreduce_residual_rmsnorm(codes, spec, T, H, res.clone(), r_out,
                                                         gam, 1e-5, y, requant_out=payload)
            return send, fuse
        if qtag or btag:
            nb = fcomm.codes_bytes(spec, T, H) if qtag else fcomm.tagged_bytes(T, H)
            blocks = [torch.empty(nb, dtype=torch.uint8, device=dev) for _ in range(P)]
            st = torch.zeros(2, dtype=torch.int32, device=dev)
            send = (fcomm.bind_group_quantize_tagged(xset, spec, epoch, blocks) if qtag
                    else fcomm.bind_pack_tagged_multi(xset, epoch, blocks))
            send()
            payload = fcomm.alloc_qtensor(fcomm.QSpec(synth.base_format(fmt), G), T, H, dev) \
                if qtag else None
            fuse = fcomm.bind_allreduce_residual_rmsnorm(blocks, spec, T, H, res.clone(), r_out,
                                                         gam, 1e-5, y, requant_out=payload,
                                                         expected_epoch=epoch, d_status=st)
            return send, fuse
        return None, fcomm.bind_allreduce_residual_rmsnorm(xset, spec, T, H, res.clone(), r_out,
                                                           gam, 1e-5, y)

    fits = fused_in + 4 * E < 2 * L2_BYTES
    k = 1 if fused_in >= 2 * L2_BYTES else -(-2 * L2_BYTES // fused_in) + 1
    cold = k <= 64
    k = min(k, 64)
    sets = [make_set(xs)] + [make_set([x.clone() for x in xs]) for _ in range(k - 1)]
    send, fuse = sets[0]
    calls = max(calls, k)
    fm, fp10, fp90 = stream_timed([f for _, f in sets], calls, reps)
    gb = lambda nbytes, us: nbytes / us / 1e3
    line = {"sweep": True, "message_bytes": msg, "hidden": H, "tokens": T, "P": P,
            "format": synth.FMT_NAMES[fmt],
            "fused_us": round(fm, 3), "fused_us_p10": round(fp10, 3), "fused_us_p90": round(fp90, 3),
            "fused_GBps": round(gb(fused_bytes, fm), 1),
            "fused_frac": round(gb(fused_bytes, fm) / peak, 4),
            "fused_frac_nominal": round(gb(fused_bytes, fm) / NOMINAL_HBM_GBS, 4),
            "sets": k, "calls_per_rep": calls, "reps": reps, "inputs_cold": cold,
            "peak_kind": kind}
    if held:
        hu, fh, _ = device_timed(fuse, reps, scrub=flush if fits else None)
        line.update(fused_held_us=round(hu, 2), fused_held_frac=round(gb(fused_bytes, hu) / peak, 4),
                    fused_host_us=round(fh, 2),
                    held_scrub="read-only" if fits else "none (inputs larger than L2)")
    if sender_bytes:
        sm, sp10, sp90 = stream_timed([s for s, _ in sets], calls, reps)
        line.update(sender_us=round(sm, 3), sender_us_p10=round(sp10, 3),
                    sender_us_p90=round(sp90, 3),
                    sender_GBps=round(gb(sender_bytes, sm), 1),
                    sender_frac=round(gb(sender_bytes, sm) / peak, 4),
                    sender_frac_nominal=round(gb(sender_bytes, sm) / NOMINAL_HBM_GBS, 4))
        if held:
            line.update(sender_held_us=round(device_timed(send, reps, scrub=flush if fits else None)[0], 2))
    del xs, res, gam, send, fuse, sets
    torch.cuda.empty_cache()
    return line


def run_sweep(args):
    """Message-size sweep of the fused kernel (and the sender).

    Inputs are seeded N(0,1) bf16 generated on the device (a measurement,
    not a parity case); the calls are bound once (fcomm.Bound).  Each point
    is timed two ways:

    * steady (the reported figure): `--calls` calls (at least 50) back to
      back between one pair of CUDA events, cycling through k buffer sets
      whose inputs together exceed twice L2 (so every call reads cold
      inputs and meets its predecessor's dirty outputs, as in a stream of
      all-reduce calls); k is capped at 64 for the smallest messages, whose
      inputs then stay in L2 ("inputs_cold": false).  Median, p10 and p90
      over the repetitions.
    * held: one call per event pair after a read-only L2 scrub (cold
      inputs, clean L2), median of the repetitions; the event clock's tick
      (about 2 us) bounds its resolution.

    The host's cost of issuing one call is reported beside them."""
    import torch
    from quantized_reduce_rmsnorm_gb300 import fcomm
    fcomm.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    gen = torch.Generator(device=dev)
    for msg, H, T, P, fmt, G in sweep_selection(args):
        if T == 0:
            continue
        line = measure_point(msg, H, T, P, fmt, G, calls=args.calls, flush=flush, gen=gen)
        print(json.dumps(line), flush=True)


SELECTOR_POINTS = [  # (rows, hidden, P): on and off the measured grid of sizes, P and hidden
    (64, 8192, 4), (192, 8192, 4), (1024, 8192, 4), (3072, 8192, 4), (6144, 8192, 4),
    (64, 8192, 8), (768, 8192, 8), (4096, 8192, 8), (256, 4096, 2), (2048, 4096, 2),
    (512, 8192, 3), (2048, 8192, 6), (1024, 5120, 8), (8192, 5120, 4), (16384, 8192, 2),
]


def selector_check(points, calls=50, reps=5):
    """For each (rows, hidden, P): every encoding's measured step (sender +
    fused steady device time, as in the sweep) beside the protocol
    selector's estimate for one GPU, the selector's pick and the measured
    fastest.  Returns one dict per point."""
    import torch
    from quantized_reduce_rmsnorm_gb300 import fcomm, synth
    fcomm.load()
    gen = torch.Generator(device=torch.device("cuda", torch.cuda.current_device()))
    encs = synth.SWEEP_FORMATS + synth.SWEEP_TAGGED_FORMATS
    out = []
    for rows, H, P in points:
        meas, est = {}, {}
        for fmt, G in encs:
            r = measure_point(2 * rows * H, H, rows, P, fmt, G, calls=calls, reps=reps, gen=gen,
                              held=False)
            name = synth.FMT_NAMES[fmt]
            meas[name] = r["fused_us"] + (r.get("sender_us") or 0.0)
            est[name] = fcomm.protocol_estimate(rows, H, P, fcomm.QSpec(fmt, G))
        pick, pick_est = fcomm.select_protocol(rows, H, P, 4)
        pick_name = synth.FMT_NAMES[pick.fmt]
        fastest = min(meas, key=meas.get)
        out.append({"selector": True, "rows": rows, "hidden": H, "P": P,
                    "message_bytes": 2 * rows * H,
                    "measured_us": {k: round(v, 2) for k, v in meas.items()},
                    "estimate_us": {k: round(v, 2) for k, v in est.items()},
                    "est_error": {k: round(est[k] / meas[k] - 1, 3) for k in meas},
                    "pick": pick_name, "fastest": fastest,
                    "pick_over_fastest": round(meas[pick_name] / meas[fastest], 4)})
    return out


def run_split_table(args):
    """bench.py --split-table: two token subsets on two streams at the even
    boundary and at the wave-aware one (fc_token_split), on row counts around
    multiples of the fused kernel's wave, for a tagged and two quantized
    workloads; steady device time per step (each subset's fused call on its
    own stream, the sender before them), 20 steps per pair of events."""
    import torch
    from quantized_reduce_rmsnorm_gb300 import fcomm, synth
    from quantized_reduce_rmsnorm_gb300.pipeline import Pipeline
    fcomm.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    cases = [synth.Workload("split-bf16-tagged", P=8, T=0, H=5120, fmt=synth.FMT_BF16_TAGGED, group=0,
                            splits=2),
             synth.Workload("split-int8", P=8, T=0, H=8192, fmt=synth.FMT_INT8_SYM, group=128, splits=2),
             synth.Workload("split-int4", P=4, T=0, H=8192, fmt=synth.FMT_INT4_ASYM, group=32, splits=2)]
    for base in cases:
        _, wave = fcomm.token_split(fcomm.QSpec(base.fmt, base.group), base.P, 4096, base.H)
        for T in (2 * wave - wave // 4, 2 * wave + 16, 2 * wave + wave // 4, 2 * wave + wave // 2,
                  3 * wave + wave // 3):
            w = synth.Workload(**{**base.__dict__, "T": int(T)})
            inp = synth.make_inputs(w, seed=5)
            res = {}
            for mode in ("even", "wave"):
                pipe = Pipeline(w, inp, device=dev, split=mode)
                m, p10, p90 = stream_timed([pipe.step], 20, 5)
                res[mode] = (m, p10, p90, pipe.bounds)
                del pipe
            print(json.dumps({"split_table": True, "workload": w.name, "P": w.P, "tokens": w.T,
                              "hidden": w.H, "wave_rows": wave,
                              "even_us": round(res["even"][0], 2), "even_bounds": res["even"][3],
                              "wave_us": round(res["wave"][0], 2), "wave_bounds": res["wave"][3],
                              "wave_over_even": round(res["wave"][0] / res["even"][0], 4),
                              "p10_p90_even": [round(v, 2) for v in res["even"][1:3]],
                              "p10_p90_wave": [round(v, 2) for v in res["wave"][1:3]]}), flush=True)
            torch.cuda.empty_cache()


def run_selector(args):
    """bench.py --selector: the protocol selector against measurements (one GPU)."""
    import torch
    torch.cuda.set_device(0)
    for line in selector_check(SELECTOR_POINTS, calls=args.calls):
        print(json.dumps(line), flush=True)


def sweep_report(path):
    """Markdown table of the sweep's JSON lines (bench.py --sweep ... > path)."""
    rows = [json.loads(l) for l in open(path) if l.startswith("{") and '"sweep"' in l]
    peak, kind = peaks()
    print("| message | H | tokens | P | format | fused us (p10-p90) | fused frac | of 8 TB/s "
          "| held us | sets | cold | sender us (p10-p90) | sender frac |")
    print("|---|---|---|---|---|---|---|---|---|---|---|---|---|")
    for r in rows:
        snd = (f"{r['sender_us']:.2f} ({r['sender_us_p10']:.2f}-{r['sender_us_p90']:.2f})"
               if r.get("sender_us") is not None else "-")
        sf = f"{r['sender_frac']:.3f}" if r.get("sender_frac") is not None else "-"
        print(f"| {r['message_bytes']} | {r['hidden']} | {r['tokens']} | {r['P']} | {r['format']} "
              f"| {r['fused_us']:.2f} ({r['fused_us_p10']:.2f}-{r['fused_us_p90']:.2f}) "
              f"| {r['fused_frac']:.3f} | {r['fused_frac_nominal']:.3f} | {r['fused_held_us']:.2f} "
              f"| {r['sets']} | {'yes' if r['inputs_cold'] else 'no'} | {snd} | {sf} |")
    print()
    for fmt in ("bf16", "int8_sym_g128", "int4_asym_g32", "bf16_tagged", "int8_sym_g128_tagged",
                "int4_asym_g32_tagged"):
        for lo, label in ((16 << 20, "16 MB and more"), (64 << 20, "64 MB and more")):
            sel = [r for r in rows if r["format"] == fmt and r["message_bytes"] >= lo]
            if not sel:
                continue
            f = sorted(r["fused_frac"] for r in sel)
            below = [r for r in sel if r["fused_frac"] < 0.70]
            print(f"* {fmt}, messages of {label}: fused fraction of the {kind} peak min / median / max "
                  f"{f[0]:.3f} / {statistics.median(f):.3f} / {f[-1]:.3f}; "
                  f"{len(below)} of {len(sel)} points below 0.70"
                  + ("" if not below else " (" + ", ".join(
                      f"{r['message_bytes'] >> 20} MB H={r['hidden']} P={r['P']}: {r['fused_frac']:.3f}"
                      for r in below) + ")"))


def run_gather(args):
    """The standalone quantized all-gather (fc_allgather_dequant): P shard
    payloads of a prefill-sized and a decode-sized tensor (quantized on the
    device from seeded N(0,1) bf16), gathered and dequantized to bf16 and to
    fp32.  Timed as the sweep times the fused call: `--calls` bound calls
    back to back per pair of CUDA events, cycling through buffer sets whose
    payloads and outputs together exceed twice L2 (at most 64 sets), median
    and p10/p90 over 7 repetitions; plus one held call after a read-only L2
    scrub."""
    import torch
    from quantized_reduce_rmsnorm_gb300 import fcomm, synth
    fcomm.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    peak, kind = peaks()
    flush = torch.empty(2 * L2_BYTES // 4, dtype=torch.float32, device=dev)
    gen = torch.Generator(device=dev)
    for name, T, H, P, spec in (("prefill", 8192, 8192, 4, fcomm.INT4_G32),
                                ("prefill", 8192, 8192, 4, fcomm.INT8_G128),
                                ("decode", 64, 8192, 8, fcomm.INT8_G128)):
        E = T * H
        qs = fcomm.codes_bytes(spec, T, H) + fcomm.groups(spec, T, H) * (8 if spec.fmt == fcomm.FMT_INT4_ASYM else 4)
        for odt, osz in ((torch.bfloat16, 2), (torch.float32, 4)):
            alg = qs + osz * E
            n_sets = max(1, min(64, -(-2 * L2_BYTES // alg) + 1))
            calls, keep = [], []
            for k in range(n_sets):
                gen.manual_seed((T ^ P) + 7919 * k)
                x = torch.randn(T, H, generator=gen, device=dev).to(torch.bfloat16)
                whole = fcomm.alloc_qtensor(spec, T, H, dev)
                fcomm.group_quantize(x, spec, whole)
                del x
                out = torch.empty(T, H, dtype=odt, device=dev)
                calls.append(fcomm.bind_allgather_dequant(fcomm.shard_views(whole, spec, T, H, P),
                                                          spec, T, H, out))
                keep.append(whole)
            med, p10, p90 = stream_timed(calls, max(args.calls, 50), 7)
            held = device_timed(calls[0], 7, warm=2, scrub=flush)[0]
            print(json.dumps({"gather": True, "workload": name, "rows": T, "hidden": H, "P": P,
                              "format": synth.FMT_NAMES[spec.fmt], "out": str(odt).split(".")[-1],
                              "us": round(med, 2), "us_p10": round(p10, 2), "us_p90": round(p90, 2),
                              "held_us": round(held, 2), "sets": n_sets,
                              "inputs_cold": n_sets * alg > 2 * L2_BYTES,
                              "alg_bytes": alg, "GB/s": round(alg / med / 1e3, 1),
                              "frac": round(alg / med / 1e3 / peak, 4),
                              "frac_nominal": round(alg / med / 1e3 / NOMINAL_HBM_GBS, 4),
                              "peak_kind": kind}), flush=True)
            del calls, keep
            torch.cuda.empty_cache()


def run_overlap(args):
    """The fused reduce + residual + RMSNorm with its grid capped at max_ctas
    CTAs (one per SM), alone and concurrently with a bf16 GEMM standing in for
    the other token subset's compute (TokenWeave, abstract: communication and
    RMSNorm on 2-8 SMs, overlapped with the other subset's computation)."""
    import torch
    from quantized_reduce_rmsnorm_gb300 import fcomm, synth
    from quantized_reduce_rmsnorm_gb300.pipeline import Pipeline
    fcomm.load()
    dev = torch.device("cuda", 0)
    torch.cuda.set_device(dev)
    base = synth.WORKLOADS[args.workload]
    w = synth.Workload(**{**base.__dict__, "T": base.T // max(1, base.splits), "splits": 1})
    pipe = Pipeline(w, synth.make_inputs(w, seed=0), device=dev)
    pipe.sender(torch.cuda.current_stream(dev))
    g = torch.Generator(device=dev)
    g.manual_seed(0)
    A = torch.randn(4096, 8192, generator=g, device=dev).to(torch.bfloat16)
    B = torch.randn(8192, 8192, generator=g, device=dev).to(torch.bfloat16)
    C = torch.empty(4096, 8192, dtype=torch.bfloat16, device=dev)
    s_ar, s_mm = torch.cuda.Stream(dev), torch.cuda.Stream(dev)

    def fused(cap, st):
        fcomm.allreduce_residual_rmsnorm(
            pipe.blocks if w.fmt == synth.FMT_BF16_TAGGED else (pipe.codes if pipe.payload is not None else pipe.x),
            pipe.spec, w.T, w.H, pipe.residual, pipe.residual_out, pipe.gamma, w.eps, pipe.y,
            requant_out=pipe.payload, expected_epoch=pipe.epoch,
            d_status=pipe.status[0] if pipe.status is not None else None, max_ctas=cap, stream=st)

    def gemm(st):
        with torch.cuda.stream(st):
            torch.matmul(A, B, out=C)

    def timed(fn, reps=10):
        return device_timed(fn, reps, warm=3)[0]

    def both(cap):
        cur = torch.cuda.current_stream(dev)
        ev0 = torch.cuda.Event()
        ev0.record(cur)
        s_ar.wait_event(ev0), s_mm.wait_event(ev0)
        e_ar0, e_ar1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e_ar0.record(s_ar)
        fused(cap, s_ar)
        e_ar1.record(s_ar)
        gemm(s_mm)
        cur.wait_stream(s_ar), cur.wait_stream(s_mm)
        both.last_ar = e_ar1, e_ar0

    t_mm = timed(lambda: gemm(torch.cuda.current_stream(dev)))
    peak, _ = peaks()
    alg = pipe.alg_bytes()["fused"]
    for cap in (2, 4, 8, 16, 32, 64, 0):
        t_ar = timed(lambda: fused(cap, torch.cuda.current_stream(dev)))
        t_both = timed(lambda: both(cap))
        e1, e0 = both.last_ar
        t_ar_conc = e0.elapsed_time(e1) * 1e3
        hidden = (t_ar + t_mm - t_both) / min(t_ar, t_mm)
        print(json.dumps({"overlap": True, "workload": f"{w.name} subset {w.T}x{w.H} P={w.P}",
                          "max_ctas": cap or "all", "fused_alone_us": round(t_ar, 1),
                          "fused_alone_GBps": round(alg / t_ar / 1e3, 1),
                          "gemm_alone_us": round(t_mm, 1), "both_us": round(t_both, 1),
                          "fused_during_gemm_us": round(t_ar_conc, 1),
                          "overlap_of_shorter": round(hidden, 3)}), flush=True)


def main():
    args = parse()
    if args.report_sweep:
        sweep_report(args.report_sweep)
        return
    if args.selector:
        run_selector(args)
        return
    if args.split_table:
        run_split_table(args)
        return
    if args.gather:
        run_gather(args)
        return
    if args.overlap:
        run_overlap(args)
        return
    if args.sweep:
        run_sweep(args)
        return
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
