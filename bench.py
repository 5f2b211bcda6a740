#!/usr/bin/env python3
"""Benchmark of the fused N-way reduce + residual add + RMSNorm (+ per-token FP8) path.

Metric: microseconds per call under CUDA-graph replay, and the achieved HBM bandwidth of
the fused kernel as a fraction of the measured GB300 copy bandwidth.

Headline workload: the largest single-GPU configuration, N=8 bf16 partials of 4096 x 6144
(48 MiB each), residual in/out, plain RMSNorm, bf16 output (554 MB moved per call).  The
gemma + per-token FP8 + bf16 mirror call on N=4, 2800 x 6144 (every step of the path in
one call) is timed the same way as a second named entry.  A "step" is one replay of a CUDA
graph holding `calls_per_step` calls that rotate over buffer sets larger than L2 together,
the methodology of the pages' benchmarks (k calls captured per graph, replays timed with
CUDA events).  The JSON line ends with a compact per-configuration summary (every workload
of the five configurations: us/call HBM-cold and L2-warm, GB/s, fraction of peak).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun each rank runs an independent replica on its own GPU (the path has no
exchange between GPUs); rank 0 prints one JSON line.
"""
from __future__ import annotations

import argparse
import ctypes
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

HEADLINE = "n8_m4096_h6144_bf16_plain"
SECOND = "n4_m2800_h6144_bf16_gemma_fp8"
METRIC = "us/call (CUDA-graph replay) and achieved HBM GB/s, fused reduce+RMSNorm"
UNIT = "us/call"
SMI_FIELDS = ("timestamp,index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")


# ---------------------------------------------------------------------------
# ranks (replicas)
# ---------------------------------------------------------------------------

def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def init_dist(world: int, backend: str, timeout_s: float | None = None):
    """Join the replicas' process group.  A bounded timeout (default 600 s, or
    AR_BENCH_PG_TIMEOUT seconds) turns a rank that died or never arrives into an error at the
    next barrier or reduction on the others, instead of a wait of torch's default length."""
    import datetime
    import torch.distributed as dist
    if world > 1 and not dist.is_initialized():
        if timeout_s is None:
            timeout_s = float(os.environ.get("AR_BENCH_PG_TIMEOUT", "600"))
        dist.init_process_group(backend, timeout=datetime.timedelta(seconds=timeout_s))
    return dist


def barrier(world: int):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(value: float, world: int, device=None) -> float:
    """Largest value over all ranks (the slowest replica sets the job's time)."""
    if world == 1:
        return value
    import torch
    import torch.distributed as dist
    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_us_per_call(max_elapsed_ms: float, calls_per_rank: int, world: int) -> float:
    """Whole-job time per call: the slowest rank's elapsed time over all calls of all ranks."""
    return max_elapsed_ms * 1000.0 / (calls_per_rank * world)


# ---------------------------------------------------------------------------
# clocks during the timed region
# ---------------------------------------------------------------------------

class ClockSampler:
    def __init__(self, gpu_index: int, interval_ms: int = 50):
        self.gpu, self.interval, self.proc, self.path = gpu_index, interval_ms, None, None

    def start(self):
        import shutil
        import tempfile
        if not shutil.which("nvidia-smi"):
            return
        fd, self.path = tempfile.mkstemp(prefix="clocks_", suffix=".csv")
        os.close(fd)
        self.proc = subprocess.Popen(
            ["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={SMI_FIELDS}", "--format=csv,noheader,nounits",
             "-lms", str(self.interval)], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)

    def stop(self, t0: float, t1: float):
        if self.proc is None:
            return None
        time.sleep(self.interval / 1000.0 * 2)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 10:
                    continue
                try:
                    ts = time.mktime(time.strptime(parts[0].split(".")[0], "%Y/%m/%d %H:%M:%S"))
                    frac = float("0." + parts[0].split(".")[1]) if "." in parts[0] else 0.0
                    rows.append((ts + frac, float(parts[2]), float(parts[3]), parts[5:]))
                except (ValueError, IndexError):
                    continue
        os.unlink(self.path)
        inside = [r for r in rows if t0 - 0.05 <= r[0] <= t1 + 0.05]
        window = "timed"
        if not inside:
            inside, window = rows, "run (no sample fell inside the timed region)"
        if not inside:
            return None
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in inside for i, v in enumerate(r[3][1:5]) if v.lower() == "active"})
        return {"sm_mhz": statistics.median(r[1] for r in inside), "sm_max_mhz": max(r[2] for r in inside),
                "reasons": reasons, "samples": len(inside), "window": window}


# ---------------------------------------------------------------------------
# our path
# ---------------------------------------------------------------------------

def measured_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            pk = json.load(f)
        return float(pk["hbm_gbs"]), "measured"
    except (OSError, KeyError, ValueError):
        return 6800.0, "fallback"


def _code_only(text: str) -> str:
    """C/CUDA source with comments removed and whitespace collapsed (what the compiler sees)."""
    import re
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", " ", text)
    return " ".join(text.split())


def kernel_source_hash() -> str:
    """Hash of the library's sources, comments and layout left out, so that a recorded DRAM
    traffic figure stays attached to the code it was measured on."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "tensor_all_reduce_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        if f.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, f), encoding="utf-8") as fh:
                h.update(f.encode() + b"\0" + _code_only(fh.read()).encode())
    return h.hexdigest()[:16]


def recorded_traffic(workload: str):
    """DRAM bytes per launch from the committed ncu summary, if taken on the current kernels."""
    path = os.path.join(ROOT, "profiles", "dram_traffic.txt")
    if not os.path.exists(path):
        return None
    cur = kernel_source_hash()
    with open(path) as f:
        for line in f:
            if line.startswith("#") or not line.strip():
                continue
            kv = dict(tok.split("=", 1) for tok in line.split())
            if kv.get("workload") == workload and kv.get("kernel_src") == cur:
                return int(kv["bytes_per_launch"])
    return None


class FusedSets:
    """R buffer sets for one fused workload, carved from one slab per role."""

    def __init__(self, wl, sets: int, dev):
        import torch
        from tensor_all_reduce_gb300 import synth
        self.wl, self.R = wl, sets
        t = synth.TORCH_DTYPES[wl.dtype]
        m, h, n = wl.m, wl.h, wl.n
        inp = wl.inputs()
        hp = h + wl.pad                     # padded rows: [m, h] views of [m, h + pad] buffers
        self.parts = torch.empty((sets, n, m, hp), dtype=t, device=dev)[..., :h]
        self.res = torch.empty((sets, m, hp), dtype=t, device=dev)[..., :h] if wl.residual else None
        self.w = inp["weight"].to(dev)
        want_y = wl.mirror or not wl.quant
        self.out = (torch.empty((sets, m, hp), dtype=torch.float32 if wl.out_fp32 else t, device=dev)[..., :h]
                    if want_y else None)
        self.ro = torch.empty((sets, m, hp), dtype=t, device=dev)[..., :h] if wl.residual else None
        self.q = torch.empty((sets, m, hp), dtype=torch.uint8, device=dev)[..., :h] if wl.quant else None
        ns = m * (h // wl.group) if wl.group else m
        self.sc = torch.empty((sets, ns), dtype=torch.float32, device=dev) if wl.quant else None
        for k in range(n):
            self.parts[:, k].copy_(inp["partials"][k].to(dev).unsqueeze(0).expand(sets, m, h))
        if self.res is not None:
            self.res.copy_(inp["residual"].to(dev).unsqueeze(0).expand(sets, m, h))

    def call(self, ctx, i: int):
        r = i % self.R
        wl = self.wl
        ctx.fused_reduce_rmsnorm(list(self.parts[r].unbind(0)), None if self.res is None else self.res[r], self.w,
                                 eps=1e-6, gemma=wl.gemma, quant=wl.quant,
                                 out=None if self.out is None else self.out[r],
                                 residual_out=None if self.ro is None else self.ro[r],
                                 q_out=None if self.q is None else self.q[r],
                                 scale_out=None if self.sc is None else self.sc[r],
                                 want_out=self.out is not None, want_residual_out=self.ro is not None,
                                 skip_norm=wl.skip_norm, out_fp32=wl.out_fp32, group_size=wl.group)


class BatchSets:
    """`k` independent calls of one fused workload per step, either as one batched launch or
    as k separate launches, rotating over R sets of k buffer sets."""

    def __init__(self, wl, k: int, sets: int, dev, batched: bool):
        self.inner = FusedSets(wl, k * sets, dev)
        self.k, self.R, self.batched = k, sets, batched

    def call(self, ctx, i: int):
        base = (i % self.R) * self.k
        if not self.batched:
            for j in range(self.k):
                self.inner.call(ctx, base + j)
            return
        f, wl = self.inner, self.inner.wl
        calls = []
        for j in range(self.k):
            r = base + j
            calls.append({"partials": list(f.parts[r].unbind(0)), "residual": None if f.res is None else f.res[r],
                          "weight": f.w, "eps": 1e-6, "gemma": wl.gemma, "quant": wl.quant,
                          "out": None if f.out is None else f.out[r], "residual_out": None if f.ro is None else f.ro[r],
                          "q_out": None if f.q is None else f.q[r], "scale_out": None if f.sc is None else f.sc[r]})
        ctx.fused_reduce_rmsnorm_batch(calls)


class ReduceSets:
    def __init__(self, wl, sets: int, dev):
        import torch
        from tensor_all_reduce_gb300 import synth
        self.wl, self.R = wl, sets
        t = synth.TORCH_DTYPES[wl.dtype]
        parts = synth.reduce_inputs(wl.n, wl.numel, wl.dtype, wl.seed)
        self.parts = torch.empty((sets, wl.n, wl.numel), dtype=t, device=dev)
        for k in range(wl.n):
            self.parts[:, k].copy_(parts[k].to(dev).unsqueeze(0).expand(sets, wl.numel))
        self.out = torch.empty((sets, wl.numel), dtype=t, device=dev)

    def call(self, ctx, i: int):
        r = i % self.R
        ctx.reduce_sum(list(self.parts[r].unbind(0)), out=self.out[r])


def rotation_sets(footprint: int, l2: int, cap: int = 4096) -> int:
    """Buffer sets whose total footprint covers L2 three times (HBM-cold replays)."""
    return max(1, min(cap, math.ceil(3 * l2 / max(footprint, 1))))


def time_graph(sets, ctx, calls: int, steps: int, warmup: int, world: int, sampler=None):
    """Capture `calls` calls in one graph; replay `warmup` untimed, then time `steps` replays."""
    import torch
    for i in range(min(calls, sets.R)):
        sets.call(ctx, i)                   # eager warm-up of every buffer set
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(g, stream=s):
        for i in range(calls):
            sets.call(ctx, i)
    torch.cuda.current_stream().wait_stream(s)
    for _ in range(warmup):
        g.replay()
    torch.cuda.synchronize()
    barrier(world)
    torch.cuda.synchronize()
    # one event between consecutive replays: the total and every step's own duration
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(steps + 1)]
    t0 = time.time()
    evs[0].record()
    for i in range(steps):
        g.replay()
        evs[i + 1].record()
    evs[-1].synchronize()
    t1 = time.time()
    torch.cuda.synchronize()
    barrier(world)
    elapsed_ms = evs[0].elapsed_time(evs[-1])
    step_ms = [evs[i].elapsed_time(evs[i + 1]) for i in range(steps)]
    del g
    return elapsed_ms, t0, t1, step_ms


def _host_buffers(wl):
    """Pinned host inputs and outputs of one call of the workload."""
    import torch
    from tensor_all_reduce_gb300 import synth
    inp = wl.inputs()
    t = synth.TORCH_DTYPES[wl.dtype]
    m, h = wl.m, wl.h
    ins = {"partials": [p.pin_memory() for p in inp["partials"]],
           "residual": inp["residual"].pin_memory() if inp["residual"] is not None else None,
           "weight": None if wl.skip_norm else inp["weight"].pin_memory()}
    outs = {"out": torch.empty((m, h), dtype=torch.float32 if wl.out_fp32 else t, pin_memory=True)
            if (wl.mirror or not wl.quant) else None,
            "residual_out": torch.empty((m, h), dtype=t, pin_memory=True) if wl.residual else None,
            "q_out": torch.empty((m, h), dtype=torch.uint8, pin_memory=True) if wl.quant else None,
            "scale_out": torch.empty((m, h // wl.group) if wl.group else (m,), dtype=torch.float32, pin_memory=True)
            if wl.quant else None}
    nbytes = lambda xs: sum(x.numel() * x.element_size() for x in xs if x is not None)
    return ins, outs, nbytes(ins["partials"] + [ins["residual"], ins["weight"]]), nbytes(outs.values())


def _time_steps(step, steps: int):
    import torch
    for _ in range(2):
        step()
    torch.cuda.synchronize()
    start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    start.record()
    for _ in range(steps):
        step()
    end.record()
    end.synchronize()
    return start.elapsed_time(end) * 1000.0 / steps


def e2e_fused(ctx, wl, steps: int, dev):
    """Same metric end to end through the C-ABI call on HOST buffers (ar_fused_reduce_rmsnorm_host):
    the inputs sit in pinned host memory, the kernel reads them across the CPU-GPU link and
    writes every output into pinned host memory, so each step's whole host->device and
    device->host traffic is inside the timed region.  Returns (us per call, bytes in, bytes out)."""
    import torch
    import tensor_all_reduce_gb300 as tar
    from tensor_all_reduce_gb300 import synth
    ins, outs, h2d, d2h = _host_buffers(wl)
    ptr = lambda x: None if x is None else x.data_ptr()
    code = {"bf16": tar.AR_DTYPE_BF16, "fp16": tar.AR_DTYPE_F16}[wl.dtype]
    args = tar.make_fused_args([p.data_ptr() for p in ins["partials"]], ptr(ins["residual"]),
                               ptr(outs["residual_out"]), ptr(ins["weight"]), ptr(outs["out"]), 1e-6, wl.gemma,
                               wl.quant, ptr(outs["q_out"]), ptr(outs["scale_out"]), wl.m, wl.h, code,
                               skip_norm=wl.skip_norm, out_fp32=wl.out_fp32, group_size=wl.group)
    stream = torch.cuda.current_stream().cuda_stream
    us = _time_steps(lambda: tar.ar_fused_reduce_rmsnorm_host(ctx.handle, args, stream), steps)
    return us, h2d, d2h


def e2e_copy_engines(ctx, wl, steps: int, dev):
    """The same call with explicit copies instead: pinned host inputs copied to device buffers,
    the device-memory call, the outputs copied back (for comparison with e2e_fused)."""
    import torch
    ins, outs, _, _ = _host_buffers(wl)
    d_ins = {k: (None if v is None else [p.to(dev) for p in v] if k == "partials" else v.to(dev))
             for k, v in ins.items()}
    d_outs = {k: (None if v is None else torch.empty(v.shape, dtype=v.dtype, device=dev)) for k, v in outs.items()}

    def step():
        for d, hh in zip(d_ins["partials"], ins["partials"]):
            d.copy_(hh, non_blocking=True)
        for k in ("residual", "weight"):
            if ins[k] is not None:
                d_ins[k].copy_(ins[k], non_blocking=True)
        ctx.fused_reduce_rmsnorm(d_ins["partials"], d_ins["residual"], d_ins["weight"], eps=1e-6, gemma=wl.gemma,
                                 quant=wl.quant, want_out=wl.mirror or not wl.quant, want_residual_out=wl.residual,
                                 skip_norm=wl.skip_norm,
                                 out_fp32=wl.out_fp32, group_size=wl.group, **d_outs)
        for k, hh in outs.items():
            if hh is not None:
                hh.copy_(d_outs[k], non_blocking=True)

    return _time_steps(step, steps)


# ---------------------------------------------------------------------------
# the oracle on the host cores (CPU baseline and the reference arm)
# ---------------------------------------------------------------------------

class OracleInputs:
    """A workload's inputs in the oracle's storage convention, drawn once (outside any timing)."""

    def __init__(self, wl):
        from tensor_all_reduce_gb300 import synth
        self.wl = wl
        inp = wl.inputs()
        self.parts = [synth.bits(p) for p in inp["partials"]]
        self.res = synth.bits(inp["residual"]) if inp["residual"] is not None else None
        self.w = None if wl.skip_norm else synth.bits(inp["weight"])

    def call(self, orc, a: int = 0, b: int | None = None):
        """One oracle call on rows [a, b) (the whole call by default)."""
        wl = self.wl
        b = wl.m if b is None else b
        parts = [p[a:b] for p in self.parts]
        res = None if self.res is None else self.res[a:b]
        if wl.skip_norm or wl.out_fp32 or wl.group:
            orc.fused_ex(parts, res, self.w, 1e-6, wl.gemma, wl.quant, wl.dtype, skip_norm=wl.skip_norm,
                         out_fp32=wl.out_fp32, group=wl.group)
        else:
            orc.fused(parts, res, self.w, 1e-6, wl.gemma, wl.quant, wl.dtype)


def timed_oracle_s(inputs, orc, rows: int) -> float:
    """Seconds of one oracle call on the first `rows` rows."""
    t = time.perf_counter()
    inputs.call(orc, 0, rows)
    return time.perf_counter() - t


def cpu_model() -> str:
    """The host CPU as /proc/cpuinfo names it (model name, else implementer and part)."""
    info = {}
    try:
        with open("/proc/cpuinfo") as f:
            for line in f:
                k, _, v = line.partition(":")
                info.setdefault(k.strip(), v.strip())
    except OSError:
        pass
    if info.get("model name"):
        return info["model name"]
    if info.get("CPU part"):
        return f"{os.uname().machine} (implementer {info.get('CPU implementer', '?')}, part {info['CPU part']})"
    return os.uname().machine


def host_cores() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else (os.cpu_count() or 1)


def rows_for_budget(wl, per_call_s: float, calls: int, budget_s: float) -> int:
    """Whole calls when `calls` of them fit in the budget, else the most rows that do."""
    if per_call_s * calls <= budget_s:
        return wl.m
    return max(1, min(wl.m, int(budget_s / calls / (per_call_s / wl.m))))


def oracle_all_cores_us(inputs, orc, runs: int = 3):
    """Whole calls with the rows partitioned over every host core: each thread runs the same
    serial oracle on its own contiguous block of rows (rows are independent; the C call
    releases the GIL).  Returns (us per call, threads)."""
    from concurrent.futures import ThreadPoolExecutor
    cores = host_cores()
    m = inputs.wl.m
    bounds = [m * k // cores for k in range(cores + 1)]

    def block(k):
        if bounds[k + 1] > bounds[k]:
            inputs.call(orc, bounds[k], bounds[k + 1])

    samples = []
    with ThreadPoolExecutor(cores) as ex:
        for _ in range(runs):
            t = time.perf_counter()
            list(ex.map(block, range(cores)))
            samples.append((time.perf_counter() - t) * 1e6)
    return statistics.median(samples), cores


def cpu_baseline(wl, budget_s: float = 30.0, runs: int = 3):
    """The serial oracle (one thread, pinned to one core) on whole calls of the workload,
    median of `runs` (fewer whole calls, or a row sample, if they would exceed the budget);
    beside it the same oracle with the rows partitioned over all host cores."""
    import oracle
    orc = oracle.get()
    inputs = OracleInputs(wl)
    probe_rows = min(wl.m, 16)
    per_call_s = timed_oracle_s(inputs, orc, probe_rows) * wl.m / probe_rows
    runs = max(1, min(runs, int(budget_s / max(per_call_s, 1e-9))))
    rows = rows_for_budget(wl, per_call_s, runs, budget_s)
    pinned = hasattr(os, "sched_setaffinity")
    if pinned:
        cpus = os.sched_getaffinity(0)
        os.sched_setaffinity(0, {min(cpus)})            # this thread only, restored below
    try:
        samples = [timed_oracle_s(inputs, orc, rows) * 1e6 * wl.m / rows for _ in range(runs)]
    finally:
        if pinned:
            os.sched_setaffinity(0, cpus)
    mt_us, cores = oracle_all_cores_us(inputs, orc)
    value = statistics.median(samples)
    fp = wl.algorithmic_bytes()
    what = "whole calls" if rows == wl.m else f"{rows} of {wl.m} rows per run, scaled to a full call"
    return {"value": round(value, 3), "unit": UNIT, "cores": 1, "kind": "oracle", "cpu": cpu_model(),
            "gbs": round(fp / (value * 1e-6) / 1e9, 4),
            "sample": f"serial C oracle, {what}, one thread pinned to one core, median of {runs} runs",
            "all_cores": {"value": round(mt_us, 3), "unit": UNIT, "cores": cores,
                          "gbs": round(fp / (mt_us * 1e-6) / 1e9, 4),
                          "sample": f"the same oracle on whole calls, the rows split in {cores} contiguous blocks "
                                    f"over {cores} threads, median of 3 runs"}}


def workload_config(wl, world: int) -> dict:
    """The `config` object of both arms' JSON lines: what the workload is."""
    fp = wl.algorithmic_bytes()
    cfg = {"workload": wl.name, "n_partials": wl.n, "m": wl.m, "h": wl.h, "dtype": wl.dtype, "gemma": wl.gemma,
           "residual": wl.residual, "fp8_per_token": wl.quant and not wl.group, "bf16_mirror": wl.quant and wl.mirror,
           "bytes_per_call": fp,
           "l2": f"inputs larger than L2 ({fp / 1e6:.0f} MB per call against a 126 MiB L2), buffer sets "
                 f"rotating over at least three times L2",
           "parallelism": "replicas" if world > 1 else "single GPU"}
    return cfg


def run_reference(args, world, rank):
    """The reference arm: the serial oracle (the pages hold no installable code) on the host
    cores, on the same workload, metric and unit.  Each step is one whole call when warm-up and
    steps fit in about two and a half minutes, else the same row sample every step (the value is
    then scaled to a full call); ms_per_step is the time a step actually took."""
    import oracle
    from tensor_all_reduce_gb300 import synth
    if rank != 0:
        return 0
    wl = synth.by_name(args.workload)
    orc = oracle.get()
    inputs = OracleInputs(wl)
    probe_rows = min(wl.m, 16)
    per_call_s = timed_oracle_s(inputs, orc, probe_rows) * wl.m / probe_rows
    rows = rows_for_budget(wl, per_call_s, args.steps + args.warmup, 150.0)
    for _ in range(args.warmup):
        timed_oracle_s(inputs, orc, rows)
    step_s = [timed_oracle_s(inputs, orc, rows) for _ in range(args.steps)]
    value = statistics.median(step_s) * 1e6 * wl.m / rows
    if rows == wl.m:
        sample = f"serial C oracle, one whole call per step, median of {args.steps} steps"
    else:
        sample = (f"serial C oracle on the first {rows} of {wl.m} rows per step, median of {args.steps} steps, "
                  f"scaled to a full call")
    line = {"impl": "reference", "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": args.gpus,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(sum(step_s) / len(step_s) * 1e3, 3),
            "higher_is_better": False, "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype,
            "data": "synthetic", "config": workload_config(wl, world), "rows_per_step": rows,
            "cpu_baseline": {"value": round(value, 3), "unit": UNIT, "cores": 1, "kind": "oracle", "cpu": cpu_model(),
                             "sample": sample},
            "e2e": {"value": round(value, 3), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}
    print(json.dumps(line), flush=True)
    return 0


# ---------------------------------------------------------------------------
# main
# ---------------------------------------------------------------------------

def time_workload(ctx, dev, wl, l2, peak, steps: int = 5, warmup: int = 2):
    """us/call of one workload, HBM-cold (buffer sets rotating over three times L2) and
    L2-warm (the same buffers every call), with GB/s and the fraction of peak."""
    import torch
    from tensor_all_reduce_gb300 import synth
    fused = isinstance(wl, synth.FusedWorkload)
    fp = wl.algorithmic_bytes()
    R = rotation_sets(fp, l2)
    calls = max(64, R)
    sets = (FusedSets if fused else ReduceSets)(wl, R, dev)
    ms, *_ = time_graph(sets, ctx, calls, steps=steps, warmup=warmup, world=1)
    cold = ms * 1000 / (steps * calls)
    variant = ctx.last_variant
    del sets
    torch.cuda.empty_cache()
    sets = (FusedSets if fused else ReduceSets)(wl, 1, dev)
    ms, *_ = time_graph(sets, ctx, 64, steps=steps, warmup=warmup, world=1)
    warm = ms * 1000 / (steps * 64)
    del sets
    torch.cuda.empty_cache()
    gbs = fp / (cold * 1e-6) / 1e9
    return {"workload": wl.name, "variant": variant, "us_per_call_cold": round(cold, 3),
            "us_per_call_l2_warm": round(warm, 3), "bytes_per_call": fp, "gbs_cold": round(gbs, 1),
            "frac_of_peak_cold": round(gbs / peak, 4), "rotation_sets": R}


def config_workloads():
    """Every workload of the five configurations, in order: C1 (N=4, 16 x 6144 plain), C2
    (reduce-only 1023/1024/1025 x 512, fp16 and fp32), C3 (decode 1/16/64/256 x 6144), C4
    (gemma + FP8 + mirror at 1024/2800 x 6144 and 1024 x 7168), C5 (N=8, 4096 x 6144)."""
    from tensor_all_reduce_gb300 import synth
    return ([("C1", w) for w in synth.small_fused()] + [("C2", w) for w in synth.reduce_only()]
            + [("C3", w) for w in synth.decode_sweep()] + [("C4", w) for w in synth.gemma_fp8()]
            + [("C5", w) for w in synth.large_m()])


def configs_summary(ctx, dev, l2, peak):
    """Compact per-configuration table: {"C4 n4_m2800_h6144_bf16_gemma_fp8": [variant, us cold,
    us L2-warm, GB/s cold, fraction of peak cold], ...}."""
    out = {}
    for tag, wl in config_workloads():
        e = time_workload(ctx, dev, wl, l2, peak)
        out[f"{tag} {wl.name}"] = [e["variant"], e["us_per_call_cold"], e["us_per_call_l2_warm"], e["gbs_cold"],
                                   e["frac_of_peak_cold"]]
    return out


def sweep(ctx, dev, l2, peak):
    """The workloads outside the five configurations (wide rows, the further forms of the fused
    call, the large plain sums) and 8 decode calls batched against 8 launches."""
    import torch
    from tensor_all_reduce_gb300 import synth
    out = [time_workload(ctx, dev, wl, l2, peak)
           for wl in synth.wide_rows() + synth.mid_batch() + synth.options() + synth.padded_rows()
           + synth.reduce_large()]
    # 8 independent decode calls (16 x 6144 each): one batched launch against 8 launches
    wl = synth.FusedWorkload("n4_m16_h6144_bf16_decode", 4, 16, 6144, seed=1236)
    k = 8
    R = rotation_sets(k * wl.algorithmic_bytes(), l2, cap=64)
    for batched in (True, False):
        sets = BatchSets(wl, k, R, dev, batched)
        ms, *_ = time_graph(sets, ctx, max(R, 32), steps=5, warmup=2, world=1)
        cold = ms * 1000 / (5 * max(R, 32))
        variant = ctx.last_variant
        del sets
        sets = BatchSets(wl, k, 1, dev, batched)
        ms, *_ = time_graph(sets, ctx, 32, steps=5, warmup=2, world=1)
        warm = ms * 1000 / (5 * 32)
        del sets
        torch.cuda.empty_cache()
        out.append({"workload": f"{k}x_{wl.name}_{'batched' if batched else 'separate'}", "variant": variant,
                    "us_per_call_cold": round(cold, 3), "us_per_call_l2_warm": round(warm, 3),
                    "bytes_per_call": k * wl.algorithmic_bytes(), "unit_note": "one step = 8 calls", "rotation_sets": R})
    return out


def run_env(ctx, dev) -> dict:
    """Facts about the run: the device, the CUDA runtime and driver, the library's hash, the host."""
    import torch
    import tensor_all_reduce_gb300 as tar
    props = torch.cuda.get_device_properties(dev)
    env = {"device": props.name, "sm_count": ctx.info(tar.AR_INFO_SM_COUNT), "l2_bytes": ctx.info(tar.AR_INFO_L2_BYTES),
           "hbm_bytes": props.total_memory, "cc": f"{props.major}.{props.minor}", "torch": torch.__version__,
           "cuda_runtime_torch": torch.version.cuda, "host_cores": host_cores(), "host_cpu": cpu_model()}
    try:
        rt, drv = ctypes.c_int(), ctypes.c_int()
        cudart = ctypes.CDLL("libcudart.so.13") if os.path.exists("/usr/local/cuda/lib64/libcudart.so.13") else None
        if cudart is not None and cudart.cudaRuntimeGetVersion(ctypes.byref(rt)) == 0:
            env["cuda_runtime"] = rt.value
        if cudart is not None and cudart.cudaDriverGetVersion(ctypes.byref(drv)) == 0:
            env["cuda_driver"] = drv.value
    except OSError:
        pass
    try:
        out = subprocess.run(["nvidia-smi", "--query-gpu=driver_version", "--format=csv,noheader", "-i",
                              str(dev.index or 0)], capture_output=True, text=True, timeout=20)
        if out.returncode == 0:
            env["nvidia_driver"] = out.stdout.strip()
    except (OSError, subprocess.TimeoutExpired):
        pass
    with open(tar.LIB_PATH, "rb") as f:
        env["libar_sha256"] = hashlib.sha256(f.read()).hexdigest()
    env["kernel_src_hash"] = kernel_source_hash()
    return env


def timed_headline(ctx, dev, wl, l2, args, world, rank):
    """The CUDA-graph measurement of one workload as the bench line reports it."""
    import torch
    fp = wl.algorithmic_bytes()
    R = max(2, rotation_sets(fp, l2, cap=64))
    calls = max(args.calls_per_step, R)
    sets = FusedSets(wl, R, dev)
    sampler = ClockSampler(dev.index or 0) if rank == 0 else None
    if sampler:
        sampler.start()
    elapsed_ms, t0, t1, step_ms = time_graph(sets, ctx, calls, args.steps, args.warmup, world)
    clocks = sampler.stop(t0, t1) if sampler else None
    variant = ctx.last_variant
    del sets
    torch.cuda.empty_cache()
    return {"elapsed_ms": elapsed_ms, "step_ms": step_ms, "clocks": clocks, "variant": variant, "R": R,
            "calls": calls, "fp": fp}


def run_case(args, dev):
    """--case NAME: `case_calls` eager calls of one named workload (fused or plain reduce) over
    buffer sets rotating across three times L2, timed with CUDA events; prints one JSON line.
    A short, self-contained run for profiling one kernel launch at a time."""
    import torch
    import tensor_all_reduce_gb300 as tar
    from tensor_all_reduce_gb300 import synth
    wl = synth.by_name(args.case)
    if args.case_rows and isinstance(wl, synth.FusedWorkload):   # the same call on fewer rows
        import dataclasses
        wl = dataclasses.replace(wl, m=args.case_rows, name=f"{wl.name} ({args.case_rows} rows)")
    with tar.Context(dev.index or 0) as ctx:
        ctx.set_option(tar.AR_OPT_FORCE_VARIANT, args.force_variant)
        l2 = ctx.info(tar.AR_INFO_L2_BYTES)
        fused = isinstance(wl, synth.FusedWorkload)
        if args.case_batch and fused:       # `case_batch` independent calls of the workload, one launch
            R = rotation_sets(args.case_batch * wl.algorithmic_bytes(), l2, cap=64)
            sets = BatchSets(wl, args.case_batch, R, dev, batched=True)
        else:
            R = rotation_sets(wl.algorithmic_bytes(), l2, cap=64)
            sets = (FusedSets if fused else ReduceSets)(wl, R, dev)
        for i in range(args.warmup):
            sets.call(ctx, i)
        torch.cuda.synchronize()
        start, end = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record()
        for i in range(args.case_calls):
            sets.call(ctx, args.warmup + i)
        end.record()
        end.synchronize()
        us = start.elapsed_time(end) * 1000.0 / max(args.case_calls, 1)
        print(json.dumps({"case": wl.name, "variant": ctx.last_variant, "calls": args.case_calls, "warmup": args.warmup,
                          "batch": args.case_batch, "buffer_sets": R, "us_per_call_eager": round(us, 3),
                          "bytes_per_call": wl.algorithmic_bytes() * max(1, args.case_batch)}), flush=True)
    return 0


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=100)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--workload", default=HEADLINE)
    p.add_argument("--calls-per-step", type=int, default=500)
    p.add_argument("--no-sweep", action="store_true", help="skip the per-configuration summary and the sweep")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--e2e-steps", type=int, default=20)
    p.add_argument("--case", default=None, help="run only `--case-calls` eager calls of this workload")
    p.add_argument("--case-calls", type=int, default=3)
    p.add_argument("--case-rows", type=int, default=0, help="with --case: run the fused workload on this many rows")
    p.add_argument("--case-batch", type=int, default=0,
                   help="with --case: each call is this many independent calls of the workload in one batched launch")
    p.add_argument("--force-variant", type=int, default=0,
                   help="with --case: AR_OPT_FORCE_VARIANT (0 auto, 1 row, 2 cluster, 3 staged, 4 element-wise)")
    args = p.parse_args(argv)
    world, rank, local = dist_env()
    if args.impl == "reference":
        return run_reference(args, world, rank)

    import torch
    import tensor_all_reduce_gb300 as tar
    from tensor_all_reduce_gb300 import synth
    if not torch.cuda.is_available():
        print(json.dumps({"error": "no CUDA device"}))
        return 1
    torch.cuda.set_device(local)
    dev = torch.device("cuda", local)
    if args.case:
        import __graft_entry__
        __graft_entry__.build()
        return run_case(args, dev)
    init_dist(world, "nccl")
    import __graft_entry__
    if rank == 0:
        __graft_entry__.build()
    barrier(world)
    ctx = tar.Context(local)
    l2 = ctx.info(tar.AR_INFO_L2_BYTES)
    peak, peak_kind = measured_peaks()
    wl = synth.by_name(args.workload)

    hl = timed_headline(ctx, dev, wl, l2, args, world, rank)
    fp, calls = hl["fp"], hl["calls"]
    max_ms = max_over_ranks(hl["elapsed_ms"], world, dev)
    launches = args.steps * calls
    value = job_us_per_call(max_ms, launches, world)
    per_launch_us = hl["elapsed_ms"] * 1000.0 / launches    # this rank's average launch duration
    achieved = fp / (per_launch_us * 1e-6) / 1e9

    e2e_us, h2d, d2h = e2e_fused(ctx, wl, args.e2e_steps, dev)
    e2e_us = max_over_ranks(e2e_us, world, dev) / world
    copy_us = e2e_copy_engines(ctx, wl, args.e2e_steps, dev)

    second = None
    if args.workload != SECOND:
        wl2 = synth.by_name(SECOND)
        s2 = timed_headline(ctx, dev, wl2, l2, args, 1, 1)
        us2 = s2["elapsed_ms"] * 1000.0 / (args.steps * s2["calls"])
        gbs2 = s2["fp"] / (us2 * 1e-6) / 1e9
        second = {"workload": wl2.name, "value": round(us2, 3), "unit": UNIT, "variant": s2["variant"],
                  "achieved_gbs": round(gbs2, 1), "frac": round(gbs2 / peak, 4), "bytes_per_call": s2["fp"],
                  "traffic": recorded_traffic(wl2.name), "calls_per_step": s2["calls"], "buffer_sets": s2["R"],
                  "per_step_median": round(statistics.median(s2["step_ms"]) * 1000.0 / s2["calls"], 3)}

    extra = {}
    if rank == 0 and not args.no_sweep:
        extra["sweep"] = sweep(ctx, dev, l2, peak)
        extra["configs"] = configs_summary(ctx, dev, l2, peak)
    cpu = None
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        cpu = cpu_baseline(wl)
    env = run_env(ctx, dev) if rank == 0 else None
    ctx.close()
    if rank == 0:
        step_ms = hl["step_ms"]
        line = {
            "metric": METRIC, "value": round(value, 3), "unit": UNIT, "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": round(max_ms / args.steps, 4), "higher_is_better": False,
            "scaling": "weak", "vs_baseline": None, "dtype": wl.dtype, "data": "synthetic",
            "config": workload_config(wl, world),
            "timing": {"calls_per_step": calls, "buffer_sets": hl["R"], "variant": hl["variant"],
                       "method": "CUDA-graph replays of calls_per_step calls rotating over buffer_sets sets, "
                                 "CUDA events on the replaying stream"},
            "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                         "frac": round(achieved / peak, 4), "traffic": recorded_traffic(wl.name),
                         "peak_kind": peak_kind, "algorithmic_bytes_per_launch": fp},
            "e2e": {"value": round(e2e_us, 3), "unit": UNIT, "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                    "api": "ar_fused_reduce_rmsnorm_host",
                    "note": "one C-ABI call per step on pinned host buffers: the kernel reads the inputs from and "
                            "writes the outputs to host memory across the CPU-GPU link",
                    "copy_engines_us": round(copy_us, 3)},
            "per_step": {"median": round(statistics.median(step_ms) * 1000.0 / calls, 3),
                         "min": round(min(step_ms) * 1000.0 / calls, 3),
                         "max": round(max(step_ms) * 1000.0 / calls, 3), "unit": UNIT,
                         "note": "rank 0's replays one by one (CUDA events between replays)"},
            "gpu_launches": launches,
            "clocks": hl["clocks"],
            "env": env,
        }
        if cpu is not None:
            line["cpu_baseline"] = cpu
        if second is not None:
            line["second"] = second
        if "sweep" in extra:
            line["sweep"] = extra["sweep"]
            line["configs_fields"] = ["variant", "us_cold", "us_l2_warm", "gbs_cold", "frac_of_peak_cold"]
            line["configs"] = extra["configs"]          # last: the end of the line is what a log tail keeps
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()
    return 0


if __name__ == "__main__":
    sys.exit(main())
