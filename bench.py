#!/usr/bin/env python
"""NVFP4 quantize throughput on GB300: GB/s and fraction of the HBM roofline.

Default workload: 2D NVFP4 quantize of an 8192 x 5120 BF16 N(0,1) matrix
(seed 1), row-wise and column-wise outputs, scales in the cuBLAS 128x4
layout.  One step = one full quantize call (amax + fused cast: every row of
the hot path for this workload; for 1D/2D one persistent kernel launch).  Bytes per step = input read once + FP4
codes + E4M3 scales written (3.125 B per element for BF16 row+col).

Timing: W untimed warm-up steps; then K steps, each bracketed by CUDA events
on the launching stream, with a 256 MiB buffer written between steps to
flush the L2 (129 MB) so every step starts with x in HBM; barrier +
synchronize on both sides; the max over ranks is reported.  SM clocks are
sampled with nvidia-smi during the timed region.

--impl reference times the CPU oracle (single-threaded C) on a bounded
sample of the same workload; under torchrun only rank 0 runs it.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import re
import statistics
import subprocess
import sys
import tempfile
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

BYTES_PER_ELEM = {  # algorithmic bytes per element: input once + outputs
    ("bf16", "rowcol"): 2 + 2 * (0.5 + 1 / 16),
    ("fp32", "rowcol"): 4 + 2 * (0.5 + 1 / 16),
    ("bf16", "row"): 2 + 0.5 + 1 / 16,
}
FALLBACK_HBM_GBS = 6800.0


def workload_bytes(spec) -> float:
    import torch
    dt = "bf16" if spec["dtype"] == torch.bfloat16 else "fp32"
    dirs = "row" if spec["mode"] == "row_scaled" else "rowcol"
    extra = 4.0 / spec["N"] if spec["mode"] == "row_scaled" else 0.0   # per-row amax
    return spec["M"] * spec["N"] * (BYTES_PER_ELEM[(dt, dirs)] + extra)


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return FALLBACK_HBM_GBS, "fallback"


def kernel_source_hash(source: str) -> str:
    """Hash of what a kernel is built from: its source file in csrc/, the
    local headers it includes (transitively) and the build script (flags)."""
    pkg = os.path.join(ROOT, "nvfp4_block_scaled_amax_gb300")
    dirs = [os.path.join(pkg, "csrc"), os.path.join(ROOT, "include")]
    seen, todo = {}, [source]
    while todo:
        name = todo.pop()
        if name in seen:
            continue
        path = next((os.path.join(d, name) for d in dirs if os.path.exists(os.path.join(d, name))), None)
        if path is None:
            continue
        with open(path, "rb") as f:
            seen[name] = f.read()
        todo += re.findall(r'#include "([^"]+)"', seen[name].decode())
    h = hashlib.sha256()
    for name in sorted(seen):
        h.update(name.encode() + seen[name])
    with open(os.path.join(pkg, "build.py"), "rb") as f:
        h.update(f.read())
    return h.hexdigest()[:16]


def ncu_traffic(workload: str):
    """DRAM bytes per call from the committed ncu summary, if it was taken on
    the current sources of that kernel (else None)."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    if not os.path.exists(path):
        return None
    with open(path) as f:
        d = json.load(f)
    e = d.get(workload)
    if not e or e.get("kernel_hash") != kernel_source_hash(e.get("source", "")):
        return None
    return e.get("dram_bytes_per_call")


class ClockSampler:
    """nvidia-smi clocks / throttle reasons sampled every 100 ms."""

    FIELDS = "clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,clocks_event_reasons.hw_slowdown," \
             "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown," \
             "clocks_event_reasons.sw_power_cap"

    def __init__(self, gpu_index: int):
        self.path = tempfile.mktemp(suffix=".csv")
        self.gpu = gpu_index
        self.proc = None

    def __enter__(self):
        try:
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", "-i", str(self.gpu), f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "100"],
                                         stdout=self.f, stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        if self.proc is not None:
            time.sleep(0.2)
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        rows = []
        with open(self.path) as f:
            for ln in f:
                p = [v.strip() for v in ln.split(",")]
                if len(p) == 8 and p[0].replace(".", "").isdigit():
                    rows.append(p)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[0]) for r in rows]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[4 + i].lower() == "active"})
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": float(rows[0][1]), "samples": len(rows),
                "power_w_max": max(float(r[2]) for r in rows if r[2].replace(".", "").isdigit()),
                "reasons": reasons}


# ---------------------------------------------------------------------------
# GPU arm
# ---------------------------------------------------------------------------

def run_step_fn(nv, spec, x, q, mask):
    mode = spec["mode"]
    sw = spec["swizzled"]

    def step():
        nv.quantize(x, mode, rowwise=True, colwise=mode != "row_scaled", swizzled=sw, sign_mask=mask, out=q)
    return step


class L2Flush:
    """Between timed steps: write a 256 MiB buffer (twice the 129 MB L2), then
    read another 256 MiB buffer, so the step starts with none of its data in
    L2 and no dirty lines of the flush buffer left to write back during it."""

    def __init__(self, dev):
        import torch
        self.w = torch.empty(256 << 20, dtype=torch.uint8, device=dev)
        self.r = torch.ones(32 << 20, dtype=torch.int64, device=dev)
        self.sink = torch.empty((), dtype=torch.int64, device=dev)

    def __call__(self, k):
        import torch
        self.w.fill_(k & 0xFF)
        torch.sum(self.r, dim=0, out=self.sink)


def time_steps(step, steps, flush, stream):
    """Per-step device time (ms) from CUDA events on the launching stream.
    The flush kernels before each step keep the GPU busy long enough for the
    host to enqueue the step, so the events bracket device work only."""
    import torch
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    # A ~1 ms device-side spin first, so that the host is already several
    # steps ahead when the first timed step starts (otherwise the first
    # step's events can include the host's enqueue time).
    if hasattr(torch.cuda, "_sleep"):
        torch.cuda._sleep(2_000_000)
    for k in range(steps):
        flush(k)
        starts[k].record(stream)
        step()
        ends[k].record(stream)
    torch.cuda.synchronize()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)]


def host_us_per_call(step, n=200):
    """Host-side cost of one call (no synchronization inside)."""
    import torch
    torch.cuda.synchronize()
    t0 = time.perf_counter()
    for _ in range(n):
        step()
    t = time.perf_counter() - t0
    torch.cuda.synchronize()
    return round(1e6 * t / n, 2)


def host_costs(nv, spec, x, q, mask, step, stream):
    """Host microseconds per call, three ways: the Python ``quantize``; a
    ``QuantizePlan`` bound once to the tensors; the C entry point itself,
    called through ctypes with its arguments built once (argument checks,
    tensor-map lookup and the kernel launch)."""
    import ctypes

    from nvfp4_block_scaled_amax_gb300 import _lib
    mode = spec["mode"]
    colwise = mode != "row_scaled"
    plan = nv.QuantizePlan(x, mode, rowwise=True, colwise=colwise, swizzled=spec["swizzled"], sign_mask=mask,
                           out=q)
    sp = stream.cuda_stream
    plan_us = host_us_per_call(lambda: plan(sp))
    L = _lib.load()
    fn, args = plan._fn, plan._args + (ctypes.c_void_p(sp),)
    c_us = host_us_per_call(lambda: fn(*args))
    return {"python_quantize": host_us_per_call(step), "python_plan": plan_us, "c_abi_via_ctypes": c_us}


def steady_state(nv, spec, x_host, dev, stream, steps):
    """The same quantize called back to back with no L2 flush, rotating over
    three input and three output sets (3 x (input + outputs) > the 129 MB
    L2), so each call's reads come from HBM and the previous calls' dirty
    outputs are written back while it runs: ms per call from two events
    around all the calls."""
    import torch
    mode = spec["mode"]
    colwise = mode != "row_scaled"
    mask = 0
    if mode == "rht":
        from nvfp4_block_scaled_amax_gb300 import inputs
        mask = inputs.sign_mask_from_seed(spec["seed"])
    xs = [x_host.to(dev) for _ in range(3)]
    qs = [nv.empty(spec["M"], spec["N"], colwise=colwise, row_scaled=mode == "row_scaled",
                   swizzled=spec["swizzled"], device=dev) for _ in range(3)]
    calls = [(lambda xi=xi, qi=qi: nv.quantize(xi, mode, colwise=colwise, swizzled=spec["swizzled"],
                                               sign_mask=mask, out=qi)) for xi, qi in zip(xs, qs)]
    n = max(30, 3 * steps)
    for k in range(9):
        calls[k % 3]()
    torch.cuda.synchronize()
    if hasattr(torch.cuda, "_sleep"):
        torch.cuda._sleep(2_000_000)
    s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    s.record(stream)
    for k in range(n):
        calls[k % 3]()
    e.record(stream)
    torch.cuda.synchronize()
    ms = s.elapsed_time(e) / n
    gbs = workload_bytes(spec) / (ms / 1e3) / 1e9
    peak, _ = measured_peaks()
    del xs, qs
    torch.cuda.empty_cache()
    return {"ms_per_call": round(ms, 5), "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4), "calls": n,
            "how": "back to back, no flush; 3 input and output sets rotated (more than L2 in all)"}


def bench_ours(args, rank, world, local_rank):
    import torch
    import torch.distributed as dist

    import nvfp4_block_scaled_amax_gb300 as nv
    from nvfp4_block_scaled_amax_gb300 import inputs

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    spec = inputs.WORKLOADS[args.workload]
    M, N = spec["M"], spec["N"]
    mask = inputs.sign_mask_from_seed(spec["seed"]) if spec["mode"] == "rht" else 0
    x_host = inputs.make(spec)
    x = x_host.to(dev)
    q = nv.empty(M, N, rowwise=True, colwise=spec["mode"] != "row_scaled", row_scaled=spec["mode"] == "row_scaled",
                 swizzled=spec["swizzled"], device=dev)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream(dev)
    step = run_step_fn(nv, spec, x, q, mask)
    bytes_step = workload_bytes(spec)

    # warm-up in the timed pattern (flush, events, step): the first flush +
    # step pair of a process runs slower once
    time_steps(step, args.warmup, flush, stream)
    torch.cuda.synchronize()
    if world > 1:
        dist.barrier()
    with ClockSampler(local_rank) as clocks:
        torch.cuda.synchronize()
        if world > 1:
            dist.barrier()
        t0 = time.perf_counter()
        times = time_steps(step, args.steps, flush, stream)
        if world > 1:
            dist.barrier()
        wall = time.perf_counter() - t0
    total_ms = sum(times)
    if world > 1:
        t = torch.tensor([total_ms], device=dev)
        dist.all_reduce(t, op=dist.ReduceOp.MAX)
        total_ms = float(t.item())
    single = spec["mode"] in ("1d", "2d")
    gpu_launches = args.steps * (1 if single or spec["mode"] == "row_scaled" else 3)

    # The same work through the two-pass path (zero + amax kernels, then the
    # cast kernel), and its two halves, also L2-flushed: for comparison.
    split = {}
    if spec["mode"] != "row_scaled" and not args.no_split:
        two = lambda: nv.quantize(x, spec["mode"], swizzled=spec["swizzled"], sign_mask=mask, out=q,  # noqa
                                  path="two_pass")
        amax_fn = (lambda: nv.compute_amax_rht(x, mask, q.amax_row, q.amax_col)) if spec["mode"] == "rht" else \
            (lambda: nv.compute_amax(x, q.amax_row, q.amax_col))
        cast_fn = lambda: nv.quantize(x, spec["mode"], swizzled=spec["swizzled"], sign_mask=mask, out=q,  # noqa
                                      skip_amax=True)
        split["two_pass_ms"] = statistics.mean(time_steps(two, args.steps, flush, stream))
        split["amax_ms"] = statistics.mean(time_steps(amax_fn, args.steps, flush, stream))
        tc = []
        for k in range(args.steps):   # the cast reads x after the amax pass, as in the two-pass call
            flush(k)
            amax_fn()
            s, e = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            s.record(stream)
            cast_fn()
            e.record(stream)
            tc.append((s, e))
        torch.cuda.synchronize()
        split["cast_ms"] = statistics.mean([s.elapsed_time(e) for s, e in tc])
        split = {k: round(v, 5) for k, v in split.items()}

    # e2e: host buffers through the public API, copies inside the timed region
    e2e = None if args.no_e2e else bench_e2e(nv, spec, x_host, q, mask, args, dev, flush)
    host_us = host_costs(nv, spec, x, q, mask, step, stream)
    steady = steady_state(nv, spec, x_host, dev, stream, args.steps)

    peak, peak_kind = measured_peaks()
    ms_per_step = total_ms / args.steps
    value = world * bytes_step * args.steps / (total_ms / 1e3) / 1e9
    per_gpu = bytes_step / (ms_per_step / 1e3) / 1e9
    result = {
        "metric": "NVFP4 quantize GB/s and % HBM roofline, 8192x5120 BF16 row+col, 1 GB300",
        "value": round(value, 1), "unit": "GB/s", "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "step_ms": {"min": round(min(times), 5), "median": round(statistics.median(times), 5),
                    "max": round(max(times), 5)},
        "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16" if spec["dtype"] == torch.bfloat16 else "f32",
        "data": "synthetic (seeded torch.randn N(0,1), generated on the host)",
        "config": {"workload": args.workload, "mode": spec["mode"], "M": M, "N": N,
                   "rowwise": True, "colwise": spec["mode"] != "row_scaled", "swizzled": spec["swizzled"],
                   "bytes_per_step": bytes_step,
                   "l2": "flushed between steps (256 MiB write, then 256 MiB read of another buffer)",
                   "parallelism": f"replicas x{world} (one independent matrix per GPU)"},
        "roofline": {"bound": "hbm",
                     "kernel": "fused_kernel (one launch: amax, grid barrier, cast)" if single else
                     "quantize call (zero + amax + cast kernels)",
                     "achieved": round(per_gpu, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(per_gpu / peak, 4), "peak_kind": f"{peak_kind} (MEASURED_PEAKS.json hbm_gbs)"
                     if peak_kind == "measured" else "fallback 6.8 TB/s",
                     "traffic": ncu_traffic(args.workload), "two_pass_ms": split},
        "e2e": e2e,
        "gpu_launches": gpu_launches,
        "host_us_per_call": host_us["c_abi_via_ctypes"],
        "host_us": host_us,
        "steady_state": steady,
        "wall_s_timed": round(wall, 3),
    }
    if rank == 0:
        result["clocks"] = clocks.summary()
        if args.variants:
            result["variants"] = bench_variants(nv, inputs, args, dev, flush, stream)
        if not args.no_cpu_baseline:
            result["cpu_baseline"] = cpu_baseline(spec, x_host, args.cpu_budget)
    return result


def bench_e2e(nv, spec, x_host, q, mask, args, dev, flush):
    """Same metric through the public API with host buffers: every step copies
    its input from pinned host memory to the device, quantizes it and copies
    all of its outputs back to pinned host memory, inside the timed region.
    Measured two ways: one step at a time (copy in, quantize, copy out,
    serialised; L2 flushed between steps; mean per step), and as a stream of
    steps on two device buffer sets and three streams, so that step k + 1's
    copy in overlaps step k's quantize and copy out (the host link carries
    both directions at once); `value` is the stream's: K steps' bytes over
    the time from the first copy in to the last copy out."""
    import torch
    stream = torch.cuda.current_stream(dev)
    xh = x_host.pin_memory()
    colwise = spec["mode"] != "row_scaled"

    def outputs(qq):
        return [t for t in (qq.data_row, qq.scale_row, qq.amax_row, qq.data_col, qq.scale_col, qq.amax_col)
                if t is not None]

    def quantize(xd, qq):
        nv.quantize(xd, spec["mode"], rowwise=True, colwise=colwise, swizzled=spec["swizzled"],
                    sign_mask=mask, out=qq)

    xd = torch.empty_like(xh, device=dev)
    outs = outputs(q)
    hosts = [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in outs]
    h2d = xh.numel() * xh.element_size()
    d2h = sum(t.numel() * t.element_size() for t in outs)

    def step():
        xd.copy_(xh, non_blocking=True)
        quantize(xd, q)
        for h, t in zip(hosts, outs):
            h.copy_(t, non_blocking=True)

    for _ in range(max(1, args.warmup)):
        step()
    times = time_steps(step, args.steps, flush, stream)
    ms_serial = statistics.mean(times)

    # the stream of steps: buffer set k % 2; events order each set's reuse
    sets = []
    for _ in range(2):
        qq = nv.empty(spec["M"], spec["N"], colwise=colwise, row_scaled=spec["mode"] == "row_scaled",
                      swizzled=spec["swizzled"], device=dev)
        oo = outputs(qq)
        sets.append({"x": torch.empty_like(xh, device=dev), "q": qq, "outs": oo,
                     "hosts": [torch.empty(t.shape, dtype=t.dtype, pin_memory=True) for t in oo],
                     "in": torch.cuda.Event(), "done": torch.cuda.Event(), "out": torch.cuda.Event()})
    s_in, s_q, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    for st in sets:  # every event recorded once, so that the first waits are satisfied
        for ev in ("in", "done", "out"):
            st[ev].record(stream)

    def enqueue(k):
        st = sets[k % 2]
        s_in.wait_event(st["done"])       # step k - 2's quantize has read this input buffer
        with torch.cuda.stream(s_in):
            st["x"].copy_(xh, non_blocking=True)
            st["in"].record(s_in)
        s_q.wait_event(st["in"])
        s_q.wait_event(st["out"])         # step k - 2's outputs have been copied out
        with torch.cuda.stream(s_q):
            quantize(st["x"], st["q"])
            st["done"].record(s_q)
        s_out.wait_event(st["done"])
        with torch.cuda.stream(s_out):
            for h, t in zip(st["hosts"], st["outs"]):
                h.copy_(t, non_blocking=True)
            st["out"].record(s_out)

    n = max(args.steps, 6)
    for k in range(4):
        enqueue(k)
    torch.cuda.synchronize()
    t0, t1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    t0.record(s_in)
    for k in range(n):
        enqueue(k)
    for st_ in (s_in, s_q):
        s_out.wait_stream(st_)
    t1.record(s_out)
    torch.cuda.synchronize()
    ms_stream = t0.elapsed_time(t1) / n
    wb = workload_bytes(spec)
    return {"value": round(wb / (ms_stream / 1e3) / 1e9, 1), "unit": "GB/s",
            "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h, "ms_per_step": round(ms_stream, 4),
            "how": f"{n} steps streamed on two buffer sets: step k+1's copy in overlaps step k's quantize "
                   "and copy out (three CUDA streams, pinned host buffers)",
            "serial": {"value": round(wb / (ms_serial / 1e3) / 1e9, 1), "unit": "GB/s",
                       "ms_per_step": round(ms_serial, 4),
                       "how": "one step at a time: copy in, quantize, copy out; L2 flushed between steps"}}


def bench_variants(nv, inputs, args, dev, flush, stream):
    """The other workloads, fewer steps: GB/s and fraction of the HBM peak."""
    import torch
    peak, _ = measured_peaks()
    out = {}
    steps = max(5, args.steps // 4)
    for name, spec in inputs.WORKLOADS.items():
        if name == args.workload:
            continue
        x = inputs.make(spec).to(dev)
        mask = inputs.sign_mask_from_seed(spec["seed"]) if spec["mode"] == "rht" else 0
        q = nv.empty(spec["M"], spec["N"], colwise=spec["mode"] != "row_scaled",
                     row_scaled=spec["mode"] == "row_scaled", swizzled=spec["swizzled"], device=dev)
        step = run_step_fn(nv, spec, x, q, mask)
        for _ in range(3):
            step()
        ms = statistics.median(time_steps(step, steps, flush, stream))
        gbs = workload_bytes(spec) / (ms / 1e3) / 1e9
        out[name] = {"ms": round(ms, 5), "GB/s": round(gbs, 1), "frac": round(gbs / peak, 4)}
        if spec["mode"] == "rht":  # the single-pass alternative (x read from HBM once)
            sp = lambda: nv.quantize(x, "rht", swizzled=spec["swizzled"], sign_mask=mask, out=q,  # noqa
                                     path="single_pass")
            for _ in range(3):
                sp()
            sms = statistics.median(time_steps(sp, steps, flush, stream))
            sgbs = workload_bytes(spec) / (sms / 1e3) / 1e9
            out[name + "_single_pass"] = {"ms": round(sms, 5), "GB/s": round(sgbs, 1), "frac": round(sgbs / peak, 4)}
        if spec["mode"] in ("2d", "1d") and spec["M"] == 8192:
            dq = lambda: nv.dequantize(q.data_row, q.scale_row, q.amax_row, swizzled=spec["swizzled"])  # noqa
            for _ in range(3):
                dq()
            dms = statistics.median(time_steps(dq, steps, flush, stream))
            dbytes = spec["M"] * spec["N"] * (0.5 + 1 / 16 + 2)
            out[name + "_dequant"] = {"ms": round(dms, 5), "GB/s": round(dbytes / (dms / 1e3) / 1e9, 1),
                                      "frac": round(dbytes / (dms / 1e3) / 1e9 / peak, 4)}
        del x, q
        torch.cuda.empty_cache()
    # stochastic rounding: inputs.SR with its random bytes (1 byte per
    # element read on top of the plain quantize's traffic)
    spec = inputs.SR
    x = inputs.make(spec).to(dev)
    rb = inputs.random_bytes(spec["M"], spec["N"], seed=spec["rbits_seed"]).to(dev)
    q = nv.empty(spec["M"], spec["N"], swizzled=spec["swizzled"], device=dev)
    sstep = lambda: nv.quantize_sr(x, rb, spec["mode"], swizzled=spec["swizzled"], out=q)  # noqa
    for _ in range(3):
        sstep()
    sms = statistics.median(time_steps(sstep, steps, flush, stream))
    sbytes = spec["M"] * spec["N"] * (BYTES_PER_ELEM[("bf16", "rowcol")] + 1.0)
    out[f"sr_{spec['mode']}_{spec['M']}x{spec['N']}_bf16"] = {
        "ms": round(sms, 5), "GB/s": round(sbytes / (sms / 1e3) / 1e9, 1),
        "frac": round(sbytes / (sms / 1e3) / 1e9 / peak, 4)}
    del x, rb, q
    torch.cuda.empty_cache()
    # grouped quantize: the members of inputs.GROUPED (8192 x 5120 in all),
    # each with its own amax, in three launches
    spec = inputs.GROUPED
    splits, N = spec["splits"], spec["N"]
    x = inputs.make_grouped(spec).to(dev)
    outs = [nv.empty(m, N, swizzled=spec["swizzled"], device=dev) for m in splits]
    gstep = lambda: nv.quantize_grouped(x, splits, spec["mode"], swizzled=spec["swizzled"], out=outs)  # noqa
    for _ in range(3):
        gstep()
    gms = statistics.median(time_steps(gstep, steps, flush, stream))
    dt = "bf16" if spec["dtype"] == torch.bfloat16 else "fp32"
    gbytes = sum(splits) * N * BYTES_PER_ELEM[(dt, "rowcol")]
    gname = f"grouped_{len(splits)}_members_{sum(splits)}x{N}_{dt}_{spec['mode']}"
    out[gname] = {"ms": round(gms, 5), "GB/s": round(gbytes / (gms / 1e3) / 1e9, 1),
                  "frac": round(gbytes / (gms / 1e3) / 1e9 / peak, 4)}
    del x, outs
    torch.cuda.empty_cache()
    return out


# ---------------------------------------------------------------------------
# CPU oracle arm
# ---------------------------------------------------------------------------

def _oracle_sample(spec, x_host, rows):
    import numpy as np
    import torch
    xs = x_host[:rows].contiguous()
    xb = xs.view(torch.int16).numpy().view(np.uint16) if xs.dtype == torch.bfloat16 else xs.numpy()
    return xb


def time_oracle(spec, x_host, rows):
    import oracle
    xb = _oracle_sample(spec, x_host, rows)
    mask = 0
    if spec["mode"] == "rht":
        from nvfp4_block_scaled_amax_gb300 import inputs
        mask = inputs.sign_mask_from_seed(spec["seed"])
    t0 = time.perf_counter()
    oracle.quantize(spec["mode"], xb, colwise=spec["mode"] != "row_scaled", sign_mask=mask)
    return time.perf_counter() - t0


def host_cpu():
    """The host's logical core count and CPU model name (lscpu, else
    /proc/cpuinfo, else the platform string)."""
    import platform
    model = None
    try:
        out = subprocess.run(["lscpu"], capture_output=True, text=True, timeout=10).stdout
        for ln in out.splitlines():
            if ln.strip().lower().startswith("model name"):
                model = ln.split(":", 1)[1].strip()
                break
    except (OSError, subprocess.SubprocessError):
        pass
    if model is None and os.path.exists("/proc/cpuinfo"):
        with open("/proc/cpuinfo") as f:
            for ln in f:
                if ln.lower().startswith("model name"):
                    model = ln.split(":", 1)[1].strip()
                    break
    return {"host_cores": os.cpu_count(), "cpu_model": model or platform.processor() or platform.machine()}


def cpu_baseline(spec, x_host, budget_s):
    import oracle
    oracle.build()
    M, N = spec["M"], spec["N"]
    rows = 64
    t = time_oracle(spec, x_host, rows)
    target = max(64, min(M, int(rows * budget_s / max(t, 1e-3)) // 16 * 16))
    t = time_oracle(spec, x_host, target)
    frac = target / M
    gbs = workload_bytes(spec) * frac / t / 1e9
    return {"value": round(gbs, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"first {target} of {M} rows ({N} columns), {t:.1f} s, single-threaded C oracle",
            **host_cpu()}


def bench_reference(args, rank):
    from nvfp4_block_scaled_amax_gb300 import inputs
    import oracle
    oracle.build()
    spec = inputs.WORKLOADS[args.workload]
    x_host = inputs.make(spec)
    M, N = spec["M"], spec["N"]
    # size each step so the whole run stays within a few minutes
    probe = time_oracle(spec, x_host, 32)
    per_step_budget = max(0.5, 120.0 / max(1, args.steps + args.warmup))
    rows = max(16, min(M, int(32 * per_step_budget / max(probe, 1e-3)) // 16 * 16))
    for _ in range(args.warmup):
        time_oracle(spec, x_host, rows)
    times = [time_oracle(spec, x_host, rows) for _ in range(args.steps)]
    total = sum(times)
    bytes_step = workload_bytes(spec) * rows / M
    value = bytes_step * args.steps / total / 1e9
    sample = f"first {rows} of {M} rows ({N} columns) per step, single-threaded C oracle"
    return {"metric": "NVFP4 quantize GB/s and % HBM roofline, 8192x5120 BF16 row+col, 1 GB300",
            "value": round(value, 5), "unit": "GB/s", "n_gpus": 1, "steps": args.steps, "warmup": args.warmup,
            "ms_per_step": round(1e3 * total / args.steps, 3), "higher_is_better": True, "scaling": "weak",
            "vs_baseline": None, "dtype": "bf16", "data": "synthetic (seeded torch.randn N(0,1))",
            "config": {"workload": args.workload, "mode": spec["mode"], "M": M, "N": N,
                       "swizzled": spec["swizzled"]},
            "impl": "reference",
            "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": 1, "kind": "oracle",
                             "sample": sample, **host_cpu()},
            "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0}}


def main():
    p = argparse.ArgumentParser(description=__doc__.split("\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=50)
    p.add_argument("--warmup", type=int, default=5)
    p.add_argument("--impl", choices=["ours", "reference"], default="ours")
    p.add_argument("--workload", default="2d_8192x5120_bf16")
    p.add_argument("--variants", action="store_true", default=True)
    p.add_argument("--no-variants", dest="variants", action="store_false")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-split", action="store_true")
    p.add_argument("--cpu-budget", type=float, default=15.0, help="seconds of oracle work for cpu_baseline")
    args = p.parse_args()
    args.warmup = max(3, args.warmup)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank == 0:
            print(json.dumps(bench_reference(args, rank)), flush=True)
        return

    if world > 1:
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    result = bench_ours(args, rank, world, local_rank)
    if rank == 0:
        print(json.dumps(result), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.barrier()
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
