#!/usr/bin/env python
"""Benchmark of the row-exact few-row quantized mat-vec on GB300.

Metric: achieved HBM GB/s (algorithmic weight + x + y bytes per call, over
the device time of the calls) and us per call, m = 1..8.  One "step" is one
pass of the whole path over the workload: one call per listed m.

Default workload: Q6_K weights n = 128256, k = 4096 (431 MB, the largest
configuration that fits one GPU), batch 1, m in {1, 4, 8} (W ~ N(0, 0.02)
quantized to Q6_K, x ~ N(0, 1)), synthetic and seeded.  Weights are read
cold: every call uses the next copy of a ring of weight copies totalling
>= 4x the L2 size.  The same line carries per-m tables of the other
configurations (key "workloads"; --no-extra skips them).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME] [--impl reference]

Under torchrun (N > 1) every rank runs the same workload on its own GPU
(replicas: the path needs no exchange); rank 0 prints max-over-ranks timing.
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
sys.path.insert(0, ROOT)

# name: (format, n, k, batch, m list, token-major grouped, config index for seeds)
WORKLOADS = {
    "f16_n256_k512_m1": ("f16", 256, 512, 1, [1], False, 0),
    "q8_0_n4096_k4096_m1-8": ("q8_0", 4096, 4096, 1, list(range(1, 9)), False, 1),
    "q4_K_n14336_k4096_m1-8": ("q4_K", 14336, 4096, 1, list(range(1, 9)), False, 2),
    "q6_K_n128256_k4096_m1,4,8": ("q6_K", 128256, 4096, 1, [1, 4, 8], False, 3),
    "q5_0_grouped_b16_n1024_k4096_m8": ("q5_0", 1024, 4096, 16, [8], True, 4),
    # same formats at >= 64 MB of weights
    "f16_n8192_k4096_m1-8": ("f16", 8192, 4096, 1, list(range(1, 9)), False, 5),
    "q8_0_n16384_k4096_m1-8": ("q8_0", 16384, 4096, 1, list(range(1, 9)), False, 6),
    "q4_K_n28672_k4096_m1-8": ("q4_K", 28672, 4096, 1, list(range(1, 9)), False, 7),
    "q5_0_grouped_b32_n1024_k4096_m8": ("q5_0", 1024, 4096, 32, [8], True, 8),
    # more than 8 input rows (rem_matvec_many: one pass over W per group of 8 rows on the SIMT
    # engine, of 16 rows on the tensor-core engine)
    "q4_K_n14336_k4096_m16,32": ("q4_K", 14336, 4096, 1, [16, 32], False, 9),
    "q8_0_n16384_k4096_m16,32": ("q8_0", 16384, 4096, 1, [16, 32], False, 14),
    "q6_K_n128256_k4096_m16": ("q6_K", 128256, 4096, 1, [16], False, 15),
    # dense weights under the same row contract
    "bf16_n8192_k4096_m1-8": ("bf16", 8192, 4096, 1, list(range(1, 9)), False, 11),
    "f32_n4096_k4096_m1-8": ("f32", 4096, 4096, 1, list(range(1, 9)), False, 12),
    # affine group quantization (4-bit codes, f16 scale and bias per 64 values)
    "a4_g64_n14336_k4096_m1-8": ("a4_g64", 14336, 4096, 1, list(range(1, 9)), False, 13),
    # fused epilogue y = W.x + bias (rem_matvec_axpby, one bias vector for all rows)
    "q8_0_n4096_k4096_m1-8_bias": ("q8_0", 4096, 4096, 1, list(range(1, 9)), False, 10),
    # profiling size of the Q6_K path: 215 MB of weights (above the L2), for ncu captures
    "q6_K_n65536_k4096_m1,8": ("q6_K", 65536, 4096, 1, [1, 8], False, 16),
    # the tensor-core engine on request (rem_matvec_sched) where the default is the lanes-over-rows one
    "q5_0_grouped_b16_n1024_k4096_m1-8_tc": ("q5_0", 1024, 4096, 16, list(range(1, 9)), True, 4, "tc"),
    "q5_0_n28672_k4096_m1-8_tc": ("q5_0", 28672, 4096, 1, list(range(1, 9)), False, 17, "tc"),
    "q8_0_n28672_k4096_m1-8_tc": ("q8_0", 28672, 4096, 1, list(range(1, 9)), False, 18, "tc"),
}
# workloads that run the epilogue alpha * W.x + beta * c with c a bias vector
EPILOGUE = {"q8_0_n4096_k4096_m1-8_bias": (1.0, 1.0)}
# the largest configuration that fits one GPU (431 MB of Q6_K weights)
DEFAULT = "q6_K_n128256_k4096_m1,4,8"
# the other configurations timed in the same run, one per-m table each
EXTRA = ["f16_n256_k512_m1", "q8_0_n4096_k4096_m1-8", "q4_K_n14336_k4096_m1-8", "q5_0_grouped_b16_n1024_k4096_m8",
         "f16_n8192_k4096_m1-8", "q8_0_n16384_k4096_m1-8", "q4_K_n28672_k4096_m1-8", "q5_0_grouped_b32_n1024_k4096_m8",
         "q4_K_n14336_k4096_m16,32", "q8_0_n16384_k4096_m16,32", "q6_K_n128256_k4096_m16",
         "bf16_n8192_k4096_m1-8", "f32_n4096_k4096_m1-8", "a4_g64_n14336_k4096_m1-8", "q8_0_n4096_k4096_m1-8_bias",
         "q5_0_grouped_b16_n1024_k4096_m1-8_tc", "q5_0_n28672_k4096_m1-8_tc", "q8_0_n28672_k4096_m1-8_tc"]
METRIC = "achieved HBM GB/s (% of GB300 peak) and us/call, m=1..8 quantized mat-vec"


def peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), float(d.get("sm_max_mhz", 2070.0)), "measured"
    return 6800.0, 2070.0, "fallback"


def kernel_sources_sha256() -> str:
    """Digest of the CUDA sources and the public header (what a DRAM-traffic
    figure measured by ncu depends on)."""
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "quantized_few_row_gb300", "csrc")
    for name in sorted(os.listdir(csrc)):
        if name.endswith((".cu", ".cuh", ".h")):
            with open(os.path.join(csrc, name), "rb") as f:
                h.update(name.encode() + b"\0" + f.read())
    with open(os.path.join(ROOT, "include", "rem.h"), "rb") as f:
        h.update(b"rem.h\0" + f.read())
    return h.hexdigest()


def profiled_traffic(workload: str):
    """DRAM bytes per launch (read + write, averaged over one step's
    launches) recorded under profiles/ for this workload, if the recording was
    made from the current kernel sources; else None."""
    path = os.path.join(ROOT, "profiles", f"rem_mv_{workload}.md")
    if not os.path.exists(path):
        return None
    rec = {}
    with open(path) as f:
        for line in f:
            line = line.strip().strip("`")
            for key in ("kernel_sources_sha256", "dram_bytes_per_launch"):
                if line.startswith(key + ":"):
                    rec[key] = line.split(":", 1)[1].strip()
    if rec.get("kernel_sources_sha256") != kernel_sources_sha256() or "dram_bytes_per_launch" not in rec:
        return None
    return float(rec["dram_bytes_per_launch"])


def affine_group_size(fmt):
    """Group size of an affine weight type name ("a4_g64" -> 64), else 0."""
    return int(fmt.split("_g")[1]) if fmt.startswith("a") else 0


def call_bytes(fmt, n, k, batch, m, row_bytes):
    """Algorithmic bytes of one call: every weight once (affine: codes plus the
    binary16 scale and bias of every group), x and y once."""
    gs = affine_group_size(fmt)
    wrow = row_bytes + (4 * (k // gs) if gs else 0)
    return batch * n * wrow + 4 * batch * m * k + 4 * batch * m * n


class Clocks:
    """nvidia-smi sampling of SM clocks and throttle reasons while running."""
    Q = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
         "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
         "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index: int):
        self.index = index
        self.proc = None
        self.path = None

    def start(self):
        try:
            fd, self.path = tempfile.mkstemp(suffix=".csv")
            os.close(fd)
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.Q}", "--format=csv,noheader,nounits",
                 "-lms", "50"], stdout=open(self.path, "w"), stderr=subprocess.DEVNULL)
        except (OSError, FileNotFoundError):
            self.proc = None
            return
        # nvidia-smi takes a moment to start: wait (at most 5 s) for its first
        # sample so that the timed region that follows is sampled
        t_end = time.time() + 5.0
        while time.time() < t_end and self.proc.poll() is None and os.path.getsize(self.path) == 0:
            time.sleep(0.02)

    def stop(self, busy_mhz_floor: float = 0.0):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        rows = []
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) >= 9:
                    rows.append(parts)
        os.unlink(self.path)
        if not rows:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["no samples"]}
        sm = [float(r[1]) for r in rows if r[1].replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if r[2].replace(".", "").isdigit()]
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        reasons = sorted({names[i] for r in rows for i in range(4) if r[5 + i].lower() == "active"})
        loaded = [s for s in sm if s >= busy_mhz_floor] or sm
        return {"sm_mhz": statistics.median(loaded) if loaded else None, "sm_max_mhz": max(mx) if mx else None,
                "samples": len(rows), "reasons": reasons}


# ---------------------------------------------------------------- our arm

def max_over_ranks(seconds: float, world: int, device) -> float:
    """The slowest rank's time (all ranks call it; world 1 returns its own)."""
    if world <= 1:
        return seconds
    import torch
    t = torch.tensor([seconds], dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return float(t.item())


def job_throughput(bytes_per_step: int, steps: int, seconds: float, world: int) -> float:
    """Whole-job GB/s: every replica processes the same step bytes; time is the slowest rank's."""
    return world * bytes_per_step * steps / seconds / 1e9


class Workload:
    """One configuration on the device: weights quantized on the device (a ring
    of copies totalling >= 4x the L2 size, so calls read them cold), inputs,
    outputs, and call(slot, m) through the library's public C ABI."""

    def __init__(self, name, dev, rem, inputs, l2):
        import torch
        fmt, n, k, batch, ms, grouped, ci = WORKLOADS[name][:7]
        # an engine requested explicitly (the tensor cores for Q8_0 / Q5_0), else the library's choice
        forced = WORKLOADS[name][7] if len(WORKLOADS[name]) > 7 else None
        self.sched = rem.Schedule(engine=1 if forced == "tc" else 0) if forced else None
        self.name, self.fmt, self.n, self.k, self.batch, self.ms, self.grouped = name, fmt, n, k, batch, ms, grouped
        self.rem = rem
        self.rb = rem.rem_row_bytes(fmt, k)
        wbytes = self.rb * n * batch
        self.wbytes = wbytes
        mmax = max(ms)
        gs = affine_group_size(fmt)
        self.gs = gs
        ring = max(1, math.ceil(4 * l2 / wbytes))
        if gs:
            # affine: random codes, f16 scales ~ 0.02*3/15 and biases ~ -0.02*3 per group (device-side, seeded)
            g = torch.Generator(device=dev)
            g.manual_seed(1000 + ci)
            w0 = torch.randint(0, 256, (wbytes,), dtype=torch.uint8, device=dev, generator=g)
            ng = batch * n * (k // gs)
            scales = (torch.rand(ng, device=dev, generator=g) * 0.004 + 0.002).half()
            biases = (torch.rand(ng, device=dev, generator=g) * -0.06).half()
            ring = max(1, math.ceil(4 * l2 / (wbytes + 4 * ng)))
        else:
            # weights: N(0, 0.02) drawn on the device, quantized by the library
            wf = inputs.torch_normal((batch * n, k), 1000 + ci, inputs.W_STD, dev)
            w0 = torch.empty(wbytes, dtype=torch.uint8, device=dev)
            rem.check(rem.rem_quantize(wf, fmt, batch * n, k, w0))
            del wf
        self.ring = ring
        self.wring = [w0] + [w0.clone() for _ in range(ring - 1)]
        self.sring = [scales] + [scales.clone() for _ in range(ring - 1)] if gs else None
        self.bring = [biases] + [biases.clone() for _ in range(ring - 1)] if gs else None
        if grouped:   # token-major: x [m, batch*k], y [m, batch*n]
            self.x = inputs.torch_normal((mmax, batch * k), 2000 + ci, inputs.X_STD, dev)
            self.y = torch.empty((mmax, batch * n), dtype=torch.float32, device=dev)
            self.xbs, self.ybs = k, n
        else:         # batch-major: x [batch, m, k]
            self.x = inputs.torch_normal((batch, mmax, k), 2000 + ci, inputs.X_STD, dev)
            self.y = torch.empty((batch, mmax, n), dtype=torch.float32, device=dev)
            self.xbs, self.ybs = mmax * k, mmax * n
        self.epi = EPILOGUE.get(name)
        self.bias = inputs.torch_normal((batch, n), 3000 + ci, inputs.X_STD, dev) if self.epi else None
        self.engine = self.sched.engine if self.sched is not None else rem.rem_engine_of(fmt, batch * n, k)
        torch.cuda.synchronize()

    def call(self, slot, m, stream=None, xv=None, yv=None):
        """One library call for m input rows on ring slot `slot`; xv / yv: a
        packed per-call segment ([batch, m, k] batch-major or [m, batch*k]
        token-major) instead of the resident buffers."""
        rem, fmt, n, k, batch = self.rem, self.fmt, self.n, self.k, self.batch
        xs, ys = (self.x, self.y) if xv is None else (xv, yv)
        if xv is None:
            xb, yb = self.xbs, self.ybs
        else:
            xb, yb = (k, n) if self.grouped else (m * k, m * n)
        w = self.wring[slot]
        if self.gs:
            return rem.rem_matvec_affine(w, self.sring[slot], self.bring[slot], fmt, n, k, batch, xs, m, k, xb, ys,
                                         n, yb, 0, stream)
        if self.epi:
            return rem.rem_matvec_axpby(w, fmt, n, k, batch, xs, m, k, xb, ys, n, yb, self.epi[0], self.epi[1],
                                        self.bias, 0, n, stream)
        if self.sched is not None:
            xrs, yrs = (batch * k, batch * n) if self.grouped else (k, n)
            return rem.rem_matvec_sched(w, fmt, n, k, batch, xs, m, xrs, xb, ys, yrs, yb, self.sched, stream)
        if m > 8:
            xrs, yrs = (batch * k, batch * n) if self.grouped else (k, n)
            return rem.rem_matvec_many(w, fmt, n, k, batch, xs, m, xrs, xb, ys, yrs, yb, 0, stream)
        return rem.rem_matvec(w, fmt, n, k, batch, xs, m, xb, ys, yb, stream)

    def bytes(self, m):
        extra = 4 * self.batch * self.n if self.epi else 0     # the bias vector, read once per call
        return call_bytes(self.fmt, self.n, self.k, self.batch, m, self.rb) + extra

    def launches(self, m):
        per = 8 if self.engine != 1 else 16
        return (m + per - 1) // per

    def free(self):
        self.wring = self.sring = self.bring = None
        self.x = self.y = self.bias = None


def time_per_m(wl, stream, budget_s=2e-3):
    """Device microseconds per call for each m: a CUDA graph of one call per
    ring slot (cold weights), replayed until about budget_s of work is timed
    with events on the launching stream.  Also returns the same on one weight
    copy (warm, for comparison only) and the plan of the last call."""
    import torch
    per_m, warm, plans = {}, {}, {}
    for m in wl.ms:
        with torch.cuda.stream(stream):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
                for slot in range(wl.ring):
                    wl.rem.check(wl.call(slot, m))
            plans[m] = wl.rem.rem_last_plan()
            for _ in range(3):
                g.replay()
            stream.synchronize()
            t0 = time.perf_counter()
            g.replay()
            stream.synchronize()
            one = max(1e-6, time.perf_counter() - t0)
            reps = max(3, min(2000, int(budget_s / one) + 3))
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(reps):
                g.replay()
            e1.record(stream)
        stream.synchronize()
        per_m[m] = e0.elapsed_time(e1) * 1e3 / (reps * wl.ring)
        with torch.cuda.stream(stream):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
                for _ in range(16):
                    wl.rem.check(wl.call(0, m))
            for _ in range(2):
                g.replay()
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            for _ in range(10):
                g.replay()
            e1.record(stream)
        stream.synchronize()
        warm[m] = e0.elapsed_time(e1) * 1e3 / (10 * 16)
    return per_m, warm, plans


def per_m_table(wl, per_m, hbm, fp32_peak):
    out = {}
    for m in wl.ms:
        b = wl.bytes(m)
        gbs = b / (per_m[m] * 1e-6) / 1e9
        tfl = 2.0 * m * wl.batch * wl.n * wl.k / (per_m[m] * 1e-6) / 1e12
        out[str(m)] = {"us": round(per_m[m], 3), "gbs": round(gbs, 1), "hbm_frac": round(gbs / hbm, 4),
                       "fp32_tflops": round(tfl, 2), "fp32_frac": round(tfl / fp32_peak, 4)}
    return out


def run_ours(args, rank, world, local_rank):
    import torch

    import quantized_few_row_gb300 as rem
    from quantized_few_row_gb300 import inputs

    torch.cuda.set_device(local_rank)
    dev = torch.device("cuda", local_rank)
    rem.build()
    rem.load()
    props = torch.cuda.get_device_properties(dev)
    l2 = int(getattr(props, "L2_cache_size", 128 << 20))
    wl = Workload(args.workload, dev, rem, inputs, l2)
    ms = wl.ms
    fmt, n, k, batch = wl.fmt, wl.n, wl.k, wl.batch
    ring = wl.ring

    # first calls outside any capture (device set-up, schedule caches)
    for m in ms:
        rem.check(wl.call(0, m))
    torch.cuda.synchronize()
    # host cost of a call (argument checks, plan and tensor-map caches, the
    # launch) through the Python binding, on a stream that is not captured
    side = torch.cuda.Stream(device=dev)
    with torch.cuda.stream(side):
        for m in ms:
            rem.check(wl.call(0, m, side))
        side.synchronize()
        reps = 200
        t0 = time.perf_counter()
        for i in range(reps):
            rem.check(wl.call(0, ms[i % len(ms)], side))
        host_us = (time.perf_counter() - t0) * 1e6 / reps
        side.synchronize()

    stream = torch.cuda.Stream(device=dev)
    C = len(ms)
    period = ring // math.gcd(C, ring)
    graphs = []
    with torch.cuda.stream(stream):
        for sidx in range(period):
            g = torch.cuda.CUDAGraph()
            with torch.cuda.graph(g, stream=stream, capture_error_mode="relaxed"):
                for c, m in enumerate(ms):
                    rem.check(wl.call((sidx * C + c) % ring, m))
            graphs.append(g)
    torch.cuda.synchronize()

    clocks = Clocks(local_rank)
    clocks.start()
    with torch.cuda.stream(stream):
        for s in range(args.warmup):
            graphs[s % period].replay()
    stream.synchronize()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with torch.cuda.stream(stream):
        ev0.record(stream)
        for s in range(args.steps):
            graphs[(args.warmup + s) % period].replay()
        ev1.record(stream)
    stream.synchronize()
    torch.cuda.synchronize()
    elapsed = max_over_ranks(ev0.elapsed_time(ev1) / 1e3, world, dev)
    if world > 1:
        torch.distributed.barrier()

    step_bytes = sum(wl.bytes(m) for m in ms)
    value = job_throughput(step_bytes, args.steps, elapsed, world)

    # per-m device time (cold ring, graph of one call per ring slot), and warm for comparison
    per_m, per_m_warm, plans = time_per_m(wl, stream)
    clk = clocks.stop(busy_mhz_floor=0.0)

    # end to end through the public binding: each step's inputs (one x segment per call, packed) go
    # host->device in one copy, every call writes its own y segment, and the step's outputs come back
    # device->host in one copy.  The copies run on a second stream with two device buffers each, the
    # way a caller streams steps: step s's outputs come back and step s+2's inputs go over while
    # step s+1 computes; every step's copies lie inside the timed region, which ends when the last
    # step's outputs are on the host.
    xoff, yoff = [0], [0]
    for m in ms:
        xoff.append(xoff[-1] + batch * m * k)
        yoff.append(yoff[-1] + batch * m * n)
    xh = torch.empty(xoff[-1], dtype=torch.float32).pin_memory()
    for i, m in enumerate(ms):
        src = wl.x[:m].reshape(-1) if wl.grouped else wl.x[:, :m].reshape(-1)
        xh[xoff[i]:xoff[i + 1]].copy_(src.cpu())
    yh = torch.empty(yoff[-1], dtype=torch.float32).pin_memory()
    xp = [torch.empty(xoff[-1], dtype=torch.float32, device=dev) for _ in range(2)]
    yp = [torch.empty(yoff[-1], dtype=torch.float32, device=dev) for _ in range(2)]
    h2d = 4 * xoff[-1]
    d2h = 4 * yoff[-1]
    e2e_steps = max(1, min(args.steps, 200))
    torch.cuda.synchronize()
    cur = torch.cuda.current_stream(dev)
    cps = torch.cuda.Stream(dev)
    x_in = [torch.cuda.Event() for _ in range(2)]      # buffer b holds its step's inputs
    y_out = [torch.cuda.Event() for _ in range(2)]     # buffer b's outputs are on the host
    done = [torch.cuda.Event() for _ in range(2)]      # the calls of buffer b's step have run
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record(cur)
    cps.wait_event(t0)

    def put(b):
        with torch.cuda.stream(cps):
            xp[b].copy_(xh, non_blocking=True)
            x_in[b].record(cps)

    for b in range(min(2, e2e_steps)):
        put(b)
    slot = 0
    for s in range(e2e_steps):
        b = s % 2
        cur.wait_event(x_in[b])
        if s >= 2:
            cur.wait_event(y_out[b])
        for i, m in enumerate(ms):
            rem.check(wl.call(slot % ring, m, cur, xp[b][xoff[i]:xoff[i + 1]], yp[b][yoff[i]:yoff[i + 1]]))
            slot += 1
        done[b].record(cur)
        cps.wait_event(done[b])
        with torch.cuda.stream(cps):
            yh.copy_(yp[b], non_blocking=True)
            y_out[b].record(cps)
        if s + 2 < e2e_steps:
            put(b)
    cur.wait_event(y_out[(e2e_steps - 1) % 2])
    t1.record(cur)
    torch.cuda.synchronize()
    e2e_elapsed = max_over_ranks(t0.elapsed_time(t1) / 1e3, world, dev)
    e2e_value = job_throughput(step_bytes, e2e_steps, e2e_elapsed, world)
    # the packed path computes what the device-resident layout does, bit for bit (same W, same split)
    for i, m in enumerate(ms):
        rem.check(wl.call(0, m))
        ref = (wl.y[:m] if wl.grouped else wl.y[:, :m]).reshape(-1).cpu()
        if not torch.equal(ref.view(torch.int32), yh[yoff[i]:yoff[i + 1]].view(torch.int32)):
            raise RuntimeError(f"end-to-end outputs for m={m} differ from the device-resident call")

    hbm, sm_max, peak_kind = peaks()
    fp32_peak = props.multi_processor_count * 128 * 2 * sm_max * 1e6 / 1e12   # TFLOP/s, plain FMA pipe
    per_step_launches = sum(wl.launches(m) for m in ms)
    launches = args.steps * per_step_launches
    avg_launch_s = elapsed / launches
    achieved = (step_bytes / per_step_launches) / avg_launch_s / 1e9
    kernel_s = sum(per_m[m] for m in ms) * 1e-6
    achieved_kernel = step_bytes / kernel_s / 1e9
    engine = {0: "simt (lanes over rows, FP32 pipe)", 1: "tc (tcgen05 tensor cores)"}.get(wl.engine, "?")
    res = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "GB/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(elapsed / args.steps * 1e3, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f32 accumulate over %s weights" % fmt,
        "data": "synthetic (seeded W ~ N(0,0.02) quantized on device, x ~ N(0,1))",
        "config": {"workload": args.workload, "format": fmt, "n": n, "k": k, "batch": batch, "m": ms,
                   "token_major": wl.grouped, "engine": engine,
                   "l2": f"cold: weight ring of {ring} copies x {wl.wbytes} B (>= 4x L2)",
                   "timed": "CUDA graphs of one step each, events on the launching stream",
                   "parallelism": f"replicas x{world}"},
        "per_m_us": {str(m): round(per_m[m], 3) for m in ms},
        "per_m_warm_us": {str(m): round(per_m_warm[m], 3) for m in ms},
        "per_m": per_m_table(wl, per_m, hbm, fp32_peak),
        "plans": {str(m): plans[m] for m in ms},
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": hbm, "unit": "GB/s",
                     "frac": round(achieved / hbm, 4),
                     "basis": "step: algorithmic bytes of the step's launches over the timed graph replays "
                              "(gaps between replays included)",
                     "achieved_kernel": round(achieved_kernel, 1), "frac_kernel": round(achieved_kernel / hbm, 4),
                     "basis_kernel": "kernel: the same bytes over the sum of the per-m CUDA-event launch times "
                                     "(graphs of back-to-back calls on cold weights)",
                     "traffic": profiled_traffic(args.workload),
                     "peak_source": f"{peak_kind} hbm_gbs", "kernel": "rem_tc_kernel / rem_mv_kernel (all m of the step)",
                     "fp32_peak_tflops": round(fp32_peak, 1)},
        "e2e": {"value": round(e2e_value, 2), "unit": "GB/s", "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "steps": e2e_steps,
                "path": "packed step inputs pinned -> device (1 copy), one library call per m, packed outputs -> pinned host "
                        "(1 copy), un-captured; copies on a second stream, two device buffers, overlapping "
                        "the neighbouring steps' calls"},
        "host_us_per_call": round(host_us, 2),
        "host_us_basis": "wall time per library call through the Python (ctypes) binding, stream not captured",
        "gpu_launches": launches,
        "clocks": clk,
    }
    wl.free()
    del graphs
    torch.cuda.empty_cache()

    # the other configurations, one table each (per-m device time on cold weights)
    if not args.no_extra:
        extra = {}
        for name in EXTRA:
            if name == args.workload:
                continue
            w2 = Workload(name, dev, rem, inputs, l2)
            for m in w2.ms:
                rem.check(w2.call(0, m))
            torch.cuda.synchronize()
            pm, warm, pl = time_per_m(w2, stream, budget_s=1e-3)
            extra[name] = {"engine": {0: "simt", 1: "tc"}.get(w2.engine, "?"),
                           "weight_bytes": w2.wbytes,
                           "per_m": per_m_table(w2, pm, hbm, fp32_peak),
                           "per_m_warm_us": {str(m): round(warm[m], 3) for m in w2.ms}}
            w2.free()
            del w2
            torch.cuda.empty_cache()
        res["workloads"] = extra
    return res


# ---------------------------------------------------------------- the oracle on host cores

def oracle_sample(fmt, n, k, batch, ms, grouped, ci, seconds: float):
    """Time the oracle on a bounded sample of weight rows; returns
    (GB/s of algorithmic bytes, cores, description)."""
    import numpy as np

    import oracle
    from quantized_few_row_gb300 import inputs

    oracle.build()
    rows_total = batch * n
    mmax = max(ms)
    x = inputs.activations(mmax, k, 2000 + ci)
    gs = affine_group_size(fmt)
    bits = int(fmt[1]) if gs else 0
    rbytes = k * bits // 8 if gs else oracle.row_bytes(fmt, k)
    nbytes_per = lambda rows: sum(call_bytes(fmt, rows, k, 1, m, rbytes) for m in ms)

    def prepare(rows):
        v = inputs.weights(rows, k, 1000 + ci)
        w = oracle.affine_quantize(v, bits, gs) if gs else oracle.quantize(v, fmt)
        return w, np.arange(rows, dtype=np.uint64)

    def sweep(w, idx, rows):
        t0 = time.perf_counter()
        for m in ms:
            if gs:
                oracle.affine_matvec_rows(*w, bits, gs, rows, k, x, m, k, 0, idx)
            else:
                oracle.matvec_rows(w, fmt, rows, k, x, m, k, 0, idx)
        return time.perf_counter() - t0

    # grow the row sample until one sweep takes a measurable time, then
    # repeat sweeps until about `seconds` of oracle work has been timed
    rows = min(rows_total, 64)
    w, idx = prepare(rows)
    dt = sweep(w, idx, rows)
    while dt < 0.5 and rows < rows_total:
        rows = min(rows_total, rows * 4)
        w, idx = prepare(rows)
        dt = sweep(w, idx, rows)
    total, reps = dt, 1
    while total < seconds:
        total += sweep(w, idx, rows)
        reps += 1
    value = reps * nbytes_per(rows) / total / 1e9
    return value, oracle.threads(), (f"{rows} of {rows_total} weight rows, m in {ms}, {reps} sweeps, "
                                     f"{total:.2f} s")


def oracle_sample_one_core(workload: str, seconds: float):
    """oracle_sample on one host thread (a child process with OMP_NUM_THREADS=1)."""
    env = dict(os.environ, OMP_NUM_THREADS="1")
    code = ("import json, bench; fmt, n, k, batch, ms, g, ci = bench.WORKLOADS[%r][:7]; "
            "print(json.dumps(bench.oracle_sample(fmt, n, k, batch, ms, g, ci, %r)))" % (workload, seconds))
    r = subprocess.run([sys.executable, "-c", code], cwd=ROOT, env=env, capture_output=True, text=True,
                       timeout=int(20 * seconds) + 300)
    if r.returncode != 0:
        return None
    v, cores, desc = json.loads(r.stdout.strip().splitlines()[-1])
    return {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle", "sample": desc}


def run_reference(args):
    fmt, n, k, batch, ms, grouped, ci = WORKLOADS[args.workload][:7]
    per_step = max(0.2, 60.0 / max(1, args.steps + args.warmup))
    vals = []
    for s in range(args.warmup + args.steps):
        v, cores, desc = oracle_sample(fmt, n, k, batch, ms, grouped, ci, per_step)
        if s >= args.warmup:
            vals.append(v)
    value = statistics.median(vals)
    return {
        "impl": "reference", "metric": METRIC, "value": round(value, 4), "unit": "GB/s", "n_gpus": 1,
        "steps": args.steps, "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64 accumulate over exact f32 weights", "data": "synthetic",
        "config": {"workload": args.workload, "format": fmt, "n": n, "k": k, "batch": batch, "m": ms},
        "cpu_baseline": {"value": round(value, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(value, 4), "unit": "GB/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--workload", default=DEFAULT, choices=sorted(WORKLOADS))
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--cpu-seconds", type=float, default=8.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--no-extra", action="store_true", help="time only the selected workload")
    args = ap.parse_args()
    if args.warmup < 3:
        args.warmup = 3

    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))

    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args)), flush=True)
        return

    if world > 1:
        import torch
        torch.cuda.set_device(local_rank)
        torch.distributed.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    res = run_ours(args, rank, world, local_rank)
    if rank == 0:
        if args.no_cpu_baseline:
            res["cpu_baseline"] = None
        else:
            fmt, n, k, batch, ms, grouped, ci = WORKLOADS[args.workload][:7]
            v, cores, desc = oracle_sample(fmt, n, k, batch, ms, grouped, ci, args.cpu_seconds)
            res["cpu_baseline"] = {"value": round(v, 4), "unit": "GB/s", "cores": cores, "kind": "oracle",
                                   "sample": desc}
            res["cpu_baseline_1core"] = oracle_sample_one_core(args.workload, min(4.0, args.cpu_seconds))
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch
        torch.distributed.barrier()
        torch.distributed.destroy_process_group()


if __name__ == "__main__":
    main()
