#!/usr/bin/env python
"""Benchmark of the FP8 scaled-quantize + scaled-GEMM hot path on GB300.

One step = one pass of the path over one batch of the blockwise workload
(4096 x 4096 x 4096): cast-transpose X [4096, 4096] bf16 ~ N(0,1) with 1 % of
columns x100 into row- and column-wise E4M3 with 1x128 scales, cast-transpose
W [4096, 4096] ~ N(0, 0.02) with 128x128 scales, then Y = X W^T (FP8 GEMM,
FP32 accumulation, BF16 out).  Inputs are resident in HBM; L2 is flushed
between timed steps because the inputs fit in L2: a 256 MiB write, then a
256 MiB read, so that the timed region starts from a cold L2 that holds no
dirty lines of the flush (their write-back would otherwise land on the first
kernel of the step).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Prints one JSON line (rank 0).  Besides the step it reports, by default, every
recipe's kernels at the sizes the targets are stated for (`per_recipe`: each a
median of >= 50 event-timed launches with L2 flushed before each), a sustained
window of back-to-back steps for the clock record, the same step end to end
through the C ABI with host buffers (`e2e`), and the CPU oracle timed on the
host cores (`cpu_baseline`).  --impl reference times the CPU oracle on the
whole step instead; --cpu-baseline-sweep [SIZE ...] times the oracle's casts of
every recipe on one thread and on every core (no GPU).
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
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

import numpy as np
import torch

M = N = K = 4096
WORKLOAD = "blockwise fprop 4096x4096x4096: X 1x128 E4M3 (row+col), W 128x128 E4M3 (row+col), Y=XW^T bf16"
METRIC = "FP8 scaled-GEMM TFLOPS & quantize GB/s per recipe, % of GB300 roofline"
UNIT = "TFLOP/s"
FLUSH_BYTES = 256 << 20
KERNEL_REPS = 50          # event-timed launches per kernel figure (median reported)
SUSTAIN_S = 1.5           # back-to-back steps after the timed region, for the clock record
# DRAM bytes (dram__bytes_read.sum + dram__bytes_write.sum) of one blockwise GEMM launch at
# 4096^3 from an ncu capture of the current kernel version; None when not captured for it
TRAFFIC_GEMM = 34_121_472 + 2_049_536


def peaks():
    p = {"hbm_gbs": 6800.0, "bf16_tflops": 1900.0, "bf16_tflops_sustained": 1700.0, "source": "fallback"}
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        with open(path) as f:
            d = json.load(f)
        for k in ("hbm_gbs", "bf16_tflops", "bf16_tflops_sustained"):
            if k in d:
                p[k] = float(d[k])
        p["source"] = "measured"
    return p


def fp8_peak_of(pk):
    """Dense FP8 = 2 x dense BF16 (the nominal 4.5 / 2.25 PFLOP/s ratio), from the burst figure."""
    return 2.0 * pk["bf16_tflops"]


# ------------------------------------------------------------------ clocks
class ClockSampler:
    """nvidia-smi samples every 50 ms, each stamped with the host clock when read, so
    that a window of the run (the timed steps, the sustained steps, the per-recipe
    kernels) can be summarised on its own."""

    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
    REASONS = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]

    def __init__(self, gpu_index: int, out_path: str | None):
        self.gpu = gpu_index
        self.out_path = out_path
        self.proc = None
        self.samples = []       # (host time, raw line)

    def start(self):
        try:
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "50"],
                                         stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            threading.Thread(target=self._read, daemon=True).start()
        except (OSError, ValueError):
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.samples.append((time.monotonic(), line.strip()))

    def stop(self):
        if self.proc is None:
            return
        time.sleep(0.12)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        if self.out_path:
            with open(self.out_path, "w") as f:
                f.write("\n".join(f"{t:.3f},{ln}" for t, ln in self.samples) + "\n")

    def summary(self, windows):
        """Median SM clock, max clock, power and active throttle reasons over the samples
        read inside any of the (t0, t1) windows (host monotonic seconds)."""
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"], "samples": 0}
        sm, smax, pw, reasons = [], [], [], set()
        for t, ln in self.samples:
            if not any(a <= t <= b for a, b in windows):
                continue
            parts = [p.strip() for p in ln.split(",")]
            if len(parts) < 9:
                continue
            try:
                sm.append(float(parts[1]))
                smax.append(float(parts[2]))
                pw.append(float(parts[3]))
            except ValueError:
                continue
            for nm, v in zip(self.REASONS, parts[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(nm)
        return {"sm_mhz": statistics.median(sm) if sm else None, "sm_max_mhz": max(smax) if smax else None,
                "power_w_max": max(pw) if pw else None, "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ distributed
def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif torch.cuda.is_available():
        torch.cuda.set_device(0)
    return rank, world, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(v: float, world: int) -> float:
    if world == 1:
        return v
    import torch.distributed as dist
    t = torch.tensor([v], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ------------------------------------------------------------------ our arm
class Path:
    """Buffers and launches of one step of the blockwise workload."""

    def __init__(self, fq, x, w):
        self.fq = fq
        R, F = fq.Recipe, fq.Format
        self.R, self.F = R, F
        dev = x.device
        self.x, self.w = x, w
        self.qx = torch.empty((M, K), dtype=torch.uint8, device=dev)
        self.sx = torch.empty((M, K // 128), dtype=torch.float32, device=dev)
        self.qxt = torch.empty((K, M), dtype=torch.uint8, device=dev)
        self.sxt = torch.empty((K, M // 128), dtype=torch.float32, device=dev)
        self.qw = torch.empty((N, K), dtype=torch.uint8, device=dev)
        self.sw = torch.empty((N // 128, K // 128), dtype=torch.float32, device=dev)
        self.qwt = torch.empty((K, N), dtype=torch.uint8, device=dev)
        self.swt = torch.empty((K // 128, N // 128), dtype=torch.float32, device=dev)
        self.y = torch.empty((M, N), dtype=torch.bfloat16, device=dev)
        self.launches_per_step = 2

    def cast_x(self):
        self.fq.fp8_cast_transpose(self.x, self.R.BLOCK_1x128, self.F.E4M3, None, None, self.qx, self.sx, self.qxt,
                                   self.sxt)

    def cast_w(self):
        self.fq.fp8_cast_transpose(self.w, self.R.BLOCK_128x128, self.F.E4M3, None, None, self.qw, self.sw, self.qwt,
                                   self.swt)

    def casts(self):
        # both casts in one launch (fp8_cast_transpose_multi; a kernel compiled for this pairing):
        # one grid start and one tail instead of two (the step 94.2-94.7 against 94.7-96.0 us)
        R, F = self.R, self.F
        self.fq.fp8_cast_transpose_multi([(self.x, R.BLOCK_1x128, F.E4M3, None, None, self.qx, self.sx, self.qxt, self.sxt),
                                          (self.w, R.BLOCK_128x128, F.E4M3, None, None, self.qw, self.sw, self.qwt, self.swt)])

    def gemm(self):
        self.fq.fp8_scaled_gemm(self.qx, self.F.E4M3, self.R.BLOCK_1x128, self.sx, self.qw, self.F.E4M3,
                                self.R.BLOCK_128x128, self.sw, self.y)

    def step(self):
        self.casts()
        self.gemm()


def bytes_cast(recipe_name, r, c, in_bytes=2):
    """Algorithmic bytes of a row + column cast-transpose of an r x c matrix: the input read
    (2 B per element for bf16, 4 B for float32) and 1 B + 1 B written per element, plus the
    scale arrays of both copies."""
    extra = {"TENSOR": 0, "BLOCK_1x128": 2 * (r * c // 128) * 4, "BLOCK_128x128": 2 * (r * c // 16384) * 4,
             "MX_1x32": 2 * (r * c // 32), "MX_1x32_TILED": 2 * (r * c // 32)}[recipe_name]
    return (in_bytes + 2) * r * c + extra


class L2Flush:
    """Between timed regions: write a buffer larger than L2 (evicting every input),
    then read another one, so that the write's dirty lines are written back before the
    next timed region instead of during its first kernel (measured: up to 8 us on a
    cast of 268 MB)."""

    def __init__(self, dev):
        self.w = torch.empty(FLUSH_BYTES, dtype=torch.uint8, device=dev)
        self.r = torch.ones(FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
        self.out = torch.empty((), dtype=torch.float32, device=dev)

    def __call__(self):
        self.w.zero_()
        torch.amax(self.r, dim=0, out=self.out)


def _capture(fn):
    """Capture `fn` (a sequence of C-ABI calls on the current stream) in a CUDA graph."""
    g = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        fn()                     # warm: attributes and caches set outside the capture
    torch.cuda.current_stream().wait_stream(side)
    torch.cuda.synchronize()
    with torch.cuda.graph(g):
        fn()
    torch.cuda.synchronize()
    return g


def time_kernel(fn, reps=KERNEL_REPS, flush=None, warm=10):
    """Median of `reps` launches, each alone between two events on the launching stream,
    L2 flushed before each (the flush is enqueued ahead of the first event, so the host
    enqueues the launch while the flush runs and the events see the kernel alone)."""
    s = torch.cuda.current_stream()
    for _ in range(warm):
        fn()
    es = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(reps)]
    for a, b in es:
        if flush is not None:
            flush()
        a.record(s)
        fn()
        b.record(s)
    torch.cuda.synchronize()
    return statistics.median(a.elapsed_time(b) for a, b in es)


def time_in_step(path, steps, flush):
    """The GEMM as it runs inside the step: a graph of the step's two launches with an
    event-record node before and after the GEMM (external events, so that they are nodes
    of the graph), replayed `steps` times with L2 flushed before each replay.  Returns the
    GEMM's times in ms, or None where this torch cannot record events inside a graph."""
    try:
        ea = torch.cuda.Event(enable_timing=True, external=True)
        eb = torch.cuda.Event(enable_timing=True, external=True)
    except TypeError:
        return None

    def body():
        path.casts()
        ea.record()
        path.gemm()
        eb.record()

    g = _capture(body)
    ts = []
    for _ in range(steps):
        flush()
        g.replay()
        torch.cuda.synchronize()
        ts.append(ea.elapsed_time(eb))
    return ts


def run_ours(args, rank, world):
    import scaled_quantize_gemm_amax_gb300 as fq
    from scaled_quantize_gemm_amax_gb300 import build as fqbuild
    from scaled_quantize_gemm_amax_gb300 import workloads as wl

    fqbuild.build()
    fq.load_library()
    dev = torch.device("cuda", torch.cuda.current_device())
    x, w = wl.cfg2_blockwise(dev)
    path = Path(fq, x, w)
    flush = L2Flush(dev)
    stream = torch.cuda.current_stream()
    clocks = ClockSampler(torch.cuda.current_device(), args.clocks_csv)
    clocks.start()

    # the timed step is one CUDA graph of the two launches (no host launch cost inside it)
    g_step = _capture(path.step)
    for _ in range(args.warmup):
        g_step.replay()
        flush()
    torch.cuda.synchronize()
    assert fq.fp8_get_device_status() == fq.Status.OK

    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(args.steps)]
    time.sleep(0.2)
    barrier(world)
    torch.cuda.synchronize()
    t_timed0 = time.monotonic()
    for i in range(args.steps):
        ev[i][0].record(stream)
        g_step.replay()
        ev[i][1].record(stream)
        flush()          # outside the step's events: L2 does not carry inputs across steps
    torch.cuda.synchronize()
    t_timed1 = time.monotonic()
    barrier(world)
    st = fq.fp8_get_device_status()
    assert st == fq.Status.OK, st
    step_times = [a.elapsed_time(b) for a, b in ev]
    step_ms = max_over_ranks(statistics.mean(step_times), world)
    sustained = run_sustained(fq, wl, dev, x, w, path)

    # per-kernel breakdown of the step: each launch alone, L2 flushed before it (the two casts
    # also one at a time, for their own rates)
    t_cc = time_kernel(path.casts, flush=flush)
    t_cx = time_kernel(path.cast_x, flush=flush)
    t_cw = time_kernel(path.cast_w, flush=flush)
    g_ms = time_kernel(path.gemm, flush=flush)
    g_in_step = time_in_step(path, KERNEL_REPS, flush)

    flops = 2.0 * M * N * K
    pk = peaks()
    fp8_peak = fp8_peak_of(pk)
    gemm_tflops = flops / (g_ms * 1e-3) / 1e12
    cx_gbs = bytes_cast("BLOCK_1x128", M, K) / (t_cx * 1e-3) / 1e9
    cw_gbs = bytes_cast("BLOCK_128x128", N, K) / (t_cw * 1e-3) / 1e9
    cc_gbs = (bytes_cast("BLOCK_1x128", M, K) + bytes_cast("BLOCK_128x128", N, K)) / (t_cc * 1e-3) / 1e9
    value = world * flops / (step_ms * 1e-3) / 1e12

    result = {
        "metric": METRIC, "value": round(value, 2), "unit": UNIT, "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(step_ms, 5), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "fp8-e4m3 (fp32 accumulate, bf16 out)",
        "data": "synthetic (seeded N(0,1) + 1% columns x100 / N(0,0.02))",
        "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K, "recipe": "blockwise 1x128 x 128x128",
                   "l2": "flushed between steps (256 MiB write, then 256 MiB read)", "launch": "one CUDA graph per step",
                   "parallelism": f"replicas x{world}"},
        "step_ms_median": round(statistics.median(step_times), 5),
        "kernels": {
            "stat": f"median of {KERNEL_REPS} launches, L2 flushed before each",
            "cast_transpose_x_and_w (the step's one two-job launch)": {
                "us": round(t_cc * 1e3, 2), "GB/s": round(cc_gbs, 1), "frac_hbm": round(cc_gbs / pk["hbm_gbs"], 4)},
            "cast_transpose_x_1x128": {"us": round(t_cx * 1e3, 2), "GB/s": round(cx_gbs, 1),
                                       "frac_hbm": round(cx_gbs / pk["hbm_gbs"], 4)},
            "cast_transpose_w_128x128": {"us": round(t_cw * 1e3, 2), "GB/s": round(cw_gbs, 1),
                                         "frac_hbm": round(cw_gbs / pk["hbm_gbs"], 4)},
            "gemm_blockwise": {"us": round(g_ms * 1e3, 2), "TFLOP/s": round(gemm_tflops, 1),
                               "frac_fp8": round(gemm_tflops / fp8_peak, 4)},
        },
        "roofline": {"bound": "tensor", "achieved": round(gemm_tflops, 1), "peak": round(fp8_peak, 1),
                     "unit": "TFLOP/s", "frac": round(gemm_tflops / fp8_peak, 4), "traffic": TRAFFIC_GEMM,
                     "peak_source": f"{pk['source']}: 2 x bf16 burst ({pk['bf16_tflops']})"},
        "gpu_launches": path.launches_per_step * args.steps,
        "sustained": {k: v for k, v in sustained.items() if k not in ("t0", "t1")},
    }
    if g_in_step:
        m_in, med_in = statistics.mean(g_in_step), statistics.median(g_in_step)
        tf_in = flops / (m_in * 1e-3) / 1e12
        result["kernels"]["gemm_blockwise_in_step"] = {
            "us": round(m_in * 1e3, 2), "us_median": round(med_in * 1e3, 2), "TFLOP/s": round(tf_in, 1),
            "frac_fp8": round(tf_in / fp8_peak, 4),
            "stat": f"mean of {len(g_in_step)} replays of the step as a graph with events around the GEMM node, "
                    "L2 flushed before each (operands as the casts leave them)"}
    t_pr0 = time.monotonic()
    if not args.no_per_recipe:
        result["per_recipe"] = run_per_recipe(fq, wl, dev, flush)
    t_pr1 = time.monotonic()
    clocks.stop()
    ck = clocks.summary([(t_timed0, t_timed1), (sustained["t0"], sustained["t1"])])
    ck["window"] = "the timed steps and the sustained back-to-back steps that follow them"
    ck["timed_region_samples"] = clocks.summary([(t_timed0, t_timed1)])["samples"]
    result["clocks"] = ck
    if not args.no_per_recipe:
        result["per_recipe"]["clocks"] = clocks.summary([(t_pr0, t_pr1)])
    result["quality_vs_bf16"] = quality_vs_bf16(fq, x, w)
    if not args.no_e2e:
        result["e2e"] = run_e2e(fq, x, w, args, world)
    if rank == 0 and world == 1 and not args.no_cpu_baseline:
        result["cpu_baseline"] = cpu_baseline(x, w)
    return result


def run_sustained(fq, wl, dev, x, w, path):
    """Back-to-back steps for about SUSTAIN_S seconds, rotating over four input sets
    (the first is the timed step's own) so that each step's inputs come from HBM
    without a flush between steps: 4 x 64 MiB of bf16 inputs plus their FP8 copies
    exceed L2.  Timed with two events around the whole window; it gives the clock
    sampler a window under load."""
    paths = [path] + [Path(fq, x.roll(i, 0).contiguous(), w.roll(i, 0).contiguous()) for i in (1, 2, 3)]
    graphs = [_capture(p.step) for p in paths]
    stream = torch.cuda.current_stream()
    for g in graphs:
        g.replay()
    torch.cuda.synchronize()
    # size the window from one round's time
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(stream)
    for g in graphs:
        g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    per_round_s = max(e0.elapsed_time(e1) * 1e-3, 1e-5)
    rounds = max(1, int(SUSTAIN_S / per_round_s))
    t0 = time.monotonic()
    e0.record(stream)
    for _ in range(rounds):
        for g in graphs:
            g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    t1 = time.monotonic()
    assert fq.fp8_get_device_status() == fq.Status.OK
    n = rounds * len(graphs)
    ms = e0.elapsed_time(e1) / n
    return {"steps": n, "seconds": round(e0.elapsed_time(e1) * 1e-3, 3), "ms_per_step": round(ms, 5),
            "TFLOP/s": round(2.0 * M * N * K / (ms * 1e-3) / 1e12, 1),
            "inputs": "four input sets in turn (512 MiB of bf16 with their FP8 copies), no flush", "t0": t0, "t1": t1}


def quality_vs_bf16(fq, x, w):
    """Informative only (no parity claim): ||Y_fp8 - Y_bf16||_F / ||Y_bf16||_F on the bench's
    X, W for each recipe pairing, Y_bf16 being the BF16 product with FP32 accumulation that the
    FP8 path replaces (computed by torch's matmul, outside the path)."""
    R, F = fq.Recipe, fq.Format
    y_ref = (x @ w.t()).double()
    nref = torch.linalg.norm(y_ref)
    out = {}
    for name, ra, rb in (("per_tensor_current", R.TENSOR, R.TENSOR), ("blockwise", R.BLOCK_1x128, R.BLOCK_128x128),
                         ("mxfp8", R.MX_1x32_TILED, R.MX_1x32_TILED)):
        sa_t = sb_t = None
        if ra == R.TENSOR:
            sa_t, sb_t = torch.empty(1, device=x.device), torch.empty(1, device=x.device)
            for t, sc in ((x, sa_t), (w, sb_t)):
                am = torch.empty(1, device=x.device)
                fq.fp8_amax(t, am)
                fq.fp8_compute_scale(am, F.E4M3, sc, torch.empty(1, device=x.device))
        qa, sa, _, _ = fq.cast_transpose(x, ra, F.E4M3, sa_t, col=False)
        qb, sb, _, _ = fq.cast_transpose(w, rb, F.E4M3, sb_t, col=False)
        y = fq.scaled_gemm(qa, F.E4M3, ra, sa, qb, F.E4M3, rb, sb)
        out[name] = round(float(torch.linalg.norm(y.double() - y_ref) / nref), 6)
    out["note"] = "relative Frobenius difference from the BF16 product (X with 1 % of columns x100), E4M3"
    return out


def run_per_recipe(fq, wl, dev, flush):
    """Every recipe's kernels at the sizes the targets are stated for: cast-transpose
    (row + column copies) of each recipe and the amax at 8192^2, 16384^2 and 32768^2;
    the GEMM of each recipe pairing at 4096^3 and 8192^3, the MXFP8 LLaMA-7B linears,
    the blockwise weight-gradient pairing, and the per-tensor (delayed-scaling)
    GPT-175B linears' fprop / dgrad / wgrad; dequantization, the fused output
    quantization and the FP8 gradient all-reduce.  Each figure is the median of
    KERNEL_REPS launches with L2 flushed before each."""
    R, F, O = fq.Recipe, fq.Format, fq.OutDtype
    pk = peaks()
    hbm = pk["hbm_gbs"]
    fp8 = fp8_peak_of(pk)
    out = {"stat": f"median of {KERNEL_REPS} launches, L2 flushed before each",
           "peaks": {"hbm_GB/s": hbm, "fp8_TFLOP/s": fp8, "source": pk["source"]},
           "cast_transpose": {}, "amax": {}, "gemm": {}, "dequantize": {}, "fused_gemm_amax": {}, "allreduce": {}}

    def bw(us_ms, nbytes):
        gbs = nbytes / (us_ms * 1e-3) / 1e9
        return {"us": round(us_ms * 1e3, 2), "GB/s": round(gbs, 1), "frac_hbm": round(gbs / hbm, 4)}

    def tf(us_ms, flops):
        t = flops / (us_ms * 1e-3) / 1e12
        return {"us": round(us_ms * 1e3, 2), "TFLOP/s": round(t, 1), "frac_fp8": round(t / fp8, 4)}

    one = torch.ones(1, dtype=torch.float32, device=dev)
    # ---- cast-transpose and amax (bandwidth sweep inputs: N(0,1), 0.1 % of elements x1000)
    for size in (8192, 16384, 32768):
        x = wl.cfg5_sweep(size, dev)
        for rec in (R.TENSOR, R.BLOCK_1x128, R.BLOCK_128x128, R.MX_1x32_TILED):
            sc = one if rec == R.TENSOR else None
            qr, sr, qc, scol = fq.cast_transpose(x, rec, F.E4M3, sc)
            ms = time_kernel(lambda: fq.fp8_cast_transpose(x, rec, F.E4M3, sc, None, qr, sr, qc, scol), flush=flush)
            out["cast_transpose"][f"{rec.name}_{size}"] = bw(ms, bytes_cast(rec.name, size, size))
            del qr, sr, qc, scol
        amax = torch.empty(1, dtype=torch.float32, device=dev)
        ms = time_kernel(lambda: fq.fp8_amax(x, amax), flush=flush)
        out["amax"][str(size)] = bw(ms, 2 * size * size)
        if size == 16384:
            for rec in (R.TENSOR, R.BLOCK_1x128, R.BLOCK_128x128, R.MX_1x32_TILED):
                sc = one if rec == R.TENSOR else None
                q, sq, _, _ = fq.cast_transpose(x, rec, F.E4M3, sc, col=False)
                y = torch.empty((size, size), dtype=torch.bfloat16, device=dev)
                ms = time_kernel(lambda: fq.fp8_dequantize(q, rec, F.E4M3, sq, y), flush=flush)
                out["dequantize"][f"{rec.name}_{size}"] = bw(ms, 3 * size * size + sq.numel() * sq.element_size())
                del q, sq, y
        del x
        torch.cuda.empty_cache()

    # ---- the FP32 master copy of a weight quantized directly (binary32 input, 4 B read per element)
    out["cast_transpose_f32"] = {}
    w32 = wl.normal_bf16((8192, 8192), 7, 0.02, dev).float()
    for rec in (R.TENSOR, R.BLOCK_1x128, R.BLOCK_128x128, R.MX_1x32_TILED):
        sc = one if rec == R.TENSOR else None
        qr, sr, qc, scol = fq.cast_transpose(w32, rec, F.E4M3, sc)
        ms = time_kernel(lambda: fq.fp8_cast_transpose_f32(w32, rec, F.E4M3, sc, None, qr, sr, qc, scol), flush=flush)
        out["cast_transpose_f32"][f"{rec.name}_8192"] = bw(ms, bytes_cast(rec.name, 8192, 8192, in_bytes=4))
        del qr, sr, qc, scol
    del w32

    # ---- GEMMs
    shapes = [("tensor_4096", R.TENSOR, R.TENSOR, (4096, 4096, 4096), F.E4M3, F.E4M3, O.BF16),
              ("tensor_8192", R.TENSOR, R.TENSOR, (8192, 8192, 8192), F.E4M3, F.E4M3, O.BF16),
              ("blockwise_4096", R.BLOCK_1x128, R.BLOCK_128x128, (4096, 4096, 4096), F.E4M3, F.E4M3, O.BF16),
              ("blockwise_8192", R.BLOCK_1x128, R.BLOCK_128x128, (8192, 8192, 8192), F.E4M3, F.E4M3, O.BF16),
              # K / 128 odd: the 256 x 160 pair tiles with 128-deep stages
              ("blockwise_4096x4096x4224", R.BLOCK_1x128, R.BLOCK_128x128, (4096, 4096, 4224), F.E4M3, F.E4M3, O.BF16),
              ("blockwise_wgrad_4096", R.BLOCK_1x128, R.BLOCK_1x128, (4096, 4096, 4096), F.E4M3, F.E4M3, O.FP32),
              ("blockwise_wgrad_8192", R.BLOCK_1x128, R.BLOCK_1x128, (8192, 8192, 8192), F.E4M3, F.E4M3, O.FP32),
              ("mx_4096", R.MX_1x32_TILED, R.MX_1x32_TILED, (4096, 4096, 4096), F.E4M3, F.E4M3, O.BF16),
              ("mx_8192", R.MX_1x32_TILED, R.MX_1x32_TILED, (8192, 8192, 8192), F.E4M3, F.E4M3, O.BF16)]
    shapes += [(f"mx_llama7b_{k}", R.MX_1x32_TILED, R.MX_1x32_TILED, v, F.E4M3, F.E4M3, O.BF16)
               for k, v in wl.CFG3_SHAPES.items()]
    # GPT-175B linears (2048 tokens), per-tensor (delayed) scaling: fprop E4M3 x E4M3 -> bf16,
    # dgrad E5M2 dY x E4M3 W -> bf16, wgrad E5M2 dY^T x E4M3 X^T -> fp32
    t = wl.CFG4_TOKENS
    for lin, (fin, fout) in wl.CFG4_LINEARS.items():
        shapes += [(f"gpt175b_{lin}_fprop", R.TENSOR, R.TENSOR, (t, fout, fin), F.E4M3, F.E4M3, O.BF16),
                   (f"gpt175b_{lin}_dgrad", R.TENSOR, R.TENSOR, (t, fin, fout), F.E5M2, F.E4M3, O.BF16),
                   (f"gpt175b_{lin}_wgrad", R.TENSOR, R.TENSOR, (fout, fin, t), F.E5M2, F.E4M3, O.FP32)]
    qkv_in, qkv_out = wl.CFG4_LINEARS["qkv"]
    shapes += [("gpt175b_qkv_wgrad_blockwise", R.BLOCK_1x128, R.BLOCK_1x128, (qkv_out, qkv_in, t), F.E5M2, F.E4M3,
                O.FP32)]
    for name, ra, rb, (m, n, k), fa, fb, od in shapes:
        a = wl.normal_bf16((m, k), 1, 1.0, dev)
        b = wl.normal_bf16((n, k), 2, 0.02, dev)
        qa, sa, _, _ = fq.cast_transpose(a, ra, fa, one if ra == R.TENSOR else None, col=False)
        qb, sb, _, _ = fq.cast_transpose(b, rb, fb, one if rb == R.TENSOR else None, col=False)
        del a, b
        c = torch.empty((m, n), dtype=torch.float32 if od == O.FP32 else torch.bfloat16, device=dev)
        ms = time_kernel(lambda: fq.fp8_scaled_gemm(qa, fa, ra, sa, qb, fb, rb, sb, c, od), flush=flush)
        out["gemm"][name] = dict(tf(ms, 2.0 * m * n * k), M=m, N=n, K=k)
        del qa, qb, sa, sb, c

    # ---- fused output quantization (per-tensor, delayed scale) against the unfused chain
    s = 8192
    a = wl.normal_bf16((s, s), 1, 1.0, dev)
    b = wl.normal_bf16((s, s), 2, 0.02, dev)
    qa, sa, _, _ = fq.cast_transpose(a, R.TENSOR, F.E4M3, one, col=False)
    qb, sb, _, _ = fq.cast_transpose(b, R.TENSOR, F.E4M3, one, col=False)
    c = torch.empty((s, s), dtype=torch.bfloat16, device=dev)
    c_q = torch.empty((s, s), dtype=torch.uint8, device=dev)
    c_amax = torch.empty(1, dtype=torch.float32, device=dev)
    c_sinv = torch.empty(1, dtype=torch.float32, device=dev)
    c_scale = torch.full((1,), 64.0, dtype=torch.float32, device=dev)
    ms = time_kernel(lambda: fq.fp8_scaled_gemm_amax(qa, F.E4M3, R.TENSOR, sa, qb, F.E4M3, R.TENSOR, sb, None,
                                                     O.BF16, c_amax, c_scale, F.E4M3, c_q, c_sinv), flush=flush)

    def unfused():
        fq.fp8_scaled_gemm(qa, F.E4M3, R.TENSOR, sa, qb, F.E4M3, R.TENSOR, sb, c)
        fq.fp8_quantize(c, R.TENSOR, F.E4M3, c_scale, c_amax, c_q, c_sinv)

    ms_u = time_kernel(unfused, flush=flush)
    out["fused_gemm_amax"]["tensor_8192"] = dict(tf(ms, 2.0 * s ** 3), unfused_us=round(ms_u * 1e3, 2))
    del a, b, qa, qb, c, c_q

    # ---- FP8 gradient all-reduce: 8 ranks' 8192^2 gradients ~ N(0, 1e-3): amax pass (2 B/elem),
    # then cast and sum (2 B read + 1 B payload per rank element, 4 B per reduced element)
    kr, n = 8, 8192 * 8192
    g = (torch.randn((kr, n), generator=torch.Generator(device=dev).manual_seed(9), device=dev) * 1e-3).to(
        torch.bfloat16)
    amax = torch.empty(1, dtype=torch.float32, device=dev)
    q = torch.empty((kr, n), dtype=torch.uint8, device=dev)
    si = torch.empty(1, dtype=torch.float32, device=dev)
    red = torch.empty(n, dtype=torch.float32, device=dev)
    ms = time_kernel(lambda: fq.fp8_allreduce_sum(g, F.E5M2, amax, q, si, red), flush=flush)
    out["allreduce"]["8x8192^2"] = bw(ms, kr * n * 2 + kr * n * 3 + 4 * n)
    del g, q, red
    torch.cuda.synchronize()
    assert fq.fp8_get_device_status() == fq.Status.OK
    torch.cuda.empty_cache()
    return out


def run_e2e(fq, x, w, args, world):
    """The same step through the public API with host buffers: every step copies X and W
    from pinned host memory, runs the three calls, and copies Y back to pinned host
    memory, all inside the timed region.  Consecutive steps overlap on three streams
    (copy in, compute, copy out) with two sets of device buffers."""
    xh = x.cpu().pin_memory()
    wh = w.cpu().pin_memory()
    paths = [Path(fq, torch.empty_like(x), torch.empty_like(w)) for _ in range(2)]
    yh = [torch.empty((M, N), dtype=torch.bfloat16).pin_memory() for _ in range(2)]
    s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
    comp = torch.cuda.current_stream()
    ev = lambda: torch.cuda.Event()
    in_done, comp_done, out_done = [ev(), ev()], [ev(), ev()], [ev(), ev()]
    steps = max(4, min(args.steps, 64))

    def run(n):
        for i in range(n):
            b = i % 2
            p = paths[b]
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(comp_done[b])          # buffer b's previous step has been consumed
                p.x.copy_(xh, non_blocking=True)
                p.w.copy_(wh, non_blocking=True)
                in_done[b].record(s_in)
            comp.wait_event(in_done[b])
            if i >= 2:
                comp.wait_event(out_done[b])              # buffer b's previous result has left
            p.step()
            comp_done[b].record(comp)
            with torch.cuda.stream(s_out):
                s_out.wait_event(comp_done[b])
                yh[b].copy_(p.y, non_blocking=True)
                out_done[b].record(s_out)

    run(4)
    torch.cuda.synchronize()
    barrier(world)
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    e0.record(comp)
    s_in.wait_event(e0)
    s_out.wait_event(e0)
    run(steps)
    comp.wait_stream(s_in)
    comp.wait_stream(s_out)
    e1.record(comp)
    torch.cuda.synchronize()
    ms = max_over_ranks(e0.elapsed_time(e1) / steps, world)
    # the last results did reach the host
    assert torch.equal(yh[(steps - 1) % 2], paths[(steps - 1) % 2].y.cpu())
    return {"value": round(world * 2.0 * M * N * K / (ms * 1e-3) / 1e12, 2), "unit": UNIT,
            "ms_per_step": round(ms, 4), "steps": steps, "overlap": "copy-in / compute / copy-out streams",
            "h2d_bytes_per_step": int(xh.numel() * 2 + wh.numel() * 2), "d2h_bytes_per_step": int(M * N * 2)}


# ------------------------------------------------------------------ oracle (CPU) legs
def _bits(t):
    return t.contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def _oracle_quantize_rows(oracle, xh, kind, threads):
    """Row-wise oracle quantization of xh by `threads` host threads, each on its own run
    of 128-row slabs (the oracle's C functions release the interpreter lock while they
    run; the slabs are independent for the 1x128 and 128x128 recipes, so the result is
    the single call's, byte for byte)."""
    rows = xh.shape[0]
    per = -(-(rows // 128) // threads) * 128
    bounds = [(r0, min(rows, r0 + per)) for r0 in range(0, rows, per)]
    res = [None] * len(bounds)

    def work(i):
        r0, r1 = bounds[i]
        res[i] = oracle.quantize_rowwise(np.ascontiguousarray(xh[r0:r1]), kind, oracle.E4M3)

    ts = [threading.Thread(target=work, args=(i,)) for i in range(len(bounds))]
    for t in ts:
        t.start()
    for t in ts:
        t.join()
    return np.concatenate([r[0] for r in res]), np.concatenate([r[1] for r in res])


def _oracle_step(oracle, xh, wh, threads, gemm=True):
    """One step of the workload on the oracle: X 1x128 and W 128x128, row-wise and
    column-wise copies (quantization on `threads` host threads), then the GEMM
    C = deq(X) deq(W)^T in float64 (the library matmul on its own thread pool).
    Returns (quantize seconds, GEMM seconds)."""
    t0 = time.perf_counter()
    qx, sx = _oracle_quantize_rows(oracle, xh, oracle.KIND_1x128, threads)
    _oracle_quantize_rows(oracle, oracle.transpose_bf16(xh), oracle.KIND_1x128, threads)
    qw, sw = _oracle_quantize_rows(oracle, wh, oracle.KIND_128x128, threads)
    _oracle_quantize_rows(oracle, oracle.transpose_bf16(wh), oracle.KIND_128x128, threads)
    t1 = time.perf_counter()
    if gemm:
        oracle.scaled_gemm(qx, oracle.E4M3, oracle.KIND_1x128, sx, qw, oracle.E4M3, oracle.KIND_128x128, sw)
    return t1 - t0, time.perf_counter() - t1


def cpu_baseline(x, w):
    """The oracle as it stands on the host cores, on the whole step: quantization on
    one thread and on every core (threads over 128-row slabs), the float64 GEMM on the
    matmul library's thread pool (all cores).  value = the step's flops / the
    all-core step time."""
    import oracle
    oracle.build()
    xh, wh = _bits(x), _bits(w)
    cores = os.cpu_count()
    tq1, _ = _oracle_step(oracle, xh, wh, 1, gemm=False)
    tq, tg = _oracle_step(oracle, xh, wh, cores)
    step_s = tq + tg
    return {"value": round(2.0 * M * N * K / step_s / 1e12, 6), "unit": UNIT, "cores": cores, "kind": "oracle",
            "sample": (f"the whole step on the oracle, measured once: quantization of X and W (row + column "
                       f"copies) {tq1:.3f} s on 1 thread, {tq:.3f} s on {cores} threads; float64 GEMM of the full "
                       f"4096^3 product {tg:.3f} s on the matmul library's threads; all-core step {step_s:.3f} s"),
            "single_thread_quantize_s": round(tq1, 4), "all_core_quantize_s": round(tq, 4),
            "gemm_s": round(tg, 4), "all_core_step_s": round(step_s, 4)}


def _oracle_cast_both(oracle, xh, kind, threads, scale=None):
    """Row + column copies of xh on the oracle, `threads` host threads: each thread takes
    a run of 128-row slabs for the row-wise copy and a run of 128-column slabs (its slab
    transposed, then the row-wise recipe: the column-wise copy's definition) for the
    column-wise one.  Returns the (q, s) pieces of each copy in order (slabs of the
    row-wise copy's rows, then of the column-wise copy's rows), not joined."""
    rows, cols = xh.shape

    def runs(n):
        per = -(-(n // 128) // threads) * 128
        return [(a, min(n, a + per)) for a in range(0, n, per)]

    jobs = ([(lambda r0=r0, r1=r1: np.ascontiguousarray(xh[r0:r1])) for r0, r1 in runs(rows)] +
            [(lambda c0=c0, c1=c1: oracle.transpose_bf16(np.ascontiguousarray(xh[:, c0:c1]))) for c0, c1 in runs(cols)])
    out = [None] * len(jobs)

    def work(i):
        out[i] = oracle.quantize_rowwise(jobs[i](), kind, oracle.E4M3, scale)

    ts = [threading.Thread(target=work, args=(i,)) for i in range(len(jobs))]
    for i in range(0, len(ts), threads):
        for t in ts[i:i + threads]:
            t.start()
        for t in ts[i:i + threads]:
            t.join()
    n_row = len(runs(rows))
    return out[:n_row], out[n_row:]


def cpu_baseline_sweep(sizes):
    """The oracle's casts (row + column copies, E4M3) for every recipe on s x s inputs of
    the bandwidth-sweep recipe (N(0, 1), 0.1 % of elements x1000, generated on the host):
    one thread and every core for s <= 16384, every core only above (one run each).
    Per-tensor current scaling includes its amax and scale.  GB/s counts the same
    algorithmic bytes as the GPU casts.  Needs no GPU."""
    import oracle
    from scaled_quantize_gemm_amax_gb300 import workloads as wl
    oracle.build()
    cores = os.cpu_count()
    recipes = (("TENSOR", oracle.KIND_TENSOR), ("BLOCK_1x128", oracle.KIND_1x128),
               ("BLOCK_128x128", oracle.KIND_128x128), ("MX_1x32", oracle.KIND_MX))
    rows = []
    for s in sizes:
        xh = _bits(wl.cfg5_sweep(s, "cpu"))
        for name, kind in recipes:
            for threads in ((1, cores) if s <= 16384 else (cores,)):
                t0 = time.perf_counter()
                scale = None
                if kind == oracle.KIND_TENSOR:
                    scale = oracle.tensor_scale(oracle.amax(xh), oracle.E4M3)[0]
                _oracle_cast_both(oracle, xh, kind, threads, scale)
                sec = time.perf_counter() - t0
                gbs = bytes_cast(name, s, s) / sec / 1e9
                rows.append({"size": s, "recipe": name, "threads": threads, "s": round(sec, 4),
                             "GB/s": round(gbs, 4)})
                print(f"# oracle cast {name} {s}^2 on {threads} thread(s): {sec:.3f} s, {gbs:.3f} GB/s",
                      file=sys.stderr, flush=True)
        del xh
    return {"kind": "oracle", "what": "row + column casts, E4M3, every recipe", "cores": cores,
            "host": os.uname().machine, "inputs": "s x s ~ N(0, 1), 0.1 % of elements x1000, host generator",
            "runs": rows}


def run_reference(args, rank, world):
    """The oracle as the reference arm: every step is the whole workload on the host
    cores (see _oracle_step), measured, not extrapolated."""
    import oracle
    from scaled_quantize_gemm_amax_gb300 import workloads as wl

    if rank != 0:
        return None
    x, w = wl.cfg2_blockwise("cpu")
    xh, wh = _bits(x), _bits(w)
    oracle.build()
    cores = os.cpu_count()
    for _ in range(args.warmup):
        _oracle_step(oracle, xh, wh, cores)
    times = []
    t_start = time.perf_counter()
    for _ in range(args.steps):
        tq, tg = _oracle_step(oracle, xh, wh, cores)
        times.append((tq, tg))
    wall = time.perf_counter() - t_start
    step_s = wall / args.steps
    value = 2.0 * M * N * K / step_s / 1e12
    info = (f"each step the whole workload on the oracle: quantization of X and W (row + column copies) on "
            f"{cores} threads (median {statistics.median(t for t, _ in times):.3f} s), float64 GEMM of the full "
            f"4096^3 product on the matmul library's threads (median {statistics.median(g for _, g in times):.3f} s)")
    return {"impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": UNIT, "n_gpus": 1,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(step_s * 1e3, 3),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 oracle (fp8 codes)",
            "data": "synthetic (seeded, CPU generator)",
            "config": {"workload": WORKLOAD, "M": M, "N": N, "K": K, "recipe": "blockwise 1x128 x 128x128",
                       "parallelism": f"cpu x{cores} threads"},
            "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": cores, "kind": "oracle",
                             "sample": info},
            "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "wall_s": round(wall, 2)}


CASES = ("cast_tensor", "cast_1x128", "cast_128x128", "cast_mx", "cast_f32_tensor", "cast_f32_1x128", "cast_f32_128x128",
         "cast_f32_mx", "amax", "amax_f32", "gemm_tensor", "gemm_block", "gemm_mx",
         "gemm_block_wgrad", "gemm_amax", "dequant_tensor", "dequant_1x128", "dequant_128x128", "dequant_mx", "allreduce",
         "cast_step")


def run_case(args):
    """One kernel in a loop (for profiling): cast cases on a size x size input of the
    bandwidth sweep, GEMM cases at size^3.  Prints the median time as JSON."""
    import scaled_quantize_gemm_amax_gb300 as fq
    from scaled_quantize_gemm_amax_gb300 import build as fqbuild
    from scaled_quantize_gemm_amax_gb300 import workloads as wl

    fqbuild.build()
    fq.load_library()
    R, F = fq.Recipe, fq.Format
    dev = torch.device("cuda", 0)
    s = args.size
    flush = L2Flush(dev)
    pk = peaks()
    if args.case == "cast_step":
        # the step's one launch of both casts (X 1x128, W 128x128, row + col) on its 4096^2 inputs
        x, w = wl.cfg2_blockwise(dev)
        path = Path(fq, x, w)
        ms = time_kernel(path.casts, reps=args.steps, flush=flush)
        nbytes = bytes_cast("BLOCK_1x128", M, K) + bytes_cast("BLOCK_128x128", N, K)
        res = {"case": args.case, "size": M, "us": round(ms * 1e3, 2), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1)}
        res["frac_hbm"] = round(res["GB/s"] / pk["hbm_gbs"], 4)
    elif args.case.startswith("cast") or args.case.startswith("amax"):
        x = wl.cfg5_sweep(s, dev) if s in wl.CFG5_SIZES else wl.normal_bf16((s, s), 5, 1.0, dev)
        f32 = "f32" in args.case
        if f32:
            x = x.float()
        rec = {"cast_tensor": R.TENSOR, "cast_1x128": R.BLOCK_1x128, "cast_128x128": R.BLOCK_128x128,
               "cast_mx": R.MX_1x32_TILED, "amax": None, "amax_f32": None, "cast_f32_tensor": R.TENSOR,
               "cast_f32_1x128": R.BLOCK_1x128, "cast_f32_128x128": R.BLOCK_128x128,
               "cast_f32_mx": R.MX_1x32_TILED}[args.case]
        if rec is None:
            amax = torch.empty(1, dtype=torch.float32, device=dev)
            fn = (lambda: fq.fp8_amax_f32(x, amax)) if f32 else (lambda: fq.fp8_amax(x, amax))
            nbytes = (4 if f32 else 2) * s * s
        else:
            scale = torch.ones(1, dtype=torch.float32, device=dev) if rec == R.TENSOR else None
            qr, sr, qc, sc = fq.cast_transpose(x, rec, F.E4M3, scale)
            cast = fq.fp8_cast_transpose_f32 if f32 else fq.fp8_cast_transpose
            fn = lambda: cast(x, rec, F.E4M3, scale, None, qr, sr, qc, sc)
            nbytes = bytes_cast(rec.name, s, s, in_bytes=4 if f32 else 2)
        ms = time_kernel(fn, reps=args.steps, flush=flush)
        res = {"case": args.case, "size": s, "us": round(ms * 1e3, 2), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1)}
        res["frac_hbm"] = round(res["GB/s"] / pk["hbm_gbs"], 4)
    elif args.case.startswith("dequant"):
        # FP8 -> BF16 of an s x s row-wise copy: 1 B read + 2 B written per element (+ scales)
        x = wl.cfg5_sweep(s, dev) if s in wl.CFG5_SIZES else wl.normal_bf16((s, s), 5, 1.0, dev)
        rec = {"dequant_tensor": R.TENSOR, "dequant_1x128": R.BLOCK_1x128, "dequant_128x128": R.BLOCK_128x128,
               "dequant_mx": R.MX_1x32_TILED}[args.case]
        scale = torch.ones(1, dtype=torch.float32, device=dev) if rec == R.TENSOR else None
        q, sq, _, _ = fq.cast_transpose(x, rec, F.E4M3, scale, col=False)
        y = torch.empty((s, s), dtype=torch.bfloat16, device=dev)
        ms = time_kernel(lambda: fq.fp8_dequantize(q, rec, F.E4M3, sq, y), reps=args.steps, flush=flush)
        nbytes = 3 * s * s + sq.numel() * sq.element_size()
        res = {"case": args.case, "size": s, "us": round(ms * 1e3, 2), "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1)}
        res["frac_hbm"] = round(res["GB/s"] / pk["hbm_gbs"], 4)
    elif args.case == "allreduce":
        # 8 ranks' size x size gradients: amax pass (2 B/elem) + cast and sum (2 B read, 1 B payload per
        # rank element, 4 B per reduced element)
        k, n = 8, s * s
        g = (torch.randn((k, n), generator=torch.Generator(device=dev).manual_seed(9), device=dev) * 1e-3).to(
            torch.bfloat16)
        amax = torch.empty(1, dtype=torch.float32, device=dev)
        q = torch.empty((k, n), dtype=torch.uint8, device=dev)
        si = torch.empty(1, dtype=torch.float32, device=dev)
        out = torch.empty(n, dtype=torch.float32, device=dev)
        ms = time_kernel(lambda: fq.fp8_allreduce_sum(g, F.E5M2, amax, q, si, out), reps=args.steps, flush=flush)
        nbytes = k * n * 2 + k * n * 3 + 4 * n
        res = {"case": args.case, "size": s, "ranks": k, "us": round(ms * 1e3, 2),
               "GB/s": round(nbytes / (ms * 1e-3) / 1e9, 1)}
        res["frac_hbm"] = round(res["GB/s"] / pk["hbm_gbs"], 4)
    elif args.case == "gemm_amax":
        # per-tensor GEMM whose epilogue writes C's FP8 copy (delayed scale) and amax, against
        # the unfused chain: GEMM to bf16, then amax and the per-tensor cast of C
        a = wl.normal_bf16((s, s), 1, 1.0, dev)
        b = wl.normal_bf16((s, s), 2, 0.02, dev)
        sc1 = torch.ones(1, dtype=torch.float32, device=dev)
        qa, sa, _, _ = fq.cast_transpose(a, R.TENSOR, F.E4M3, sc1, col=False)
        qb, sb, _, _ = fq.cast_transpose(b, R.TENSOR, F.E4M3, sc1, col=False)
        c = torch.empty((s, s), dtype=torch.bfloat16, device=dev)
        c_q = torch.empty((s, s), dtype=torch.uint8, device=dev)
        c_amax = torch.empty(1, dtype=torch.float32, device=dev)
        c_sinv = torch.empty(1, dtype=torch.float32, device=dev)
        c_scale = torch.full((1,), 64.0, dtype=torch.float32, device=dev)
        fused = lambda: fq.fp8_scaled_gemm_amax(qa, F.E4M3, R.TENSOR, sa, qb, F.E4M3, R.TENSOR, sb, None,
                                                fq.OutDtype.BF16, c_amax, c_scale, F.E4M3, c_q, c_sinv)

        def unfused():
            fq.fp8_scaled_gemm(qa, F.E4M3, R.TENSOR, sa, qb, F.E4M3, R.TENSOR, sb, c)
            fq.fp8_quantize(c, R.TENSOR, F.E4M3, c_scale, c_amax, c_q, c_sinv)

        ms = time_kernel(fused, reps=args.steps, flush=flush)
        ms_u = time_kernel(unfused, reps=args.steps, flush=flush)
        tf = 2.0 * s ** 3 / (ms * 1e-3) / 1e12
        res = {"case": args.case, "size": s, "us": round(ms * 1e3, 2), "TFLOP/s": round(tf, 1),
               "frac_fp8": round(tf / fp8_peak_of(pk), 4), "unfused_us": round(ms_u * 1e3, 2)}
    else:
        # gemm_block_wgrad: the weight-gradient pairing, 1x128 x 1x128 (a scale per row of B), FP32 out
        ra = {"gemm_tensor": R.TENSOR, "gemm_block": R.BLOCK_1x128, "gemm_mx": R.MX_1x32_TILED,
              "gemm_block_wgrad": R.BLOCK_1x128}[args.case]
        rb = {"gemm_tensor": R.TENSOR, "gemm_block": R.BLOCK_128x128, "gemm_mx": R.MX_1x32_TILED,
              "gemm_block_wgrad": R.BLOCK_1x128}[args.case]
        od = fq.OutDtype.FP32 if args.case == "gemm_block_wgrad" else fq.OutDtype.BF16
        m, n, k = (args.size, args.size, args.size) if args.mnk is None else args.mnk
        a = wl.normal_bf16((m, k), 1, 1.0, dev)
        b = wl.normal_bf16((n, k), 2, 0.02, dev)
        sc1 = torch.ones(1, dtype=torch.float32, device=dev)
        qa, sa, _, _ = fq.cast_transpose(a, ra, F.E4M3, sc1 if ra == R.TENSOR else None, col=False)
        qb, sb, _, _ = fq.cast_transpose(b, rb, F.E4M3, sc1 if rb == R.TENSOR else None, col=False)
        c = torch.empty((m, n), dtype=torch.float32 if od == fq.OutDtype.FP32 else torch.bfloat16, device=dev)
        ms = time_kernel(lambda: fq.fp8_scaled_gemm(qa, F.E4M3, ra, sa, qb, F.E4M3, rb, sb, c, od), reps=args.steps,
                         flush=flush)
        tf = 2.0 * m * n * k / (ms * 1e-3) / 1e12
        res = {"case": args.case, "M": m, "N": n, "K": k, "us": round(ms * 1e3, 2), "TFLOP/s": round(tf, 1),
               "frac_fp8": round(tf / fp8_peak_of(pk), 4)}
    assert fq.fp8_get_device_status() == fq.Status.OK
    print(json.dumps(res), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--case", choices=CASES, default=None, help="time one kernel in a loop (profiling)")
    ap.add_argument("--size", type=int, default=4096)
    ap.add_argument("--mnk", type=int, nargs=3, default=None, help="GEMM cases: M N K instead of size^3")
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--no-per-recipe", action="store_true", help="skip the per-recipe kernel figures")
    ap.add_argument("--no-e2e", action="store_true")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--clocks-csv", default=None, help="also write the raw clock samples of the run here")
    ap.add_argument("--cpu-baseline-sweep", type=int, nargs="*", default=None, metavar="SIZE",
                    help="time the oracle's casts on the host cores at these sizes (default: the bandwidth "
                         "sweep's sizes) and print them as one JSON line; no GPU")
    args = ap.parse_args()
    if args.cpu_baseline_sweep is not None:
        from scaled_quantize_gemm_amax_gb300 import workloads as wl
        print(json.dumps(cpu_baseline_sweep(args.cpu_baseline_sweep or wl.CFG5_SIZES)), flush=True)
        return
    if args.warmup < 3:
        args.warmup = 3
    if args.case is not None:
        run_case(args)
        return
    rank, world, _ = dist_setup(args)
    if args.impl == "reference":
        res = run_reference(args, rank, world)
    else:
        res = run_ours(args, rank, world)
    if rank == 0 and res is not None:
        print(json.dumps(res), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
