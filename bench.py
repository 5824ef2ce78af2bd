#!/usr/bin/env python3
"""Benchmark of the BF16 attention leaf on GB300.

One step = one call of the hot path (attn_dense_fwd, or attn_prefix_fwd for
the prefix workload) over one batch of seeded synthetic bf16 inputs.  The
metric is TFLOP/s with FLOPs = 4 * B * H * Nq * Nkv * D (2*D per score for
Q K^T, 2*D for P V).  The default workload is the largest single-GPU one,
dense B=1 N=32768 H=32 D=128 (inputs N(0, 0.5^2)).

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload ID]
    python bench.py --impl reference ...   # the FP64 CPU oracle, same metric

Rank 0 prints one JSON line.  Under torchrun (N > 1) each rank runs an
independent replica of the workload on its own GPU (no collective on the data
path); the value is all ranks' FLOPs over the slowest rank's time.
"""
from __future__ import annotations

import argparse
import json
import os
import statistics
import subprocess
import sys
import tempfile
import threading
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import numpy as np  # noqa: E402

import workloads  # noqa: E402

METRIC = "attention fwd TFLOP/s and % of GB300 BF16 tensor peak (h32, d128/d64)"
UNIT = "TFLOP/s"
FALLBACK_BF16_TFLOPS = 1900.0
L2_FLUSH_BYTES = 512 << 20   # > 126 MB L2: written between timed iterations
KERNEL_NAME = "ncp::attn_fwd_kernel"


# ----------------------------------------------------------------------------
# Helpers
# ----------------------------------------------------------------------------

def log(*a):
    print(*a, file=sys.stderr, flush=True)


def dist_env():
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    return world, rank, local


def measured_peaks():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return {"bf16_tflops": FALLBACK_BF16_TFLOPS, "hbm_gbs": 6800.0}, "fallback"


def kernel_source_hash() -> str:
    import hashlib
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "non_causal_prefix_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        path = os.path.join(csrc, f)
        if os.path.isfile(path) and f.endswith((".cu", ".cuh", ".h")):
            with open(path, "rb") as fh:
                h.update(fh.read())
    return h.hexdigest()[:16]


def recorded_profile(workload_name: str) -> dict:
    """The committed ncu figures of one launch of the workload's kernel
    (profiles/traffic.json), if they were taken on the current kernel source;
    else {}.  Keys: dram_bytes_per_launch, and where captured
    tensor_pipe_active_pct and duration_us."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            doc = json.load(f)
    except (OSError, ValueError):
        return {}
    ent = doc.get(workload_name)
    if not ent or ent.get("kernel_source_hash") != kernel_source_hash():
        return {}
    return ent


def recorded_traffic(workload_name: str):
    """DRAM bytes per launch from the committed ncu summary, if it was taken
    on the current kernel source (else None)."""
    return recorded_profile(workload_name).get("dram_bytes_per_launch")


NOMINAL_HBM_GBS = 8000.0


def ncu_fields(workload_name: str, hbm_peak_gbs: float) -> dict:
    """The ncu figures the line carries beside the roofline: tensor-pipe
    utilisation and DRAM GB/s (against the nominal 8 TB/s and the measured
    copy bandwidth), from one ncu capture of the current source; None where
    no such capture is recorded."""
    ent = recorded_profile(workload_name)
    dram = ent.get("dram_bytes_per_launch")
    dur = ent.get("duration_us")
    gbs = dram / (dur * 1e-6) / 1e9 if dram and dur else None
    return {
        "tensor_pipe_active_pct": ent.get("tensor_pipe_active_pct"),
        "dram_gbs": round(gbs, 1) if gbs else None,
        "dram_frac_of_8tbs": round(gbs / NOMINAL_HBM_GBS, 4) if gbs else None,
        "dram_frac_of_measured": round(gbs / hbm_peak_gbs, 4) if gbs else None,
        "ncu_source": "profiles/traffic.json (one ncu launch, --clock-control none)"
                      if ent else None,
    }


class ClockSampler:
    """nvidia-smi sampling of SM clock and throttle reasons in the background."""

    FIELDS = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index: int):
        import torch
        self.gpu_id = None
        try:
            self.gpu_id = "GPU-" + str(torch.cuda.get_device_properties(device_index).uuid)
        except Exception:
            self.gpu_id = None
        self.proc = None
        self.lines = []
        self.window = None

    def mark(self, t0: float, t1: float):
        """Host wall-clock bounds of the timed region."""
        self.window = (t0, t1)

    def start(self):
        cmd = ["nvidia-smi", f"--query-gpu={self.FIELDS}", "--format=csv,noheader,nounits",
               "-lms", "50"]
        if self.gpu_id:
            cmd.insert(1, f"--id={self.gpu_id}")
        try:
            self.proc = subprocess.Popen(cmd, stdout=subprocess.PIPE, stderr=subprocess.DEVNULL,
                                         text=True)
        except OSError:
            self.proc = None
            return
        self.thread = threading.Thread(target=self._read, daemon=True)
        self.thread.start()
        time.sleep(0.3)

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append((time.time(), line.strip()))

    def stop(self):
        if not self.proc:
            return None
        time.sleep(0.25)
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
        self.thread.join(timeout=2)
        return summarize_clocks(self.lines, self.window)


def summarize_clocks(lines, window):
    """Median SM clock, max clock, throttle reasons seen and sample counts from
    timestamped nvidia-smi CSV lines (the ClockSampler.FIELDS columns), taken
    over the timed region `window` = (t0, t1) host seconds; None without a
    usable sample."""
    sm, mx, power, reasons = [], [], [], set()
    names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
    in_window = 0
    if window is not None and lines:
        t0, t1 = window
        # nvidia-smi prints a sample shortly after taking it: allow 0.1 s of lag.
        inside = [(t, x) for t, x in lines if t0 <= t <= t1 + 0.1]
        in_window = len(inside)
        if inside:
            lines = inside
        else:
            # The timed region was shorter than the sampling period: keep
            # the samples nearest to it (same kernel, taken during the
            # warm-up just before and the runs just after).
            mid = 0.5 * (t0 + t1)
            lines = sorted(lines, key=lambda tx: abs(tx[0] - mid))[:4]
    for _, line in lines:
        parts = [p.strip() for p in line.split(",")]
        if len(parts) < 8:
            continue
        try:
            sm.append(float(parts[0]))
            mx.append(float(parts[1]))
            power.append(float(parts[2]))
        except ValueError:
            continue
        for n, v in zip(names, parts[4:8]):
            if v.lower().startswith("active"):
                reasons.add(n)
    if not sm:
        return None
    return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
            "reasons": sorted(reasons), "samples": len(sm), "samples_in_timed_region": in_window,
            "power_w_max": max(power) if power else None}


def max_over_ranks(value: float, device=None) -> float:
    """Maximum of ``value`` over the ranks of the default process group (the
    value itself when there is no group or a single rank)."""
    import torch
    import torch.distributed as dist
    if not (dist.is_available() and dist.is_initialized()) or dist.get_world_size() == 1:
        return value
    t = torch.tensor([float(value)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def job_throughput(world: int, steps: int, flops_per_step: int, slowest_ms: float) -> float:
    """Whole-job TFLOP/s: every rank runs ``steps`` steps of its own replica;
    the job takes as long as the slowest rank."""
    return world * steps * flops_per_step / (slowest_ms / 1e3) / 1e12


# ----------------------------------------------------------------------------
# GPU arm
# ----------------------------------------------------------------------------

def make_call(ncp, w, dev_in, out):
    if w.kind == "dense":
        q, k, v = dev_in
        return lambda stream=None: ncp.attn_dense_fwd(q, k, v, out, stream)
    if w.kind == "cross":
        q, k, v = dev_in
        return lambda stream=None: ncp.attn_dense_cross_fwd(q, k, v, out, stream)
    if w.kind == "masked_prefix":
        q, kc, vc, kp, vp = dev_in
        ids = workloads.image_ids(w).to(q.device)
        valid = workloads.key_valid(w).to(q.device)
        return lambda stream=None: ncp.attn_masked_prefix_fwd(q, kc, vc, kp, vp, ids, valid,
                                                              w.sm_scale, out, stream)
    if w.kind == "block_causal":
        q, k, v = dev_in
        ids = workloads.image_ids(w).to(q.device)
        return lambda stream=None: ncp.attn_block_causal_fwd(q, k, v, ids, out, stream)
    q, kp, vp, kc, vc = dev_in
    return lambda stream=None: ncp.attn_prefix_fwd(q, kp, vp, kc, vc, out, stream)


def time_device(torch, call, flush, steps, warmup, stream):
    """Per-launch device time (ms) with CUDA events on the launching stream;
    the L2 is flushed (a 512 MiB write) before every launch, outside the
    events."""
    for _ in range(warmup):
        flush.add_(1)
        call(stream)
    torch.cuda.synchronize()
    starts = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    ends = [torch.cuda.Event(enable_timing=True) for _ in range(steps)]
    t0 = time.time()
    with torch.cuda.stream(stream):
        for i in range(steps):
            flush.add_(1)
            starts[i].record(stream)
            call(stream)
            ends[i].record(stream)
    torch.cuda.synchronize()
    t1 = time.time()
    return [s.elapsed_time(e) for s, e in zip(starts, ends)], (t0, t1)


def time_graph(torch, call, stream, iters, reps=5):
    """Per-launch device time (ms) of `iters` back-to-back launches captured in
    one CUDA graph on `stream` and replayed: the median over `reps` replays,
    timed with CUDA events on that stream.  No L2 flush runs between the
    launches, so inputs that fit in L2 stay there (warm timing)."""
    call(stream)  # a splitting call captures the workspace its stream used last
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=stream):
        for _ in range(iters):
            call(stream)
    with torch.cuda.stream(stream):
        g.replay()
    torch.cuda.synchronize()
    ts = []
    for _ in range(reps):
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        with torch.cuda.stream(stream):
            a.record(stream)
            g.replay()
            b.record(stream)
        torch.cuda.synchronize()
        ts.append(a.elapsed_time(b) / iters)
    del g
    return statistics.median(ts)


def time_e2e(torch, ncp, w, host_in, steps, warmup, stream):
    """Host-to-host time per step through the C-ABI call: every step copies its
    inputs in from pinned host memory, runs the call and copies the output back
    to pinned host memory.  Two buffer sets and three streams (copies in,
    compute, copies out) let step i's compute overlap step i+1's input copy and
    step i-1's output copy, as a serving loop would; the CUDA events bracket
    all ``steps`` steps, copies included.  Also returns the bandwidth of one
    step's input copy and of its output copy, each timed alone before the
    loop (GB/s): the link these copies go over sets the floor of a step."""
    nbuf = 2
    h2d_stream, d2h_stream = torch.cuda.Stream(), torch.cuda.Stream()
    dev_in = [[torch.empty_like(t, device="cuda") for t in host_in] for _ in range(nbuf)]
    dev_out = [torch.empty_like(dev_in[0][0]) for _ in range(nbuf)]
    host_out = [torch.empty_like(host_in[0]).pin_memory() for _ in range(nbuf)]
    calls = [make_call(ncp, w, dev_in[i], dev_out[i]) for i in range(nbuf)]
    in_ready = [torch.cuda.Event() for _ in range(nbuf)]
    computed = [torch.cuda.Event() for _ in range(nbuf)]
    out_done = [torch.cuda.Event() for _ in range(nbuf)]

    def one(step):
        i = step % nbuf
        with torch.cuda.stream(h2d_stream):
            h2d_stream.wait_event(computed[i])      # inputs of step - nbuf consumed
            for d, h in zip(dev_in[i], host_in):
                d.copy_(h, non_blocking=True)
            in_ready[i].record(h2d_stream)
        stream.wait_event(in_ready[i])
        stream.wait_event(out_done[i])              # output of step - nbuf copied out
        calls[i](stream)
        computed[i].record(stream)
        with torch.cuda.stream(d2h_stream):
            d2h_stream.wait_event(computed[i])
            host_out[i].copy_(dev_out[i], non_blocking=True)
            out_done[i].record(d2h_stream)

    # The copies alone, once warm: one step's inputs in, one output out.
    copy_gbs = {}
    for name, pairs in (("h2d", list(zip(dev_in[0], host_in))), ("d2h", [(host_out[0], dev_out[0])])):
        for rep in range(2):
            a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            with torch.cuda.stream(h2d_stream):
                a.record(h2d_stream)
                for dst, src in pairs:
                    dst.copy_(src, non_blocking=True)
                b.record(h2d_stream)
            torch.cuda.synchronize()
        nbytes = sum(src.numel() * src.element_size() for _, src in pairs)
        copy_gbs[name] = round(nbytes / (a.elapsed_time(b) / 1e3) / 1e9, 1)
    for s in range(warmup):
        one(s)
    torch.cuda.synchronize()
    start = torch.cuda.Event(enable_timing=True)
    end = torch.cuda.Event(enable_timing=True)
    start.record(h2d_stream)
    for s in range(steps):
        one(s)
    d2h_stream.wait_event(computed[(steps - 1) % nbuf])
    end.record(d2h_stream)
    torch.cuda.synchronize()
    h2d = sum(t.numel() * t.element_size() for t in host_in)
    d2h = host_out[0].numel() * host_out[0].element_size()
    return start.elapsed_time(end) / steps, h2d, d2h, copy_gbs


def cpu_oracle_sample(w, inputs_cpu, target_s: float):
    """The oracle, as it stands, on sampled output rows of workload ``w``:
    FP64 TFLOP/s over the sample and the threads it used."""
    import oracle
    cores = len(os.sched_getaffinity(0))
    oracle.set_threads(cores)
    bits = [workloads.bf16_bits(t) for t in inputs_cpu]
    if w.kind in ("dense", "cross"):
        fn = oracle.dense_attention_rows
    elif w.kind == "prefix":
        fn = oracle.prefix_attention_rows
    elif w.kind == "masked_prefix":
        ids = workloads.image_ids(w).numpy()
        valid = workloads.key_valid(w).numpy().astype(np.uint8)
        scale = float(np.float32(w.sm_scale))
        fn = lambda *a: oracle.masked_prefix_attention_rows(  # noqa: E731
            *a[:-1], ids, valid, scale, a[-1])
    else:
        ids = workloads.image_ids(w).numpy()
        fn = lambda *a: oracle.block_causal_attention_rows(*a[:-1], ids, a[-1])  # noqa: E731
    total_rows = w.B * w.Nq * w.H
    flops_per_row = 4 * w.visible_pairs * w.D / w.Nq  # mean over rows
    rng = np.random.default_rng(0)
    n = min(total_rows, 256)
    t0 = time.perf_counter()
    fn(*bits, rng.integers(0, total_rows, n))
    dt = time.perf_counter() - t0
    n2 = int(min(total_rows, max(n, n * target_s / max(dt, 1e-6))))
    rows = rng.integers(0, total_rows, n2)
    t0 = time.perf_counter()
    fn(*bits, rows)
    dt = time.perf_counter() - t0
    return {
        "value": n2 * flops_per_row / dt / 1e12,
        "unit": UNIT,
        "cores": oracle.max_threads(),
        "kind": "oracle",
        "sample": f"{n2} of {total_rows} output rows (b,q,h) of {w.describe()}, "
                  f"{dt:.1f} s of FP64 C/OpenMP",
        "seconds": dt,
    }


def run_gpu(args):
    import torch
    world, rank, local = dist_env()
    if world > 1:
        import torch.distributed as tdist
        torch.cuda.set_device(local)
        tdist.init_process_group("nccl")
    else:
        torch.cuda.set_device(0)
    import non_causal_prefix_gb300 as ncp
    if rank == 0 or world == 1:
        ncp.build(quiet=True)
    if world > 1:
        torch.distributed.barrier()
    ncp.load_library()

    w = workloads.WORKLOADS[args.workload]
    host_in = workloads.make_inputs(w)
    dev_in = [t.cuda() for t in host_in]
    out = torch.empty_like(dev_in[0])
    call = make_call(ncp, w, dev_in, out)
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device="cuda")
    stream = torch.cuda.Stream()

    clocks = ClockSampler(torch.cuda.current_device())
    clocks.start()
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    times, window = time_device(torch, call, flush, args.steps, args.warmup, stream)
    torch.cuda.synchronize()
    if world > 1:
        torch.distributed.barrier()
    clocks.mark(*window)
    status, _ = ncp.device_status(stream)
    if status != ncp.ATTN_OK:
        raise RuntimeError(f"device status after timing: {ncp.status_string(status)}")

    total_ms = max_over_ranks(sum(times), device="cuda")
    value = job_throughput(world, args.steps, w.flops, total_ms)
    ms_per_step = total_ms / args.steps

    # End to end through the public API with host buffers.
    host_pinned = [t.pin_memory() for t in host_in]
    e2e_ms, h2d, d2h, copy_gbs = time_e2e(torch, ncp, w, host_pinned, max(4, args.steps), 3,
                                           stream)
    e2e_ms = max_over_ranks(e2e_ms, device="cuda")
    e2e_value = job_throughput(world, 1, w.flops, e2e_ms)
    clock_info = clocks.stop()

    peaks, peak_src = measured_peaks()
    peak = float(peaks.get("bf16_tflops", FALLBACK_BF16_TFLOPS))
    hbm_peak = float(peaks.get("hbm_gbs", 6800.0))
    # `value` and `roofline.achieved` both use the mean launch time (total
    # over the K timed launches); the median, the statistic of the pages'
    # audit timing, is reported beside them.
    mean_ms = statistics.mean(times)
    median_ms = statistics.median(times)
    achieved = w.flops / (mean_ms / 1e3) / 1e12
    achieved_median = w.flops / (median_ms / 1e3) / 1e12
    line = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(ms_per_step, 5),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "bf16",
        "data": "synthetic (seeded N(0, sigma^2) rounded to bf16)",
        "config": {
            "workload": w.name,
            "shape": w.describe(),
            "flops_per_step": w.flops,
            "l2": "512 MiB buffer written before every timed launch (inputs < L2)",
            "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
        },
        "timing": {
            "statistic": "value and roofline.achieved: mean of the K per-launch CUDA-event "
                         "times; *_median: their median",
            "mean_ms": round(mean_ms, 5),
            "median_ms": round(median_ms, 5),
            "min_ms": round(min(times), 5),
            "max_ms": round(max(times), 5),
            "value_median": round(achieved_median * world, 2),
        },
        "roofline": {
            "bound": "tensor",
            "achieved": round(achieved, 2),
            "achieved_median": round(achieved_median, 2),
            "peak": peak,
            "unit": UNIT,
            "frac": round(achieved / peak, 4),
            "frac_median": round(achieved_median / peak, 4),
            "peak_source": f"{peak_src} bf16_tflops (burst; kernel timed alone)",
            "kernel": KERNEL_NAME + ("<128>" if w.D == 128 else "<64>"),
            "traffic": recorded_traffic(w.name),
            "algorithmic_bytes": w.hbm_bytes,
            **ncu_fields(w.name, hbm_peak),
        },
        "e2e": {"value": round(e2e_value, 2), "unit": UNIT, "h2d_bytes_per_step": h2d,
                "d2h_bytes_per_step": d2h, "ms_per_step": round(e2e_ms, 4),
                "copy_gbs_alone": copy_gbs},
        "gpu_launches": args.steps,
        "clocks": clock_info,
    }

    if not args.no_configs and rank == 0 and world == 1:
        line["per_config"] = per_config(torch, ncp, flush, stream, peak, args)
    if rank == 0 and world == 1 and not args.no_cpu:
        line["cpu_baseline"] = cpu_oracle_sample(w, host_in, args.cpu_seconds)
        line["cpu_baseline"].pop("seconds", None)
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank == 0:
        print(json.dumps(line), flush=True)


# The audit timing of the kernel pages: at least 10 warm-up calls, then the
# median of at least 50 per-call CUDA-event samples.
CONFIG_WARMUP = 10
CONFIG_SAMPLES = 50


def per_config(torch, ncp, flush, stream, peak, args):
    """Device TFLOP/s of every synthetic workload (context for the line): the
    median, mean and min of CONFIG_SAMPLES per-launch CUDA-event times after
    CONFIG_WARMUP warm-up launches, with the L2 flushed before each launch,
    and graph_us, the per-launch time of graph_iters back-to-back launches
    replayed from one CUDA graph (warm L2)."""
    res = {}
    for cid, w in workloads.WORKLOADS.items():
        dev_in = [t.cuda() for t in workloads.make_inputs(w)]
        out = torch.empty_like(dev_in[0])
        call = make_call(ncp, w, dev_in, out)
        times, _ = time_device(torch, call, flush, CONFIG_SAMPLES, CONFIG_WARMUP, stream)
        us = statistics.median(times) * 1e3
        tf = w.flops / (us / 1e6) / 1e12
        iters = max(1, min(50, int(2000.0 / us)))
        g_us = time_graph(torch, call, stream, iters) * 1e3
        res[w.name] = {"median_us": round(us, 2), "mean_us": round(statistics.mean(times) * 1e3, 2),
                       "min_us": round(min(times) * 1e3, 2), "samples": len(times),
                       "warmup": CONFIG_WARMUP,
                       "tflops": round(tf, 1), "frac_of_peak": round(tf / peak, 4),
                       "graph_us": round(g_us, 2), "graph_iters": iters,
                       "tensor_pipe_active_pct": recorded_profile(w.name).get(
                           "tensor_pipe_active_pct")}
        del dev_in, out
    torch.cuda.empty_cache()
    return res


# ----------------------------------------------------------------------------
# Reference arm: the FP64 oracle on the host cores
# ----------------------------------------------------------------------------

def run_reference(args):
    world, rank, _ = dist_env()
    if rank != 0:
        return
    import oracle
    oracle.build()
    w = workloads.WORKLOADS[args.workload]
    inputs = workloads.make_inputs(w)
    per_step = max(1.0, 90.0 / max(1, args.steps + args.warmup))
    for _ in range(args.warmup):
        cpu_oracle_sample(w, inputs, per_step / 4)
    vals, secs = [], []
    samples = []
    for _ in range(args.steps):
        r = cpu_oracle_sample(w, inputs, per_step)
        vals.append(r["value"])
        secs.append(r["seconds"])
        samples.append(r)
    value = statistics.median(vals)
    last = samples[-1]
    line = {
        "metric": METRIC,
        "value": round(value, 6),
        "unit": UNIT,
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(1e3 * statistics.mean(secs), 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": "f64",
        "data": "synthetic (seeded N(0, sigma^2) rounded to bf16)",
        "impl": "reference",
        "config": {"workload": w.name, "shape": w.describe(), "flops_per_step": w.flops},
        "cpu_baseline": {"value": round(value, 6), "unit": UNIT, "cores": last["cores"],
                         "kind": "oracle", "sample": last["sample"]},
        "e2e": {"value": round(value, 6), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def main():
    ap = argparse.ArgumentParser(description=__doc__,
                                 formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=50)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", type=int, default=5, choices=sorted(workloads.WORKLOADS))
    ap.add_argument("--no-configs", action="store_true", help="skip the per-config table")
    ap.add_argument("--no-cpu", action="store_true", help="skip the CPU oracle baseline")
    ap.add_argument("--cpu-seconds", type=float, default=15.0)
    args = ap.parse_args()
    if args.warmup < 3:
        ap.error("--warmup must be >= 3")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_gpu(args)


if __name__ == "__main__":
    main()
