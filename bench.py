#!/usr/bin/env python3
"""Benchmark of the Gated DeltaNet forward recurrence on B300.

One step = one chunked prefill forward (gdn_chunk_fwd) over the prefill
workload: B=4 sequences x T=4096 tokens, H_qk=16, H_v=32, d_k=d_v=128, bf16
q/k/v, fp32 g/beta and state, chunk 64, zero initial state, bf16 output plus
fp32 final states. value = tokens/s over all ranks. The same JSON line also
carries the two other prefill workloads, each measured the same way: `long`
(B=1, T=65536, h0 ~ N(0, 0.02)) and `varlen` (64 packed sequences, lengths
U{128..8192}, per-sequence initial states); the decode step (256 sequences x 32 heads x 128x128 fp32 states,
1000 consecutive in-place steps, bf16 token inputs) in GB/s, the output
epilogue and input prologue in GB/s, the gradient of the prefill
workload (gdn_chunk_bwd) in tokens/s against the fp32 CUDA-core peak, and the
per-channel-decay variant (KDA) prefill and decode.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own independent copy of the
workload (the work shards by sequence with no exchange: weak scaling); the
timed region is bracketed by barriers and the max over ranks is reported.
Every timed leg records one CUDA event per launch on the launching stream and
reports the mean over the bracketed region (the value), the median with a 95%
confidence interval, and its first call in the process separately (cold).
`e2e` runs the same call on host buffers: each step copies its inputs from
pinned host memory and its outputs back, with the copies of one step
overlapping the previous step's call.
--impl reference times the fp64 CPU oracle (test infrastructure) on a bounded
sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import threading
import time

# The gradient oracle's CPU baseline is numpy; keep its BLAS on one thread so
# the reported core count is the one used (set before numpy is first imported).
os.environ.setdefault("OPENBLAS_NUM_THREADS", "1")

import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

import gdn_inputs  # noqa: E402

METRIC = "GDN prefill tokens/s and decode GB/s on 1 B300, % of roofline"
PEAKS_FALLBACK = {"hbm_gbs": 6400.0, "bf16_tflops": 1800.0, "bf16_tflops_sustained": 1400.0}
KERNEL_SOURCES = ["gdn_chunk_tc.cuh", "gdn_tc_ptx.cuh", "gdn_common.cuh"]
TRAFFIC_FILE = os.path.join(ROOT, "profiles", "chunk_tc_prefill_ncu.txt")


# --------------------------------------------------------------------------- helpers
PEAK_SOURCE = "fallback"
WL = gdn_inputs.WORKLOADS


def load_peaks():
    """The machine's measured peaks (copy bandwidth, bf16 dense) or the fallback."""
    global PEAK_SOURCE
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            peaks = json.load(f)
        PEAK_SOURCE = "measured"
        return peaks
    except (OSError, ValueError):
        PEAK_SOURCE = "fallback"
        return dict(PEAKS_FALLBACK)


def kernel_sha():
    """Hash of the prefill kernel's sources (ties recorded ncu counters to them)."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "gated_deltanet_recurrence_05_b300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic(key="dram_bytes_per_launch"):
    """DRAM bytes per prefill launch from the committed ncu summary (`key`: the
    prefill workload's, or `dram_bytes_per_launch_long`), or None if the
    summary is absent or was taken on other kernel sources."""
    try:
        kv = {}
        with open(TRAFFIC_FILE) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_sha256") != kernel_sha():
            return None
        return float(kv[key])
    except (OSError, KeyError, ValueError):
        return None


def prefill_algorithmic(w, out_bytes=2):
    """Algorithmic bytes and FLOPs of one prefill forward (each input read once,
    each output written once; FLOPs of the chunked method, per token and value
    head: 6 dk dv + 2C(dk + 2dv) + 4C dk / G + 2C^2/3)."""
    T = sum(w["lengths"])
    hq, hv, dk, dv = w["h_qk"], w["h_v"], w["d_k"], w["d_v"]
    N = len(w["lengths"])
    in_b = 2 if w["dtype"] == "bf16" else 4
    bytes_ = T * (2 * hq * dk * in_b + hv * dv * in_b + 2 * hv * 4 + hv * dv * out_bytes)
    bytes_ += N * hv * dk * dv * 4  # final states written
    if w["h0"] is not None:
        bytes_ += N * hv * dk * dv * 4
    C, G = 64, hv // hq
    flops = T * hv * (6 * dk * dv + 2 * C * (dk + 2 * dv) + 4 * C * dk / G + 2 * C * C / 3)
    return bytes_, flops


def decode_algorithmic(n, hq, hv, dk, dv):
    """Bytes of one decode step: the state read and written once, one bf16
    token of q, k, v, a bf16 output, fp32 g and beta."""
    return 2 * n * hv * dk * dv * 4 + n * (2 * hq * dk * 2 + hv * dv * 2 + hv * dv * 2 + 2 * hv * 4)


class ClockSampler:
    """Samples SM clocks and throttle reasons with nvidia-smi while running."""

    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.QUERY}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.thread = threading.Thread(target=self._read, daemon=True)
            self.thread.start()
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def _read(self):
        for line in self.proc.stdout:
            self.lines.append(line.strip())

    def __exit__(self, *exc):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
            self.thread.join(timeout=2)

    def summary(self):
        sm, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in self.lines:
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sm.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for name, val in zip(names, f[5:9]):
                if val.lower() == "active":
                    reasons.add(name)
        if not sm:
            return None
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sm)}


def dist_setup(args):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if (args.impl == "ours" and torch.cuda.is_available()) else "gloo"
        if backend == "nccl":
            torch.cuda.set_device(local)
        dist.init_process_group(backend=backend)
    elif args.impl == "ours" and torch.cuda.is_available():
        torch.cuda.set_device(local)
    return world, rank, local


def barrier(world):
    if world > 1:
        import torch.distributed as dist
        dist.barrier()


def max_over_ranks(x, world, device):
    """Max of a float over all ranks (every rank gets the result)."""
    if world == 1:
        return float(x)
    import torch.distributed as dist
    t = torch.tensor([float(x)], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def aggregate_throughput(units_per_rank, world, max_seconds):
    """Whole-job throughput: units processed on all ranks / slowest rank's time."""
    return units_per_rank * world / max_seconds


def cu_of(w):
    return torch.tensor([0] + torch.cumsum(torch.tensor(w["lengths"]), 0).tolist(), dtype=torch.int32)


# --------------------------------------------------------------------------- timing helpers
def median_ci95(xs):
    """Median of the samples and a distribution-free 95% confidence interval
    for it: the order statistics (j, k) with P(j <= Binom(n, 1/2) < k) >= 0.95,
    as narrow as possible and symmetric (for n < 6 no pair reaches 0.95 and
    the interval is the whole range)."""
    xs = sorted(float(x) for x in xs)
    n = len(xs)
    if n == 0:
        return None
    med = statistics.median(xs)
    lo, hi = 0, n - 1
    for j in range(n // 2, -1, -1):
        k = n - 1 - j
        cover = sum(math.comb(n, i) for i in range(j + 1, k + 1)) / 2.0 ** n
        if cover >= 0.95:
            lo, hi = j, k
            break
    return {"median": med, "ci95": [xs[lo], xs[hi]], "n": n, "ci_method": "order statistics (binomial)"}


def timed_launches(fn, reps, stream, dev, world):
    """Run fn(i) for i < reps on `stream` with one CUDA event before each call
    and one after the last (all on the launching stream), bracketed by a
    barrier and device synchronisations. Returns (mean ms per call over the
    whole bracketed region, list of per-call ms). The calls must be issued on
    the current stream (where the spin runs)."""
    evs = [torch.cuda.Event(enable_timing=True) for _ in range(reps + 1)]
    barrier(world)
    torch.cuda.synchronize(dev)
    # a short device-side spin before the first event, so that the host has
    # queued the first launches by the time it ends: the events then time the
    # device work, not the host's latency to enqueue the first call
    torch.cuda._sleep(2_000_000)
    for i in range(reps):
        evs[i].record(stream)
        fn(i)
    evs[reps].record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    per = [evs[i].elapsed_time(evs[i + 1]) for i in range(reps)]
    return evs[0].elapsed_time(evs[reps]) / reps, per


def warm_up(fn, n, stream, dev, min_seconds=0.05):
    """At least n untimed calls, and more until `min_seconds` of them have run
    (so that clocks have settled after any idle time). Returns the count."""
    t = time.perf_counter()
    k = 0
    while k < n or time.perf_counter() - t < min_seconds:
        fn()
        k += 1
        if k % 16 == 0:
            torch.cuda.synchronize(dev)
    torch.cuda.synchronize(dev)
    return k


def cold_call(fn, stream, dev):
    """Time one call that nothing has warmed (first call of this workload in
    the process): device time between events and host wall time to its end."""
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize(dev)
    t = time.perf_counter()
    e0.record(stream)
    fn()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    return {"device_ms": e0.elapsed_time(e1), "host_wall_ms": (time.perf_counter() - t) * 1e3}


# --------------------------------------------------------------------------- oracle (CPU) leg
def oracle_sample(w, target_s=12.0, threads=0):
    """Time the fp64 oracle on a bounded sample of the workload: whole sequences
    of a subset of (sequence, value-head) pairs. Returns tokens/s (pair-tokens/s
    divided by H_v), the thread count and a description of the sample."""
    import oracle
    # explicit thread counts on every call: the oracle's OpenMP setting persists
    cores = len(os.sched_getaffinity(0)) if threads <= 0 else threads
    N, hv = len(w["lengths"]), w["h_v"]
    cu = cu_of(w)
    # the longest sequence first, so that the probe sees a representative pair
    n0 = max(range(N), key=lambda n: w["lengths"][n])
    t = time.perf_counter()
    oracle.recurrent(w["q"], w["k"], w["v"], w["g"], w["beta"], h0=w["h0"], cu_seqlens=cu,
                     pairs=[(n0, 0)], threads=1)
    one = (time.perf_counter() - t) / max(w["lengths"][n0], 1)   # s per pair-token, one thread
    mean_len = max(1.0, sum(w["lengths"]) / N)
    n_pairs = max(cores, int(target_s * cores / max(one * mean_len, 1e-6)))
    n_pairs = max(1, min(n_pairs, N * hv))
    pairs = [(i // hv % N, i % hv) for i in range(n_pairs)]
    t = time.perf_counter()
    oracle.recurrent(w["q"], w["k"], w["v"], w["g"], w["beta"], h0=w["h0"], cu_seqlens=cu,
                     pairs=pairs, threads=cores)
    dt = time.perf_counter() - t
    pair_tokens = sum(w["lengths"][n] for n, _ in pairs)
    return pair_tokens / hv / dt, cores, (
        f"{n_pairs} of {N * hv} (sequence, value-head) pairs, whole sequences "
        f"({pair_tokens} pair-tokens), fp64 recurrence, {dt:.1f} s")


def oracle_baseline(w, target_s):
    """The oracle on all host cores (bounded sample) and on one core (one
    whole pair), both in tokens/s of the workload (pair-tokens / H_v)."""
    import oracle
    tok_s, cores, sample = oracle_sample(w, target_s=target_s)
    N, hv = len(w["lengths"]), w["h_v"]
    n0 = max(range(N), key=lambda n: w["lengths"][n])
    t = time.perf_counter()
    oracle.recurrent(w["q"], w["k"], w["v"], w["g"], w["beta"], h0=w["h0"], cu_seqlens=cu_of(w),
                     pairs=[(n0, 0)], threads=1)
    dt1 = time.perf_counter() - t
    return {"value": tok_s, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample,
            "value_1thread": w["lengths"][n0] / hv / dt1,
            "sample_1thread": f"one whole pair ({w['lengths'][n0]} tokens) on 1 thread, {dt1:.2f} s"}


# --------------------------------------------------------------------------- GPU legs
def e2e_pipelined(host_in, dev_in, run, dev_out, host_out, steps, dev, world):
    """End to end through the C ABI with HOST buffers: every step copies its
    inputs from pinned host memory to the device, runs the call and copies its
    outputs back to pinned host memory. Copies and calls go on three streams
    with double-buffered device inputs and outputs, so that the copies of one
    step overlap the call of the previous one (as a caller streaming batches
    would run it). Returns seconds per step (max over ranks)."""
    s_in, s_run, s_out = (torch.cuda.Stream(dev) for _ in range(3))
    ev_in = [torch.cuda.Event() for _ in range(2)]
    ev_run = [torch.cuda.Event() for _ in range(2)]
    ev_out = [torch.cuda.Event() for _ in range(2)]

    def go(n):
        for i in range(n):
            b = i & 1
            with torch.cuda.stream(s_in):
                if i >= 2:
                    s_in.wait_event(ev_run[b])       # the call of step i - 2 has read buffer b
                for key, t in host_in.items():
                    dev_in[b][key].copy_(t, non_blocking=True)
                ev_in[b].record(s_in)
            s_run.wait_event(ev_in[b])
            if i >= 2:
                s_run.wait_event(ev_out[b])          # outputs b of step i - 2 are back on the host
            run(dev_in[b], dev_out[b], s_run)
            ev_run[b].record(s_run)
            with torch.cuda.stream(s_out):
                s_out.wait_event(ev_run[b])
                for key, t in host_out.items():
                    t.copy_(dev_out[b][key], non_blocking=True)
                ev_out[b].record(s_out)
        torch.cuda.synchronize(dev)

    go(2)  # warm the streams and buffers
    barrier(world)
    torch.cuda.synchronize(dev)
    t0 = time.perf_counter()
    go(steps)
    sec = (time.perf_counter() - t0) / steps
    return max_over_ranks(sec, world, dev)


def workload_config(name, w, world):
    """The `config` object of a prefill line (the same for both arms)."""
    lengths = w["lengths"]
    N, T = len(lengths), sum(lengths)
    seq = f"T={T // N}" if w["cu_seqlens"] is None else \
        f"{N} packed sequences, lengths U{{{WL[name].len_lo}..{WL[name].len_hi}}} (seed 0: {T} tokens)"
    h0 = "h0 ~ N(0, 0.02)" if w["h0"] is not None else "zero h0"
    return {"workload": f"{name}: B={N}, {seq}, H_qk={w['h_qk']}, H_v={w['h_v']}, d_k=d_v={w['d_k']}, chunk 64, "
                        f"bf16 q/k/v/o, fp32 g/beta/state, {h0}",
            "global_batch": N * world, "seq_len": T // N, "parallelism": f"replicas x{world}",
            "l2": "inputs larger than L2 (126 MB) every step; no flush"}


def run_prefill_leg(args, name, dev, peaks, world, rank, steps, cpu_seconds, main=False):
    """One prefill workload (gdn_chunk_fwd, bf16 o, fp32 final states) timed
    over `steps` launches with inputs resident in HBM; plus its cold first call,
    the median and 95% CI of the per-launch times, the roofline, the oracle on
    the host cores and the pipelined end-to-end throughput through the C ABI."""
    import gated_deltanet_recurrence_05_b300 as gdn
    w = gdn_inputs.make_workload(name, seed=args.seed + rank)
    lengths = w["lengths"]
    N, T = len(lengths), sum(lengths)
    dd = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in w.items()}
    order = gdn.plan_seq_order(w["cu_seqlens"]).to(dev) if w["cu_seqlens"] is not None else None
    o = torch.empty(T, w["h_v"], w["d_v"], dtype=torch.bfloat16, device=dev)
    fs = torch.empty(N, w["h_v"], w["d_k"], w["d_v"], dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def call(inp, o_, fs_, s_):
        gdn.chunk_fwd(inp["q"], inp["k"], inp["v"], inp["g"], inp["beta"], inp.get("h0"), dd["cu_seqlens"],
                      num_seqs=None if w["cu_seqlens"] is not None else N, seq_order=order,
                      out=o_, final_state_out=fs_, stream=s_)

    def step(_i=0):
        call(dd, o, fs, stream)

    cold = cold_call(step, stream, dev)
    with ClockSampler(dev.index) as clk:
        # warm-up inside the sampled window, right before the timed launches
        # (the sampler's start-up would otherwise leave the GPU idle in between)
        warm = warm_up(step, args.warmup, stream, dev)
        if gdn.get_device_error() != 0:
            raise RuntimeError(f"device error during the {name} warm-up")
        ms, per = timed_launches(step, steps, stream, dev, world)
    if gdn.get_device_error() != 0:
        raise RuntimeError(f"device error during the timed {name} region")
    ms_max = max_over_ranks(ms, world, dev)
    value = aggregate_throughput(T, world, ms_max / 1e3)

    bytes_, flops = prefill_algorithmic(w)
    gbs = bytes_ / (ms / 1e3) / 1e9
    tfs = flops / (ms / 1e3) / 1e12
    ridge = peaks["bf16_tflops"] * 1e12 / (peaks["hbm_gbs"] * 1e9)
    roofline = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(gbs / peaks["hbm_gbs"], 4),
                "traffic": (args.traffic if main and args.traffic is not None else
                            recorded_traffic() if name == "prefill" else
                            recorded_traffic("dram_bytes_per_launch_long") if name == "long" else None),
                "peak_source": PEAK_SOURCE, "algorithmic_bytes_per_launch": int(bytes_),
                "arithmetic_intensity_flop_per_byte": round(flops / bytes_, 1),
                "ridge_flop_per_byte": round(ridge, 1),
                "frac_of_min_roof": round(tfs * 1e12 / min(peaks["bf16_tflops"] * 1e12,
                                                           flops / bytes_ * peaks["hbm_gbs"] * 1e9), 4),
                "tensor": {"achieved_tflops": round(tfs, 1), "peak_tflops": peaks["bf16_tflops"],
                           "frac": round(tfs / peaks["bf16_tflops"], 4),
                           "algorithmic_flops_per_launch": flops}}

    e2e = None
    if not args.skip_e2e:
        keys = [k for k in ("q", "k", "v", "g", "beta", "h0") if w.get(k) is not None]
        host_in = {k: w[k].contiguous().pin_memory() for k in keys}
        dev_in = [{k: dd[k] for k in keys}, {k: torch.empty_like(dd[k]) for k in keys}]
        dev_out = [{"o": o, "fs": fs}, {"o": torch.empty_like(o), "fs": torch.empty_like(fs)}]
        host_out = {"o": torch.empty(o.shape, dtype=o.dtype).pin_memory(),
                    "fs": torch.empty(fs.shape, dtype=fs.dtype).pin_memory()}
        h2d = sum(t.numel() * t.element_size() for t in host_in.values())
        d2h = sum(t.numel() * t.element_size() for t in host_out.values())
        n_e2e = max(3, min(steps, 10 if T <= 20000 else 4))
        sec = e2e_pipelined(host_in, dev_in, lambda i, o_, s_: call(i, o_["o"], o_["fs"], s_), dev_out, host_out,
                            n_e2e, dev, world)
        if gdn.get_device_error() != 0:
            raise RuntimeError(f"device error in the {name} end-to-end run")
        e2e = {"value": aggregate_throughput(T, world, sec), "unit": "tokens/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h), "steps": n_e2e,
               "how": "C ABI call on host buffers: pinned H2D of the step's inputs, the call, D2H of o and the "
                      "final states, every step; copies of one step overlap the previous step's call "
                      "(three streams, double-buffered device tensors)"}

    cpu = None
    if rank == 0 and world == 1 and not args.skip_cpu_baseline:
        cpu = oracle_baseline(w, cpu_seconds)

    cfg = workload_config(name, w, world)
    return {
        "value": value, "unit": "tokens/s", "ms_per_step": ms_max, "steps": steps, "config": cfg,
        "workload": cfg["workload"], "tokens": T,
        "timing": _timing(per, ms), "cold_first_call": cold,
        "warmup_calls_run": warm,
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": steps,
        "clocks": clk.summary(),
    }


def run_ours(args, world, rank, local):
    dev = torch.device("cuda", local)
    peaks = load_peaks()
    main = run_prefill_leg(args, args.workload, dev, peaks, world, rank, args.steps, args.cpu_seconds, main=True)
    legs = {}
    if not args.skip_long_varlen and args.workload == "prefill":
        for name in ("long", "varlen"):
            legs[name] = run_prefill_leg(args, name, dev, peaks, world, rank, max(3, min(args.steps, 10)),
                                         args.cpu_seconds)
            torch.cuda.empty_cache()
    o_shape = (main["tokens"], 32, 128)
    decode = None if args.skip_decode else run_decode(args, dev, peaks, world)
    epilogue = None if args.skip_epilogue else run_epilogue(args, dev, peaks, world, o_shape)
    gated = None
    if epilogue is not None and args.workload == "prefill":
        sep = main["ms_per_step"] * 1e3 + epilogue["standalone"]["us_per_launch"]
        gated = run_gated_prefill(args, dev, peaks, world, sep)
    w = gdn_inputs.make_workload("prefill", seed=args.seed + rank)
    dd = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in w.items()}
    prologue = None if args.skip_epilogue else run_prologue(args, dev, peaks, world, w)
    backward = None if args.skip_backward else run_backward(args, dev, peaks, world, w, dd)
    kda = None if args.skip_kda else run_kda(args, dev, peaks, world, w, dd)
    launches = main["gpu_launches"]
    return {
        "metric": METRIC, "value": main["value"], "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": main["ms_per_step"], "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": main["config"],
        "roofline": main["roofline"], "cpu_baseline": main["cpu_baseline"], "e2e": main["e2e"],
        "gpu_launches": launches, "clocks": main["clocks"], "timing": main["timing"],
        "cold_first_call": main["cold_first_call"],
        "long": legs.get("long"), "varlen": legs.get("varlen"),
        "decode": decode, "epilogue": epilogue, "gated_prefill": gated, "prologue": prologue,
        "backward": backward, "kda": kda,
    }


def _timing(per, mean_ms, unit_scale=1.0, unit="ms per launch"):
    t = median_ci95([x * unit_scale for x in per])
    t.update(unit=unit, mean=mean_ms * unit_scale)
    if len(per) <= 32:
        t["samples"] = [round(x * unit_scale, 4) for x in per]
    return t


def run_gated_prefill(args, dev, peaks, world, separate_us):
    """The prefill and the layer's output epilogue through one call
    (gdn_chunk_fwd_gated: the prefill kernel, then the epilogue kernel in place
    on o) on the prefill workload; `separate_us` is the sum of the two lines
    measured on their own."""
    import gated_deltanet_recurrence_05_b300 as gdn
    w = gdn_inputs.make_workload("prefill", seed=args.seed)
    lengths = w["lengths"]
    N, T = len(lengths), sum(lengths)
    dd = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in w.items()}
    gen = torch.Generator().manual_seed(args.seed + 99)
    z = torch.randn(T, w["h_v"], w["d_v"], generator=gen).to(torch.bfloat16).to(dev)
    wn = (torch.randn(w["d_v"], generator=gen) * 0.2).to(dev)
    o = torch.empty(T, w["h_v"], w["d_v"], dtype=torch.bfloat16, device=dev)
    fs = torch.empty(N, w["h_v"], w["d_k"], w["d_v"], dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step(_i=0):
        gdn.chunk_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["h0"], None, num_seqs=N, out=o,
                      final_state_out=fs, gate=z, norm_weight=wn, stream=stream)

    cold = cold_call(step, stream, dev)
    for _ in range(args.warmup):
        step()
    ms, per = timed_launches(step, args.steps, stream, dev, world)
    if gdn.get_device_error() != 0:
        raise RuntimeError("device error in the gated prefill")
    us = max_over_ranks(ms * 1e3, world, dev)
    bytes_, flops = prefill_algorithmic(w)
    bytes_ += z.numel() * 2 + wn.numel() * 4
    gbs = bytes_ / (us / 1e6) / 1e9
    tfs = flops / (us / 1e6) / 1e12
    return {"workload": "prefill workload, then the output epilogue in place on o (bf16 gate [T, H_v, d_v], fp32 "
                        "norm weight), one gdn_chunk_fwd_gated call per step",
            "us_per_step": us, "tokens_per_s": T * world / (us / 1e6), "gpu_launches": 2 * args.steps,
            "separate_us": separate_us, "timing": _timing(per, ms, 1e3, "us per step"), "cold_first_call": cold,
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4), "algorithmic_bytes_per_launch": int(bytes_),
                         "tensor": {"achieved_tflops": round(tfs, 1), "peak_tflops": peaks["bf16_tflops"],
                                    "frac": round(tfs / peaks["bf16_tflops"], 4)}}}


def run_decode(args, dev, peaks, world):
    """Consecutive in-place decode steps on 256 x 32 states of 128x128."""
    import gated_deltanet_recurrence_05_b300 as gdn
    wl = gdn_inputs.WORKLOADS["decode"]
    steps = args.decode_steps
    d = gdn_inputs.make_workload("decode", steps=steps, seed=args.seed)
    dd = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    state = dd["state"].clone()
    o = torch.empty(wl.num_seqs, wl.h_v, wl.d_v, dtype=torch.bfloat16, device=dev)
    stream = torch.cuda.current_stream(dev)

    def one(t):
        gdn.decode_step(dd["q"][t], dd["k"][t], dd["v"][t], dd["g"][t], dd["beta"][t], state,
                        out=o, stream=stream)

    cold = cold_call(lambda: one(0), stream, dev)
    with ClockSampler(dev.index) as clk:
        warm_up(lambda: one(1), 3, stream, dev)
        state.copy_(dd["state"])
        ms, per = timed_launches(one, steps, stream, dev, world)
    if gdn.get_device_error() != 0:
        raise RuntimeError("device error in decode")
    us = max_over_ranks(ms * 1e3, world, dev)
    b = decode_algorithmic(wl.num_seqs, wl.h_qk, wl.h_v, wl.d_k, wl.d_v)
    gbs = b / (us / 1e6) / 1e9
    graph = decode_graph(gdn, dd, state, o, steps, b, peaks, dev, world)
    return {"workload": f"decode: {wl.num_seqs} sequences x H_v={wl.h_v} (H_qk={wl.h_qk}) x 128x128 fp32 "
                        f"states (512 MiB, > L2), bf16 token inputs and output, {steps} in-place steps",
            "us_per_step": us, "steps_per_s": 1e6 / us, "tokens_per_s": wl.num_seqs * 1e6 / us * world,
            "GB_per_s": gbs * world, "gpu_launches": steps, "clocks": clk.summary(),
            "timing": _timing(per, ms, 1e3, "us per step"), "cold_first_call": cold, "graph": graph,
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4), "algorithmic_bytes_per_launch": int(b)}}


def decode_graph(gdn, dd, state, o, steps, b, peaks, dev, world):
    """The same `steps` consecutive decode steps (each its own pregenerated
    token) captured once through the C ABI into a CUDA Graph and replayed as
    one launch; timed with CUDA events around a replay after one untimed
    replay. Returns the per-step time, or the capture's error message."""
    try:
        cg = torch.cuda.CUDAGraph()
        side = torch.cuda.Stream(dev)
        side.wait_stream(torch.cuda.current_stream(dev))
        with torch.cuda.graph(cg, stream=side):
            cap = torch.cuda.current_stream(dev)
            for t in range(steps):
                gdn.decode_step(dd["q"][t], dd["k"][t], dd["v"][t], dd["g"][t], dd["beta"][t], state,
                                out=o, stream=cap)
    except Exception as e:  # a capture the runtime refused: report it, keep the run
        torch.cuda.synchronize(dev)
        return {"error": f"{type(e).__name__}: {e}"[:300]}
    stream = torch.cuda.current_stream(dev)
    state.copy_(dd["state"])
    cg.replay()                      # untimed
    e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    torch.cuda.synchronize(dev)
    e0.record(stream)
    cg.replay()
    e1.record(stream)
    torch.cuda.synchronize(dev)
    barrier(world)
    if gdn.get_device_error() != 0:
        raise RuntimeError("device error in the decode graph")
    us = max_over_ranks(e0.elapsed_time(e1) * 1e3 / steps, world, dev)
    gbs = b / (us / 1e6) / 1e9
    del cg
    return {"steps": steps, "gpu_launches": steps, "us_per_step": us, "GB_per_s": gbs * world,
            "frac": round(gbs / peaks["hbm_gbs"], 4),
            "how": f"{steps} decode steps captured into one CUDA Graph through the C ABI, replayed once untimed "
                   f"and once timed (CUDA events around the replay)"}


def run_epilogue(args, dev, peaks, world, o_shape):
    """The GDN output epilogue (zero-centred RMSNorm x sigmoid gate): standalone
    on a tensor shaped like the prefill output, and fused into the decode step."""
    import gated_deltanet_recurrence_05_b300 as gdn
    gen = torch.Generator().manual_seed(args.seed + 99)
    o = torch.randn(o_shape, generator=gen).to(torch.bfloat16).to(dev)
    z = torch.randn(o.shape, generator=gen).to(torch.bfloat16).to(dev)
    wn = (torch.randn(o.shape[-1], generator=gen) * 0.2).to(dev)
    y = torch.empty_like(o)
    stream = torch.cuda.current_stream(dev)
    reps = max(3, args.steps)
    launch = lambda i=0: gdn.gated_rmsnorm(o, z, wn, out=y, stream=stream)
    cold = cold_call(launch, stream, dev)
    for _ in range(3):
        launch()
    ms, per = timed_launches(launch, reps, stream, dev, world)
    us = max_over_ranks(ms * 1e3, world, dev)
    b = 3 * o.numel() * o.element_size() + wn.numel() * 4
    gbs = b / (us / 1e6) / 1e9
    out = {"standalone": {"workload": f"gated RMSNorm on a bf16 tensor shaped like the prefill output {list(o.shape)} "
                                      f"(gate bf16, weight fp32), > L2 every launch",
                          "us_per_launch": us, "GB_per_s": gbs * world, "gpu_launches": reps,
                          "timing": _timing(per, ms, 1e3, "us per launch"), "cold_first_call": cold,
                          "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                                       "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                                       "algorithmic_bytes_per_launch": int(b)}}}
    del o, z, y
    if not args.skip_decode:
        wl = gdn_inputs.WORKLOADS["decode"]
        steps = min(args.decode_steps, 200)
        d = gdn_inputs.make_workload("decode", steps=steps, seed=args.seed)
        dd = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
        state = dd["state"].clone()
        od = torch.empty(wl.num_seqs, wl.h_v, wl.d_v, dtype=torch.bfloat16, device=dev)
        zd = torch.randn(steps, wl.num_seqs, wl.h_v, wl.d_v, generator=gen).to(torch.bfloat16).to(dev)
        wd = (torch.randn(wl.d_v, generator=gen) * 0.2).to(dev)

        def one(t):
            gdn.decode_step(dd["q"][t], dd["k"][t], dd["v"][t], dd["g"][t], dd["beta"][t], state, out=od,
                            gate=zd[t], norm_weight=wd, stream=stream)

        for t in range(min(3, steps)):
            one(t)
        torch.cuda.synchronize(dev)
        state.copy_(dd["state"])
        ms_d, per_d = timed_launches(one, steps, stream, dev, world)
        if gdn.get_device_error() != 0:
            raise RuntimeError("device error in the gated decode")
        us_d = max_over_ranks(ms_d * 1e3, world, dev)
        bd = decode_algorithmic(wl.num_seqs, wl.h_qk, wl.h_v, wl.d_k, wl.d_v) + zd[0].numel() * 2 + wd.numel() * 4
        gbd = bd / (us_d / 1e6) / 1e9
        out["fused_decode"] = {"workload": "the decode workload with the epilogue fused (gate bf16 per step)",
                               "us_per_step": us_d, "gpu_launches": steps,
                               "timing": _timing(per_d, ms_d, 1e3, "us per step"),
                               "roofline": {"bound": "hbm", "achieved": round(gbd, 1), "peak": peaks["hbm_gbs"],
                                            "unit": "GB/s", "frac": round(gbd / peaks["hbm_gbs"], 4),
                                            "algorithmic_bytes_per_launch": int(bd)}}
    return out


def run_prologue(args, dev, peaks, world, w):
    """The GDN input prologue (causal depthwise conv K=4, silu, per-head L2 norm
    for q and k) on the three projections of the prefill workload."""
    import gated_deltanet_recurrence_05_b300 as gdn
    T = sum(w["lengths"])
    N = len(w["lengths"])
    gen = torch.Generator().manual_seed(args.seed + 77)
    shapes = [(w["h_qk"] * w["d_k"], w["d_k"]), (w["h_qk"] * w["d_k"], w["d_k"]), (w["h_v"] * w["d_v"], 0)]
    bufs = []
    for C, ng in shapes:
        x = torch.randn(T, C, generator=gen).to(torch.bfloat16).to(dev)
        wt = (torch.randn(C, 4, generator=gen) * 0.5).to(dev)
        bufs.append((x, wt, torch.empty_like(x), ng))
    stream = torch.cuda.current_stream(dev)
    cu = w["cu_seqlens"].to(dev) if w["cu_seqlens"] is not None else None

    def step(_i=0):
        for x, wt, y, ng in bufs:
            gdn.short_conv(x, wt, cu_seqlens=cu, num_seqs=N, norm_group=ng, out=y, stream=stream)

    cold = cold_call(step, stream, dev)
    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    reps = max(3, args.steps)
    ms, per = timed_launches(step, reps, stream, dev, world)
    if gdn.get_device_error() != 0:
        raise RuntimeError("device error in the prologue")
    us = max_over_ranks(ms * 1e3, world, dev)
    b = sum(2 * x.numel() * x.element_size() + wt.numel() * 4 for x, wt, _, _ in bufs)
    gbs = b / (us / 1e6) / 1e9
    return {"workload": f"short conv (K=4) + silu (+ L2 norm per head for q, k) on the q, k [{T}, "
                        f"{shapes[0][0]}] and v [{T}, {shapes[2][0]}] bf16 projections of the prefill workload",
            "us_per_step": us, "GB_per_s": gbs * world, "gpu_launches": 3 * reps,
            "timing": _timing(per, ms, 1e3, "us per step (three launches)"), "cold_first_call": cold,
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4), "algorithmic_bytes_per_launch": int(b)}}


def backward_algorithmic(T, h_v, d_k, d_v):
    """FLOPs of the gradient by the reverse-order chain rule with the states at
    hand, per token and value head: the forward quantities it needs (S^T k,
    the rank-1 state update, S dO) and the reverse step (D += q dO^T, D^T k,
    D e, S de, D <- a (D - k de^T)): eight passes of one multiply-add per state
    element, 16 d_k d_v FLOPs."""
    return 16.0 * d_k * d_v * T * h_v


# fp32 CUDA-core peak of the B300: 148 SMs x 128 fp32 lanes x 2 FLOP per FMA x 2032 MHz
SIMT_FP32_TFLOPS = 148 * 128 * 2 * 2.032e9 / 1e12


def run_backward(args, dev, peaks, world, w, dd):
    """The gradient (gdn_chunk_bwd) of the prefill workload: bf16 dO ~ N(0,1),
    dS_T ~ N(0, 0.05), workspace allocated once outside the timed region."""
    import gated_deltanet_recurrence_05_b300 as gdn
    lengths = w["lengths"]
    N, T = len(lengths), sum(lengths)
    h_qk, h_v, d_k, d_v = w["h_qk"], w["h_v"], w["d_k"], w["d_v"]
    gr = gdn_inputs.make_grads(w, dtype="bf16", dht_std=0.05, seed=args.seed)
    do, dht = gr["do"].to(dev), gr["dht"].to(dev)
    f32 = dict(dtype=torch.float32, device=dev)
    outs = (torch.empty(T, h_qk, d_k, **f32), torch.empty(T, h_qk, d_k, **f32), torch.empty(T, h_v, d_v, **f32),
            torch.empty(T, h_v, **f32), torch.empty(T, h_v, **f32), torch.empty(N, h_v, d_k, d_v, **f32))
    ws = torch.empty(gdn.chunk_bwd_workspace_size(N, T, h_qk, h_v, d_k, d_v), dtype=torch.uint8, device=dev)
    cu = dd["cu_seqlens"]
    stream = torch.cuda.current_stream(dev)

    def step():
        gdn.chunk_bwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], do, dd["h0"], dht, cu,
                      num_seqs=None if cu is not None else N, out=outs, workspace=ws, stream=stream)

    cold = cold_call(step, stream, dev)
    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    reps = max(3, min(args.steps, 10))
    ms, per = timed_launches(lambda i: step(), reps, stream, dev, world)
    if gdn.get_device_error() != 0:
        raise RuntimeError("device error in the backward")
    us = max_over_ranks(ms * 1e3, world, dev)
    flops = backward_algorithmic(T, h_v, d_k, d_v)
    tfs = flops / (us / 1e6) / 1e12

    cpu = None
    if world == 1 and not args.skip_cpu_baseline:
        import oracle
        n_tok = min(4096, lengths[0])
        sl = slice(0, n_tok)
        t0 = time.perf_counter()
        oracle.recurrent_backward(w["q"][sl, :1], w["k"][sl, :1], w["v"][sl, :1], w["g"][sl, :1],
                                  w["beta"][sl, :1], gr["do"][sl, :1])
        sec = time.perf_counter() - t0
        cores = int(os.environ.get("OPENBLAS_NUM_THREADS", "0")) or os.cpu_count()
        cpu = {"value": n_tok / sec / h_v, "unit": "tokens/s", "cores": cores, "kind": "oracle",
               "sample": f"{n_tok} tokens of one (sequence, value head) pair, scaled to all {h_v} value heads"}
    return {"workload": f"gradient of the prefill workload (B={N}, T={T // N}, H_qk={h_qk}, H_v={h_v}, "
                        f"d=128, bf16 q/k/v/dO, fp32 g/beta/dS_T, fp32 gradients)",
            "us_per_step": us, "tokens_per_s": T * world / (us / 1e6),
            "gpu_launches": reps * (2 if h_v > h_qk else 1), "cpu_baseline": cpu,
            "timing": _timing(per, ms, 1e3, "us per gradient step"), "cold_first_call": cold,
            "roofline": {"bound": "alu", "achieved": round(tfs, 2), "peak": round(SIMT_FP32_TFLOPS, 1),
                         "unit": "TFLOP/s", "frac": round(tfs / SIMT_FP32_TFLOPS, 4),
                         "peak_source": "derived: 148 SMs x 128 fp32 lanes x 2 FLOP x 2032 MHz",
                         "algorithmic_flops_per_launch": flops}}


def run_kda(args, dev, peaks, world, w, dd):
    """The per-channel-decay variant (KDA): the prefill workload with one
    log-decay per key channel (g = -softplus(N(0,1) + 2) per channel), and
    in-place decode steps on the decode workload's 256 x 32 states with
    per-channel decays drawn per step."""
    import gated_deltanet_recurrence_05_b300 as gdn
    lengths = w["lengths"]
    N, T = len(lengths), sum(lengths)
    h_v, d_k, d_v = w["h_v"], w["d_k"], w["d_v"]
    g = gdn_inputs.make_channel_decay((T, h_v, d_k), g_shift=2.0, seed=args.seed).to(dev)
    o = torch.empty(T, h_v, d_v, dtype=torch.bfloat16, device=dev)
    fs = torch.empty(N, h_v, d_k, d_v, dtype=torch.float32, device=dev)
    cu = dd["cu_seqlens"]
    stream = torch.cuda.current_stream(dev)

    def prefill():
        gdn.kda_chunk_fwd(dd["q"], dd["k"], dd["v"], g, dd["beta"], dd["h0"], cu,
                          num_seqs=None if cu is not None else N, out=o, final_state_out=fs, stream=stream)

    timings = {}

    def timed(fn, reps, key):
        ms, per = timed_launches(fn, reps, stream, dev, world)
        if gdn.get_device_error() != 0:
            raise RuntimeError("device error in KDA")
        timings[key] = _timing(per, ms, 1e3, "us per launch")
        return max_over_ranks(ms * 1e3, world, dev)

    cold = cold_call(prefill, stream, dev)
    for _ in range(3):
        prefill()
    reps = max(3, min(args.steps, 10))
    us_pf = timed(lambda i: prefill(), reps, "prefill")
    flops = 6.0 * d_k * d_v * T * h_v   # the two reads of the state and its update, per token and head
    tfs = flops / (us_pf / 1e6) / 1e12
    tf32_peak = peaks["bf16_tflops"] * (1.1 / 2.25)

    wl = gdn_inputs.WORKLOADS["decode"]
    steps = 100
    t = gdn_inputs.make_workload("decode", steps=steps, seed=args.seed)
    tt = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in t.items()}
    gd = gdn_inputs.make_channel_decay((steps, wl.num_seqs, wl.h_v, wl.d_k), seed=args.seed).to(dev)
    state = tt["state"].clone()
    od = torch.empty(wl.num_seqs, wl.h_v, wl.d_v, dtype=torch.bfloat16, device=dev)

    def dstep(i):
        gdn.kda_decode_step(tt["q"][i], tt["k"][i], tt["v"][i], gd[i], tt["beta"][i], state, out=od,
                            stream=stream)

    for i in range(3):
        dstep(i)
    state.copy_(tt["state"])
    us_dec = timed(dstep, steps, "decode")
    # the decode step's bytes with g per key channel instead of one per head
    b = decode_algorithmic(wl.num_seqs, wl.h_qk, wl.h_v, wl.d_k, wl.d_v) + wl.num_seqs * wl.h_v * (wl.d_k - 1) * 4
    gbs = b / (us_dec / 1e6) / 1e9
    return {"prefill": {"workload": f"KDA prefill: the prefill workload (B={N}, T={T // N}) with per-channel "
                                    f"fp32 log-decays [T, {h_v}, {d_k}], bf16 o, fp32 final states",
                        "us_per_launch": us_pf, "tokens_per_s": T * world / (us_pf / 1e6), "gpu_launches": reps,
                        "timing": timings["prefill"], "cold_first_call": cold,
                        "roofline": {"bound": "tensor", "achieved": round(tfs, 2), "peak": peaks["bf16_tflops"],
                                     "unit": "TFLOP/s", "frac": round(tfs / peaks["bf16_tflops"], 4),
                                     "peak_source": "measured (bf16, the fp16 rate): the state products run on "
                                                    "fp16 warp MMA as three passes over split operands (fp32 "
                                                    "accuracy), the intra-chunk scores on tf32",
                                     "tf32_peak": round(tf32_peak, 1),
                                     "fp32_simt_peak": round(SIMT_FP32_TFLOPS, 1),
                                     "frac_of_fp32_simt": round(tfs / SIMT_FP32_TFLOPS, 4),
                                     "algorithmic_flops_per_launch": flops}},
            "decode": {"workload": f"KDA decode: {wl.num_seqs} x {wl.h_v} states of 128x128 fp32, per-channel "
                                   f"decays, {steps} in-place steps",
                       "us_per_step": us_dec, "GB_per_s": gbs * world, "gpu_launches": steps,
                       "timing": timings["decode"],
                       "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                                    "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                                    "algorithmic_bytes_per_launch": int(b)}}}


def run_reference(args, world, rank):
    """The oracle as it stands, timed on the host cores (bounded sample)."""
    if rank != 0:
        return None
    w = gdn_inputs.make_workload(args.workload, seed=args.seed)
    N, T = len(w["lengths"]), sum(w["lengths"])
    per_step = []
    cores, sample = 1, ""
    for _ in range(max(args.steps, 1)):
        tok_s, cores, sample = oracle_sample(w, target_s=max(2.0, args.cpu_seconds / max(args.steps, 1)))
        per_step.append(tok_s)
    value = statistics.median(per_step)
    return {"metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
            "warmup": args.warmup, "ms_per_step": T / value * 1e3, "higher_is_better": True,
            "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
            "config": workload_config(args.workload, w, world),
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": sample, "per_step": per_step},
            "e2e": {"value": value, "unit": "tokens/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
            "gpu_launches": 0}


def main(argv=None):
    ap = argparse.ArgumentParser(description=__doc__, formatter_class=argparse.RawDescriptionHelpFormatter)
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", choices=["ours", "reference"], default="ours")
    ap.add_argument("--workload", choices=["prefill", "long", "varlen"], default="prefill")
    ap.add_argument("--seed", type=int, default=0)
    ap.add_argument("--decode-steps", type=int, default=1000)
    ap.add_argument("--cpu-seconds", type=float, default=12.0)
    ap.add_argument("--traffic", type=float, default=None,
                    help="DRAM bytes per launch of the prefill kernel from an ncu capture")
    ap.add_argument("--skip-decode", action="store_true")
    ap.add_argument("--skip-epilogue", action="store_true", help="skip the epilogue and prologue lines")
    ap.add_argument("--skip-e2e", action="store_true")
    ap.add_argument("--skip-backward", action="store_true", help="skip the gradient line")
    ap.add_argument("--skip-kda", action="store_true", help="skip the per-channel-decay (KDA) lines")
    ap.add_argument("--skip-cpu-baseline", action="store_true")
    ap.add_argument("--skip-long-varlen", action="store_true", help="skip the long and varlen prefill lines")
    args = ap.parse_args(argv)
    args.warmup = max(args.warmup, 3)
    world, rank, local = dist_setup(args)
    line = run_reference(args, world, rank) if args.impl == "reference" else run_ours(args, world, rank, local)
    if rank == 0 and line is not None:
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
