#!/usr/bin/env python3
"""Benchmark of the Gated DeltaNet forward recurrence on B300.

One step = one chunked prefill forward (gdn_chunk_fwd) over the prefill
workload: B=4 sequences x T=4096 tokens, H_qk=16, H_v=32, d_k=d_v=128, bf16
q/k/v, fp32 g/beta and state, chunk 64, zero initial state, bf16 output plus
fp32 final states. value = tokens/s over all ranks. The same JSON line also
carries the decode step (256 sequences x 32 heads x 128x128 fp32 states,
1000 consecutive in-place steps, bf16 token inputs) in GB/s, the output
epilogue and input prologue in GB/s, the gradient of the prefill
workload (gdn_chunk_bwd) in tokens/s against the fp32 CUDA-core peak, and the
per-channel-decay variant (KDA) prefill and decode.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--impl ours|reference]

Under torchrun (N > 1) every rank runs its own independent copy of the
workload (the work shards by sequence with no exchange: weak scaling); the
timed region is bracketed by barriers and the max over ranks is reported.
--impl reference times the fp64 CPU oracle (test infrastructure) on a bounded
sample of the same workload on the host cores.
"""
from __future__ import annotations

import argparse
import hashlib
import json
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
def load_peaks():
    try:
        with open(os.path.join(ROOT, "MEASURED_PEAKS.json")) as f:
            return json.load(f), "measured"
    except (OSError, ValueError):
        return dict(PEAKS_FALLBACK), "fallback"


def kernel_sha():
    """Hash of the prefill kernel's sources (ties recorded ncu counters to them)."""
    h = hashlib.sha256()
    for name in KERNEL_SOURCES:
        with open(os.path.join(ROOT, "gated_deltanet_recurrence_05_b300", "csrc", name), "rb") as f:
            h.update(f.read())
    return h.hexdigest()[:16]


def recorded_traffic():
    """DRAM bytes per prefill launch from the committed ncu summary, or None if
    the summary is absent or was taken on other kernel sources."""
    try:
        kv = {}
        with open(TRAFFIC_FILE) as f:
            for line in f:
                if ":" in line and not line.startswith("#"):
                    k, v = line.split(":", 1)
                    kv[k.strip()] = v.strip()
        if kv.get("kernel_sha256") != kernel_sha():
            return None
        return float(kv["dram_bytes_per_launch"])
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
    t = time.perf_counter()
    oracle.recurrent(w["q"], w["k"], w["v"], w["g"], w["beta"], h0=w["h0"], cu_seqlens=cu,
                     pairs=[(0, 0)], threads=1)
    one = time.perf_counter() - t
    n_pairs = max(cores, int(target_s * cores / max(one, 1e-3)))
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


# --------------------------------------------------------------------------- GPU legs
def run_ours(args, world, rank, local):
    import gated_deltanet_recurrence_05_b300 as gdn
    dev = torch.device("cuda", local)
    peaks, peak_kind = load_peaks()
    w = gdn_inputs.make_workload(args.workload, seed=args.seed + rank)
    lengths = w["lengths"]
    N, T = len(lengths), sum(lengths)
    dd = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in w.items()}
    order = gdn.plan_seq_order(w["cu_seqlens"]).to(dev) if w["cu_seqlens"] is not None else None
    o = torch.empty(T, w["h_v"], w["d_v"], dtype=torch.bfloat16, device=dev)
    fs = torch.empty(N, w["h_v"], w["d_k"], w["d_v"], dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream(dev)

    def step():
        gdn.chunk_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["h0"], dd["cu_seqlens"],
                      num_seqs=None if w["cu_seqlens"] is not None else N, seq_order=order,
                      out=o, final_state_out=fs, stream=stream)

    for _ in range(args.warmup):
        step()
    torch.cuda.synchronize(dev)
    if gdn.get_device_error() != 0:
        raise RuntimeError("device error during warm-up")
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(local) as clk:
        barrier(world)
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        for _ in range(args.steps):
            step()
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
    if gdn.get_device_error() != 0:
        raise RuntimeError("device error during the timed region")
    ms = ev0.elapsed_time(ev1) / args.steps
    ms_max = max_over_ranks(ms, world, dev)
    value = aggregate_throughput(T, world, ms_max / 1e3)

    bytes_, flops = prefill_algorithmic(w)
    gbs = bytes_ / (ms / 1e3) / 1e9
    tfs = flops / (ms / 1e3) / 1e12
    roofline = {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                "frac": round(gbs / peaks["hbm_gbs"], 4),
                "traffic": args.traffic if args.traffic is not None else recorded_traffic(),
                "peak_source": peak_kind, "algorithmic_bytes_per_launch": int(bytes_),
                "tensor": {"achieved_tflops": round(tfs, 1), "peak_tflops": peaks["bf16_tflops"],
                           "frac": round(tfs / peaks["bf16_tflops"], 4),
                           "algorithmic_flops_per_launch": flops}}

    # end to end through the C ABI with host buffers: H2D of the step's inputs
    # from pinned memory, the call, D2H of the outputs, all inside the timed region
    e2e = None
    if not args.skip_e2e:
        host = {k: w[k].pin_memory() for k in ("q", "k", "v", "g", "beta")}
        o_h = torch.empty(o.shape, dtype=o.dtype).pin_memory()
        fs_h = torch.empty(fs.shape, dtype=fs.dtype).pin_memory()
        h2d = sum(t.numel() * t.element_size() for t in host.values())
        d2h = o.numel() * o.element_size() + fs.numel() * fs.element_size()

        def e2e_step():
            for key, t in host.items():
                dd[key].copy_(t, non_blocking=True)
            step()
            o_h.copy_(o, non_blocking=True)
            fs_h.copy_(fs, non_blocking=True)

        e2e_step()
        torch.cuda.synchronize(dev)
        n_e2e = max(2, min(args.steps, 10))
        barrier(world)
        torch.cuda.synchronize(dev)
        t0 = time.perf_counter()
        for _ in range(n_e2e):
            e2e_step()
        torch.cuda.synchronize(dev)
        e2e_s = max_over_ranks((time.perf_counter() - t0) / n_e2e, world, dev)
        e2e = {"value": aggregate_throughput(T, world, e2e_s), "unit": "tokens/s",
               "h2d_bytes_per_step": int(h2d), "d2h_bytes_per_step": int(d2h)}

    decode = None if args.skip_decode else run_decode(args, dev, peaks, world)
    epilogue = None if args.skip_epilogue else run_epilogue(args, dev, peaks, world, o)
    prologue = None if args.skip_epilogue else run_prologue(args, dev, peaks, world, w)
    backward = None if args.skip_backward else run_backward(args, dev, peaks, world, w, dd)
    kda = None if args.skip_kda else run_kda(args, dev, peaks, world, w, dd)

    cpu = None
    if rank == 0 and world == 1 and not args.skip_cpu_baseline:
        tok_s, cores, sample = oracle_sample(w, target_s=args.cpu_seconds)
        cpu = {"value": tok_s, "unit": "tokens/s", "cores": cores, "kind": "oracle", "sample": sample}

    seq = f"T={T // N}" if w["cu_seqlens"] is None else f"lengths U{{{min(lengths)}..{max(lengths)}}}"
    return {
        "metric": METRIC, "value": value, "unit": "tokens/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": ms_max, "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "bf16", "data": "synthetic",
        "config": {"workload": f"{args.workload}: B={N}, {seq}, H_qk={w['h_qk']}, H_v={w['h_v']}, "
                               f"d_k=d_v={w['d_k']}, chunk 64, bf16 q/k/v/o, fp32 g/beta/state",
                   "global_batch": N * world, "seq_len": T // N, "parallelism": f"replicas x{world}",
                   "l2": "inputs larger than L2 (126 MB) every step; no flush"},
        "roofline": roofline, "cpu_baseline": cpu, "e2e": e2e, "gpu_launches": args.steps,
        "clocks": clk.summary(), "decode": decode, "epilogue": epilogue, "prologue": prologue,
        "backward": backward, "kda": kda,
    }


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

    def run(n0, n1):
        for t in range(n0, n1):
            gdn.decode_step(dd["q"][t], dd["k"][t], dd["v"][t], dd["g"][t], dd["beta"][t], state,
                            out=o, stream=stream)

    run(0, min(3, steps))
    torch.cuda.synchronize(dev)
    state.copy_(dd["state"])
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    with ClockSampler(dev.index) as clk:
        barrier(world)
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        run(0, steps)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        barrier(world)
    if gdn.get_device_error() != 0:
        raise RuntimeError("device error in decode")
    us = ev0.elapsed_time(ev1) * 1e3 / steps
    us = max_over_ranks(us, world, dev)
    b = decode_algorithmic(wl.num_seqs, wl.h_qk, wl.h_v, wl.d_k, wl.d_v)
    gbs = b / (us / 1e6) / 1e9
    return {"workload": f"decode: {wl.num_seqs} sequences x H_v={wl.h_v} (H_qk={wl.h_qk}) x 128x128 fp32 "
                        f"states (512 MiB, > L2), bf16 token inputs and output, {steps} in-place steps",
            "us_per_step": us, "steps_per_s": 1e6 / us, "tokens_per_s": wl.num_seqs * 1e6 / us * world,
            "GB_per_s": gbs * world, "gpu_launches": steps, "clocks": clk.summary(),
            "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"], "unit": "GB/s",
                         "frac": round(gbs / peaks["hbm_gbs"], 4), "algorithmic_bytes_per_launch": int(b)}}


def run_epilogue(args, dev, peaks, world, o):
    """The GDN output epilogue (zero-centred RMSNorm x sigmoid gate): standalone
    on the prefill output, and fused into the decode step."""
    import gated_deltanet_recurrence_05_b300 as gdn
    gen = torch.Generator().manual_seed(args.seed + 99)
    z = torch.randn(o.shape, generator=gen).to(torch.bfloat16).to(dev)
    wn = (torch.randn(o.shape[-1], generator=gen) * 0.2).to(dev)
    y = torch.empty_like(o)
    stream = torch.cuda.current_stream(dev)
    reps = max(3, args.steps)
    for _ in range(3):
        gdn.gated_rmsnorm(o, z, wn, out=y, stream=stream)
    torch.cuda.synchronize(dev)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    ev0.record(stream)
    for _ in range(reps):
        gdn.gated_rmsnorm(o, z, wn, out=y, stream=stream)
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    us = max_over_ranks(ev0.elapsed_time(ev1) * 1e3 / reps, world, dev)
    b = 3 * o.numel() * o.element_size() + wn.numel() * 4
    gbs = b / (us / 1e6) / 1e9
    out = {"standalone": {"workload": f"gated RMSNorm on the prefill output {list(o.shape)} bf16 (gate bf16, "
                                      f"weight fp32), > L2 every launch",
                          "us_per_launch": us, "GB_per_s": gbs * world, "gpu_launches": reps,
                          "roofline": {"bound": "hbm", "achieved": round(gbs, 1), "peak": peaks["hbm_gbs"],
                                       "unit": "GB/s", "frac": round(gbs / peaks["hbm_gbs"], 4),
                                       "algorithmic_bytes_per_launch": int(b)}}}
    if not args.skip_decode:
        wl = gdn_inputs.WORKLOADS["decode"]
        steps = min(args.decode_steps, 200)
        d = gdn_inputs.make_workload("decode", steps=steps, seed=args.seed)
        dd = {k: (v.to(dev) if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
        state = dd["state"].clone()
        od = torch.empty(wl.num_seqs, wl.h_v, wl.d_v, dtype=torch.bfloat16, device=dev)
        zd = torch.randn(steps, wl.num_seqs, wl.h_v, wl.d_v, generator=gen).to(torch.bfloat16).to(dev)
        wd = (torch.randn(wl.d_v, generator=gen) * 0.2).to(dev)

        def run(n0, n1):
            for t in range(n0, n1):
                gdn.decode_step(dd["q"][t], dd["k"][t], dd["v"][t], dd["g"][t], dd["beta"][t], state, out=od,
                                gate=zd[t], norm_weight=wd, stream=stream)

        run(0, min(3, steps))
        torch.cuda.synchronize(dev)
        state.copy_(dd["state"])
        barrier(world)
        ev0.record(stream)
        run(0, steps)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        if gdn.get_device_error() != 0:
            raise RuntimeError("device error in the gated decode")
        us_d = max_over_ranks(ev0.elapsed_time(ev1) * 1e3 / steps, world, dev)
        bd = decode_algorithmic(wl.num_seqs, wl.h_qk, wl.h_v, wl.d_k, wl.d_v) + zd[0].numel() * 2 + wd.numel() * 4
        gbd = bd / (us_d / 1e6) / 1e9
        out["fused_decode"] = {"workload": "the decode workload with the epilogue fused (gate bf16 per step)",
                               "us_per_step": us_d, "gpu_launches": steps,
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

    def step():
        for x, wt, y, ng in bufs:
            gdn.short_conv(x, wt, cu_seqlens=w["cu_seqlens"].to(dev) if w["cu_seqlens"] is not None else None,
                           num_seqs=N, norm_group=ng, out=y, stream=stream)

    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    reps = max(3, args.steps)
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    ev0.record(stream)
    for _ in range(reps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    if gdn.get_device_error() != 0:
        raise RuntimeError("device error in the prologue")
    us = max_over_ranks(ev0.elapsed_time(ev1) * 1e3 / reps, world, dev)
    b = sum(2 * x.numel() * x.element_size() + wt.numel() * 4 for x, wt, _, _ in bufs)
    gbs = b / (us / 1e6) / 1e9
    return {"workload": f"short conv (K=4) + silu (+ L2 norm per head for q, k) on the q, k [{T}, "
                        f"{shapes[0][0]}] and v [{T}, {shapes[2][0]}] bf16 projections of the prefill workload",
            "us_per_step": us, "GB_per_s": gbs * world, "gpu_launches": 3 * reps,
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

    for _ in range(3):
        step()
    torch.cuda.synchronize(dev)
    reps = max(3, min(args.steps, 10))
    ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    barrier(world)
    ev0.record(stream)
    for _ in range(reps):
        step()
    ev1.record(stream)
    torch.cuda.synchronize(dev)
    if gdn.get_device_error() != 0:
        raise RuntimeError("device error in the backward")
    us = max_over_ranks(ev0.elapsed_time(ev1) * 1e3 / reps, world, dev)
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

    def timed(fn, reps):
        ev0, ev1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        barrier(world)
        torch.cuda.synchronize(dev)
        ev0.record(stream)
        for i in range(reps):
            fn(i)
        ev1.record(stream)
        torch.cuda.synchronize(dev)
        if gdn.get_device_error() != 0:
            raise RuntimeError("device error in KDA")
        return max_over_ranks(ev0.elapsed_time(ev1) * 1e3 / reps, world, dev)

    for _ in range(3):
        prefill()
    reps = max(3, min(args.steps, 10))
    us_pf = timed(lambda i: prefill(), reps)
    flops = 6.0 * d_k * d_v * T * h_v   # S^T (a o k), S^T (a o q), the decayed rank-1 update
    tfs = flops / (us_pf / 1e6) / 1e12

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
    us_dec = timed(dstep, steps)
    # the decode step's bytes with g per key channel instead of one per head
    b = decode_algorithmic(wl.num_seqs, wl.h_qk, wl.h_v, wl.d_k, wl.d_v) + wl.num_seqs * wl.h_v * (wl.d_k - 1) * 4
    gbs = b / (us_dec / 1e6) / 1e9
    return {"prefill": {"workload": f"KDA prefill: the prefill workload (B={N}, T={T // N}) with per-channel "
                                    f"fp32 log-decays [T, {h_v}, {d_k}], bf16 o, fp32 final states",
                        "us_per_launch": us_pf, "tokens_per_s": T * world / (us_pf / 1e6), "gpu_launches": reps,
                        "roofline": {"bound": "alu", "achieved": round(tfs, 2), "peak": round(SIMT_FP32_TFLOPS, 1),
                                     "unit": "TFLOP/s", "frac": round(tfs / SIMT_FP32_TFLOPS, 4),
                                     "peak_source": "derived: 148 SMs x 128 fp32 lanes x 2 FLOP x 2032 MHz",
                                     "algorithmic_flops_per_launch": flops}},
            "decode": {"workload": f"KDA decode: {wl.num_seqs} x {wl.h_v} states of 128x128 fp32, per-channel "
                                   f"decays, {steps} in-place steps",
                       "us_per_step": us_dec, "GB_per_s": gbs * world, "gpu_launches": steps,
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
            "config": {"workload": f"{args.workload}: B={N}, T={T // N}, H_qk={w['h_qk']}, H_v={w['h_v']}, "
                                   f"d_k=d_v={w['d_k']}", "global_batch": N, "seq_len": T // N,
                       "parallelism": "host cores"},
            "impl": "reference",
            "cpu_baseline": {"value": value, "unit": "tokens/s", "cores": cores, "kind": "oracle",
                             "sample": sample},
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
