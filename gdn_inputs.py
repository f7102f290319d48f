"""Seeded synthetic inputs for the Gated DeltaNet (GDN) forward recurrence.

This module only draws random numbers and lays them out; it holds none of the
recurrence's arithmetic. Both the fp64 CPU oracle (under ``oracle/``) and the
CUDA path take their inputs from here, so the two sides always see identical
values.

Workloads (the five synthetic cases of the GDN hot path; distributions follow
the problem statement of the recurrence: q, k ~ N(0,1) then L2-normalised per
head, v ~ N(0,1), beta = sigmoid(N(0,1)), g = -softplus(N(0,1) + shift),
alpha = exp(g), initial states N(0, 0.02) where one is given):

=============  ===============================================================
``tiny``       B=1, T=64, H_qk=H_v=2, d_k=d_v=16, fp32, chunk 16, zero state
``prefill``    B=4, T=4096, H_qk=16, H_v=32, d=128, bf16 q/k/v, shift=+2
``long``       B=1, T=65536, H_qk=16, H_v=32, d=128, bf16, h0 ~ N(0,0.02)
``decode``     256 sequences x 32 v-heads, 128x128 fp32 states ~ N(0,0.02),
               one bf16 token per step, 1000 steps
``varlen``     64 sequences, lengths ~ U{128..8192}, packed by cu_seqlens
=============  ===============================================================

Draw order (fixed, one ``torch.Generator`` seeded with ``seed``): sequence
lengths (varlen only) -> q -> k -> v -> beta-raw -> g-raw -> h0. Every value is
drawn in fp32 and then cast to the storage dtype. The incoming gradients of a
backward problem (``make_grads``) come from a second generator, so drawing
them leaves the forward inputs unchanged.

Layouts (dense, row-major):
  q, k : [T_total, H_qk, d_k]      v : [T_total, H_v, d_v]
  g, beta : [T_total, H_v] fp32    h0 : [N, H_v, d_k, d_v] fp32
  cu_seqlens : [N+1] int32 (None for B equal-length sequences)
"""
from __future__ import annotations

import dataclasses
from typing import Optional

import torch

__all__ = ["Workload", "WORKLOADS", "make_prefill", "make_decode", "make_workload", "make_grads",
           "make_channel_decay"]


@dataclasses.dataclass(frozen=True)
class Workload:
    name: str
    kind: str                 # "prefill" or "decode"
    h_qk: int
    h_v: int
    d_k: int
    d_v: int
    dtype: str                # "f32" or "bf16" (q, k, v)
    chunk: int = 64
    g_shift: float = 0.0      # g = -softplus(N(0,1) + g_shift)
    h0_std: float = 0.0       # 0 => zero initial state
    batch: int = 0            # equal-length batch (cu_seqlens None)
    seqlen: int = 0
    num_seqs: int = 0         # varlen / decode sequence count
    len_lo: int = 0           # varlen lengths ~ U{len_lo..len_hi}
    len_hi: int = 0
    steps: int = 0            # decode steps


WORKLOADS = {
    "tiny": Workload("tiny", "prefill", 2, 2, 16, 16, "f32", chunk=16,
                     batch=1, seqlen=64),
    "prefill": Workload("prefill", "prefill", 16, 32, 128, 128, "bf16", chunk=64,
                        g_shift=2.0, batch=4, seqlen=4096),
    "long": Workload("long", "prefill", 16, 32, 128, 128, "bf16", chunk=64,
                     h0_std=0.02, batch=1, seqlen=65536),
    "decode": Workload("decode", "decode", 16, 32, 128, 128, "bf16",
                       h0_std=0.02, num_seqs=256, steps=1000),
    "varlen": Workload("varlen", "prefill", 16, 32, 128, 128, "bf16", chunk=64,
                       h0_std=0.02, num_seqs=64, len_lo=128, len_hi=8192),
}

_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def _unit_rows(x: torch.Tensor) -> torch.Tensor:
    """L2-normalise the last dimension (input recipe: unit-norm q and k)."""
    n = torch.sqrt((x * x).sum(-1, keepdim=True)).clamp_min(1e-12)
    return x / n


def _gen(seed: int) -> torch.Generator:
    gen = torch.Generator(device="cpu")
    gen.manual_seed(int(seed))
    return gen


def make_prefill(*, h_qk: int, h_v: int, d_k: int, d_v: int, dtype: str = "bf16",
                 batch: int = 0, seqlen: int = 0, lengths=None, len_range=None,
                 num_seqs: int = 0, g_shift: float = 0.0, h0_std: float = 0.0,
                 seed: int = 0) -> dict:
    """Draw one prefill problem.

    Exactly one of (batch, seqlen), ``lengths`` (explicit list) or
    (``num_seqs``, ``len_range``) selects the sequence layout. Returns a dict of
    CPU tensors plus ``lengths`` (list of ints) and ``cu_seqlens`` (int32 or
    None when the batch is equal-length and given as (batch, seqlen)).
    """
    gen = _gen(seed)
    if len_range is not None:
        lo, hi = len_range
        lens = torch.randint(lo, hi + 1, (num_seqs,), generator=gen).tolist()
        packed = True
    elif lengths is not None:
        lens = [int(x) for x in lengths]
        packed = True
    else:
        lens = [int(seqlen)] * int(batch)
        packed = False
    total = int(sum(lens))
    q = _unit_rows(torch.randn(total, h_qk, d_k, generator=gen))
    k = _unit_rows(torch.randn(total, h_qk, d_k, generator=gen))
    v = torch.randn(total, h_v, d_v, generator=gen)
    beta = torch.sigmoid(torch.randn(total, h_v, generator=gen))
    g = -torch.nn.functional.softplus(torch.randn(total, h_v, generator=gen) + g_shift)
    n = len(lens)
    if h0_std > 0:
        h0 = torch.randn(n, h_v, d_k, d_v, generator=gen) * h0_std
    else:
        h0 = None
    cu = None
    if packed:
        cu = torch.zeros(n + 1, dtype=torch.int32)
        if n:
            cu[1:] = torch.cumsum(torch.tensor(lens, dtype=torch.int64), 0).to(torch.int32)
    dt = _DT[dtype]
    return dict(q=q.to(dt).contiguous(), k=k.to(dt).contiguous(), v=v.to(dt).contiguous(),
                g=g.contiguous(), beta=beta.contiguous(), h0=h0, cu_seqlens=cu,
                lengths=lens, h_qk=h_qk, h_v=h_v, d_k=d_k, d_v=d_v, dtype=dtype)


def make_decode(*, num_seqs: int, h_qk: int, h_v: int, d_k: int, d_v: int,
                steps: int, dtype: str = "bf16", g_shift: float = 0.0,
                h0_std: float = 0.02, seed: int = 0) -> dict:
    """Draw ``steps`` decode tokens for ``num_seqs`` sequences and their states.

    q, k: [steps, N, H_qk, d_k]; v: [steps, N, H_v, d_v]; g, beta: [steps, N, H_v];
    state: [N, H_v, d_k, d_v] fp32.
    """
    gen = _gen(seed)
    q = _unit_rows(torch.randn(steps, num_seqs, h_qk, d_k, generator=gen))
    k = _unit_rows(torch.randn(steps, num_seqs, h_qk, d_k, generator=gen))
    v = torch.randn(steps, num_seqs, h_v, d_v, generator=gen)
    beta = torch.sigmoid(torch.randn(steps, num_seqs, h_v, generator=gen))
    g = -torch.nn.functional.softplus(torch.randn(steps, num_seqs, h_v, generator=gen) + g_shift)
    state = torch.randn(num_seqs, h_v, d_k, d_v, generator=gen) * h0_std
    dt = _DT[dtype]
    return dict(q=q.to(dt).contiguous(), k=k.to(dt).contiguous(), v=v.to(dt).contiguous(),
                g=g.contiguous(), beta=beta.contiguous(), state=state.contiguous(),
                h_qk=h_qk, h_v=h_v, d_k=d_k, d_v=d_v, dtype=dtype)


def make_workload(name: str, seed: int = 0, steps: Optional[int] = None) -> dict:
    """Draw the named workload (see the table in the module docstring)."""
    w = WORKLOADS[name]
    if w.kind == "decode":
        return make_decode(num_seqs=w.num_seqs, h_qk=w.h_qk, h_v=w.h_v, d_k=w.d_k, d_v=w.d_v,
                           steps=w.steps if steps is None else steps, dtype=w.dtype,
                           g_shift=w.g_shift, h0_std=w.h0_std, seed=seed)
    if w.num_seqs:
        return make_prefill(h_qk=w.h_qk, h_v=w.h_v, d_k=w.d_k, d_v=w.d_v, dtype=w.dtype,
                            num_seqs=w.num_seqs, len_range=(w.len_lo, w.len_hi),
                            g_shift=w.g_shift, h0_std=w.h0_std, seed=seed)
    return make_prefill(h_qk=w.h_qk, h_v=w.h_v, d_k=w.d_k, d_v=w.d_v, dtype=w.dtype,
                        batch=w.batch, seqlen=w.seqlen, g_shift=w.g_shift,
                        h0_std=w.h0_std, seed=seed)


def make_grads(problem: dict, *, dtype: str = "f32", dht_std: float = 0.0, seed: int = 0) -> dict:
    """Incoming gradients for a backward problem drawn by ``make_prefill``:
    dO ~ N(0, 1) shaped like v (stored in ``dtype``) and, when dht_std > 0,
    dS_T ~ N(0, dht_std) shaped like the states (fp32; None otherwise).
    Drawn from its own generator seeded with ``seed + 7919``."""
    gen = _gen(seed + 7919)
    v = problem["v"]
    n = len(problem["lengths"])
    do = torch.randn(v.shape, generator=gen)
    dht = None
    if dht_std > 0:
        dht = torch.randn(n, v.shape[1], problem["q"].shape[2], v.shape[2], generator=gen) * dht_std
    return dict(do=do.to(_DT[dtype]).contiguous(), dht=dht)


def make_channel_decay(shape, *, g_shift: float = 0.0, seed: int = 0) -> torch.Tensor:
    """Per-key-channel log-decays for the per-channel-decay variant (KDA):
    g = -softplus(N(0, 1) + g_shift) of the given shape ([T, H_v, d_k] for a
    prefill, [N, H_v, d_k] for a decode step), fp32, from its own generator
    seeded with ``seed + 104729``."""
    gen = _gen(seed + 104729)
    return (-torch.nn.functional.softplus(torch.randn(tuple(shape), generator=gen) + g_shift)).contiguous()
