"""fp64 CPU oracle for the Gated DeltaNet forward recurrence.

TEST INFRASTRUCTURE ONLY: the tests, the smoke check and the benchmark's
CPU-baseline / reference leg may import this package; the product (the CUDA
library and its Python binding) never does, and the two share no code.

The arithmetic lives in ``gdn_oracle.c`` (plain C, fp64, sequential per
(sequence, value-head) pair, OpenMP across pairs). This module only marshals
numpy / torch CPU arrays into it and back.

  recurrent(...)  token-by-token gated delta rule (the oracle proper)
  chunked(...)    the chunkwise algebra, used only to pin that algebra
  gated_rmsnorm(...)  the output epilogue (zero-centred RMSNorm times a
                  sigmoid gate), numpy fp64, in ``epilogue.py``
  short_conv(...), short_conv_step(...)  the input prologue (causal
                  depthwise conv, SiLU, per-head L2 norm), in ``prologue.py``
  recurrent_backward(...)  the gradient of the recurrence (reverse-order chain
                  rule, numpy fp64), in ``backward.py``
  kda_recurrent(...)  the per-key-channel-decay variant (KDA), numpy fp64, in
                  ``kda.py``

Both return ``(o, S)``: with ``pairs=None`` o is [T_total, H_v, d_v] and S is
[N, H_v, d_k, d_v] (float64 numpy); with ``pairs=[(n, h), ...]`` they are
lists with one [len_n, d_v] / [d_k, d_v] array per requested pair.

Parity status: every function here is pinned by ``tests/test_oracle_pins.py``
(closed forms, invariants and a hand-worked example; see that file).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

from .backward import chunked_backward, recurrent_backward  # noqa: F401
from .epilogue import gated_rmsnorm, rms_normalize, sigmoid  # noqa: F401
from .kda import kda_chunked, kda_recurrent  # noqa: F401
from .prologue import l2_normalize_groups, short_conv, short_conv_step, silu  # noqa: F401

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "gdn_oracle.c")
_LIB_PATH = os.path.join(_HERE, "_gdn_oracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle with gcc (fp64, -O2, OpenMP). Returns the .so path."""
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _declare(lib):
    P, I32, D = ctypes.c_void_p, ctypes.c_int32, ctypes.c_double
    common = [P, P, P, ctypes.c_int, P, P, P, P, I32, I32, I32, I32, I32, D]
    tail = [P, I32, P, P, P, I32]
    lib.gdn_oracle_recurrent.argtypes = common + tail
    lib.gdn_oracle_recurrent.restype = ctypes.c_int
    lib.gdn_oracle_chunked.argtypes = common + [I32] + tail
    lib.gdn_oracle_chunked.restype = ctypes.c_int
    lib.gdn_oracle_max_threads.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    with _lock:
        if _lib is None:
            _lib = _declare(ctypes.CDLL(build()))
    return _lib


def max_threads() -> int:
    return int(_load().gdn_oracle_max_threads())


def _as_np(x, kind):
    """torch/numpy -> contiguous numpy. kind 'qkv' keeps bf16 as raw uint16."""
    if x is None:
        return None, None
    try:
        import torch
        if isinstance(x, torch.Tensor):
            x = x.detach().cpu().contiguous()
            if kind == "qkv":
                if x.dtype == torch.bfloat16:
                    return x.view(torch.int16).numpy().view(np.uint16), 1
                return x.to(torch.float32).numpy(), 0
            if kind == "i32":
                return x.to(torch.int32).numpy(), None
            return x.to(torch.float32).numpy(), None
    except ImportError:  # pragma: no cover
        pass
    x = np.ascontiguousarray(x)
    if kind == "qkv":
        if x.dtype == np.uint16:
            return x, 1
        return np.ascontiguousarray(x, dtype=np.float32), 0
    if kind == "i32":
        return np.ascontiguousarray(x, dtype=np.int32), None
    return np.ascontiguousarray(x, dtype=np.float32), None


def _run(fn, q, k, v, g, beta, h0, cu_seqlens, scale, pairs, threads, chunk=None):
    qn, dt_q = _as_np(q, "qkv")
    kn, dt_k = _as_np(k, "qkv")
    vn, dt_v = _as_np(v, "qkv")
    if not (dt_q == dt_k == dt_v):
        raise ValueError("q, k, v must share one dtype")
    gn, _ = _as_np(g, "f32")
    bn, _ = _as_np(beta, "f32")
    hn, _ = _as_np(h0, "f32")
    total, h_qk, d_k = qn.shape
    h_v, d_v = vn.shape[1], vn.shape[2]
    if cu_seqlens is None:
        cun = np.array([0, total], dtype=np.int32)
    else:
        cun, _ = _as_np(cu_seqlens, "i32")
    N = cun.shape[0] - 1
    if scale is None:
        scale = 1.0 / math.sqrt(d_k)
    full = pairs is None
    if full:
        pairs = [(n, h) for n in range(N) for h in range(h_v)]
    pairs = [(int(n), int(h)) for n, h in pairs]
    pr = np.array(pairs, dtype=np.int32).reshape(-1, 2)
    lens = [int(cun[n + 1] - cun[n]) for n, _ in pairs]
    offs = np.zeros(len(pairs), dtype=np.int64)
    if pairs:
        offs[1:] = np.cumsum(lens)[:-1]
    o = np.zeros((max(1, int(sum(lens))), d_v), dtype=np.float64)
    S = np.zeros((max(1, len(pairs)), d_k, d_v), dtype=np.float64)
    ptr = lambda a: None if a is None else a.ctypes.data_as(ctypes.c_void_p)
    args = [ptr(qn), ptr(kn), ptr(vn), dt_q, ptr(gn), ptr(bn), ptr(hn), ptr(cun), N,
            h_qk, h_v, d_k, d_v, float(scale)]
    if chunk is not None:
        args.append(int(chunk))
    args += [ptr(pr), len(pairs), ptr(offs), ptr(o), ptr(S), int(threads)]
    rc = fn(*args)
    if rc != 0:
        raise ValueError(f"oracle rejected its arguments (code {rc})")
    if full:
        o_full = np.zeros((total, h_v, d_v), dtype=np.float64)
        S_full = np.zeros((N, h_v, d_k, d_v), dtype=np.float64)
        for p, (n, h) in enumerate(pairs):
            a, b = int(cun[n]), int(cun[n + 1])
            o_full[a:b, h, :] = o[offs[p]:offs[p] + (b - a)]
            S_full[n, h] = S[p]
        return o_full, S_full
    return ([o[offs[p]:offs[p] + lens[p]].copy() for p in range(len(pairs))],
            [S[p].copy() for p in range(len(pairs))])


class Oracle:
    """The two oracle forms bound to one compiled copy of ``gdn_oracle.c``.

    The module-level functions use the copy built from the committed source;
    the pin tests also bind deliberately broken copies (built from an edited
    source in a temporary folder) to show that the pins catch those mistakes.
    """

    def __init__(self, lib):
        self._lib = _declare(lib)

    def recurrent(self, q, k, v, g, beta, h0=None, cu_seqlens=None, scale=None, pairs=None,
                  threads=0):
        """Token-by-token gated delta rule in fp64 (see gdn_oracle.c)."""
        return _run(self._lib.gdn_oracle_recurrent, q, k, v, g, beta, h0, cu_seqlens, scale,
                    pairs, threads)

    def chunked(self, q, k, v, g, beta, h0=None, cu_seqlens=None, scale=None, pairs=None,
                threads=0, chunk=64):
        """Chunkwise algebra in fp64 (see gdn_oracle.c); equals ``recurrent`` up to rounding."""
        return _run(self._lib.gdn_oracle_chunked, q, k, v, g, beta, h0, cu_seqlens, scale, pairs,
                    threads, chunk=chunk)


def load_variant(so_path: str) -> "Oracle":
    """Bind an oracle compiled elsewhere (used by the pin tests' planted mistakes)."""
    return Oracle(ctypes.CDLL(so_path))


def recurrent(q, k, v, g, beta, h0=None, cu_seqlens=None, scale=None, pairs=None, threads=0):
    """Token-by-token gated delta rule in fp64 (see gdn_oracle.c)."""
    return _run(_load().gdn_oracle_recurrent, q, k, v, g, beta, h0, cu_seqlens, scale, pairs, threads)


def chunked(q, k, v, g, beta, h0=None, cu_seqlens=None, scale=None, pairs=None, threads=0, chunk=64):
    """Chunkwise algebra in fp64 (see gdn_oracle.c); equals ``recurrent`` up to rounding."""
    return _run(_load().gdn_oracle_chunked, q, k, v, g, beta, h0, cu_seqlens, scale, pairs,
                threads, chunk=chunk)


def decode_steps(q, k, v, g, beta, state, scale=None, threads=0):
    """Run ``steps`` decode tokens through the recurrence, one token per step.

    q, k: [steps, N, H_qk, d_k]; v: [steps, N, H_v, d_v]; g, beta: [steps, N, H_v];
    state: [N, H_v, d_k, d_v]. Returns (o [steps, N, H_v, d_v], final state).
    Implemented as a prefill of N sequences of length ``steps`` (the decode step
    is the same recurrence applied to one token).
    """
    import torch
    steps, N = q.shape[0], q.shape[1]
    perm = lambda x: x.transpose(0, 1).reshape(N * steps, *x.shape[2:]).contiguous()
    cu = torch.arange(0, N + 1, dtype=torch.int32) * steps
    o, S = recurrent(perm(q), perm(k), perm(v), perm(g), perm(beta), h0=state, cu_seqlens=cu,
                     scale=scale, threads=threads)
    o = o.reshape(N, steps, *o.shape[1:]).transpose(1, 0, 2, 3)
    return np.ascontiguousarray(o), S
