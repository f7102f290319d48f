"""fp64 CPU oracle of the GDN input prologue (test infrastructure only).

The pages say only that the GDN layer adds "short causal convolutions" to the
gated delta rule ("Qwen3.8-Next design: hybrid attention, residuals and
n-gram embeddings", podcast transcript segment 14); q and k enter the rule
L2-normalised (the recurrence's inputs). The plainest reading, used here and
by the CUDA path:

  u[t, c] = sum_{i=0}^{K-1} w[c, i] * x[t - (K - 1) + i, c]     (per channel c)
  s[t, c] = silu(u[t, c]) = u / (1 + exp(-u))
  y[t, :] = s[t, :] grouped in heads of `norm_group` channels, each head
            divided by sqrt(sum of its squares + eps)   (q and k; none for v)

x[t'] is the sequence's own past: before the first token of a sequence it is
the caller's conv state (the K - 1 inputs that preceded it) or zero. The
final state holds the last K - 1 inputs of each sequence (fewer tokens than
that keep the older state entries). A decode step applies the same formula to
one token with the state as its past and shifts the state by one.

Every step is a direct fp64 evaluation on the exact input values; the
sequences, taps and channels are looped over plainly.

Parity status: pinned by ``tests/test_oracle_prologue.py`` (a hand-worked
example, closed forms, invariants, two independent forms of the same filter,
and planted mistakes).
"""
from __future__ import annotations

import numpy as np

from .epilogue import _f64


def silu(u):
    """u * sigmoid(u), fp64, finite for large |u|."""
    u = _f64(u)
    out = np.empty_like(u)
    pos = u >= 0
    out[pos] = u[pos] / (1.0 + np.exp(-u[pos]))
    eu = np.exp(u[~pos])
    out[~pos] = u[~pos] * eu / (1.0 + eu)
    return out


def l2_normalize_groups(s, group: int, eps: float = 1e-6):
    """Divide each run of `group` consecutive channels by sqrt(sum sq + eps)."""
    s = _f64(s)
    sh = s.shape
    g = s.reshape(*sh[:-1], sh[-1] // group, group)
    g = g / np.sqrt(np.sum(g * g, axis=-1, keepdims=True) + eps)
    return g.reshape(sh)


def _finish(u, activation, norm_group, eps):
    s = silu(u) if activation == "silu" else u
    return l2_normalize_groups(s, norm_group, eps) if norm_group else s


def short_conv(x, w, cu_seqlens=None, state0=None, activation="silu", norm_group=0, eps=1e-6):
    """Causal depthwise conv over the tokens of each sequence, then SiLU and
    (norm_group > 0) L2 normalisation per head.

    x: [T, C]; w: [C, K]; cu_seqlens: [N + 1] or None (one sequence);
    state0: [N, C, K - 1] or None (zeros). Returns (y [T, C], state [N, C, K - 1]).
    """
    x = _f64(x)
    w = _f64(w)
    T, C = x.shape
    K = w.shape[1]
    cu = [0, T] if cu_seqlens is None else [int(v) for v in np.asarray(cu_seqlens).tolist()]
    N = len(cu) - 1
    st0 = np.zeros((N, C, K - 1)) if state0 is None else _f64(state0)
    u = np.zeros((T, C))
    state = np.zeros((N, C, K - 1))
    for n in range(N):
        t0, t1 = cu[n], cu[n + 1]
        # the sequence's inputs preceded by its K - 1 past inputs
        past = st0[n].T                               # [K - 1, C], oldest first
        seq = np.concatenate([past, x[t0:t1]], axis=0)
        for t in range(t1 - t0):
            for i in range(K):
                u[t0 + t] += w[:, i] * seq[t + i]
        state[n] = seq[len(seq) - (K - 1):].T if K > 1 else state[n]
    return _finish(u, activation, norm_group, eps), state


def short_conv_step(x, w, state, activation="silu", norm_group=0, eps=1e-6):
    """One token per sequence. x: [N, C]; w: [C, K]; state: [N, C, K - 1]
    (oldest first). Returns (y [N, C], new state [N, C, K - 1])."""
    x = _f64(x)
    w = _f64(w)
    st = _f64(state)
    K = w.shape[1]
    u = w[:, K - 1] * x
    for i in range(K - 1):
        u = u + w[:, i] * st[:, :, i]
    new = np.concatenate([st[:, :, 1:], x[:, :, None]], axis=2) if K > 1 else st
    return _finish(u, activation, norm_group, eps), new
