"""fp64 CPU oracle of the GDN output epilogue (test infrastructure only).

The pages name the epilogue without writing it out: the GDN layer adds "a
sigmoid output gate, zero-centered RMSNorm" to the gated delta rule
("Qwen3.8-Next design: hybrid attention, residuals and n-gram embeddings",
podcast transcript segment 14), and the component list of the attention-gate
page gives the gate as sigma(x W_g) (.) o ("Qwen3.8 attention gate", component
"Output gate + sink"). The plainest reading, used here and by the CUDA path:

    y = o / sqrt(mean_j(o_j^2) + eps) * (1 + w) * sigmoid(z)

per row (one token of one value head; the mean runs over the d_v features of
that head), with

  - z    the gate pre-activation x W_g, supplied by the caller (same layout as o),
  - w    the per-feature norm weight in zero-centred form (the scale is 1 + w,
         so w = 0 is the plain RMS normalisation), shared by all heads,
  - eps  a small constant inside the square root (1e-6 by default).

The norm is applied first and the gate multiplies its result. Every step is a
direct fp64 evaluation of this formula on the exact input values (bf16 inputs
are upcast element by element); nothing is fused or reordered.

Parity status: pinned by ``tests/test_oracle_epilogue.py`` (a hand-worked
example, closed forms of special cases, invariants, and planted mistakes).
"""
from __future__ import annotations

import numpy as np


def _f64(x):
    """torch / numpy -> float64 numpy (bf16 upcast exactly through fp32)."""
    if x is None:
        return None
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu").to(torch.float32).numpy().astype(np.float64)
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def rms_normalize(x, eps: float = 1e-6):
    """x / sqrt(mean(x^2) + eps) over the last axis (fp64)."""
    x = _f64(x)
    ms = np.mean(x * x, axis=-1, keepdims=True)
    return x / np.sqrt(ms + eps)


def sigmoid(z):
    """1 / (1 + exp(-z)), fp64, written to stay finite for large |z|."""
    z = _f64(z)
    out = np.empty_like(z)
    pos = z >= 0
    out[pos] = 1.0 / (1.0 + np.exp(-z[pos]))
    ez = np.exp(z[~pos])
    out[~pos] = ez / (1.0 + ez)
    return out


def gated_rmsnorm(o, z, w=None, eps: float = 1e-6):
    """y = rms_normalize(o) * (1 + w) * sigmoid(z) over the last axis (fp64).

    o, z: [..., d] (any leading shape, e.g. [T, H_v, d_v]); w: [d] or None (= 0).
    """
    y = rms_normalize(o, eps)
    if w is not None:
        y = y * (1.0 + _f64(w))
    return y * sigmoid(z)
