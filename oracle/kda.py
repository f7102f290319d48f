"""fp64 CPU oracle of the per-channel-decay variant of the gated delta rule
(KDA) -- test infrastructure only: the tests, the smoke check and the
benchmark's CPU leg may import it; the product never does.

The pages name KDA only as the alternative to Gated DeltaNet in the linear
token-mixer slot of about three of every four layers (the "Qwen3.8 attention
gate" page, blueprint component "Gated DeltaNet / KDA") and never define it.
The reading used here and by the CUDA path is the plainest per-channel
generalisation of the gated delta rule as the podcast episode "Qwen3.8-Next
design: hybrid attention, residuals and n-gram embeddings" (transcript
segment 14) describes it -- decay the state first, then read what is stored
under the key and write only the error -- with the scalar decay replaced by
one decay per key channel:

    S~  = diag(a_t) S_{t-1}            a_t = exp(g_t), g_t in R^{d_k}
    e_t = v_t - S~^T k_t
    S_t = S~ + b_t k_t e_t^T           b_t = beta_t
    o_t = scale S_t^T q_t

with S of shape d_k x d_v (rows = key channels), the same orientation, GQA
grouping and varlen packing as the gated delta rule; g has shape
[T, H_v, d_k]. With every channel's g equal, this is the gated delta rule.
Each token is evaluated directly from these four lines in fp64 on the exact
input values (bf16 upcast element by element).

``kda_chunked`` is a second, independent form: the chunkwise algebra with
per-channel decay factors inside the inner products (the blueprint of a
chunked KDA kernel), kept only to pin that algebra against ``kda_recurrent``.

Parity status: pinned by ``tests/test_oracle_kda.py`` (a hand-worked example,
equality with the gated-delta-rule C oracle for uniform channels, the beta = 0
closed form, key-axis retrieval, planted mistakes; ``kda_chunked`` by equality
with ``kda_recurrent`` for several chunk sizes).
"""
from __future__ import annotations

import math

import numpy as np


def _f64(x):
    if x is None:
        return None
    try:
        import torch
        if isinstance(x, torch.Tensor):
            return x.detach().to("cpu").to(torch.float32).numpy().astype(np.float64)
    except ImportError:  # pragma: no cover
        pass
    return np.asarray(x, dtype=np.float64)


def _pair(q, k, v, g, b, S, scale):
    """One (sequence, value head): q, k [L, d_k]; v [L, d_v]; g [L, d_k];
    b [L]; S [d_k, d_v] (updated in place). Returns o [L, d_v]."""
    L, d_v = v.shape
    o = np.zeros((L, d_v))
    for t in range(L):
        Sd = np.exp(g[t])[:, None] * S          # each key channel decays by its own factor
        e = v[t] - Sd.T @ k[t]                  # what is missing under k_t after the decay
        S[...] = Sd + b[t] * np.outer(k[t], e)  # write only the error
        o[t] = scale * (S.T @ q[t])
    return o


def kda_recurrent(q, k, v, g, beta, h0=None, cu_seqlens=None, scale=None):
    """Token-by-token KDA in fp64. q, k [T, H_qk, d_k]; v [T, H_v, d_v];
    g [T, H_v, d_k] (per-channel log-decay); beta [T, H_v]; h0 [N, H_v, d_k, d_v]
    or None; cu_seqlens [N + 1] or None (one sequence). Returns (o [T, H_v, d_v],
    S [N, H_v, d_k, d_v])."""
    q, k, v, g, beta, h0 = (_f64(x) for x in (q, k, v, g, beta, h0))
    T, h_qk, d_k = q.shape
    h_v, d_v = v.shape[1], v.shape[2]
    cu = np.array([0, T]) if cu_seqlens is None else _f64(cu_seqlens).astype(np.int64)
    N = len(cu) - 1
    if scale is None:
        scale = 1.0 / math.sqrt(d_k)
    grp = h_v // h_qk
    o = np.zeros((T, h_v, d_v))
    S_out = np.zeros((N, h_v, d_k, d_v))
    for n in range(N):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        for h in range(h_v):
            hk = h // grp
            S = np.zeros((d_k, d_v)) if h0 is None else h0[n, h].copy()
            o[t0:t1, h] = _pair(q[t0:t1, hk], k[t0:t1, hk], v[t0:t1, h], g[t0:t1, h], beta[t0:t1, h], S,
                                float(scale))
            S_out[n, h] = S
    return o, S_out


def _pair_chunked(q, k, v, g, b, S, scale, C):
    """Chunkwise KDA for one (sequence, value head); S updated in place.

    Unrolling the rule inside a chunk (rows r, s = 0..L-1, G_r = running sum
    of g_r per key channel, E_rs = exp(G_r - G_s) per channel for s <= r):
      S_r = diag(e^{G_r}) S0 + sum_{s<=r} diag(E_rs) k_s u_s^T
    so the errors u_r = b_r e_r solve (I + A) U = diag(b) (V - (K o e^G) S0)
    with A_rs = b_r sum_i k_ri k_si E_rsi (s < r); with T = (I + A)^-1:
      W = T diag(b) (K o e^G),  U = T diag(b) V - W S0
      O = scale ((Q o e^G) S0 + P U),  P_rs = sum_i q_ri k_si E_rsi (s <= r)
      S1 = diag(e^{G_last}) S0 + (K o e^{G_last - G})^T U"""
    L_tot, d_v = v.shape
    o = np.zeros((L_tot, d_v))
    for c0 in range(0, L_tot, C):
        c1 = min(c0 + C, L_tot)
        K, Q, V, gg, bb = k[c0:c1], q[c0:c1], v[c0:c1], g[c0:c1], b[c0:c1]
        n = c1 - c0
        G = np.cumsum(gg, axis=0)                                  # [n, d_k]
        diff = G[:, None, :] - G[None, :, :]                       # [r, s, i]
        lower = np.tril(np.ones((n, n), dtype=bool))
        E = np.where(lower[:, :, None], np.exp(np.where(lower[:, :, None], diff, 0.0)), 0.0)
        KK = np.einsum("ri,si,rsi->rs", K, K, E)
        QK = np.einsum("ri,si,rsi->rs", Q, K, E)
        A = np.tril(bb[:, None] * KK, -1)
        T = np.linalg.inv(np.eye(n) + A)
        W = T @ (bb[:, None] * (K * np.exp(G)))
        U = T @ (bb[:, None] * V) - W @ S
        o[c0:c1] = scale * ((Q * np.exp(G)) @ S + np.tril(QK) @ U)
        S[...] = np.exp(G[-1])[:, None] * S + (K * np.exp(G[-1][None, :] - G)).T @ U
    return o


def kda_chunked(q, k, v, g, beta, h0=None, cu_seqlens=None, scale=None, chunk=64):
    """The chunkwise form of ``kda_recurrent`` (same arguments and returns,
    plus the chunk size); equal to it up to rounding."""
    q, k, v, g, beta, h0 = (_f64(x) for x in (q, k, v, g, beta, h0))
    T, h_qk, d_k = q.shape
    h_v, d_v = v.shape[1], v.shape[2]
    cu = np.array([0, T]) if cu_seqlens is None else _f64(cu_seqlens).astype(np.int64)
    N = len(cu) - 1
    if scale is None:
        scale = 1.0 / math.sqrt(d_k)
    grp = h_v // h_qk
    o = np.zeros((T, h_v, d_v))
    S_out = np.zeros((N, h_v, d_k, d_v))
    for n in range(N):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        for h in range(h_v):
            hk = h // grp
            S = np.zeros((d_k, d_v)) if h0 is None else h0[n, h].copy()
            if t1 > t0:
                o[t0:t1, h] = _pair_chunked(q[t0:t1, hk], k[t0:t1, hk], v[t0:t1, h], g[t0:t1, h],
                                            beta[t0:t1, h], S, float(scale), int(chunk))
            S_out[n, h] = S
    return o, S_out
