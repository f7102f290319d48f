"""fp64 CPU oracle of the gradient of the Gated DeltaNet recurrence (test
infrastructure only: the tests, the smoke check and the benchmark's CPU leg
may import it; the product never does, and the two share no code).

The pages ask for the cost of every design change "in training, prefill and
decode" (the arXiv abstract page of "On the Design of Qwen3.8-Next
Architecture", section "Abstract (arXiv)"); training needs the gradient of the
token mixer. The pages do not write that gradient out: it is fixed by the
forward rule alone (the podcast episode "Qwen3.8-Next design: hybrid
attention, residuals and n-gram embeddings", transcript segment 14, read as

    e_t = v_t - a_t S_{t-1}^T k_t               (what the decayed state misses)
    S_t = a_t S_{t-1} + b_t k_t e_t^T           a_t = exp(g_t), b_t = beta_t
    o_t = scale S_t^T q_t

with S of shape d_k x d_v, the same reading as the forward oracle). Given
the output gradient dO and the gradient dS_T of the final state (zero when
absent), the loss is L = sum_t <dO_t, o_t> + <dS_T, S_T>, and this module
returns dL/dq, dL/dk, dL/dv, dL/dg, dL/dbeta and dL/dS_0.

It applies the chain rule to the three lines above, one token at a time from
the last to the first, carrying D = dL/dS_t:

    D    += scale q_t dO_t^T                 (o_t reads S_t)
    dq_t  = scale S_t dO_t
    de    = b_t D^T k_t                      (e_t enters S_t through b_t k_t e_t^T)
    dv_t  = de
    db_t  = k_t^T D e_t
    dk_t  = b_t D e_t - a_t S_{t-1} de       (k_t in the write and in the read)
    dg_t  = a_t (<D, S_{t-1}> - k_t^T S_{t-1} de)    (a_t in the decay and in the read)
    D     = a_t (D - k_t de^T)               (dL/dS_{t-1})

and dL/dS_0 is the D left after the first token. The states S_0..S_T of the
sequence are first computed forward and kept (no recomputation, no
checkpoints). The q/k gradient of a q/k head is the sum over the value heads
that share it (contiguous groups: value head h reads q/k head h // (H_v/H_qk)).

Parity status: pinned by ``tests/test_oracle_backward.py`` against central
finite differences of the forward oracle (``gdn_oracle.c``), closed forms of
the beta = 0 case, and two homogeneity identities; planted mistakes show each
term is pinned.
"""
from __future__ import annotations

import math

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


def _pair_backward(q, k, v, g, b, do, S0, dST, scale):
    """One (sequence, value head) pair. q, k: [L, d_k]; v, do: [L, d_v];
    g, b: [L]; S0, dST: [d_k, d_v]. Returns (dq, dk, dv, dg, db, dS0)."""
    L, d_k = k.shape
    d_v = v.shape[1]
    a = np.exp(g)
    S = np.empty((L + 1, d_k, d_v))
    S[0] = S0
    E = np.empty((L, d_v))
    for t in range(L):
        E[t] = v[t] - a[t] * (S[t].T @ k[t])
        S[t + 1] = a[t] * S[t] + b[t] * np.outer(k[t], E[t])
    dq = np.zeros((L, d_k))
    dk = np.zeros((L, d_k))
    dv = np.zeros((L, d_v))
    dg = np.zeros(L)
    db = np.zeros(L)
    D = dST.copy()
    for t in range(L - 1, -1, -1):
        D += scale * np.outer(q[t], do[t])
        dq[t] = scale * (S[t + 1] @ do[t])
        de = b[t] * (D.T @ k[t])
        dv[t] = de
        db[t] = k[t] @ (D @ E[t])
        dk[t] = b[t] * (D @ E[t]) - a[t] * (S[t] @ de)
        dg[t] = a[t] * (np.sum(D * S[t]) - k[t] @ (S[t] @ de))
        D = a[t] * (D - np.outer(k[t], de))
    return dq, dk, dv, dg, db, D


def recurrent_backward(q, k, v, g, beta, do, h0=None, dht=None, cu_seqlens=None, scale=None,
                       pairs=None):
    """Gradient of L = <dO, O> + <dS_T, S_T> through the gated delta rule, fp64.

    Layouts as the forward: q, k [T, H_qk, d_k]; v, do [T, H_v, d_v];
    g, beta [T, H_v]; h0, dht [N, H_v, d_k, d_v] (None = zeros);
    cu_seqlens [N + 1] (None = one sequence of T tokens).

    With ``pairs=None`` returns a dict of full arrays: dq, dk [T, H_qk, d_k]
    (summed over the value heads of each group), dv [T, H_v, d_v],
    dg, dbeta [T, H_v], dh0 [N, H_v, d_k, d_v].
    With ``pairs=[(n, h), ...]`` returns a list with one dict per pair holding
    that value head's own contribution: dq, dk [len, d_k], dv [len, d_v],
    dg, dbeta [len], dh0 [d_k, d_v].
    """
    q, k, v, g, beta, do = (_f64(x) for x in (q, k, v, g, beta, do))
    h0, dht = _f64(h0), _f64(dht)
    T, h_qk, d_k = q.shape
    h_v, d_v = v.shape[1], v.shape[2]
    cu = np.array([0, T]) if cu_seqlens is None else _f64(cu_seqlens).astype(np.int64)
    N = len(cu) - 1
    if scale is None:
        scale = 1.0 / math.sqrt(d_k)
    grp = h_v // h_qk
    zero = np.zeros((d_k, d_v))

    def run(n, h):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        hk = h // grp
        S0 = zero if h0 is None else h0[n, h]
        dST = zero if dht is None else dht[n, h]
        r = _pair_backward(q[t0:t1, hk], k[t0:t1, hk], v[t0:t1, h], g[t0:t1, h], beta[t0:t1, h],
                           do[t0:t1, h], S0, dST, float(scale))
        return dict(zip(("dq", "dk", "dv", "dg", "dbeta", "dh0"), r))

    if pairs is not None:
        return [run(int(n), int(h)) for n, h in pairs]
    out = dict(dq=np.zeros((T, h_qk, d_k)), dk=np.zeros((T, h_qk, d_k)), dv=np.zeros((T, h_v, d_v)),
               dg=np.zeros((T, h_v)), dbeta=np.zeros((T, h_v)), dh0=np.zeros((N, h_v, d_k, d_v)))
    for n in range(N):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        for h in range(h_v):
            r = run(n, h)
            out["dq"][t0:t1, h // grp] += r["dq"]
            out["dk"][t0:t1, h // grp] += r["dk"]
            out["dv"][t0:t1, h] = r["dv"]
            out["dg"][t0:t1, h] = r["dg"]
            out["dbeta"][t0:t1, h] = r["dbeta"]
            out["dh0"][n, h] = r["dh0"]
    return out
