"""fp64 CPU oracle of the gradient of the Gated DeltaNet recurrence (test
infrastructure only: the tests, the smoke check and the benchmark's CPU leg
may import it; the product never does, and the two share no code).

The pages weigh each design change by its training cost next to its prefill
and decode cost (the arXiv abstract page of "On the Design of Qwen3.8-Next
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

``chunked_backward`` is a second, independent form: the chunkwise (WY)
algebra of the forward differentiated chunk by chunk, with the decay gradient
taken from its closed form. It exists only to pin that algebra (the blueprint
of a chunked gradient kernel) against ``recurrent_backward``.

Parity status: pinned by ``tests/test_oracle_backward.py`` against central
finite differences of the forward oracle (``gdn_oracle.c``), closed forms of
the beta = 0 case, two homogeneity identities and the decay-gradient
identity; planted mistakes show each term is pinned. ``chunked_backward`` is
pinned by equality with ``recurrent_backward`` for several chunk sizes.
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


def _pair_chunked_backward(q, k, v, g, b, do, S0, dST, scale, C):
    """Chunkwise gradient of one (sequence, value head) pair.

    Per chunk of L <= C rows (r, s = 0..L-1), with S0 the chunk's first state,
    G = running sum of g in the chunk, gam = exp(G), Gam_rs = exp(G_r - G_s):
      forward:  A = strict_lower(diag(b) (Gam o K K^T)), T = (I + A)^-1,
                Kb = diag(b gam) K, Vb = diag(b) V, W = T Kb, U = T Vb,
                Delta = U - W S0, P = lower(Gam o Q K^T) (diagonal included),
                O = scale (diag(gam) Q S0 + P Delta),
                S1 = gam_L S0 + Kd^T Delta with Kd = diag(exp(G_L - G)) K
      reverse, given dO and D = dL/dS1:
                dDelta = scale P^T dO + Kd D
                dS0    = gam_L D + scale (diag(gam) Q)^T dO - W^T dDelta
                dW = -dDelta S0^T, dU = dDelta, dP = scale dO Delta^T
                dQ = (dP o Gam o lower) K + scale diag(gam) dO S0^T
                dK = (dP o Gam o lower)^T Q + diag(exp(G_L - G)) Delta D^T
                dT = dW Kb^T + dU Vb^T, dKb = T^T dW, dVb = T^T dU
                dK += diag(b gam) dKb, dV = diag(b) dVb,
                dbeta = gam o rowdot(K, dKb) + rowdot(V, dVb)
                dA = strict_lower(-T^T dT T^T), E = dA o diag(b) Gam
                dK += E K + E^T K, dbeta += rowsum(dA o Gam o K K^T)
    The decays enter only through gam and Gam; their gradient is not traced
    here: dg comes from the closed form dg_t = <dS_T, S_T> + sum_{r>=t}
    (q_r . dq_r - v_r . dv_r). Returns (dq, dk, dv, dg, db, dS0)."""
    L_tot, d_k = k.shape
    d_v = v.shape[1]
    starts = list(range(0, L_tot, C))
    # forward over chunks: the state at every chunk start
    S = S0.copy()
    states = []
    for c0 in starts:
        states.append(S.copy())
        c1 = min(c0 + C, L_tot)
        K, V, gg, bb = k[c0:c1], v[c0:c1], g[c0:c1], b[c0:c1]
        G = np.cumsum(gg)
        Gam = np.tril(np.exp(G[:, None] - G[None, :]))
        A = np.tril(bb[:, None] * Gam * (K @ K.T), -1)
        T = np.linalg.inv(np.eye(len(gg)) + A)
        W = T @ ((bb * np.exp(G))[:, None] * K)
        U = T @ (bb[:, None] * V)
        Delta = U - W @ S
        S = np.exp(G[-1]) * S + (np.exp(G[-1] - G)[:, None] * K).T @ Delta
    ST = S
    dq = np.zeros((L_tot, d_k))
    dk = np.zeros((L_tot, d_k))
    dv = np.zeros((L_tot, d_v))
    db = np.zeros(L_tot)
    D = dST.copy()
    for c0, Sc in zip(reversed(starts), reversed(states)):
        c1 = min(c0 + C, L_tot)
        K, Q, V, gg, bb, dO = k[c0:c1], q[c0:c1], v[c0:c1], g[c0:c1], b[c0:c1], do[c0:c1]
        n = c1 - c0
        G = np.cumsum(gg)
        gam = np.exp(G)
        Gam = np.tril(np.exp(G[:, None] - G[None, :]))
        KK = K @ K.T
        A = np.tril(bb[:, None] * Gam * KK, -1)
        T = np.linalg.inv(np.eye(n) + A)
        Kb = (bb * gam)[:, None] * K
        Vb = bb[:, None] * V
        W = T @ Kb
        U = T @ Vb
        Delta = U - W @ Sc
        P = np.tril(Gam * (Q @ K.T))
        tail = np.exp(G[-1] - G)
        Kd = tail[:, None] * K
        dDelta = scale * P.T @ dO + Kd @ D
        dS0 = gam[-1] * D + scale * (gam[:, None] * Q).T @ dO - W.T @ dDelta
        dW = -dDelta @ Sc.T
        dU = dDelta
        dPG = np.tril(scale * (dO @ Delta.T) * Gam)
        dQc = dPG @ K + scale * gam[:, None] * (dO @ Sc.T)
        dKc = dPG.T @ Q + tail[:, None] * (Delta @ D.T)
        dT = dW @ Kb.T + dU @ Vb.T
        dKb = T.T @ dW
        dVb = T.T @ dU
        dKc += (bb * gam)[:, None] * dKb
        dVc = bb[:, None] * dVb
        dbc = gam * np.sum(K * dKb, axis=1) + np.sum(V * dVb, axis=1)
        dA = np.tril(-T.T @ dT @ T.T, -1)
        E = dA * bb[:, None] * Gam
        dKc += E @ K + E.T @ K
        dbc += np.sum(dA * Gam * KK, axis=1)
        dq[c0:c1], dk[c0:c1], dv[c0:c1], db[c0:c1] = dQc, dKc, dVc, dbc
        D = dS0
    per = np.sum(q * dq, axis=1) - np.sum(v * dv, axis=1)
    dg = float(np.sum(dST * ST)) + np.cumsum(per[::-1])[::-1]
    return dq, dk, dv, dg, db, D


def chunked_backward(q, k, v, g, beta, do, h0=None, dht=None, cu_seqlens=None, scale=None, pairs=None,
                     chunk=64):
    """The chunkwise form of ``recurrent_backward`` (same arguments and
    returns, plus the chunk size); equal to it up to rounding."""
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
        if t1 == t0:
            return dict(dq=np.zeros((0, d_k)), dk=np.zeros((0, d_k)), dv=np.zeros((0, d_v)), dg=np.zeros(0),
                        dbeta=np.zeros(0), dh0=dST.copy())
        r = _pair_chunked_backward(q[t0:t1, hk], k[t0:t1, hk], v[t0:t1, h], g[t0:t1, h], beta[t0:t1, h],
                                   do[t0:t1, h], S0, dST, float(scale), int(chunk))
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
