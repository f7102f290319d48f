"""The algebraic rearrangements the CUDA kernels rely on, checked in fp64
against the oracles (no GPU, no kernel code: each rearrangement is written
out here from its statement in the kernel's header comment).

  - gradient kernel (gdn_backward.cuh): phase 1 keeps the state at every
    32-token block start plus e_t, dq_t and q_t . dq_t; phase 2 rebuilds
    S_{t-1} de as S_b de plus an in-block correction
    sum_{s<t} Gam_{t-1,s} b_s (e_s . de_t) k_s applied at the block's end, and
    dg from its closed form;
  - decode kernel (gdn_decode.cuh): one pass over S gives S^T k and S^T q, and
    o = scale (alpha S^T q + (k . q) u);
  - KDA kernels (gdn_kda.cuh): the reads use a o k and a o q against the
    undecayed state and o = scale (S^T (a o q) + (k . q) u);
  - sequence segments of the tensor-core prefill (gdn_chunk_tc.cuh,
    segment_prefix_start): a segment that starts from a zero state at the
    nearest token ts where prod_{t=ts}^{a-1} alpha_t max(1, |1 - beta_t
    |k_t|^2|) <= 2^-40 reaches its first token a with a state within 2^-40
    times the spectral norm of the true state before ts.
"""
import math

import numpy as np
import pytest

import oracle

BLK = 32


def _blocked_backward(q, k, v, g, b, do, S0, dST, scale):
    """One (sequence, head) pair the way the gradient kernel computes it."""
    L, d_k = k.shape
    a = np.exp(g)
    nb = (L + BLK - 1) // BLK
    # phase 1
    S = S0.copy()
    ck, E = [], np.zeros_like(v)
    dq = np.zeros_like(q)
    qdq = np.zeros(L)
    for bi in range(nb):
        ck.append(S.copy())
        for t in range(bi * BLK, min(L, bi * BLK + BLK)):
            E[t] = v[t] - a[t] * (S.T @ k[t])
            S = a[t] * S + b[t] * np.outer(k[t], E[t])
            dq[t] = scale * (S @ do[t])
            qdq[t] = q[t] @ dq[t]
    carry = float(np.sum(dST * S))
    # phase 2
    D = dST.copy()
    dk, dv, dg, db = np.zeros_like(k), np.zeros_like(v), np.zeros(L), np.zeros(L)
    for bi in range(nb - 1, -1, -1):
        t0 = bi * BLK
        n = min(L, t0 + BLK) - t0
        Lc = np.cumsum(g[t0:t0 + n])
        Sb = ck[bi]
        DE, DK, vdv = np.zeros((n, v.shape[1])), np.zeros((n, d_k)), np.zeros(n)
        for j in range(n - 1, -1, -1):
            t = t0 + j
            D = D + scale * np.outer(q[t], do[t])
            c2 = D.T @ k[t]
            DE[j] = b[t] * c2
            dv[t] = DE[j]
            vdv[j] = v[t] @ DE[j]
            db[t] = c2 @ E[t]
            gprev = math.exp(Lc[j - 1]) if j > 0 else 1.0
            DK[j] = b[t] * (D @ E[t]) - a[t] * gprev * (Sb @ DE[j])
            D = a[t] * (D - np.outer(k[t], DE[j]))
        for j in range(n):
            corr = np.zeros(d_k)
            for s in range(j):
                corr += math.exp(Lc[j - 1] - Lc[s]) * b[t0 + s] * (E[t0 + s] @ DE[j]) * k[t0 + s]
            dk[t0 + j] = DK[j] - a[t0 + j] * corr
        x = qdq[t0:t0 + n] - vdv
        for j in range(n - 1, -1, -1):
            carry += x[j]
            dg[t0 + j] = carry
    return dq, dk, dv, dg, db, D


@pytest.mark.parametrize("L", [0, 1, 31, 32, 33, 100])
def test_gradient_kernel_blocked_algebra(L):
    rng = np.random.default_rng(L)
    d_k, d_v = 8, 6
    q = rng.standard_normal((L, d_k))
    k = rng.standard_normal((L, d_k))
    k /= np.linalg.norm(k, axis=1, keepdims=True) + 1e-300
    v = rng.standard_normal((L, d_v))
    g = -np.log1p(np.exp(rng.standard_normal(L)))
    b = 1 / (1 + np.exp(-rng.standard_normal(L)))
    do = rng.standard_normal((L, d_v))
    S0 = rng.standard_normal((d_k, d_v)) * 0.1
    dST = rng.standard_normal((d_k, d_v)) * 0.1
    scale = 1 / math.sqrt(d_k)
    got = _blocked_backward(q, k, v, g, b, do, S0, dST, scale)
    ref = oracle.recurrent_backward(q[:, None], k[:, None], v[:, None], g[:, None], b[:, None], do[:, None],
                                    h0=S0[None, None], dht=dST[None, None], scale=scale)
    refs = [ref["dq"][:, 0], ref["dk"][:, 0], ref["dv"][:, 0], ref["dg"][:, 0], ref["dbeta"][:, 0],
            ref["dh0"][0, 0]]
    for name, x, y in zip(("dq", "dk", "dv", "dg", "dbeta", "dS0"), got, refs):
        np.testing.assert_allclose(x, y, rtol=1e-10, atol=1e-12, err_msg=name)


def _token(rng, d_k=7, d_v=5, per_channel=False):
    S = rng.standard_normal((d_k, d_v))
    q, k = rng.standard_normal(d_k), rng.standard_normal(d_k)
    v = rng.standard_normal(d_v)
    g = -rng.uniform(0.0, 2.0, d_k if per_channel else None)
    b = float(rng.uniform(0.1, 0.9))
    return S, q, k, v, g, b


def test_decode_single_pass_rearrangement():
    rng = np.random.default_rng(3)
    # the C oracle reads fp32 inputs: use values that are exact in fp32
    S, q, k, v, g, b = (np.float32(x).astype(np.float64) if np.isscalar(x) else x.astype(np.float32).astype(np.float64)
                        for x in _token(rng))
    a, scale = math.exp(g), 0.37
    kS, qS = S.T @ k, S.T @ q                      # the one pass over S
    u = b * (v - a * kS)
    o = scale * (a * qS + (k @ q) * u)
    S_new = a * S + np.outer(k, u)
    f32 = lambda x: np.asarray(x, np.float32)
    o_ref, S_ref = oracle.recurrent(f32(q)[None, None], f32(k)[None, None], f32(v)[None, None], f32([[g]]),
                                    f32([[b]]), h0=f32(S)[None, None], scale=scale)
    np.testing.assert_allclose(o, o_ref[0, 0], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(S_new, S_ref[0, 0], rtol=1e-12, atol=1e-14)


def test_kda_single_pass_rearrangement():
    rng = np.random.default_rng(4)
    S, q, k, v, g, b = _token(rng, per_channel=True)
    a, scale = np.exp(g), 0.41
    ks, qs = S.T @ (a * k), S.T @ (a * q)          # reads against the undecayed state
    u = b * (v - ks)
    o = scale * (qs + (k @ q) * u)
    S_new = a[:, None] * S + np.outer(k, u)
    o_ref, S_ref = oracle.kda_recurrent(q[None, None], k[None, None], v[None, None], g[None, None], np.array([[b]]),
                                        h0=S[None, None], scale=scale)
    np.testing.assert_allclose(o, o_ref[0, 0], rtol=1e-12, atol=1e-14)
    np.testing.assert_allclose(S_new, S_ref[0, 0], rtol=1e-12, atol=1e-14)


def _prefix_start(g, beta, k, s0, a, ln_eps=-40 * math.log(2.0)):
    """The segment rule, written out token by token (fp64)."""
    acc = 0.0
    for t in range(a - 1, s0 - 1, -1):
        f = abs(1.0 - beta[t] * float(k[t] @ k[t]))
        acc += g[t] + (math.log(f) if f > 1.0 else 0.0)
        if acc <= ln_eps:
            return t
    return s0


@pytest.mark.parametrize("g_shift,k_scale", [(0.0, 1.0), (2.0, 1.0), (-5.0, 1.0), (0.0, 2.0), (None, 1.0)])
def test_segment_prefix_bound(g_shift, k_scale):
    """Run the rule (fp64, this file's own loop) from the exact state and from
    a zero state at the prefix start; at the segment's first token the two
    states differ by at most 2^-40 times the spectral norm of the true state
    before the prefix (the product of the per-token factors bounds the
    spectral norm of the map that carries a state difference forward)."""
    rng = np.random.default_rng(7)
    L, dk, dv = 3000, 16, 8
    k = rng.standard_normal((L, dk))
    k = k / np.linalg.norm(k, axis=1, keepdims=True) * k_scale
    v = rng.standard_normal((L, dv))
    beta = 1.0 / (1.0 + np.exp(-rng.standard_normal(L)))
    if g_shift is None:
        g = np.zeros(L)                      # alpha = 1: no bound is ever reached
    else:
        g = -np.log1p(np.exp(rng.standard_normal(L) + g_shift))
    S0 = rng.standard_normal((dk, dv)) * 0.5
    states = [S0]
    S = S0.copy()
    for t in range(L):
        a_ = math.exp(g[t])
        S = a_ * S + beta[t] * np.outer(k[t], v[t] - a_ * (S.T @ k[t]))
        states.append(S)                     # states[t + 1] = state after token t
    for seg_a in (700, 1500, 2999):
        ts = _prefix_start(g, beta, k, 0, seg_a)
        if g_shift is None:
            assert ts == 0                   # exact: the segment starts at the sequence start
            continue
        # the sequence's start: its initial state (exact); elsewhere a zero state
        Z = S0.copy() if ts == 0 else np.zeros((dk, dv))
        for t in range(ts, seg_a):
            a_ = math.exp(g[t])
            Z = a_ * Z + beta[t] * np.outer(k[t], v[t] - a_ * (Z.T @ k[t]))
        bound = 0.0 if ts == 0 else 2.0 ** -40 * np.linalg.norm(states[ts], 2)
        err = np.linalg.norm(Z - states[seg_a], 2)
        fp64 = 1e-12 * np.linalg.norm(states[seg_a], 2)  # rounding of the two fp64 runs
        assert err <= bound + fp64, (g_shift, k_scale, seg_a, ts, err, bound)
        # and the rule does not start earlier than it needs to
        if ts > 0 and ts < seg_a - 1:
            assert _prefix_start(g, beta, k, ts + 1, seg_a) == ts + 1  # one token fewer misses the bound
