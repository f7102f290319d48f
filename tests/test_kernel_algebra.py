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
    undecayed state and o = scale (S^T (a o q) + (k . q) u).
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
