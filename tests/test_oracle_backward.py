"""Pins of the gradient oracle (oracle.recurrent_backward).

The gradient of the gated delta rule is fixed by the forward rule alone (the
podcast episode "Qwen3.8-Next design: hybrid attention, residuals and n-gram
embeddings", transcript segment 14; training cost: "On the Design of
Qwen3.8-Next Architecture", arXiv abstract page). Nothing here re-types the
reverse recurrence the oracle uses. The pins are:

  - central finite differences (Richardson-extrapolated) of the *forward*
    oracle (gdn_oracle.c, the C recurrence), on tiny varlen + GQA problems
    whose inputs lie on a binary grid so that every perturbation is exact in
    the fp32 inputs the forward oracle reads;
  - a two-token scalar example differentiated by hand
    (tests/golden/gdn_gradient_hand_example.json);
  - the closed form of the beta = 0 case, where the state only decays
    (S_t = e^{G_t} S_0), for every gradient;
  - two homogeneity identities: o is linear in q token by token, so
    <dq, q> = <dO, O>; (O, S_T) is jointly linear in (v, S_0), so
    <dv, v> + <dS_0, S_0> = <dO, O> + <dS_T, S_T>;
  - the decay-gradient identity dg_t = <dS_T, S_T> + sum_{r >= t}
    (<dO_r, o_r> - <dv_r, v_r>), exact for this rule.

``test_planted_mistakes`` edits the oracle's source (a dropped term, a wrong
sign, a missing decay, a wrong index, a missing group sum, ...) and checks
that at least one pin rejects each edit.
"""
import inspect
import json
import math
import os

import numpy as np
import pytest

import oracle
import oracle.backward as backward_module

GRID = 2.0 ** -8       # inputs are multiples of this (exact in fp32)
STEP = 2.0 ** -11      # finite-difference step (x +- STEP, x +- STEP/2 stay exact in fp32)


def _grid(rng, shape, scale=1.0):
    return (np.round(rng.standard_normal(shape) * scale / GRID) * GRID).astype(np.float32)


def _problem(seed, lens=(3, 5), h_qk=1, h_v=2, d_k=3, d_v=2, with_state=True, beta_zero=False):
    rng = np.random.default_rng(seed)
    T, N = int(sum(lens)), len(lens)
    P = dict(
        q=_grid(rng, (T, h_qk, d_k), 0.7),
        k=_grid(rng, (T, h_qk, d_k), 0.7),
        v=_grid(rng, (T, h_v, d_v)),
        g=(-np.round(rng.uniform(0.05, 0.9, (T, h_v)) / GRID) * GRID).astype(np.float32),
        beta=(np.round(rng.uniform(0.1, 0.9, (T, h_v)) / GRID) * GRID).astype(np.float32),
        h0=_grid(rng, (N, h_v, d_k, d_v), 0.5) if with_state else None,
        cu=np.concatenate([[0], np.cumsum(lens)]).astype(np.int32),
    )
    if beta_zero:
        P["beta"] = np.zeros_like(P["beta"])
    P["do"] = _grid(rng, (T, h_v, d_v))
    P["dht"] = _grid(rng, (N, h_v, d_k, d_v), 0.5) if with_state else None
    return P


def _loss(P, **over):
    """L = <dO, O> + <dS_T, S_T> through the forward C oracle."""
    X = dict(P, **over)
    o, S = oracle.recurrent(X["q"], X["k"], X["v"], X["g"], X["beta"], h0=X["h0"],
                            cu_seqlens=X["cu"])
    L = float(np.sum(o * X["do"]))
    if X["dht"] is not None:
        L += float(np.sum(S * X["dht"]))
    return L


def _fd_grad(P, name):
    """Richardson-extrapolated central difference of _loss for every element of P[name]."""
    x0 = P[name]
    out = np.zeros(x0.shape)
    for idx in np.ndindex(x0.shape):
        def d(h):
            xp, xm = x0.copy(), x0.copy()
            xp[idx] += np.float32(h)
            xm[idx] -= np.float32(h)
            return (_loss(P, **{name: xp}) - _loss(P, **{name: xm})) / (2 * h)
        out[idx] = (4 * d(STEP / 2) - d(STEP)) / 3
    return out


def _call(fn, P):
    return fn(P["q"], P["k"], P["v"], P["g"], P["beta"], P["do"], h0=P["h0"], dht=P["dht"],
              cu_seqlens=P["cu"])


# ----------------------------------------------------------------------------
# pins: each takes fn with the signature of oracle.recurrent_backward
# ----------------------------------------------------------------------------

def _check_fd(fn, P):
    got = _call(fn, P)
    inputs = {"dq": "q", "dk": "k", "dv": "v", "dg": "g", "dbeta": "beta", "dh0": "h0"}
    for gname, iname in inputs.items():
        if P[iname] is None:
            continue
        ref = _fd_grad(P, iname)
        np.testing.assert_allclose(got[gname], ref, rtol=1e-7, atol=1e-8, err_msg=gname)


def pin_finite_differences_varlen_gqa(fn):
    """Two sequences (3 and 5 tokens), two value heads sharing one q/k head,
    d_k = 3, d_v = 2, random S_0 and dS_T: every gradient equals the
    finite-difference derivative of the forward oracle's loss."""
    _check_fd(fn, _problem(0))


def pin_finite_differences_plain(fn):
    """One sequence of 6 tokens, no GQA (H_qk = H_v = 2), d_k = 2, d_v = 3,
    zero initial state and no final-state gradient."""
    _check_fd(fn, _problem(1, lens=(6,), h_qk=2, h_v=2, d_k=2, d_v=3, with_state=False))


def pin_hand_example(fn):
    """Two scalar tokens differentiated by hand
    (tests/golden/gdn_gradient_hand_example.json)."""
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                        "gdn_gradient_hand_example.json")
    with open(path) as f:
        G = json.load(f)
    col = lambda x: np.array(x, dtype=np.float64).reshape(-1, 1, 1)
    got = fn(col(G["q"]), col(G["k"]), col(G["v"]), np.log(np.array(G["alpha"])).reshape(-1, 1),
             np.array(G["beta"]).reshape(-1, 1), col(G["dO"]),
             h0=np.full((1, 1, 1, 1), G["S0"]), dht=None, scale=1.0)
    for name, key in (("dq", "dq"), ("dk", "dk"), ("dv", "dv"), ("dg", "dg"), ("dbeta", "dbeta")):
        np.testing.assert_allclose(np.ravel(got[name]), G[key], rtol=0, atol=G["atol"], err_msg=name)
    np.testing.assert_allclose(float(got["dh0"].ravel()[0]), G["dS0"], rtol=0, atol=G["atol"])


def pin_beta_zero_closed_form(fn):
    """beta = 0: the state only decays, S_t = e^{G_t} S_0 with G_t the running
    sum of g. Then dv = 0 and dk = 0 exactly, and with
    D_t = sum_{r >= t} scale e^{G_r - G_t} q_r dO_r^T + e^{G_T - G_t} dS_T:
      dq_t    = scale e^{G_t} S_0 dO_t
      dS_0    = e^{G_1} D_1
      dg_s    = sum_{t >= s} scale e^{G_t} q_t^T S_0 dO_t + e^{G_T} <dS_T, S_0>
      dbeta_t = (D_t^T k_t) . (v_t - e^{G_t} S_0^T k_t)."""
    P = _problem(2, lens=(4, 3), h_qk=1, h_v=2, d_k=3, d_v=4, beta_zero=True)
    got = _call(fn, P)
    scale = 1.0 / math.sqrt(3)
    assert np.abs(got["dv"]).max() == 0.0 and np.abs(got["dk"]).max() == 0.0
    cu = P["cu"]
    for n in range(2):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        for h in range(2):
            g = P["g"][t0:t1, h].astype(np.float64)
            G = np.cumsum(g)
            S0 = P["h0"][n, h].astype(np.float64)
            dST = P["dht"][n, h].astype(np.float64)
            q = P["q"][t0:t1, 0].astype(np.float64)
            k = P["k"][t0:t1, 0].astype(np.float64)
            v = P["v"][t0:t1, h].astype(np.float64)
            do = P["do"][t0:t1, h].astype(np.float64)
            L = t1 - t0
            dq_ref = np.stack([scale * math.exp(G[t]) * (S0 @ do[t]) for t in range(L)])
            # both value heads read q/k head 0: its gradient is the sum of their closed forms
            if h == 0:
                dq_sum = dq_ref
            else:
                dq_sum = dq_sum + dq_ref
                np.testing.assert_allclose(got["dq"][t0:t1, 0], dq_sum, rtol=1e-12, atol=1e-13)
            D = [None] * L
            for t in range(L):
                D[t] = sum(scale * math.exp(G[r] - G[t]) * np.outer(q[r], do[r]) for r in range(t, L))
                D[t] = D[t] + math.exp(G[-1] - G[t]) * dST
            dS0 = math.exp(G[0]) * D[0]
            np.testing.assert_allclose(got["dh0"][n, h], dS0, rtol=1e-12, atol=1e-13)
            per_t = np.array([scale * math.exp(G[t]) * (q[t] @ S0 @ do[t]) for t in range(L)])
            dg_ref = np.array([per_t[s:].sum() for s in range(L)]) + math.exp(G[-1]) * np.sum(dST * S0)
            np.testing.assert_allclose(got["dg"][t0:t1, h], dg_ref, rtol=1e-12, atol=1e-13)
            db_ref = np.array([(D[t].T @ k[t]) @ (v[t] - math.exp(G[t]) * (S0.T @ k[t]))
                               for t in range(L)])
            np.testing.assert_allclose(got["dbeta"][t0:t1, h], db_ref, rtol=1e-12, atol=1e-13)


def pin_homogeneity(fn):
    """<dq, q> = <dO, O> and <dv, v> + <dS_0, S_0> = <dO, O> + <dS_T, S_T> on a
    larger problem (three sequences, GQA 2, d_k = 8, d_v = 6)."""
    P = _problem(3, lens=(9, 1, 14), h_qk=2, h_v=4, d_k=8, d_v=6)
    got = _call(fn, P)
    o, S = oracle.recurrent(P["q"], P["k"], P["v"], P["g"], P["beta"], h0=P["h0"], cu_seqlens=P["cu"])
    lo = float(np.sum(P["do"] * o))
    ls = float(np.sum(P["dht"] * S))
    np.testing.assert_allclose(float(np.sum(got["dq"] * P["q"])), lo, rtol=1e-11)
    lhs = float(np.sum(got["dv"] * P["v"]) + np.sum(got["dh0"] * P["h0"]))
    np.testing.assert_allclose(lhs, lo + ls, rtol=1e-11)


def pin_decay_gradient_identity(fn):
    """With D_t = dL/dS_t and S_t - b_t k_t v_t^T = a_t (I - b_t k_t k_t^T) S_{t-1},
    the rule gives dg_t = <D_t, S_t> - <dv_t, v_t> and <D_{t-1}, S_{t-1}> =
    dg_t + <dO_{t-1}, o_{t-1}>; unrolled from <D_T, S_T> = <dS_T, S_T> + <dO_T, o_T>:
        dg_t = <dS_T, S_T> + sum_{r >= t} (<dO_r, o_r> - <dv_r, v_r>)
    which ties dg to dv and the forward oracle's outputs (per pair)."""
    P = _problem(6, lens=(11, 6), h_qk=1, h_v=2, d_k=5, d_v=4)
    got = _call(fn, P)
    o, S = oracle.recurrent(P["q"], P["k"], P["v"], P["g"], P["beta"], h0=P["h0"], cu_seqlens=P["cu"])
    cu = P["cu"]
    for n in range(2):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        for h in range(2):
            per = np.sum(P["do"][t0:t1, h] * o[t0:t1, h], -1) - np.sum(got["dv"][t0:t1, h] * P["v"][t0:t1, h], -1)
            ref = float(np.sum(P["dht"][n, h] * S[n, h])) + np.cumsum(per[::-1])[::-1]
            np.testing.assert_allclose(got["dg"][t0:t1, h], ref, rtol=1e-11, atol=1e-12)


PINS = [pin_finite_differences_varlen_gqa, pin_finite_differences_plain, pin_hand_example,
        pin_beta_zero_closed_form, pin_homogeneity, pin_decay_gradient_identity]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(oracle.recurrent_backward)


def test_pairs_mode_matches_full():
    """The per-pair form returns each value head's own contribution; summed
    over a group it gives the full q/k gradient."""
    P = _problem(4, lens=(5, 7), h_qk=1, h_v=2, d_k=4, d_v=3)
    full = _call(oracle.recurrent_backward, P)
    parts = oracle.recurrent_backward(P["q"], P["k"], P["v"], P["g"], P["beta"], P["do"], h0=P["h0"],
                                      dht=P["dht"], cu_seqlens=P["cu"], pairs=[(1, 0), (1, 1)])
    np.testing.assert_allclose(parts[0]["dq"] + parts[1]["dq"], full["dq"][5:, 0], rtol=1e-14, atol=1e-15)
    np.testing.assert_allclose(parts[1]["dv"], full["dv"][5:, 1], rtol=0, atol=0)
    np.testing.assert_allclose(parts[0]["dh0"], full["dh0"][1, 0], rtol=0, atol=0)


def test_empty_sequence():
    """A zero-length sequence passes dS_T straight through to dS_0."""
    P = _problem(5, lens=(3, 0, 2), h_qk=1, h_v=1, d_k=2, d_v=2)
    got = _call(oracle.recurrent_backward, P)
    np.testing.assert_array_equal(got["dh0"][1], P["dht"][1].astype(np.float64))


# ----------------------------------------------------------------------------
# planted mistakes: each edit of the oracle's source must fail a pin
# ----------------------------------------------------------------------------

EDITS = {
    "dk_without_read_term": ("dk[t] = b[t] * (D @ E[t]) - a[t] * (S[t] @ de)", "dk[t] = b[t] * (D @ E[t])"),
    "dk_read_sign": ("dk[t] = b[t] * (D @ E[t]) - a[t] * (S[t] @ de)",
                     "dk[t] = b[t] * (D @ E[t]) + a[t] * (S[t] @ de)"),
    "carry_sign": ("D = a[t] * (D - np.outer(k[t], de))", "D = a[t] * (D + np.outer(k[t], de))"),
    "carry_without_decay": ("D = a[t] * (D - np.outer(k[t], de))", "D = (D - np.outer(k[t], de))"),
    "dq_from_previous_state": ("dq[t] = scale * (S[t + 1] @ do[t])", "dq[t] = scale * (S[t] @ do[t])"),
    "dg_without_read_term": ("dg[t] = a[t] * (np.sum(D * S[t]) - k[t] @ (S[t] @ de))",
                             "dg[t] = a[t] * np.sum(D * S[t])"),
    "dg_without_alpha": ("dg[t] = a[t] * (np.sum(D * S[t]) - k[t] @ (S[t] @ de))",
                         "dg[t] = (np.sum(D * S[t]) - k[t] @ (S[t] @ de))"),
    "dbeta_with_value_not_error": ("db[t] = k[t] @ (D @ E[t])", "db[t] = k[t] @ (D @ v[t])"),
    "dv_without_beta": ("de = b[t] * (D.T @ k[t])", "de = (D.T @ k[t])"),
    "no_output_gradient_in_carry": ("D += scale * np.outer(q[t], do[t])\n", "D += 0.0\n"),
    "no_group_sum": ('out["dq"][t0:t1, h // grp] += r["dq"]', 'out["dq"][t0:t1, h // grp] = r["dq"]'),
    "error_without_decay": ("E[t] = v[t] - a[t] * (S[t].T @ k[t])", "E[t] = v[t] - (S[t].T @ k[t])"),
}


def _variant(old, new):
    """The oracle's source with one edit in the recurrent form (the part of the
    module before the chunked form), bound as a new module."""
    src = inspect.getsource(backward_module)
    cut = src.index("def _pair_chunked_backward")
    head, tail = src[:cut], src[cut:]
    assert head.count(old) == 1, old
    ns = {"__name__": "backward_variant"}
    exec(compile(head.replace(old, new) + tail, "backward_variant", "exec"), ns)
    return ns["recurrent_backward"]


@pytest.mark.parametrize("edit", list(EDITS), ids=list(EDITS))
def test_planted_mistakes(edit):
    wrong = _variant(*EDITS[edit])
    failed = []
    with np.errstate(all="ignore"):
        for pin in PINS:
            try:
                pin(wrong)
            except (AssertionError, ValueError, FloatingPointError):
                failed.append(pin.__name__)
    assert failed, f"no pin catches {edit}"


# ----------------------------------------------------------------------------
# the chunkwise form of the gradient: equal to the pinned recurrent form
# ----------------------------------------------------------------------------

@pytest.mark.parametrize("chunk", [1, 2, 3, 16, 64, 200])
def test_chunked_backward_equals_recurrent(chunk):
    """The WY algebra differentiated chunk by chunk (oracle.chunked_backward)
    equals the reverse-order chain rule on ragged varlen + GQA inputs with
    S_0 and dS_T, for chunk sizes from 1 to longer than any sequence."""
    P = _problem(7, lens=(5, 0, 37, 64, 70), h_qk=1, h_v=2, d_k=8, d_v=6)
    ref = _call(oracle.recurrent_backward, P)
    got = oracle.chunked_backward(P["q"], P["k"], P["v"], P["g"], P["beta"], P["do"], h0=P["h0"],
                                  dht=P["dht"], cu_seqlens=P["cu"], chunk=chunk)
    for name in ("dq", "dk", "dv", "dg", "dbeta", "dh0"):
        scale = np.abs(ref[name]).max()
        np.testing.assert_allclose(got[name], ref[name], rtol=0, atol=1e-12 * scale, err_msg=name)


CHUNK_EDITS = {
    "no_transpose_in_dDelta": ("dDelta = scale * P.T @ dO + Kd @ D", "dDelta = scale * P @ dO + Kd @ D"),
    "dA_sign": ("dA = np.tril(-T.T @ dT @ T.T, -1)", "dA = np.tril(T.T @ dT @ T.T, -1)"),
    "dA_diagonal_kept": ("dA = np.tril(-T.T @ dT @ T.T, -1)", "dA = np.tril(-T.T @ dT @ T.T)"),
    "dK_missing_transpose_term": ("dKc += E @ K + E.T @ K", "dKc += E @ K"),
    "dS0_missing_state_term": ("dS0 = gam[-1] * D + scale", "dS0 = D + scale"),
    "dbeta_missing_A_term": ("dbc += np.sum(dA * Gam * KK, axis=1)", "dbc += 0.0"),
    "P_strict_lower": ("P = np.tril(Gam * (Q @ K.T))", "P = np.tril(Gam * (Q @ K.T), -1)"),
}


@pytest.mark.parametrize("edit", list(CHUNK_EDITS), ids=list(CHUNK_EDITS))
def test_chunked_backward_planted_mistakes(edit):
    old, new = CHUNK_EDITS[edit]
    src = inspect.getsource(backward_module)
    cut = src.index("def _pair_chunked_backward")
    head, tail = src[:cut], src[cut:]
    assert tail.count(old) == 1, old
    ns = {"__name__": "backward_variant"}
    exec(compile(head + tail.replace(old, new), "backward_variant", "exec"), ns)
    P = _problem(8, lens=(9, 20), h_qk=1, h_v=2, d_k=5, d_v=4)
    ref = _call(oracle.recurrent_backward, P)
    got = ns["chunked_backward"](P["q"], P["k"], P["v"], P["g"], P["beta"], P["do"], h0=P["h0"], dht=P["dht"],
                                 cu_seqlens=P["cu"], chunk=8)
    worst = max(float(np.abs(got[n] - ref[n]).max() / np.abs(ref[n]).max())
                for n in ("dq", "dk", "dv", "dg", "dbeta", "dh0"))
    assert worst > 1e-6, f"{edit} not caught ({worst:.1e})"
