"""Pins of the KDA oracle (oracle.kda_recurrent): the gated delta rule with one
decay per key channel (the reading stated in oracle/kda.py; the pages only
name KDA, on the "Qwen3.8 attention gate" page).

  - a two-token example worked by hand (tests/golden/kda_hand_example.json);
  - with every channel's decay equal, KDA is the gated delta rule: equality
    with the independent C oracle (oracle.recurrent) on varlen + GQA inputs;
  - beta = 0: the state only decays, row by row: S_T = diag(e^{G_T}) S_0 and
    o_t = scale (diag(e^{G_t}) S_0)^T q_t, with G the running sum of g per
    channel (d_k != d_v, so a decay applied to the wrong axis cannot pass);
  - no decay, beta = 1, keys along the coordinate axes: S_T^T e_i is the value
    last written under key i.
``test_planted_mistakes`` edits the oracle's source and checks each edit is
caught.
"""
import inspect
import json
import math
import os

import numpy as np
import pytest

import oracle
import oracle.kda as kda_module


def _golden():
    path = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", "kda_hand_example.json")
    with open(path) as f:
        return json.load(f)


def _rand(seed, lens, h_qk, h_v, d_k, d_v, grid=2.0 ** -10):
    rng = np.random.default_rng(seed)
    T = int(sum(lens))
    r = lambda shape, s=1.0: (np.round(rng.standard_normal(shape) * s / grid) * grid).astype(np.float32)
    q, k = r((T, h_qk, d_k), 0.5), r((T, h_qk, d_k), 0.5)
    v = r((T, h_v, d_v))
    beta = (np.round(rng.uniform(0.1, 0.9, (T, h_v)) / grid) * grid).astype(np.float32)
    h0 = r((len(lens), h_v, d_k, d_v), 0.3)
    cu = np.concatenate([[0], np.cumsum(lens)]).astype(np.int32)
    return q, k, v, beta, h0, cu, rng


# pins: each takes fn with the signature of oracle.kda_recurrent

def pin_hand_example(fn):
    G = _golden()
    q = np.array(G["q"], float)[:, None]
    k = np.array(G["k"], float)[:, None]
    v = np.array(G["v"], float)[:, None]
    g = np.log(np.array(G["alpha"], float))[:, None]
    b = np.array(G["beta"], float)[:, None]
    o, S = fn(q, k, v, g, b, h0=np.array(G["S0"], float)[None, None], scale=1.0)
    np.testing.assert_allclose(o[:, 0], G["o"], rtol=0, atol=G["atol"])
    np.testing.assert_allclose(S[0, 0], G["S_final"], rtol=0, atol=G["atol"])


def pin_uniform_channels_equal_gated_delta_rule(fn):
    q, k, v, beta, h0, cu, rng = _rand(1, (7, 1, 12), 2, 4, 6, 5)
    g1 = (-np.round(rng.uniform(0.05, 1.5, (len(q), 4)) * 1024) / 1024).astype(np.float32)
    o_ref, S_ref = oracle.recurrent(q, k, v, g1, beta, h0=h0, cu_seqlens=cu)
    g = np.repeat(g1[:, :, None], 6, axis=2)
    o, S = fn(q, k, v, g, beta, h0=h0, cu_seqlens=cu)
    np.testing.assert_allclose(o, o_ref, rtol=1e-12, atol=1e-13)
    np.testing.assert_allclose(S, S_ref, rtol=1e-12, atol=1e-13)


def pin_beta_zero_closed_form(fn):
    q, k, v, beta, h0, cu, rng = _rand(2, (5, 4), 1, 2, 4, 3)
    beta = np.zeros_like(beta)
    g = -rng.uniform(0.0, 1.0, (len(q), 2, 4))
    o, S = fn(q, k, v, g, beta, h0=h0, cu_seqlens=cu)
    scale = 1 / math.sqrt(4)
    for n in range(2):
        t0, t1 = int(cu[n]), int(cu[n + 1])
        for h in range(2):
            G = np.cumsum(g[t0:t1, h], axis=0)
            for t in range(t1 - t0):
                St = np.exp(G[t])[:, None] * h0[n, h]
                np.testing.assert_allclose(o[t0 + t, h], scale * St.T @ q[t0 + t, 0], rtol=1e-12, atol=1e-13)
            np.testing.assert_allclose(S[n, h], np.exp(G[-1])[:, None] * h0[n, h], rtol=1e-12, atol=1e-13)


def pin_axis_key_retrieval(fn):
    d_k, d_v = 4, 3
    keys = [2, 0, 2, 3, 1, 0]
    T = len(keys)
    k = np.zeros((T, 1, d_k))
    for t, i in enumerate(keys):
        k[t, 0, i] = 1.0
    rng = np.random.default_rng(3)
    v = rng.standard_normal((T, 1, d_v))
    q = rng.standard_normal((T, 1, d_k))
    o, S = fn(q, k, v, np.zeros((T, 1, d_k)), np.ones((T, 1)), h0=rng.standard_normal((1, 1, d_k, d_v)))
    for i in range(d_k):
        last = max(t for t in range(T) if keys[t] == i)
        np.testing.assert_allclose(S[0, 0].T @ np.eye(d_k)[i], v[last, 0], rtol=1e-12, atol=1e-13)


PINS = [pin_hand_example, pin_uniform_channels_equal_gated_delta_rule, pin_beta_zero_closed_form,
        pin_axis_key_retrieval]


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(oracle.kda_recurrent)


EDITS = {
    "decay_after_read": ("e = v[t] - Sd.T @ k[t]", "e = v[t] - S.T @ k[t]"),
    "decay_on_value_axis": ("Sd = np.exp(g[t])[:, None] * S", "Sd = S * np.exp(g[t])[None, :S.shape[1]]"),
    "no_decay_kept": ("S[...] = Sd + b[t] * np.outer(k[t], e)", "S[...] = S + b[t] * np.outer(k[t], e)"),
    "write_value_not_error": ("S[...] = Sd + b[t] * np.outer(k[t], e)", "S[...] = Sd + b[t] * np.outer(k[t], v[t])"),
    "output_before_write": ("o[t] = scale * (S.T @ q[t])", "o[t] = scale * (Sd.T @ q[t])"),
    "beta_on_read": ("e = v[t] - Sd.T @ k[t]", "e = v[t] - b[t] * (Sd.T @ k[t])"),
    "group_index": ("hk = h // grp", "hk = h % h_qk"),
}


def _variant(old, new):
    """The oracle's source with one edit in the recurrent form (the part of the
    module before the chunked form), bound as a new module."""
    src = inspect.getsource(kda_module)
    cut = src.index("def _pair_chunked")
    head, tail = src[:cut], src[cut:]
    assert head.count(old) == 1, old
    ns = {"__name__": "kda_variant"}
    exec(compile(head.replace(old, new) + tail, "kda_variant", "exec"), ns)
    return ns["kda_recurrent"]


@pytest.mark.parametrize("edit", list(EDITS), ids=list(EDITS))
def test_planted_mistakes(edit):
    wrong = _variant(*EDITS[edit])
    failed = []
    with np.errstate(all="ignore"):
        for pin in PINS:
            try:
                pin(wrong)
            except (AssertionError, ValueError, IndexError, FloatingPointError):
                failed.append(pin.__name__)
    assert failed, f"no pin catches {edit}"


# the chunkwise form (per-channel decay inside the inner products)

def _chunk_problem(seed):
    q, k, v, beta, h0, cu, rng = _rand(seed, (5, 0, 37, 64, 70), 1, 2, 8, 6)
    g = -rng.uniform(0.0, 1.2, (len(q), 2, 8))
    return q, k, v, g, beta, h0, cu


@pytest.mark.parametrize("chunk", [1, 2, 3, 16, 64, 200])
def test_kda_chunked_equals_recurrent(chunk):
    q, k, v, g, beta, h0, cu = _chunk_problem(5)
    o_ref, S_ref = oracle.kda_recurrent(q, k, v, g, beta, h0=h0, cu_seqlens=cu)
    o, S = oracle.kda_chunked(q, k, v, g, beta, h0=h0, cu_seqlens=cu, chunk=chunk)
    np.testing.assert_allclose(o, o_ref, rtol=0, atol=1e-12 * np.abs(o_ref).max())
    np.testing.assert_allclose(S, S_ref, rtol=0, atol=1e-12 * np.abs(S_ref).max())


CHUNK_EDITS = {
    "scalar_decay_per_row": ('E = np.where(lower[:, :, None], np.exp(np.where(lower[:, :, None], diff, 0.0)), 0.0)',
                             'E = np.where(lower[:, :, None], np.exp(np.where(lower[:, :, None], diff, 0.0)).mean(-1, keepdims=True), 0.0)'),
    "P_strict_lower": ("np.tril(QK) @ U", "np.tril(QK, -1) @ U"),
    "A_diagonal_kept": ("A = np.tril(bb[:, None] * KK, -1)", "A = np.tril(bb[:, None] * KK)"),
    "state_decay_missing": ("S[...] = np.exp(G[-1])[:, None] * S +", "S[...] = S +"),
    "query_decay_missing": ("o[c0:c1] = scale * ((Q * np.exp(G)) @ S", "o[c0:c1] = scale * (Q @ S"),
}


@pytest.mark.parametrize("edit", list(CHUNK_EDITS), ids=list(CHUNK_EDITS))
def test_kda_chunked_planted_mistakes(edit):
    old, new = CHUNK_EDITS[edit]
    src = inspect.getsource(kda_module)
    cut = src.index("def _pair_chunked")
    head, tail = src[:cut], src[cut:]
    assert tail.count(old) == 1, old
    ns = {"__name__": "kda_variant"}
    exec(compile(head + tail.replace(old, new), "kda_variant", "exec"), ns)
    q, k, v, g, beta, h0, cu = _chunk_problem(6)
    o_ref, S_ref = oracle.kda_recurrent(q, k, v, g, beta, h0=h0, cu_seqlens=cu)
    o, S = ns["kda_chunked"](q, k, v, g, beta, h0=h0, cu_seqlens=cu, chunk=16)
    worst = max(np.abs(o - o_ref).max() / np.abs(o_ref).max(), np.abs(S - S_ref).max() / np.abs(S_ref).max())
    assert worst > 1e-6, f"{edit} not caught ({worst:.1e})"
