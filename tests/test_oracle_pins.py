"""Pins of the fp64 CPU oracle against what the definition itself fixes.

The gated delta rule is described in words in the podcast episode
"Qwen3.8-Next design: hybrid attention, residuals and n-gram embeddings",
transcript segment 14 (decay erases part of the whole state; the delta term
reads what is stored under the current key, subtracts it and writes only the
error; the same key written twice leaves one corrected note) and segment 4
(fixed-size state, linear cost). Written out, with S of shape d_k x d_v:

    S_t = a_t (I - b_t k_t k_t^T) S_{t-1} + b_t k_t v_t^T,   o_t = scale S_t^T q_t

Nothing here re-types the oracle's loops. Each pin is one of: a hand-worked
example, a closed form of a special case (b = 0; a = b = 1 with orthonormal
keys; the same key twice), a structural invariant (linearity, head grouping,
packing, resumption), or the literal matrix form of the rule on tiny inputs.
``test_planted_mistakes`` rebuilds the oracle from its source with one
plausible mistake at a time and checks that some pin fails for every one.
"""
import math
import os
import shutil
import subprocess
import tempfile

import numpy as np
import pytest
import torch

import oracle

RNG = np.random.default_rng(1234)


def _rand_problem(total=29, h_qk=2, h_v=4, d_k=6, d_v=5, lengths=None, h0=True, g_lo=-1.5,
                  seed=0):
    rng = np.random.default_rng(seed)
    q = rng.standard_normal((total, h_qk, d_k)).astype(np.float32)
    k = rng.standard_normal((total, h_qk, d_k)).astype(np.float32)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    v = rng.standard_normal((total, h_v, d_v)).astype(np.float32)
    g = rng.uniform(g_lo, 0.0, (total, h_v)).astype(np.float32)
    b = rng.uniform(0.0, 1.0, (total, h_v)).astype(np.float32)
    n = 1 if lengths is None else len(lengths)
    S0 = (rng.standard_normal((n, h_v, d_k, d_v)) * 0.5).astype(np.float32) if h0 else None
    cu = None
    if lengths is not None:
        assert sum(lengths) == total
        cu = np.concatenate([[0], np.cumsum(lengths)]).astype(np.int32)
    return dict(q=q, k=k, v=v, g=g, beta=b, h0=S0, cu_seqlens=cu)


# ----------------------------------------------------------------------------
# pins, each taking an oracle object (the real one, or a planted-mistake copy)
# ----------------------------------------------------------------------------

def _golden(name):
    import json
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden", name)) as f:
        return json.load(f)


def pin_hand_example(orc):
    """d_k=2, d_v=3, three tokens worked by hand from the rule (scale = 1); the
    inputs, the derivation and the expected values are in
    tests/golden/gdn_rule_hand_example.json."""
    G = _golden("gdn_rule_hand_example.json")
    q = np.array(G["q"], dtype=np.float32)[:, None, :]
    k = np.array(G["k"], dtype=np.float32)[:, None, :]
    v = np.array(G["v"], dtype=np.float32)[:, None, :]
    g = np.log(np.array(G["alpha"], dtype=np.float64)).astype(np.float32)[:, None]
    b = np.array(G["beta"], dtype=np.float32)[:, None]
    S0 = np.array(G["S0"], dtype=np.float32)[None, None]
    o_exp, S_exp = np.array(G["o"]), np.array(G["S_final"])
    for fn in (orc.recurrent, lambda *a, **kw: orc.chunked(*a, chunk=2, **kw)):
        o, S = fn(q, k, v, g, b, h0=S0, scale=1.0)
        np.testing.assert_allclose(o[:, 0, :], o_exp, atol=G["atol"])
        np.testing.assert_allclose(S[0, 0], S_exp, atol=G["atol"])


def pin_literal_matrix_form(orc):
    """Brute force on tiny inputs: apply S <- a (I - b k k^T) S + b k v^T as a
    d_k x d_k matrix product per token (the rule's literal form), with GQA head
    h reading q/k head h // (H_v/H_qk)."""
    P = _rand_problem(total=11, h_qk=1, h_v=2, d_k=4, d_v=3, seed=7)
    scale = 0.37
    o, S = orc.recurrent(**P, scale=scale)
    for h in range(2):
        St = P["h0"][0, h].astype(np.float64)
        for t in range(11):
            kk = P["k"][t, 0].astype(np.float64)
            a = math.exp(float(P["g"][t, h]))
            bb = float(P["beta"][t, h])
            St = a * (np.eye(4) - bb * np.outer(kk, kk)) @ St + bb * np.outer(kk, P["v"][t, h])
            np.testing.assert_allclose(o[t, h], scale * St.T @ P["q"][t, 0], atol=1e-12)
        np.testing.assert_allclose(S[0, h], St, atol=1e-12)


def pin_beta_zero_closed_form(orc):
    """b = 0: nothing is written, the state only decays.
    S_T = exp(sum g) S0 and o_t = exp(G_t) scale S0^T q_t with G_t = g_1 + .. + g_t."""
    P = _rand_problem(total=13, seed=3)
    P["beta"][:] = 0.0
    o, S = orc.recurrent(**P)
    G = np.cumsum(P["g"].astype(np.float64), axis=0)  # [T, H_v]
    scale = 1.0 / math.sqrt(6)
    for h in range(4):
        S0 = P["h0"][0, h].astype(np.float64)
        np.testing.assert_allclose(S[0, h], math.exp(G[-1, h]) * S0, rtol=1e-12, atol=1e-14)
        for t in range(13):
            exp_o = math.exp(G[t, h]) * scale * S0.T @ P["q"][t, h // 2]
            np.testing.assert_allclose(o[t, h], exp_o, rtol=1e-11, atol=1e-14)
    oc, Sc = orc.chunked(**P, chunk=4)
    np.testing.assert_allclose(oc, o, rtol=1e-11, atol=1e-14)
    np.testing.assert_allclose(Sc, S, rtol=1e-11, atol=1e-14)


def pin_orthonormal_retrieval(orc):
    """a = b = 1, orthonormal keys k_1..k_d: every written value is retrieved
    under its key (S_T^T k_i = v_i), and writing a full basis overwrites any
    initial state: S_T = sum_i k_i v_i^T."""
    d_k, d_v = 6, 4
    Qm, _ = np.linalg.qr(RNG.standard_normal((d_k, d_k)))
    keys = Qm.T.astype(np.float32)  # rows orthonormal (to fp32 rounding)
    v = RNG.standard_normal((d_k, 1, d_v)).astype(np.float32)
    k = keys[:, None, :]
    q = keys[:, None, :]
    g = np.zeros((d_k, 1), dtype=np.float32)
    b = np.ones((d_k, 1), dtype=np.float32)
    S0 = RNG.standard_normal((1, 1, d_k, d_v)).astype(np.float32)
    for fn in (orc.recurrent, lambda *a, **kw: orc.chunked(*a, chunk=4, **kw)):
        o, S = fn(q, k, v, g, b, h0=S0, scale=1.0)
        K64 = keys.astype(np.float64)
        np.testing.assert_allclose(S[0, 0].T @ K64.T, v[:, 0, :].T, atol=2e-6)
        np.testing.assert_allclose(S[0, 0], K64.T @ v[:, 0, :].astype(np.float64), atol=2e-6)
        # the last write is also read back at its own step
        np.testing.assert_allclose(o[-1, 0], v[-1, 0], atol=2e-6)


def pin_same_key_twice(orc):
    """a = b = 1, the same unit key written twice: one corrected note.
    S_2 = S_0 + k (v_2 - S_0^T k)^T, so S_2^T k = v_2 and v_1 left no trace."""
    d_k, d_v = 5, 3
    kk = RNG.standard_normal(d_k)
    kk /= np.linalg.norm(kk)
    kk = kk.astype(np.float32)
    v = RNG.standard_normal((2, 1, d_v)).astype(np.float32)
    S0 = RNG.standard_normal((1, 1, d_k, d_v)).astype(np.float32)
    k = np.stack([kk, kk])[:, None, :]
    q = RNG.standard_normal((2, 1, d_k)).astype(np.float32)
    g = np.zeros((2, 1), dtype=np.float32)
    b = np.ones((2, 1), dtype=np.float32)
    o, S = orc.recurrent(q, k, v, g, b, h0=S0, scale=1.0)
    k64 = kk.astype(np.float64)
    S0d = S0[0, 0].astype(np.float64)
    exp_S = S0d + np.outer(k64, v[1, 0] - S0d.T @ k64)
    np.testing.assert_allclose(S[0, 0], exp_S, atol=1e-6)
    np.testing.assert_allclose(S[0, 0].T @ k64, v[1, 0], atol=1e-6)


def pin_linearity(orc):
    """For fixed q, k, g, b the outputs and final state are linear in (V, S0)."""
    P1 = _rand_problem(seed=11)
    P2 = _rand_problem(seed=12)
    for key in ("q", "k", "g", "beta"):
        P2[key] = P1[key]
    c1, c2 = 0.75, -1.25
    P3 = dict(P1)
    P3["v"] = (c1 * P1["v"].astype(np.float64) + c2 * P2["v"]).astype(np.float32)
    P3["h0"] = (c1 * P1["h0"].astype(np.float64) + c2 * P2["h0"]).astype(np.float32)
    # rounding of the combination to fp32 is the only source of difference
    o1, S1 = orc.recurrent(**P1)
    o2, S2 = orc.recurrent(**P2)
    o3, S3 = orc.recurrent(**P3)
    np.testing.assert_allclose(o3, c1 * o1 + c2 * o2, atol=5e-6)
    np.testing.assert_allclose(S3, c1 * S1 + c2 * S2, atol=5e-6)


def pin_gqa_grouping(orc):
    """H_v = 2 H_qk equals a run with q/k heads repeated so that v-head h reads
    q/k head h // 2 (contiguous groups)."""
    P = _rand_problem(total=17, h_qk=2, h_v=4, seed=21)
    o, S = orc.recurrent(**P)
    R = dict(P)
    R["q"] = np.repeat(P["q"], 2, axis=1)
    R["k"] = np.repeat(P["k"], 2, axis=1)
    o2, S2 = orc.recurrent(**R)
    np.testing.assert_allclose(o, o2, rtol=1e-13, atol=1e-15)
    np.testing.assert_allclose(S, S2, rtol=1e-13, atol=1e-15)


def pin_packing_and_resume(orc):
    """Packed sequences (cu_seqlens) equal separate runs, and a sequence split
    in two, with the first part's final state as the second's initial state,
    equals the whole run (the state is the whole carried context)."""
    lens = [5, 1, 12, 9]
    P = _rand_problem(total=sum(lens), lengths=lens, seed=31)
    o, S = orc.recurrent(**P)
    cu = P["cu_seqlens"]
    for n, L in enumerate(lens):
        a, b = cu[n], cu[n + 1]
        one = {key: P[key][a:b] for key in ("q", "k", "v", "g", "beta")}
        o1, S1 = orc.recurrent(**one, h0=P["h0"][n:n + 1])
        np.testing.assert_allclose(o[a:b], o1, rtol=1e-13, atol=1e-15)
        np.testing.assert_allclose(S[n], S1[0], rtol=1e-13, atol=1e-15)
        if L >= 4:
            m = L // 2
            first = {key: P[key][a:a + m] for key in ("q", "k", "v", "g", "beta")}
            second = {key: P[key][a + m:b] for key in ("q", "k", "v", "g", "beta")}
            oa, Sa = orc.recurrent(**first, h0=P["h0"][n:n + 1])
            ob, Sb = orc.recurrent(**second, h0=Sa.astype(np.float32))
            np.testing.assert_allclose(np.concatenate([oa, ob]), o[a:b], atol=1e-6)
            np.testing.assert_allclose(Sb[0], S[n], atol=1e-6)


def pin_chunked_equals_recurrent(orc):
    """The chunkwise algebra reproduces the token-by-token rule for every chunk
    size, including ragged last chunks and packed sequences."""
    lens = [23, 1, 40, 7]
    P = _rand_problem(total=sum(lens), lengths=lens, seed=41)
    o, S = orc.recurrent(**P)
    for C in (1, 2, 3, 16, 64):
        oc, Sc = orc.chunked(**P, chunk=C)
        np.testing.assert_allclose(oc, o, rtol=1e-9, atol=1e-12)
        np.testing.assert_allclose(Sc, S, rtol=1e-9, atol=1e-12)


def pin_fast_decay_chunks(orc):
    """Very fast decay (g = -12 per token, cumulative log-decay down to -768
    in a chunk of 64): the chunked form stays finite and equal to the rule."""
    P = _rand_problem(total=70, seed=51)
    P["g"][:] = -12.0
    o, S = orc.recurrent(**P)
    oc, Sc = orc.chunked(**P, chunk=64)
    assert np.isfinite(oc).all() and np.isfinite(Sc).all()
    np.testing.assert_allclose(oc, o, rtol=1e-9, atol=1e-12)
    np.testing.assert_allclose(Sc, S, rtol=1e-9, atol=1e-12)


def pin_default_scale(orc):
    """scale defaults to 1/sqrt(d_k) and multiplies only the output."""
    P = _rand_problem(total=9, d_k=9, seed=61)
    o, S = orc.recurrent(**P)
    o1, S1 = orc.recurrent(**P, scale=1.0)
    np.testing.assert_allclose(o, o1 / 3.0, rtol=1e-13)
    np.testing.assert_allclose(S, S1, rtol=0, atol=0)


def pin_value_columns_separate(orc):
    """Column j of the state evolves on its own (u_j = beta (v_j - alpha
    (S^T k)_j), S_:j <- alpha S_:j + k u_j): running the rule on a slice of
    the value columns (v and S_0 restricted to it) gives that slice of the
    outputs and final states, in both forms. This is what lets a kernel
    split d_v across CTAs."""
    lens = [9, 14]
    P = _rand_problem(total=sum(lens), lengths=lens, d_v=7, seed=71)
    o, S = orc.recurrent(**P)
    oc, Sc = orc.chunked(**P, chunk=4)
    for js in (slice(0, 3), slice(3, 7), slice(5, 6)):
        Q = dict(P, v=np.ascontiguousarray(P["v"][..., js]), h0=np.ascontiguousarray(P["h0"][..., js]))
        o1, S1 = orc.recurrent(**Q)
        np.testing.assert_allclose(o1, o[..., js], rtol=1e-13, atol=1e-14)
        np.testing.assert_allclose(S1, S[..., js], rtol=1e-13, atol=1e-14)
        o2, S2 = orc.chunked(**Q, chunk=4)
        np.testing.assert_allclose(o2, oc[..., js], rtol=1e-11, atol=1e-13)
        np.testing.assert_allclose(S2, Sc[..., js], rtol=1e-11, atol=1e-13)


PINS = [pin_hand_example, pin_literal_matrix_form, pin_beta_zero_closed_form,
        pin_orthonormal_retrieval, pin_same_key_twice, pin_linearity, pin_gqa_grouping,
        pin_packing_and_resume, pin_chunked_equals_recurrent, pin_fast_decay_chunks,
        pin_default_scale, pin_value_columns_separate]


class _Module:
    recurrent = staticmethod(oracle.recurrent)
    chunked = staticmethod(oracle.chunked)


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(_Module)


def test_bf16_inputs_upcast_exactly():
    """bf16 q/k/v are upcast element by element: the result equals feeding the
    same values already widened to fp32, bit for bit."""
    P = _rand_problem(total=15, seed=71)
    Pb = dict(P)
    for key in ("q", "k", "v"):
        Pb[key] = torch.from_numpy(P[key]).to(torch.bfloat16)
    Pf = dict(Pb)
    for key in ("q", "k", "v"):
        Pf[key] = Pb[key].to(torch.float32)
    o_b, S_b = oracle.recurrent(**Pb)
    o_f, S_f = oracle.recurrent(**Pf)
    assert np.array_equal(o_b, o_f) and np.array_equal(S_b, S_f)


def test_pairs_subset_matches_full():
    lens = [6, 11]
    P = _rand_problem(total=17, lengths=lens, seed=81)
    o, S = oracle.recurrent(**P)
    os_, Ss = oracle.recurrent(**P, pairs=[(1, 3), (0, 2)])
    np.testing.assert_array_equal(os_[0], o[6:17, 3])
    np.testing.assert_array_equal(Ss[1], S[0, 2])


def test_decode_steps_helper():
    """decode_steps runs one token per step per sequence through the rule."""
    import gdn_inputs
    d = gdn_inputs.make_decode(num_seqs=3, h_qk=1, h_v=2, d_k=4, d_v=3, steps=5, dtype="f32")
    o, S = oracle.decode_steps(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state"])
    st = d["state"].double().numpy().copy()
    for t in range(5):
        for n in range(3):
            oo, SS = oracle.recurrent(d["q"][t, n:n + 1], d["k"][t, n:n + 1], d["v"][t, n:n + 1],
                                      d["g"][t, n:n + 1], d["beta"][t, n:n + 1],
                                      h0=st[n:n + 1].astype(np.float32))
            np.testing.assert_allclose(o[t, n], oo[0], atol=1e-6)
            st[n] = SS[0]
    np.testing.assert_allclose(S, st, atol=1e-6)


def test_rejects_bad_arguments():
    P = _rand_problem(total=4, h_qk=3, h_v=4, seed=5)  # H_v not a multiple of H_qk
    with pytest.raises(ValueError):
        oracle.recurrent(**P)


# ----------------------------------------------------------------------------
# planted mistakes: each edit of the oracle's source must fail at least one pin
# ----------------------------------------------------------------------------

MUTANTS = {
    "read_without_decay": ("err[j] = vv[j] - alpha * read;", "err[j] = vv[j] - read;"),
    "error_sign": ("err[j] = vv[j] - alpha * read;", "err[j] = vv[j] + alpha * read;"),
    "write_without_beta": ("+ beta * kk[i] * err[j];", "+ kk[i] * err[j];"),
    "state_not_decayed": ("= alpha * S[(size_t)i * dv + j] + beta", "= S[(size_t)i * dv + j] + beta"),
    "no_output_scale": ("orow[j] = P->scale * acc;", "orow[j] = acc;"),
    "read_with_query": ("read += S[(size_t)i * dv + j] * kk[i];", "read += S[(size_t)i * dv + j] * qq[i];"),
    "output_before_write": ("/* S = alpha S + beta k error^T */",
                            "for (int j = 0; j < dv; ++j) { double acc = 0.0; for (int i = 0; i < dk; ++i) acc += S[(size_t)i * dv + j] * qq[i]; o[(size_t)(t - t0) * dv + j] = P->scale * acc; } continue;"),
    "gqa_interleaved": ("hk = h / grp;\n    double* kv", "hk = h % P->h_qk;\n    double* kv"),
    "log_decay_sign": ("double alpha = exp((double)P->g", "double alpha = exp(-(double)P->g"),
    "initial_state_ignored": ("if (!P->h0) { memset", "if (1) { memset"),
    "chunk_A_without_decay": ("a = B[r] * exp(G[r] - G[s]) * dot;", "a = B[r] * dot;"),
    "chunk_A_without_beta": ("a = B[r] * exp(G[r] - G[s]) * dot;", "a = exp(G[r] - G[s]) * dot;"),
    "chunk_mask_strict": ("for (int s = 0; s <= r; ++s) {", "for (int s = 0; s < r; ++s) {"),
    "chunk_state_gamma_first": ("double gl = gam[L - 1];", "double gl = gam[0];"),
    "chunk_W_without_gamma": ("B[s] * gam[s] * K[(size_t)s * dk + i];", "B[s] * K[(size_t)s * dk + i];"),
    "chunk_query_gamma_missing": ("OO[(size_t)r * dv + j] = gam[r] * qs;", "OO[(size_t)r * dv + j] = qs;"),
}


def _build_mutant(src_text, tmpdir, name):
    c = os.path.join(tmpdir, f"{name}.c")
    so = os.path.join(tmpdir, f"{name}.so")
    with open(c, "w") as f:
        f.write(src_text)
    subprocess.run(["gcc", "-O1", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-o", so, c, "-lm"],
                   check=True, capture_output=True)
    return oracle.load_variant(so)


def test_planted_mistakes_are_caught():
    src_path = os.path.join(os.path.dirname(oracle.__file__), "gdn_oracle.c")
    with open(src_path) as f:
        src = f.read()
    tmp = tempfile.mkdtemp(prefix="gdn_mut_")
    try:
        survivors = []
        for name, (old, new) in MUTANTS.items():
            assert src.count(old) >= 1, f"mutation site for {name} not found"
            orc = _build_mutant(src.replace(old, new, 1), tmp, name)
            caught = False
            for pin in PINS:
                try:
                    pin(orc)
                except (AssertionError, ValueError):
                    caught = True
                    break
            if not caught:
                survivors.append(name)
        assert not survivors, f"pins missed planted mistakes: {survivors}"
    finally:
        shutil.rmtree(tmp, ignore_errors=True)
