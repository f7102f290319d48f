"""Pins of the prologue oracle (oracle.short_conv / short_conv_step).

The pages give only "short causal convolutions" added to the gated delta rule
("Qwen3.8-Next design: hybrid attention, residuals and n-gram embeddings",
transcript segment 14); q and k enter the rule L2-normalised. The reading
(oracle/prologue.py): per channel u[t] = sum_i w[i] x[t - (K-1) + i] over the
sequence's own past (the caller's state, else zeros), then silu, then for q
and k an L2 norm per head. Each pin is a hand-worked example, a closed form,
an invariant, or an agreement of the two independent forms (a whole sequence
vs token-by-token steps); ``test_planted_mistakes`` checks each plausible
wrong reading is caught.
"""
import math

import numpy as np
import pytest

import oracle


def _x(T, C, seed):
    return np.random.default_rng(seed).standard_normal((T, C))


# pins take (conv, step) callables with the oracle's signatures

def pin_hand_example(conv, step):
    """One channel worked by hand (tests/golden/short_conv_hand_example.json):
    K = 3, w = (0.5, -1, 2), x = (1, 2, 3), no activation -> u = (2, 3, 4.5),
    final state (2, 3)."""
    import json
    import os
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                           "short_conv_hand_example.json")) as f:
        G = json.load(f)
    y, st = conv(np.array(G["x"])[:, None], np.array([G["w"]]), None, None, None, 0)
    np.testing.assert_allclose(y[:, 0], G["u"], rtol=0, atol=G["atol"])
    np.testing.assert_allclose(st[0, 0], G["state_final"], rtol=0, atol=0)


def pin_silu_values(conv, step):
    """Identity filter (only the current-token tap): y = silu(x); silu(0) = 0,
    silu(1) = 1 / (1 + e^-1) = 0.7310585786300049, silu(-1) = -0.2689414213699951."""
    w = np.array([[0.0, 0.0, 0.0, 1.0]])
    y, _ = conv(np.array([[0.0], [1.0], [-1.0]]), w, None, None, "silu", 0)
    np.testing.assert_allclose(y[:, 0], [0.0, 0.7310585786300049, -0.2689414213699951], rtol=0, atol=1e-15)


def pin_delay_and_sequence_start(conv, step):
    """Oldest-tap filter: y[t] = x[t - 3] inside each sequence, 0 for its first
    three tokens (zero past), no leak across packed sequences."""
    K, C = 4, 5
    w = np.zeros((C, K)); w[:, 0] = 1.0
    x = _x(13, C, 1)
    cu = np.array([0, 2, 9, 13])
    y, _ = conv(x, w, cu, None, None, 0)
    for a, b in zip(cu[:-1], cu[1:]):
        for t in range(a, b):
            want = x[t - 3] if t - 3 >= a else np.zeros(C)
            np.testing.assert_allclose(y[t], want, rtol=0, atol=0)


def pin_linearity(conv, step):
    """Without the activation the filter is linear in x (and in the state)."""
    C, K = 6, 4
    w = _x(C, K, 2)
    x1, x2 = _x(9, C, 3), _x(9, C, 4)
    s1, s2 = _x(C * (K - 1), 1, 5).reshape(1, C, K - 1), _x(C * (K - 1), 1, 6).reshape(1, C, K - 1)
    y1, _ = conv(x1, w, None, s1, None, 0)
    y2, _ = conv(x2, w, None, s2, None, 0)
    y3, _ = conv(2.0 * x1 - 3.0 * x2, w, None, 2.0 * s1 - 3.0 * s2, None, 0)
    np.testing.assert_allclose(y3, 2.0 * y1 - 3.0 * y2, rtol=1e-12, atol=1e-12)


def pin_unit_heads(conv, step):
    """norm_group = 8, eps = 0: each head of each token has unit L2 norm."""
    C, K = 24, 4
    y, _ = conv(_x(7, C, 7), _x(C, K, 8), None, None, "silu", 8, 0.0)
    n = np.sqrt(np.sum(y.reshape(7, 3, 8) ** 2, axis=-1))
    np.testing.assert_allclose(n, 1.0, rtol=0, atol=1e-12)


def pin_state_continuation(conv, step):
    """Splitting a sequence and passing the final state on gives the same
    output as one pass (including a piece shorter than K - 1)."""
    C, K = 5, 4
    w = _x(C, K, 9)
    x = _x(11, C, 10)
    s0 = _x(C * 3, 1, 11).reshape(1, C, 3)
    y_all, st_all = conv(x, w, None, s0, "silu", 0)
    ya, sa = conv(x[:2], w, None, s0, "silu", 0)
    yb, sb = conv(x[2:], w, None, sa, "silu", 0)
    np.testing.assert_allclose(np.concatenate([ya, yb]), y_all, rtol=1e-13, atol=1e-13)
    np.testing.assert_allclose(sb, st_all, rtol=0, atol=0)


def pin_steps_equal_sequence(conv, step):
    """Token-by-token decode steps reproduce the whole-sequence filter."""
    N, C, K, T = 3, 8, 4, 6
    w = _x(C, K, 12)
    xs = np.random.default_rng(13).standard_normal((T, N, C))
    s0 = np.random.default_rng(14).standard_normal((N, C, K - 1))
    st = s0.copy()
    ys = []
    for t in range(T):
        y, st = step(xs[t], w, st, "silu", 4)
        ys.append(y)
    # whole sequences: tokens of sequence n are xs[:, n]
    x_packed = xs.transpose(1, 0, 2).reshape(N * T, C)
    cu = np.arange(N + 1) * T
    y_seq, st_seq = conv(x_packed, w, cu, s0, "silu", 4)
    np.testing.assert_allclose(np.stack(ys).transpose(1, 0, 2).reshape(N * T, C), y_seq, rtol=1e-12, atol=1e-12)
    np.testing.assert_allclose(st, st_seq, rtol=0, atol=0)


PINS = [pin_hand_example, pin_silu_values, pin_delay_and_sequence_start, pin_linearity, pin_unit_heads,
        pin_state_continuation, pin_steps_equal_sequence]


def _conv(x, w, cu, s0, act, ng, eps=1e-6):
    return oracle.short_conv(x, w, cu_seqlens=cu, state0=s0, activation=act, norm_group=ng, eps=eps)


def _step(x, w, st, act, ng, eps=1e-6):
    return oracle.short_conv_step(x, w, st, activation=act, norm_group=ng, eps=eps)


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(_conv, _step)


# ---------------------------------------------------------------- planted mistakes

def _conv_flipped_taps(x, w, cu, s0, act, ng, eps=1e-6):
    return _conv(x, np.asarray(w)[:, ::-1], cu, s0, act, ng, eps)


def _conv_leaks_across_sequences(x, w, cu, s0, act, ng, eps=1e-6):
    y, st = _conv(x, w, None, None if s0 is None else np.asarray(s0)[:1], act, ng, eps)
    N = 1 if cu is None else len(cu) - 1
    return y, np.repeat(st, N, axis=0)


def _conv_norm_before_silu(x, w, cu, s0, act, ng, eps=1e-6):
    y, st = _conv(x, w, cu, s0, None, ng, eps)
    return (oracle.silu(y) if act == "silu" else y), st


def _conv_sigmoid_not_silu(x, w, cu, s0, act, ng, eps=1e-6):
    y, st = _conv(x, w, cu, s0, None, 0, eps)
    if act == "silu":
        y = oracle.sigmoid(y)
    return (oracle.l2_normalize_groups(y, ng, eps) if ng else y), st


def _conv_norm_all_channels(x, w, cu, s0, act, ng, eps=1e-6):
    y, st = _conv(x, w, cu, s0, act, 0, eps)
    return (oracle.l2_normalize_groups(y, y.shape[-1], eps) if ng else y), st


def _conv_state_not_shifted(x, w, cu, s0, act, ng, eps=1e-6):
    y, st = _conv(x, w, cu, s0, act, ng, eps)
    return y, (np.zeros_like(st) if s0 is None else np.asarray(s0, float))


MISTAKES = [_conv_flipped_taps, _conv_leaks_across_sequences, _conv_norm_before_silu, _conv_sigmoid_not_silu,
            _conv_norm_all_channels, _conv_state_not_shifted]


@pytest.mark.parametrize("wrong", MISTAKES, ids=[m.__name__ for m in MISTAKES])
def test_planted_mistakes(wrong):
    failed = []
    with np.errstate(all="ignore"):
        for pin in PINS:
            try:
                pin(wrong, _step)
            except (AssertionError, ValueError, IndexError):
                failed.append(pin.__name__)
    assert failed, f"no pin catches {wrong.__name__}"
