"""Pins of the epilogue oracle (oracle.gated_rmsnorm) against what its
definition fixes.

The epilogue is named by the pages, not written out: "a sigmoid output gate,
zero-centered RMSNorm" added to the gated delta rule ("Qwen3.8-Next design:
hybrid attention, residuals and n-gram embeddings", transcript segment 14) and
the gate sigma(x W_g) (.) o ("Qwen3.8 attention gate", component "Output gate +
sink"). The reading used (see oracle/epilogue.py):

    y = o / sqrt(mean_j o_j^2 + eps) * (1 + w) * sigmoid(z)   per row of d features

Each pin below is a hand-worked example, a closed form of a special case or an
invariant; none re-types the formula. ``test_planted_mistakes`` runs every pin
against plausible wrong readings and checks that each is caught.
"""
import math

import numpy as np
import pytest

import oracle


def _rows(n=5, d=16, seed=0, scale=1.0):
    rng = np.random.default_rng(seed)
    return rng.standard_normal((n, d)) * scale


# ----------------------------------------------------------------------------
# pins: each takes fn(o, z, w, eps) -> y
# ----------------------------------------------------------------------------

def pin_hand_example(fn):
    """One row worked by hand (tests/golden/gated_rmsnorm_hand_example.json):
    o = (3, 4), w = (0, 1), z = (0, ln 3), eps = 0 -> (0.4242640687, 1.6970562748)."""
    import json
    import os
    with open(os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden",
                           "gated_rmsnorm_hand_example.json")) as f:
        G = json.load(f)
    y = fn(np.array(G["o"]), np.array(G["z"]), np.array(G["w"]), G["eps"])
    np.testing.assert_allclose(y, G["y"], rtol=0, atol=G["atol"])


def pin_unit_rms(fn):
    """w = 0, gate fully open (z = 40: sigmoid = 1 - 4e-18), eps = 0: every row
    of the result has mean square exactly 1."""
    o = _rows(7, 24, seed=1, scale=3.0)
    y = fn(o, np.full_like(o, 40.0), None, 0.0)
    np.testing.assert_allclose(np.mean(y * y, axis=-1), 1.0, rtol=0, atol=1e-12)


def pin_eps_closed_form(fn):
    """w = 0, gate open: mean(y^2) = m / (m + eps) with m = mean(o^2)."""
    o = _rows(6, 10, seed=2, scale=0.01)
    eps = 1e-4
    m = np.mean(o * o, axis=-1)
    y = fn(o, np.full_like(o, 40.0), None, eps)
    np.testing.assert_allclose(np.mean(y * y, axis=-1), m / (m + eps), rtol=1e-12, atol=0)


def pin_constant_row(fn):
    """o = c (1, ..., 1) with c = -2.5, d = 7, z = 0, eps = 0: the RMS is |c|, so
    y = sign(c) (1 + w) / 2 exactly."""
    d = 7
    w = np.linspace(-0.5, 0.7, d)
    y = fn(np.full(d, -2.5), np.zeros(d), w, 0.0)
    np.testing.assert_allclose(y, -(1.0 + w) / 2.0, rtol=0, atol=1e-14)


def pin_scale_invariance(fn):
    """eps = 0: y(lambda o) = y(o) for lambda > 0 (a normalisation)."""
    o = _rows(4, 12, seed=3)
    z = _rows(4, 12, seed=4)
    w = np.linspace(-0.3, 0.3, 12)
    np.testing.assert_allclose(fn(37.5 * o, z, w, 0.0), fn(o, z, w, 0.0), rtol=1e-12, atol=1e-14)


def pin_odd(fn):
    """y(-o) = -y(o)."""
    o = _rows(4, 12, seed=5)
    z = _rows(4, 12, seed=6)
    np.testing.assert_allclose(fn(-o, z, None, 1e-6), -fn(o, z, None, 1e-6), rtol=0, atol=1e-14)


def pin_gate_complement(fn):
    """sigmoid(z) + sigmoid(-z) = 1: with w = 0 and eps = 0 the two gated halves
    add up to a row of mean square 1."""
    o = _rows(5, 9, seed=7)
    z = _rows(5, 9, seed=8, scale=3.0)
    s = fn(o, z, None, 0.0) + fn(o, -z, None, 0.0)
    np.testing.assert_allclose(np.mean(s * s, axis=-1), 1.0, rtol=0, atol=1e-12)


def pin_gate_saturation(fn):
    """z = -1000 closes the gate (exactly 0, no overflow); z = +1000 opens it."""
    o = _rows(2, 8, seed=9)
    assert np.all(fn(o, np.full_like(o, -1000.0), None, 1e-6) == 0.0)
    y = fn(o, np.full_like(o, 1000.0), None, 0.0)
    np.testing.assert_allclose(np.mean(y * y, axis=-1), 1.0, rtol=0, atol=1e-12)


def pin_rows_independent(fn):
    """Each row is normalised on its own: a row scaled by 1e3 next to the others
    changes nothing in them ([T, H, d] layout: the mean runs over d only)."""
    o = _rows(6, 8, seed=10).reshape(3, 2, 8)
    z = _rows(6, 8, seed=11).reshape(3, 2, 8)
    o2 = o.copy()
    o2[1, 0] *= 1e3
    y1, y2 = fn(o, z, None, 0.0), fn(o2, z, None, 0.0)
    np.testing.assert_allclose(y1, y2, rtol=1e-12, atol=1e-14)


PINS = [pin_hand_example, pin_unit_rms, pin_eps_closed_form, pin_constant_row, pin_scale_invariance,
        pin_odd, pin_gate_complement, pin_gate_saturation, pin_rows_independent]


def _oracle_fn(o, z, w, eps):
    return oracle.gated_rmsnorm(o, z, w, eps=eps)


@pytest.mark.parametrize("pin", PINS, ids=[p.__name__ for p in PINS])
def test_pin(pin):
    pin(_oracle_fn)


def test_accepts_torch_bf16():
    """bf16 tensors are upcast exactly (the values the GPU sees)."""
    import torch
    o = torch.randn(3, 2, 16).to(torch.bfloat16)
    z = torch.randn(3, 2, 16).to(torch.bfloat16)
    a = oracle.gated_rmsnorm(o, z, None)
    b = oracle.gated_rmsnorm(o.float().numpy().astype(np.float64), z.float().numpy().astype(np.float64), None)
    np.testing.assert_array_equal(a, b)


# ----------------------------------------------------------------------------
# planted mistakes: each plausible wrong reading must fail at least one pin
# ----------------------------------------------------------------------------

def _sig(z):
    return oracle.sigmoid(z)


def _mistake_sum_not_mean(o, z, w, eps):
    o = np.asarray(o, float); y = o / np.sqrt(np.sum(o * o, -1, keepdims=True) + eps)
    return (y * (1 + np.asarray(w)) if w is not None else y) * _sig(z)


def _mistake_eps_outside(o, z, w, eps):
    o = np.asarray(o, float); y = o / (np.sqrt(np.mean(o * o, -1, keepdims=True)) + eps)
    return (y * (1 + np.asarray(w)) if w is not None else y) * _sig(z)


def _mistake_weight_not_centred(o, z, w, eps):
    y = oracle.rms_normalize(o, eps)
    return (y * np.asarray(w) if w is not None else y) * _sig(z)


def _mistake_silu_gate(o, z, w, eps):
    y = oracle.rms_normalize(o, eps)
    y = y * (1 + np.asarray(w)) if w is not None else y
    return y * np.asarray(z, float) * _sig(z)


def _mistake_gate_before_norm(o, z, w, eps):
    y = oracle.rms_normalize(np.asarray(o, float) * _sig(z), eps)
    return y * (1 + np.asarray(w)) if w is not None else y


def _mistake_norm_over_all(o, z, w, eps):
    o = np.asarray(o, float); y = o / np.sqrt(np.mean(o * o) + eps)
    return (y * (1 + np.asarray(w)) if w is not None else y) * _sig(z)


def _mistake_no_square(o, z, w, eps):
    o = np.asarray(o, float); y = o / np.sqrt(np.abs(np.mean(o, -1, keepdims=True)) + eps)
    return (y * (1 + np.asarray(w)) if w is not None else y) * _sig(z)


MISTAKES = [_mistake_sum_not_mean, _mistake_eps_outside, _mistake_weight_not_centred, _mistake_silu_gate,
            _mistake_gate_before_norm, _mistake_norm_over_all, _mistake_no_square]


@pytest.mark.parametrize("wrong", MISTAKES, ids=[m.__name__ for m in MISTAKES])
def test_planted_mistakes(wrong):
    failed = []
    with np.errstate(all="ignore"):
        for pin in PINS:
            try:
                pin(wrong)
            except (AssertionError, ValueError, FloatingPointError):
                failed.append(pin.__name__)
    assert failed, f"no pin catches {wrong.__name__}"
