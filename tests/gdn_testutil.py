"""Shared helpers of the parity tests (no recurrence arithmetic here).

Tolerance rule (per tensor): max |got - ref| <= tau * RMS(ref), with
tau = 1e-4 for fp32 q/k/v and tau = 2e-2 for bf16 q/k/v (fp32 state), applied
to the outputs o and to the final states separately. When o is emitted in
bf16, the reference is rounded to bf16 first and one bf16 ulp of |ref| is
added to the bound (rounding of the output alone can approach the budget).
"""
import numpy as np
import torch

TAU_F32 = 1e-4
TAU_BF16 = 2e-2


def tau_for(dtype: str) -> float:
    return TAU_F32 if dtype == "f32" else TAU_BF16


def rms(x) -> float:
    x = np.asarray(x, dtype=np.float64)
    return float(np.sqrt(np.mean(x * x))) if x.size else 0.0


def max_err_ratio(got, ref, out_bf16=False) -> float:
    """max|got - ref| / (tau-free) RMS(ref), after the bf16 handling above."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    r = rms(ref)
    if out_bf16:
        ref_b = torch.from_numpy(ref).to(torch.bfloat16).double().numpy()
        # one bf16 ulp of |ref_b|: 2^(e - 8) for |x| in [2^(e-1), 2^e) (8 significant bits)
        _, e = np.frexp(np.abs(ref_b))
        ulp = np.ldexp(1.0, e - 8)
        excess = np.maximum(np.abs(got - ref_b) - ulp, 0.0)
        return float(excess.max() / r) if got.size else 0.0
    return float(np.abs(got - ref).max() / r) if got.size else 0.0


def assert_parity(got, ref, tau, label, out_bf16=False):
    e = max_err_ratio(got, ref, out_bf16=out_bf16)
    assert np.isfinite(np.asarray(got, dtype=np.float64)).all(), f"{label}: non-finite values"
    assert e <= tau, f"{label}: max|err| = {e:.3e} x RMS(ref) > {tau:.1e}"
    return e


def to_cuda(d: dict) -> dict:
    out = {}
    for key, val in d.items():
        out[key] = val.cuda() if isinstance(val, torch.Tensor) else val
    return out


def sample_pairs(num_seqs, h_v, count, seed=0, must=()):
    """Deterministic sample of (sequence, value-head) pairs, always including
    the first and last pair and any in ``must``."""
    rng = np.random.default_rng(seed)
    pairs = {(0, 0), (num_seqs - 1, h_v - 1), *must}
    while len(pairs) < min(count, num_seqs * h_v):
        pairs.add((int(rng.integers(num_seqs)), int(rng.integers(h_v))))
    return sorted(pairs)
