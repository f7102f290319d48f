"""GPU parity of gdn_chunk_fwd_gated: the prefill followed by the layer's
output epilogue (zero-centred RMSNorm times a sigmoid gate), run as a second
launch on o after the tensor-core or the CUDA-core prefill kernel.

Two checks per case:
  * against the oracle chain: oracle.recurrent, then oracle.gated_rmsnorm on
    its fp64 output. The prefill's own bound (max|o - o_ref| <= tau RMS(o_ref))
    carries over to y through the epilogue's derivative row by row: for a row
    with rms rho, |dy_j| <= |s_j sig(z_j)| (|do|/rho + |o_j| |o . do| / (d rho^3))
    to first order, so each row is held to that bound (with a factor 1.5 for
    the second-order terms) at |do| = tau RMS(o_ref);
  * against the GPU's own chain: the plain prefill's output put through the
    oracle epilogue. The gated call normalises what the plain call stores
    (fp32, or bf16 for a bf16 output, where y is held to the epilogue's
    tolerance plus the bf16 rounding of the stored o), so the two agree to
    the epilogue's fp32 tolerance (1e-4 of RMS).
"""
import numpy as np
import pytest
import torch

import gdn_inputs
import oracle
import gated_deltanet_recurrence_05_b300 as gdn
from gdn_testutil import TAU_BF16, TAU_F32, assert_parity, to_cuda

pytestmark = pytest.mark.gpu
EPS = 1e-6


def _gate(d, seed, weight=True):
    gen = torch.Generator().manual_seed(seed)
    z = (torch.randn(d["v"].shape, generator=gen) * 2.0).to(d["v"].dtype)
    w = torch.randn(d["v"].shape[-1], generator=gen) * 0.3 if weight else None
    return z, w


def _run(d, z, w, out_dtype=torch.float32, force_simt=False):
    dd = to_cuda(d)
    cu = dd["cu_seqlens"]
    n = None if cu is not None else len(d["lengths"])
    order = gdn.plan_seq_order(d["cu_seqlens"]).cuda() if cu is not None else None
    y, S = gdn.chunk_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["h0"], cu, num_seqs=n,
                         seq_order=order, output_dtype=out_dtype, force_simt=force_simt, gate=z.cuda(),
                         norm_weight=None if w is None else w.cuda(), eps=EPS)
    o, S2 = gdn.chunk_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["h0"], cu, num_seqs=n,
                          seq_order=order, output_dtype=out_dtype, force_simt=force_simt)
    torch.cuda.synchronize()
    assert gdn.get_device_error() == 0
    # the epilogue leaves the state alone (same arithmetic in both kernels)
    assert torch.allclose(S, S2, rtol=0, atol=1e-6 * float(S2.float().pow(2).mean().sqrt()) + 1e-30)
    return y.float().cpu().numpy(), o.float().cpu().numpy(), S.cpu().numpy()


def _check_against_oracle_chain(y, d, z, w, tau, label, y_bf16=False):
    cu = d["cu_seqlens"]
    if cu is None:
        cu = torch.tensor([0] + list(np.cumsum(d["lengths"])), dtype=torch.int32)
    o_ref, S_ref = oracle.recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"], cu_seqlens=cu)
    y_ref = oracle.gated_rmsnorm(o_ref, z, w, eps=EPS)
    dv = o_ref.shape[-1]
    do = tau * float(np.sqrt(np.mean(o_ref * o_ref)))
    rho = np.sqrt(np.mean(o_ref * o_ref, axis=-1) + EPS)                              # per row
    sg = np.abs((1.0 + (np.zeros(dv) if w is None else w.double().numpy())) * oracle.sigmoid(z.double().numpy()))
    amp = np.max(sg, axis=-1) * (1.0 / rho + np.max(np.abs(o_ref), axis=-1) * np.sum(np.abs(o_ref), axis=-1)
                                 / (dv * rho ** 3))
    bound = 1.5 * do * amp
    if y_bf16:  # the bf16 store of y adds half an ulp: at most 2^-8 |y|
        bound = bound + 2.0 ** -8 * np.max(np.abs(y_ref), axis=-1)
    err = np.max(np.abs(y - y_ref), axis=-1)
    assert np.isfinite(y).all(), f"{label}: non-finite"
    worst = float(np.max(err / bound))
    assert worst <= 1.0, f"{label}: a row exceeds its derived bound by {worst:.2f}x"
    return S_ref


@pytest.mark.parametrize("out_bf16", [False, True])
def test_gated_prefill_tensor_core_fused(out_bf16):
    """bf16 q/k/v, d = 128 (tensor-core prefill): ragged lengths incl. 0 and 1, GQA 2:1."""
    d = gdn_inputs.make_prefill(h_qk=2, h_v=4, d_k=128, d_v=128, dtype="bf16",
                                lengths=[300, 1, 0, 64, 65, 191], h0_std=0.02, seed=51)
    z, w = _gate(d, 51)
    y, o, S = _run(d, z, w, torch.bfloat16 if out_bf16 else torch.float32)
    S_ref = _check_against_oracle_chain(y, d, z, w, TAU_BF16, "y", y_bf16=out_bf16)
    assert_parity(S, S_ref, TAU_BF16, "final state")
    y_chain = oracle.gated_rmsnorm(o, z, w, eps=EPS)
    assert_parity(y, y_chain, TAU_F32, "y vs the plain kernel's o + epilogue", out_bf16=out_bf16)


def test_gated_prefill_no_weight_slow_decay():
    d = gdn_inputs.make_prefill(h_qk=1, h_v=2, d_k=128, d_v=128, dtype="bf16", lengths=[700, 129],
                                g_shift=-5.0, h0_std=0.02, seed=52)
    z, _ = _gate(d, 52, weight=False)
    y, o, _ = _run(d, z, None)
    _check_against_oracle_chain(y, d, z, None, TAU_BF16, "y")
    assert_parity(y, oracle.gated_rmsnorm(o, z, None, eps=EPS), TAU_F32, "y vs plain + epilogue")


@pytest.mark.parametrize("force_simt", [True, False])
def test_gated_prefill_chained_cuda_core(force_simt):
    """fp32 inputs (or a forced CUDA-core run): the epilogue runs as a second
    launch on o."""
    if force_simt:
        d = gdn_inputs.make_prefill(h_qk=2, h_v=4, d_k=128, d_v=128, dtype="bf16", lengths=[90, 33],
                                    h0_std=0.02, seed=53)
        tau = TAU_BF16
    else:
        d = gdn_inputs.make_prefill(h_qk=2, h_v=6, d_k=32, d_v=24, dtype="f32", lengths=[70, 1, 0, 129],
                                    h0_std=0.1, seed=53)
        tau = TAU_F32
    z, w = _gate(d, 53)
    y, o, _ = _run(d, z, w, force_simt=force_simt)
    _check_against_oracle_chain(y, d, z, w, tau, "y")
    assert_parity(y, oracle.gated_rmsnorm(o, z, w, eps=EPS), TAU_F32, "y vs plain + epilogue")


def test_gated_prefill_full_prefill_workload():
    """B=4, T=4096, H_qk=16, H_v=32, d=128 (the benchmark's gated line): every
    output row of every (sequence, head) pair."""
    d = gdn_inputs.make_workload("prefill")
    z, w = _gate(d, 54)
    y, o, _ = _run(d, z, w, torch.bfloat16)
    _check_against_oracle_chain(y, d, z, w, TAU_BF16, "y", y_bf16=True)
    assert_parity(y, oracle.gated_rmsnorm(o, z, w, eps=EPS), TAU_F32, "y vs plain + epilogue", out_bf16=True)
