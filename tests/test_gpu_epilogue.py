"""GPU parity of the output epilogue (gdn_gated_rmsnorm) and of the decode step
with the epilogue fused (gdn_decode_step_gated) against the fp64 oracle,
through the C ABI.

Tolerances (see gdn_testutil): the standalone epilogue sees exactly the
oracle's inputs and computes in fp32, so it is held to tau = 1e-4 x RMS (with
one bf16 ulp added when it writes bf16). The gated decode inherits the decode
bound (2e-2 x RMS for bf16 q/k/v, 1e-4 for fp32).
"""
import numpy as np
import pytest
import torch

import gdn_inputs
import oracle
import gated_deltanet_recurrence_05_b300 as gdn
from gdn_testutil import TAU_BF16, TAU_F32, assert_parity, to_cuda

pytestmark = pytest.mark.gpu

_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def _inputs(rows, d, dtype, seed, weight=True, scale=1.0):
    g = torch.Generator().manual_seed(seed)
    x = (torch.randn(rows, d, generator=g) * scale).to(_DT[dtype])
    z = (torch.randn(rows, d, generator=g) * 2.0).to(_DT[dtype])
    w = (torch.randn(d, generator=g) * 0.3) if weight else None
    return x, z, w


@pytest.mark.parametrize("dx", ["f32", "bf16"])
@pytest.mark.parametrize("dy", ["f32", "bf16"])
@pytest.mark.parametrize("d", [128, 64, 200, 1024, 5])
def test_gated_rmsnorm_parity(dx, dy, d):
    rows = 257  # not a multiple of the 8 rows of a CTA
    x, z, w = _inputs(rows, d, dx, seed=d + 7 * len(dx + dy))
    y = gdn.gated_rmsnorm(x.cuda(), z.cuda(), None if w is None else w.cuda(), eps=1e-6,
                          output_dtype=_DT[dy])
    assert gdn.get_device_error() == 0
    ref = oracle.gated_rmsnorm(x, z, w, eps=1e-6)
    assert_parity(y.float().cpu().numpy(), ref, TAU_F32, "y", out_bf16=(dy == "bf16"))


def test_gated_rmsnorm_in_place_and_no_weight():
    x, z, _ = _inputs(1000, 128, "bf16", seed=3, weight=False)
    ref = oracle.gated_rmsnorm(x, z, None, eps=1e-5)
    xd = x.cuda()
    y = gdn.gated_rmsnorm(xd, z.cuda(), None, eps=1e-5, out=xd)
    assert y.data_ptr() == xd.data_ptr()
    assert_parity(xd.float().cpu().numpy(), ref, TAU_F32, "y", out_bf16=True)


def test_gated_rmsnorm_edges():
    """A zero row stays zero (eps > 0), saturated gates give exactly 0 / the
    plain norm, a tiny-scale row is normalised like any other."""
    d = 128
    x = torch.randn(4, d)
    x[0] = 0.0
    x[3] *= 1e-20
    z = torch.zeros(4, d)
    z[1] = -100.0
    z[2] = 100.0
    y = gdn.gated_rmsnorm(x.cuda(), z.cuda(), None, eps=1e-6).cpu().numpy()
    assert np.all(y[0] == 0.0)
    assert np.all(y[1] == 0.0)
    np.testing.assert_allclose(np.mean(y[2].astype(np.float64) ** 2), 1.0 / (1.0 + 1e-6 / np.mean(
        x[2].double().numpy() ** 2)), rtol=1e-5)
    ref = oracle.gated_rmsnorm(x, z, None, eps=1e-6)
    np.testing.assert_allclose(y[3], ref[3], rtol=0, atol=1e-5 * np.sqrt(np.mean(ref[3] ** 2)) + 1e-30)
    empty = torch.empty(0, d, device="cuda")
    assert gdn.gated_rmsnorm(empty, empty.clone(), None).numel() == 0


def test_gated_rmsnorm_prefill_output_shape():
    """The epilogue on a prefill output of the benchmark's shape ([16384, 32,
    128] bf16, the launch configuration bench.py times); sampled rows are
    checked against the oracle."""
    T, H, d = 16384, 32, 128
    g = torch.Generator().manual_seed(11)
    x = torch.randn(T, H, d, generator=g).to(torch.bfloat16)
    z = torch.randn(T, H, d, generator=g).to(torch.bfloat16)
    w = torch.randn(d, generator=g) * 0.2
    y = gdn.gated_rmsnorm(x.cuda(), z.cuda(), w.cuda(), eps=1e-6)
    assert gdn.get_device_error() == 0
    rng = np.random.default_rng(0)
    ts = rng.integers(0, T, 512)
    hs = rng.integers(0, H, 512)
    ref = oracle.gated_rmsnorm(x[ts, hs], z[ts, hs], w, eps=1e-6)
    assert_parity(y[ts, hs].float().cpu().numpy(), ref, TAU_F32, "y", out_bf16=True)


def _gated_decode(d, steps, out_dtype, seed, weight=True):
    dd = to_cuda(d)
    N, h_v, d_v = d["v"].shape[1], d["v"].shape[2], d["v"].shape[3]
    gen = torch.Generator().manual_seed(seed)
    zs = (torch.randn(steps, N, h_v, d_v, generator=gen) * 2.0).to(d["q"].dtype)
    w = torch.randn(d_v, generator=gen) * 0.3 if weight else None
    state = dd["state"].clone()
    state_plain = dd["state"].clone()
    outs = []
    for t in range(steps):
        outs.append(gdn.decode_step(dd["q"][t], dd["k"][t], dd["v"][t], dd["g"][t], dd["beta"][t], state,
                                    output_dtype=out_dtype, gate=zs[t].cuda(),
                                    norm_weight=None if w is None else w.cuda(), eps=1e-6))
        gdn.decode_step(dd["q"][t], dd["k"][t], dd["v"][t], dd["g"][t], dd["beta"][t], state_plain)
    torch.cuda.synchronize()
    assert gdn.get_device_error() == 0
    # the epilogue does not touch the state
    assert torch.equal(state, state_plain)
    o_ref, S_ref = oracle.decode_steps(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state"])
    y_ref = oracle.gated_rmsnorm(o_ref, zs, w, eps=1e-6)
    return torch.stack(outs).float().cpu().numpy(), y_ref, state.cpu().numpy(), S_ref


@pytest.mark.parametrize("out_bf16", [False, True])
def test_decode_gated_d128(out_bf16):
    d = gdn_inputs.make_decode(num_seqs=6, h_qk=2, h_v=4, d_k=128, d_v=128, steps=5, seed=21)
    y, y_ref, S, S_ref = _gated_decode(d, 5, torch.bfloat16 if out_bf16 else torch.float32, seed=1)
    assert_parity(y, y_ref, TAU_BF16, "gated o", out_bf16=out_bf16)
    assert_parity(S, S_ref, TAU_BF16, "state")


@pytest.mark.parametrize("d_k,d_v", [(32, 16), (64, 96)])
def test_decode_gated_generic_fp32(d_k, d_v):
    d = gdn_inputs.make_decode(num_seqs=3, h_qk=1, h_v=3, d_k=d_k, d_v=d_v, steps=4, dtype="f32", seed=22)
    y, y_ref, S, S_ref = _gated_decode(d, 4, torch.float32, seed=2, weight=False)
    assert_parity(y, y_ref, TAU_F32, "gated o")
    assert_parity(S, S_ref, TAU_F32, "state")
