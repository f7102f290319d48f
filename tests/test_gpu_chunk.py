"""GPU parity of gdn_chunk_fwd (prefill) against the fp64 oracle.

Small cases are compared element by element over every output; the full-size
workloads are run in the launch configuration the benchmark uses and
compared on sampled (sequence, value-head) pairs that the oracle replays one
by one.
"""
import numpy as np
import pytest
import torch

import gdn_inputs
import oracle
import gated_deltanet_recurrence_05_b300 as gdn
from gdn_testutil import TAU_BF16, TAU_F32, assert_parity, sample_pairs, tau_for, to_cuda

pytestmark = pytest.mark.gpu


def _gpu(d, out_dtype=torch.float32, force_simt=False, chunk=0, final=True, order=None):
    dd = to_cuda(d)
    cu = dd["cu_seqlens"]
    o, S = gdn.chunk_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["h0"], cu,
                         num_seqs=None if cu is not None else len(d["lengths"]),
                         output_dtype=out_dtype, chunk_size=chunk, force_simt=force_simt,
                         output_final_state=final, seq_order=order)
    torch.cuda.synchronize()
    assert gdn.get_device_error() == 0
    return o.float().cpu().numpy(), None if S is None else S.cpu().numpy()


def _ref(d):
    return oracle.recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"],
                            cu_seqlens=d["cu_seqlens"] if d["cu_seqlens"] is not None else
                            torch.tensor([0] + list(np.cumsum(d["lengths"])), dtype=torch.int32))


def test_tiny_fp32_chunk16():
    """The tiny fp32 workload: B=1, T=64, 2 heads, d=16, chunk 16, tau = 1e-4."""
    d = gdn_inputs.make_workload("tiny")
    o, S = _gpu(d, chunk=16)
    o_ref, S_ref = _ref(d)
    assert_parity(o, o_ref, TAU_F32, "o")
    assert_parity(S, S_ref, TAU_F32, "final state")


@pytest.mark.parametrize("chunk", [16, 32, 64])
def test_fp32_varlen_gqa_chunks(chunk):
    d = gdn_inputs.make_prefill(h_qk=2, h_v=6, d_k=32, d_v=24, dtype="f32",
                                lengths=[70, 1, 0, 129, 64, 3], h0_std=0.1, seed=11)
    o, S = _gpu(d, chunk=chunk)
    o_ref, S_ref = _ref(d)
    assert_parity(o, o_ref, TAU_F32, "o")
    assert_parity(S, S_ref, TAU_F32, "final state")


@pytest.mark.parametrize("force_simt", [False, True])
def test_bf16_d128_varlen_edges(force_simt):
    """bf16 inputs, d=128 (tensor-core kernel unless forced onto CUDA cores):
    ragged lengths incl. 1 and 0, GQA 2:1, nonzero initial states, several
    chunks per sequence."""
    d = gdn_inputs.make_prefill(h_qk=2, h_v=4, d_k=128, d_v=128, dtype="bf16",
                                lengths=[300, 1, 0, 64, 65, 191], h0_std=0.02, seed=12)
    o, S = _gpu(d, force_simt=force_simt)
    o_ref, S_ref = _ref(d)
    assert_parity(o, o_ref, TAU_BF16, "o")
    assert_parity(S, S_ref, TAU_BF16, "final state")


def test_bf16_slow_decay_long_memory():
    """g = -softplus(N(0,1) - 5) (alpha ~ 0.99): the initial state and early
    tokens stay visible across many chunks."""
    d = gdn_inputs.make_prefill(h_qk=1, h_v=2, d_k=128, d_v=128, dtype="bf16",
                                lengths=[1000, 517], g_shift=-5.0, h0_std=0.02, seed=13)
    o, S = _gpu(d)
    o_ref, S_ref = _ref(d)
    assert_parity(o, o_ref, TAU_BF16, "o")
    assert_parity(S, S_ref, TAU_BF16, "final state")


def test_bf16_output_dtype():
    d = gdn_inputs.make_prefill(h_qk=2, h_v=4, d_k=128, d_v=128, dtype="bf16",
                                lengths=[200, 77], h0_std=0.02, seed=14)
    o, S = _gpu(d, out_dtype=torch.bfloat16)
    o_ref, S_ref = _ref(d)
    assert_parity(o, o_ref, TAU_BF16, "o (bf16)", out_bf16=True)
    assert_parity(S, S_ref, TAU_BF16, "final state")


def test_beta_zero_and_no_final_state():
    """beta = 0: pure decay of the initial state (closed form checked by the
    oracle pins); also exercises output_final_state=False."""
    d = gdn_inputs.make_prefill(h_qk=2, h_v=4, d_k=128, d_v=128, dtype="bf16",
                                lengths=[130, 70], h0_std=0.5, seed=15)
    d["beta"].zero_()
    o, S = _gpu(d, final=False)
    assert S is None
    o_ref, _ = _ref(d)
    assert_parity(o, o_ref, TAU_BF16, "o")


def test_in_place_final_state_and_resume():
    """final_state may alias initial_state; running a sequence in two parts
    with the state handed over equals the whole run."""
    d = gdn_inputs.make_prefill(h_qk=2, h_v=4, d_k=128, d_v=128, dtype="bf16",
                                lengths=[256], h0_std=0.02, seed=16)
    dd = to_cuda(d)
    state = dd["h0"].clone()
    outs = []
    for a, b in ((0, 100), (100, 256)):
        o, _ = gdn.chunk_fwd(dd["q"][a:b], dd["k"][a:b], dd["v"][a:b], dd["g"][a:b],
                             dd["beta"][a:b], state, output_dtype=torch.float32,
                             final_state_out=state)
        outs.append(o)
    torch.cuda.synchronize()
    o_ref, S_ref = _ref(d)
    assert_parity(torch.cat(outs).cpu().numpy(), o_ref, TAU_BF16, "o")
    assert_parity(state.cpu().numpy(), S_ref, TAU_BF16, "final state")


def test_simt_equals_tensor_core_kernel():
    """The fp32 CUDA-core kernel and the tensor-core kernel agree on the same
    bf16 inputs within the bf16 tolerance."""
    d = gdn_inputs.make_prefill(h_qk=2, h_v=4, d_k=128, d_v=128, dtype="bf16",
                                lengths=[333, 128], h0_std=0.02, seed=17)
    o1, S1 = _gpu(d, force_simt=True)
    o2, S2 = _gpu(d)
    assert_parity(o2, o1, TAU_BF16, "o")
    assert_parity(S2, S1, TAU_BF16, "final state")


def test_seq_order_permutation_is_transparent():
    d = gdn_inputs.make_prefill(h_qk=2, h_v=4, d_k=128, d_v=128, dtype="bf16",
                                lengths=[40, 300, 5, 129], h0_std=0.02, seed=18)
    order = gdn.plan_seq_order(d["cu_seqlens"]).cuda()
    o1, S1 = _gpu(d)
    o2, S2 = _gpu(d, order=order)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(S1, S2)


def test_bad_cu_seqlens_reported_on_device():
    """An out-of-range cu_seqlens entry is caught by the kernel's own bounds
    check (the unit is skipped, nothing is read out of bounds) and reported
    through gdn_get_device_error."""
    d = gdn_inputs.make_prefill(h_qk=1, h_v=2, d_k=128, d_v=128, dtype="bf16",
                                lengths=[64, 64], seed=19)
    dd = to_cuda(d)
    bad = torch.tensor([0, 64, 4096], dtype=torch.int32, device="cuda")
    gdn.chunk_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], None, bad)
    assert gdn.get_device_error() & 1
    assert gdn.get_device_error() == 0  # cleared


def _full_size(name, n_pairs, seed):
    d = gdn_inputs.make_workload(name)
    cu = d["cu_seqlens"]
    order = gdn.plan_seq_order(cu).cuda() if cu is not None else None
    o, S = _gpu(d, order=order)
    N = len(d["lengths"])
    if cu is None:
        cu = torch.tensor([0] + list(np.cumsum(d["lengths"])), dtype=torch.int32)
    pairs = sample_pairs(N, d["h_v"], n_pairs, seed=seed)
    o_ref, S_ref = oracle.recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"],
                                    cu_seqlens=cu, pairs=pairs)
    got_o = [o[int(cu[n]):int(cu[n + 1]), h] for n, h in pairs]
    got_S = [S[n, h] for n, h in pairs]
    tau = tau_for(d["dtype"])
    # the RMS is taken over the sampled pairs together
    assert_parity(np.concatenate(got_o), np.concatenate(o_ref), tau, f"{name} o")
    assert_parity(np.stack(got_S), np.stack(S_ref), tau, f"{name} final state")
    # and every sampled pair stays within twice the budget on its own
    for p, (n, h) in enumerate(pairs):
        assert_parity(got_o[p], o_ref[p], 2 * tau, f"{name} o pair {(n, h)}")


def test_full_prefill_workload_sampled():
    """B=4, T=4096, H_qk=16, H_v=32, d=128, bf16 (the prefill benchmark)."""
    _full_size("prefill", 10, seed=2)


@pytest.mark.slow
def test_full_varlen_workload_sampled():
    """64 packed sequences, lengths U{128..8192}, per-sequence initial states."""
    _full_size("varlen", 8, seed=3)


@pytest.mark.slow
def test_full_long_prefill_sampled():
    """B=1, T=65536, initial state N(0, 0.02)."""
    _full_size("long", 4, seed=4)
