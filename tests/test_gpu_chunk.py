"""GPU parity of gdn_chunk_fwd (prefill) against the fp64 oracle.

Every case is compared element by element over every output and final
state, the full-size workloads included: those run in the launch
configuration the benchmark uses, and the oracle replays all their
(sequence, value-head) pairs in batches.
"""
import numpy as np
import pytest
import torch

import gdn_inputs
import oracle
import gated_deltanet_recurrence_05_b300 as gdn
from gdn_testutil import TAU_BF16, TAU_F32, assert_parity, tau_for, to_cuda

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


class _MaxErr:
    """max|got - ref| and RMS(ref) of one tensor, accumulated pair by pair, so
    that a whole full-size output is compared without holding the oracle's
    fp64 copy of it at once; the worst ratio of a single pair to its own RMS
    is kept too."""

    def __init__(self):
        self.max_err, self.sumsq, self.count, self.worst_pair, self.finite = 0.0, 0.0, 0, (0.0, None), True

    def add(self, got, ref, key):
        got = np.asarray(got, dtype=np.float64)
        err = float(np.abs(got - ref).max()) if ref.size else 0.0
        self.finite = self.finite and bool(np.isfinite(got).all())
        self.max_err = max(self.max_err, err)
        self.sumsq += float(np.sum(ref * ref))
        self.count += ref.size
        r = float(np.sqrt(np.mean(ref * ref))) if ref.size else 0.0
        if r > 0 and err / r > self.worst_pair[0]:
            self.worst_pair = (err / r, key)

    def check(self, tau, label):
        assert self.finite, f"{label}: non-finite values"
        rms = np.sqrt(self.sumsq / max(self.count, 1))
        e = self.max_err / rms
        assert e <= tau, f"{label}: max|err| = {e:.3e} x RMS(ref) > {tau:.1e}"
        # and every (sequence, head) pair within twice the budget of its own RMS
        assert self.worst_pair[0] <= 2 * tau, f"{label}: pair {self.worst_pair[1]} at {self.worst_pair[0]:.3e}"
        return e


def _full_size_all_pairs(d, label, batch_pair_tokens=1 << 20):
    """Run the whole problem on the GPU in the benchmark's launch configuration
    (longest-first schedule for packed sequences), then replay EVERY
    (sequence, value-head) pair with the oracle, in batches of about
    ``batch_pair_tokens`` pair-tokens, and compare element by element."""
    cu = d["cu_seqlens"]
    order = gdn.plan_seq_order(cu).cuda() if cu is not None else None
    o, S = _gpu(d, order=order)
    N, hv = len(d["lengths"]), d["h_v"]
    if cu is None:
        cu = torch.tensor([0] + list(np.cumsum(d["lengths"])), dtype=torch.int32)
    cul = [int(x) for x in cu.tolist()]
    acc_o, acc_s = _MaxErr(), _MaxErr()

    def flush(batch):
        if not batch:
            return
        o_ref, S_ref = oracle.recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"],
                                        cu_seqlens=cu, pairs=batch)
        for p, (n, h) in enumerate(batch):
            acc_o.add(o[cul[n]:cul[n + 1], h], o_ref[p], (n, h))
            acc_s.add(S[n, h], S_ref[p], (n, h))

    batch, tok = [], 0
    for n in range(N):
        for h in range(hv):
            batch.append((n, h))
            tok += cul[n + 1] - cul[n]
            if tok >= batch_pair_tokens:
                flush(batch)
                batch, tok = [], 0
    flush(batch)
    assert acc_o.count == sum(d["lengths"]) * hv * d["d_v"]
    tau = tau_for(d["dtype"])
    acc_o.check(tau, f"{label} o")
    acc_s.check(tau, f"{label} final state")


def test_full_prefill_workload_all_pairs():
    """B=4, T=4096, H_qk=16, H_v=32, d=128, bf16 (the prefill benchmark):
    all 128 (sequence, head) pairs, every output and final-state element."""
    _full_size_all_pairs(gdn_inputs.make_workload("prefill"), "prefill")


@pytest.mark.slow
def test_full_varlen_workload_all_pairs():
    """64 packed sequences, lengths U{128..8192}, per-sequence initial states:
    all 2048 pairs."""
    _full_size_all_pairs(gdn_inputs.make_workload("varlen"), "varlen")


@pytest.mark.slow
def test_full_long_prefill_all_pairs():
    """B=1, T=65536, initial state N(0, 0.02): all 32 pairs (32 units for 148
    SMs: the tensor-core path splits the sequence into segments)."""
    _full_size_all_pairs(gdn_inputs.make_workload("long"), "long")


@pytest.mark.slow
def test_slow_decay_at_long_length():
    """g = -softplus(N(0,1) - 5) (alpha ~ 0.99) over one sequence of 65536
    tokens: the fp16 copy of the state is re-rounded 1024 times while old
    content stays visible; every pair of 8 value heads (GQA 2:1)."""
    d = gdn_inputs.make_prefill(h_qk=4, h_v=8, d_k=128, d_v=128, dtype="bf16", lengths=[65536],
                                g_shift=-5.0, h0_std=0.02, seed=23)
    _full_size_all_pairs(d, "slow decay, T=65536")


def test_fp16_range_overflow_is_reported():
    """The tensor-core kernel multiplies fp16 operands: values beyond 65504
    (here v ~ 1e5) cannot be represented. The kernel must not return such a
    result silently: it records GDN_DEVERR_RANGE, and the fp32 CUDA-core
    kernel (GDN_FLAG_FORCE_SIMT) computes the same inputs correctly."""
    d = gdn_inputs.make_prefill(h_qk=1, h_v=2, d_k=128, d_v=128, dtype="bf16",
                                lengths=[150, 70], h0_std=0.02, seed=21)
    d["v"] = (d["v"].float() * 1e5).to(torch.bfloat16)
    dd = to_cuda(d)
    gdn.chunk_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["h0"], dd["cu_seqlens"],
                  output_dtype=torch.float32)
    assert gdn.get_device_error() & gdn.DEVERR_RANGE
    o, S = _gpu(d, force_simt=True)
    o_ref, S_ref = _ref(d)
    assert_parity(o, o_ref, TAU_BF16, "o (CUDA-core kernel)")
    assert_parity(S, S_ref, TAU_BF16, "final state (CUDA-core kernel)")


def test_large_values_inside_fp16_range_stay_within_tolerance():
    """v ~ 1e3 and an initial state ~ 20 (all inside the fp16 range): the
    tensor-core kernel keeps its relative accuracy and reports nothing."""
    d = gdn_inputs.make_prefill(h_qk=2, h_v=4, d_k=128, d_v=128, dtype="bf16",
                                lengths=[200, 77], h0_std=0.02, seed=24)
    d["v"] = (d["v"].float() * 1e3).to(torch.bfloat16)
    d["h0"] = d["h0"] * 1e3
    o, S = _gpu(d)
    o_ref, S_ref = _ref(d)
    assert_parity(o, o_ref, TAU_BF16, "o")
    assert_parity(S, S_ref, TAU_BF16, "final state")


def _run_split(d, split):
    dd = to_cuda(d)
    o, S = gdn.chunk_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["h0"], dd["cu_seqlens"],
                         output_dtype=torch.float32, split=split)
    torch.cuda.synchronize()
    assert gdn.get_device_error() == 0
    return o.cpu().numpy(), S.cpu().numpy()


def test_sequence_segments_without_decay_are_bit_exact():
    """alpha = 1 (g = 0): no prefix ever reaches the 2^-40 bound, so every
    segment restarts at its sequence's first token with the initial state and
    computes exactly what the unsplit kernel computes for its tokens."""
    d = gdn_inputs.make_prefill(h_qk=2, h_v=4, d_k=128, d_v=128, dtype="bf16",
                                lengths=[3000, 2100], h0_std=0.02, seed=61)
    d["g"].zero_()
    o1, S1 = _run_split(d, True)
    o2, S2 = _run_split(d, False)
    np.testing.assert_array_equal(o1, o2)
    np.testing.assert_array_equal(S1, S2)


@pytest.mark.parametrize("k_scale", [1.0, 1.5])
def test_sequence_segments_match_oracle(k_scale):
    """Fewer (sequence, head) units than SMs: the sequences are split into
    segments, each started from a zero state where the decay bound allows
    (unit keys: beta |k|^2 < 1; keys of norm 1.5: factors |1 - beta |k|^2| up
    to 1.25 lengthen the prefixes). Every output and final state against the
    oracle and against the unsplit kernel."""
    d = gdn_inputs.make_prefill(h_qk=2, h_v=4, d_k=128, d_v=128, dtype="bf16",
                                lengths=[3000, 1, 0, 1500, 700, 2600], h0_std=0.02, seed=62)
    if k_scale != 1.0:
        d["k"] = (d["k"].float() * k_scale).to(torch.bfloat16)
    o, S = _run_split(d, True)
    o_ref, S_ref = _ref(d)
    assert_parity(o, o_ref, TAU_BF16, "o")
    assert_parity(S, S_ref, TAU_BF16, "final state")
    o2, S2 = _run_split(d, False)
    assert_parity(o, o2, TAU_BF16, "o vs unsplit")
    assert_parity(S, S2, TAU_BF16, "final state vs unsplit")


def _run_batch(d, N, **kw):
    dd = to_cuda(d)
    o, S = gdn.chunk_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["h0"], None, num_seqs=N,
                         output_dtype=torch.float32, **kw)
    torch.cuda.synchronize()
    assert gdn.get_device_error() == 0
    return o.cpu().numpy(), S.cpu().numpy()


@pytest.mark.parametrize("g_zero", [False, True])
def test_balanced_shares_match_oracle(g_zero):
    """Equal-length batch cut into balanced shares of 3 chunks (GDN_FLAG_BALANCE):
    16 chunks per unit, so most CTAs take the end of one (sequence, head) unit
    and the start of the next, the first piece started from a zero state after
    its prefix. Every output and final state against the oracle and the
    unsplit kernel; with alpha = 1 every piece restarts at its sequence start
    and the results equal the unsplit kernel's bit for bit."""
    N, L = 2, 1000
    d = gdn_inputs.make_prefill(h_qk=2, h_v=4, d_k=128, d_v=128, dtype="bf16", batch=N, seqlen=L, h0_std=0.02,
                                seed=64)
    assert d["cu_seqlens"] is None
    if g_zero:
        d["g"].zero_()
    o, S = _run_batch(d, N, balance=True)
    o2, S2 = _run_batch(d, N, split=False)
    if g_zero:
        np.testing.assert_array_equal(o, o2)
        np.testing.assert_array_equal(S, S2)
    else:
        o_ref, S_ref = _ref(d)
        assert_parity(o, o_ref, TAU_BF16, "o")
        assert_parity(S, S_ref, TAU_BF16, "final state")
        assert_parity(o, o2, TAU_BF16, "o vs unsplit")
        assert_parity(S, S2, TAU_BF16, "final state vs unsplit")


def test_bf16_output_segments_and_unaligned_buffer():
    """bf16 outputs with sequence segments (the rows of a segment's prefix are
    not stored) into a 16-byte aligned and a 2-byte aligned buffer: both
    against the oracle, and equal to each other bit for bit. Ragged lengths,
    GQA 2:1."""
    d = gdn_inputs.make_prefill(h_qk=2, h_v=4, d_k=128, d_v=128, dtype="bf16",
                                lengths=[3000, 1, 0, 1500, 77, 700], h0_std=0.02, seed=63)
    dd = to_cuda(d)
    T = sum(d["lengths"])
    outs = []
    for offset in (0, 1):  # elements: 0 = 16-byte aligned, 1 = 2-byte aligned
        buf = torch.full((T * 4 * 128 + 8,), float("nan"), dtype=torch.bfloat16, device="cuda")
        out = buf[offset:offset + T * 4 * 128].view(T, 4, 128)
        assert (out.data_ptr() % 16 == 0) == (offset == 0)
        gdn.chunk_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["h0"], dd["cu_seqlens"], out=out)
        torch.cuda.synchronize()
        assert gdn.get_device_error() == 0
        outs.append(out.float().cpu().numpy())
    np.testing.assert_array_equal(outs[0], outs[1])
    o_ref, _ = _ref(d)
    assert_parity(outs[0], o_ref, TAU_BF16, "o (bf16)", out_bf16=True)
