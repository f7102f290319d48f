"""GPU parity of the per-channel-decay variant (KDA: gdn_kda_chunk_fwd,
gdn_kda_decode_step) against the fp64 KDA oracle (oracle.kda_recurrent).

Both kernels keep an fp32 state (bf16 inputs widened exactly); the prefill's
products run on the warp MMA as three passes over operands split into high
and low parts (fp16 with power-of-two scales for the state products, tf32 for
the intra-chunk scores), about 22 significant bits, so outputs and final
states are held to
max|err| <= 1e-4 x RMS(ref) (the fp32 bound of the forward tests); a bf16 output is compared with the oracle
rounded to bf16 plus one bf16 ulp. Inputs: the seeded recipe of gdn_inputs
with per-channel log-decays g = -softplus(N(0,1) + shift) per key channel.
"""
import numpy as np
import pytest
import torch

import gdn_inputs
import oracle
import gated_deltanet_recurrence_05_b300 as gdn
from gdn_testutil import TAU_F32, assert_parity, to_cuda

pytestmark = pytest.mark.gpu


def _cu(d):
    if d["cu_seqlens"] is not None:
        return d["cu_seqlens"]
    return torch.tensor([0] + list(np.cumsum(d["lengths"])), dtype=torch.int32)


def _kda_gpu(d, g, out_dtype=torch.float32, order=None):
    dd = to_cuda(d)
    cu = dd["cu_seqlens"]
    o, S = gdn.kda_chunk_fwd(dd["q"], dd["k"], dd["v"], g.cuda(), dd["beta"], dd["h0"], cu,
                             num_seqs=None if cu is not None else len(d["lengths"]), output_dtype=out_dtype,
                             seq_order=order)
    torch.cuda.synchronize()
    assert gdn.get_device_error() == 0
    return o.float().cpu().numpy(), S.cpu().numpy()


def test_prefill_bf16_varlen_gqa_edges():
    d = gdn_inputs.make_prefill(h_qk=2, h_v=4, d_k=128, d_v=128, dtype="bf16",
                                lengths=[1, 31, 32, 0, 33, 100, 65], h0_std=0.02, seed=41)
    g = gdn_inputs.make_channel_decay((sum(d["lengths"]), 4, 128), seed=41)
    o, S = _kda_gpu(d, g)
    o_ref, S_ref = oracle.kda_recurrent(d["q"], d["k"], d["v"], g, d["beta"], h0=d["h0"], cu_seqlens=_cu(d))
    assert_parity(o, o_ref, TAU_F32, "o")
    assert_parity(S, S_ref, TAU_F32, "final state")


def test_prefill_sequence_segments():
    """Fewer (sequence, head) units than two per SM and long sequences: the
    prefill splits each sequence into segments, the later ones started from a
    zero state where the slowest channel's decay has shrunk the earlier tokens'
    influence below 2^-40 (see the header). Every output and final state
    against the oracle, at the fp32 bound."""
    d = gdn_inputs.make_prefill(h_qk=1, h_v=2, d_k=128, d_v=128, dtype="bf16",
                                lengths=[3000, 1, 1500, 700], h0_std=0.02, seed=44)
    g = gdn_inputs.make_channel_decay((sum(d["lengths"]), 2, 128), seed=44)
    o, S = _kda_gpu(d, g)
    o_ref, S_ref = oracle.kda_recurrent(d["q"], d["k"], d["v"], g, d["beta"], h0=d["h0"], cu_seqlens=_cu(d))
    assert_parity(o, o_ref, TAU_F32, "o")
    assert_parity(S, S_ref, TAU_F32, "final state")


def test_prefill_balanced_shares():
    """An equal-length batch with few units: the prefill cuts the tokens of the
    (sequence, q/k head) groups into balanced shares (here 288 tokens), each
    taken by the group's two value heads in neighbouring CTAs; most CTAs
    finish one unit and start the next. Every output and final state against
    the oracle, at the fp32 bound."""
    d = gdn_inputs.make_prefill(h_qk=2, h_v=4, d_k=128, d_v=128, dtype="bf16", batch=1, seqlen=20000,
                                h0_std=0.02, seed=45)
    assert d["cu_seqlens"] is None
    g = gdn_inputs.make_channel_decay((20000, 4, 128), seed=45)
    o, S = _kda_gpu(d, g)
    o_ref, S_ref = oracle.kda_recurrent(d["q"], d["k"], d["v"], g, d["beta"], h0=d["h0"], cu_seqlens=_cu(d))
    assert_parity(o, o_ref, TAU_F32, "o")
    assert_parity(S, S_ref, TAU_F32, "final state")


def test_prefill_fp32_equal_length_bf16_output_and_order():
    d = gdn_inputs.make_prefill(h_qk=2, h_v=2, d_k=128, d_v=128, dtype="f32", batch=3, seqlen=45, seed=42)
    g = gdn_inputs.make_channel_decay((135, 2, 128), g_shift=-3.0, seed=42)
    o, S = _kda_gpu(d, g, out_dtype=torch.bfloat16, order=torch.tensor([2, 0, 1], dtype=torch.int32).cuda())
    o_ref, S_ref = oracle.kda_recurrent(d["q"], d["k"], d["v"], g, d["beta"], cu_seqlens=_cu(d))
    assert_parity(o, o_ref, TAU_F32, "o (bf16)", out_bf16=True)
    assert_parity(S, S_ref, TAU_F32, "final state")


def test_prefill_strong_and_zero_decay_chunks():
    """Extreme per-channel decays: strong decays (g ~ -8 per token, so the
    state forgets within a few tokens and products of decays underflow), a
    weak stretch inside the same sequence, no decay at all (g = 0, alpha = 1),
    and half the channels strong with the other half weak in one sequence;
    every output and final state against the oracle at the fp32 bound."""
    d = gdn_inputs.make_prefill(h_qk=1, h_v=2, d_k=128, d_v=128, dtype="bf16", lengths=[200, 150, 70],
                                h0_std=0.02, seed=46)
    T = sum(d["lengths"])
    g = gdn_inputs.make_channel_decay((T, 2, 128), g_shift=8.0, seed=46)
    weak = gdn_inputs.make_channel_decay((T, 2, 128), g_shift=-3.0, seed=47)
    g[90:160] = weak[90:160]           # sequence 0: strong, weak, strong
    g[200:350] = 0.0                   # sequence 1: no decay
    g[350:, :, 64:] = weak[350:, :, 64:]  # sequence 2: channels 0-63 strong, 64-127 weak
    o, S = _kda_gpu(d, g)
    o_ref, S_ref = oracle.kda_recurrent(d["q"], d["k"], d["v"], g, d["beta"], h0=d["h0"], cu_seqlens=_cu(d))
    assert_parity(o, o_ref, TAU_F32, "o")
    assert_parity(S, S_ref, TAU_F32, "final state")


@pytest.mark.parametrize("g_shift", [2.0, 4.0])
def test_prefill_moderate_decays_within_a_chunk(g_shift):
    """Decays of the prefill benchmark's distribution (g_shift 2: the running
    decay of a 16-token chunk falls to about 2^-50) and stronger ones near the
    chunk's per-element threshold (g_shift 4): A and P pair rows scaled by
    exp(G_t) and exp(-G_s), which must keep their full range even where
    exp(G_t) alone is far below the fp16 range; every output and final state
    against the oracle at the fp32 bound."""
    d = gdn_inputs.make_prefill(h_qk=1, h_v=2, d_k=128, d_v=128, dtype="bf16", lengths=[100, 37],
                                h0_std=0.02, seed=48)
    g = gdn_inputs.make_channel_decay((137, 2, 128), g_shift=g_shift, seed=48)
    o, S = _kda_gpu(d, g)
    o_ref, S_ref = oracle.kda_recurrent(d["q"], d["k"], d["v"], g, d["beta"], h0=d["h0"], cu_seqlens=_cu(d))
    assert_parity(o, o_ref, TAU_F32, "o")
    assert_parity(S, S_ref, TAU_F32, "final state")


def test_uniform_channels_equal_gated_delta_rule():
    """Equal decays in every channel: KDA must reproduce the gated delta rule
    (the fp32 CUDA-core prefill of gdn_chunk_fwd)."""
    d = gdn_inputs.make_prefill(h_qk=1, h_v=2, d_k=128, d_v=128, dtype="bf16", lengths=[77, 40],
                                h0_std=0.02, seed=43)
    g = d["g"][:, :, None].expand(-1, -1, 128).contiguous()
    o, S = _kda_gpu(d, g)
    dd = to_cuda(d)
    o2, S2 = gdn.chunk_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["h0"], dd["cu_seqlens"],
                           output_dtype=torch.float32, force_simt=True)
    torch.cuda.synchronize()
    assert_parity(o, o2.cpu().numpy(), TAU_F32, "o vs gated delta rule")
    assert_parity(S, S2.cpu().numpy(), TAU_F32, "state vs gated delta rule")


def _decode_steps(t, g, steps):
    tt = to_cuda(t)
    state = tt["state"].clone()
    gg = g.cuda()
    outs = []
    for s in range(steps):
        outs.append(gdn.kda_decode_step(tt["q"][s], tt["k"][s], tt["v"][s], gg[s], tt["beta"][s], state,
                                        output_dtype=torch.float32))
    torch.cuda.synchronize()
    return torch.stack(outs).cpu().numpy(), state.cpu().numpy()


def _decode_ref(t, g):
    steps, N = t["q"].shape[0], t["q"].shape[1]
    perm = lambda x: x.transpose(0, 1).reshape(N * steps, *x.shape[2:]).contiguous()
    cu = torch.arange(0, N + 1, dtype=torch.int32) * steps
    o, S = oracle.kda_recurrent(perm(t["q"]), perm(t["k"]), perm(t["v"]), perm(g), perm(t["beta"]),
                                h0=t["state"], cu_seqlens=cu)
    return o.reshape(N, steps, *o.shape[1:]).transpose(1, 0, 2, 3), S


def test_decode_steps_gqa():
    t = gdn_inputs.make_decode(num_seqs=5, h_qk=2, h_v=4, d_k=128, d_v=128, steps=6, seed=44)
    g = gdn_inputs.make_channel_decay((6, 5, 4, 128), seed=44)
    o, S = _decode_steps(t, g, 6)
    o_ref, S_ref = _decode_ref(t, g)
    assert_parity(o, o_ref, TAU_F32, "decode o")
    assert_parity(S, S_ref, TAU_F32, "decode state")


def test_decode_equals_prefill():
    t = gdn_inputs.make_decode(num_seqs=3, h_qk=1, h_v=2, d_k=128, d_v=128, steps=9, seed=45)
    g = gdn_inputs.make_channel_decay((9, 3, 2, 128), seed=45)
    o_dec, S_dec = _decode_steps(t, g, 9)
    perm = lambda x: x.transpose(0, 1).reshape(27, *x.shape[2:]).contiguous()
    cu = (torch.arange(0, 4, dtype=torch.int32) * 9).cuda()
    o_pf, S_pf = gdn.kda_chunk_fwd(perm(t["q"]).cuda(), perm(t["k"]).cuda(), perm(t["v"]).cuda(),
                                   perm(g).cuda(), perm(t["beta"]).cuda(), t["state"].cuda(), cu,
                                   output_dtype=torch.float32)
    torch.cuda.synchronize()
    o_pf = o_pf.cpu().numpy().reshape(3, 9, 2, 128).transpose(1, 0, 2, 3)
    assert_parity(o_dec, o_pf, TAU_F32, "decode vs prefill o")
    assert_parity(S_dec, S_pf.cpu().numpy(), TAU_F32, "decode vs prefill state")


def test_full_size_prefill_sampled_pairs():
    """The prefill workload's shapes (B=4, T=4096, H_qk=16, H_v=32, d=128,
    bf16) with per-channel decays (shift +2, as the workload's scalar g):
    one call; sampled (sequence, value head) pairs replayed by the oracle."""
    w = gdn_inputs.WORKLOADS["prefill"]
    d = gdn_inputs.make_workload("prefill")
    g = gdn_inputs.make_channel_decay((w.batch * w.seqlen, w.h_v, 128), g_shift=2.0)
    o, S = _kda_gpu(d, g, out_dtype=torch.float32)
    T, G = w.seqlen, w.h_v // w.h_qk
    for n, h in ((0, 0), (2, 17), (3, 31)):
        t0, t1, hk = n * T, (n + 1) * T, h // G
        o_ref, S_ref = oracle.kda_recurrent(d["q"][t0:t1, hk:hk + 1], d["k"][t0:t1, hk:hk + 1],
                                            d["v"][t0:t1, h:h + 1], g[t0:t1, h:h + 1], d["beta"][t0:t1, h:h + 1])
        assert_parity(o[t0:t1, h], o_ref[:, 0], TAU_F32, f"pair ({n}, {h}) o")
        assert_parity(S[n, h], S_ref[0, 0], TAU_F32, f"pair ({n}, {h}) final state")


def test_full_size_decode_step():
    """The decode workload's shapes (256 sequences x 32 value heads, 128 x 128
    states ~ N(0, 0.02), bf16 token): one step, every pair against the oracle."""
    w = gdn_inputs.WORKLOADS["decode"]
    t = gdn_inputs.make_workload("decode", steps=1)
    g = gdn_inputs.make_channel_decay((1, w.num_seqs, w.h_v, 128))
    o, S = _decode_steps(t, g, 1)
    o_ref, S_ref = _decode_ref(t, g)
    assert_parity(o, o_ref, TAU_F32, "decode o")
    assert_parity(S, S_ref, TAU_F32, "decode state")
