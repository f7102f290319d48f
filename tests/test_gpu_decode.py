"""GPU parity of gdn_decode_step against the fp64 oracle (through the C ABI)."""
import numpy as np
import pytest
import torch

import gdn_inputs
import oracle
import gated_deltanet_recurrence_05_b300 as gdn
from gdn_testutil import TAU_BF16, TAU_F32, assert_parity, sample_pairs, to_cuda

pytestmark = pytest.mark.gpu


def _run_steps(d, steps, out_dtype=None):
    dd = to_cuda(d)
    state = dd["state"].clone()
    outs = []
    for t in range(steps):
        outs.append(gdn.decode_step(dd["q"][t], dd["k"][t], dd["v"][t], dd["g"][t], dd["beta"][t],
                                    state, output_dtype=out_dtype))
    torch.cuda.synchronize()
    assert gdn.get_device_error() == 0
    return torch.stack(outs).float().cpu().numpy(), state.cpu().numpy()


@pytest.mark.parametrize("d_k,d_v,h_qk,h_v", [(128, 128, 2, 4), (32, 16, 1, 3), (16, 48, 2, 2)])
def test_decode_fp32(d_k, d_v, h_qk, h_v):
    d = gdn_inputs.make_decode(num_seqs=5, h_qk=h_qk, h_v=h_v, d_k=d_k, d_v=d_v, steps=7,
                               dtype="f32", seed=3)
    o, S = _run_steps(d, 7)
    o_ref, S_ref = oracle.decode_steps(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state"])
    assert_parity(o, o_ref, TAU_F32, "o")
    assert_parity(S, S_ref, TAU_F32, "state")


@pytest.mark.parametrize("out_bf16", [False, True])
def test_decode_bf16_d128(out_bf16):
    d = gdn_inputs.make_decode(num_seqs=6, h_qk=2, h_v=4, d_k=128, d_v=128, steps=9, seed=5)
    o, S = _run_steps(d, 9, torch.bfloat16 if out_bf16 else torch.float32)
    o_ref, S_ref = oracle.decode_steps(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state"])
    assert_parity(o, o_ref, TAU_BF16, "o", out_bf16=out_bf16)
    assert_parity(S, S_ref, TAU_BF16, "state")


def test_decode_full_size_all_pairs():
    """256 sequences x 32 value heads x 128x128 states (512 MiB), the launch
    configuration of the decode benchmark, 16 consecutive steps, every pair
    checked against the oracle."""
    d = gdn_inputs.make_workload("decode", steps=16)
    o, S = _run_steps(d, 16, torch.float32)
    o_ref, S_ref = oracle.decode_steps(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state"])
    assert_parity(o, o_ref, TAU_BF16, "o")
    assert_parity(S, S_ref, TAU_BF16, "state")


@pytest.mark.slow
def test_decode_full_1000_steps_sampled():
    """The full decode workload: 1000 consecutive in-place steps; sampled
    (sequence, head) pairs are replayed by the oracle."""
    d = gdn_inputs.make_workload("decode")
    dd = to_cuda(d)
    state = dd["state"].clone()
    pairs = sample_pairs(256, 32, 12, seed=1)
    sel_n = [n for n, _ in pairs]
    sel_h = [h for _, h in pairs]
    got = []
    for t in range(1000):
        o = gdn.decode_step(dd["q"][t], dd["k"][t], dd["v"][t], dd["g"][t], dd["beta"][t], state,
                            output_dtype=torch.float32)
        got.append(o[sel_n, sel_h].cpu())
    torch.cuda.synchronize()
    got = torch.stack(got, 1).numpy()  # [pairs, steps, d_v]
    S = state.cpu().numpy()
    for p, (n, h) in enumerate(pairs):
        hk = h // 2
        o_ref, S_ref = oracle.recurrent(d["q"][:, n, hk:hk + 1], d["k"][:, n, hk:hk + 1],
                                        d["v"][:, n, h:h + 1], d["g"][:, n, h:h + 1],
                                        d["beta"][:, n, h:h + 1],
                                        h0=d["state"][n:n + 1, h:h + 1])
        assert_parity(got[p], o_ref[:, 0], TAU_BF16, f"o pair {(n, h)}")
        assert_parity(S[n, h], S_ref[0, 0], TAU_BF16, f"state pair {(n, h)}")


def test_decode_matches_prefill():
    """T decode steps give the same outputs and state as one prefill of the
    same T tokens (cross-kernel consistency)."""
    d = gdn_inputs.make_decode(num_seqs=2, h_qk=2, h_v=4, d_k=128, d_v=128, steps=40, seed=9,
                               dtype="f32")
    o_dec, S_dec = _run_steps(d, 40)
    dd = to_cuda(d)
    for n in range(2):
        sl = lambda x: x[:, n].contiguous()
        o_pf, S_pf = gdn.chunk_fwd(sl(dd["q"]), sl(dd["k"]), sl(dd["v"]), sl(dd["g"]),
                                   sl(dd["beta"]), dd["state"][n:n + 1].contiguous())
        torch.cuda.synchronize()
        assert_parity(o_dec[:, n], o_pf.cpu().numpy(), TAU_F32, "o decode vs prefill")
        assert_parity(S_dec[n], S_pf[0].cpu().numpy(), TAU_F32, "state decode vs prefill")


def test_decode_steps_captured_in_a_cuda_graph():
    """Consecutive decode steps issued through the C ABI inside a CUDA Graph
    capture (the way a serving loop replays them) and replayed: outputs and
    state against the oracle, and the replay equals the same steps run
    eagerly, bit for bit."""
    d = gdn_inputs.make_decode(num_seqs=6, h_qk=2, h_v=4, d_k=128, d_v=128, steps=8, seed=9)
    dd = to_cuda(d)
    state = dd["state"].clone()
    outs = torch.empty(8, 6, 4, 128, dtype=torch.float32, device="cuda")
    graph = torch.cuda.CUDAGraph()
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(graph, stream=side):
        cap = torch.cuda.current_stream()
        for t in range(8):
            gdn.decode_step(dd["q"][t], dd["k"][t], dd["v"][t], dd["g"][t], dd["beta"][t], state,
                            out=outs[t], stream=cap)
    state.copy_(dd["state"])  # the capture ran nothing; start from the initial states
    graph.replay()
    torch.cuda.synchronize()
    assert gdn.get_device_error() == 0
    o_ref, S_ref = oracle.decode_steps(d["q"], d["k"], d["v"], d["g"], d["beta"], d["state"])
    assert_parity(outs.cpu().numpy(), o_ref, TAU_BF16, "o (graph)")
    assert_parity(state.cpu().numpy(), S_ref, TAU_BF16, "state (graph)")
    o_eager, S_eager = _run_steps(d, 8, torch.float32)
    assert np.array_equal(outs.cpu().numpy(), o_eager)
    assert np.array_equal(state.cpu().numpy(), S_eager)
