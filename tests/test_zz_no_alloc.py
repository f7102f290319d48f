"""gdn_chunk_bwd_static: the gradient entry point for callers that cannot
allocate device memory (a host with a fixed memory budget, a plug-in given
tensors but no allocator, a path where cudaMalloc is not allowed). It runs the
same backward kernel as gdn_chunk_bwd on a 64 MiB scratch array built into
the library instead of a caller workspace.

The test calls it through the C ABI twice in a row, on two different
problems, and compares each result with the fp64 gradient oracle and with
gdn_chunk_bwd's (caller workspace), under the gradient tolerance of the
backward parity tests. The second call runs on whatever the first left in
the shared array. It also checks that a problem larger than the array is
refused before anything runs. The file is named so that pytest collects it
last.
"""
import ctypes

import numpy as np
import pytest
import torch

import gdn_inputs
import oracle
import gated_deltanet_recurrence_05_b300 as gdn
from gdn_testutil import assert_parity

pytestmark = pytest.mark.gpu

TAU_BWD = 1e-3           # as in tests/test_gpu_backward.py
UNSUPPORTED = 2
SCRATCH_BYTES = 64 << 20


def _problem(seed, lengths, h_qk, h_v):
    d = gdn_inputs.make_prefill(h_qk=h_qk, h_v=h_v, d_k=128, d_v=128, dtype="bf16", lengths=lengths,
                                h0_std=0.02, seed=seed)
    gr = gdn_inputs.make_grads(d, dtype="bf16", dht_std=0.05, seed=seed)
    dd = {k: (v.cuda() if isinstance(v, torch.Tensor) else v) for k, v in d.items()}
    ref = oracle.recurrent_backward(d["q"], d["k"], d["v"], d["g"], d["beta"], gr["do"], h0=d["h0"],
                                    dht=gr["dht"], cu_seqlens=d["cu_seqlens"])
    return dd, gr["do"].cuda(), gr["dht"].cuda(), ref


def _static(dd, do, dht):
    q, v = dd["q"], dd["v"]
    T, h_qk, h_v = q.shape[0], q.shape[1], v.shape[1]
    N = dd["cu_seqlens"].numel() - 1
    f32 = dict(dtype=torch.float32, device="cuda")
    outs = [torch.full((T, h_qk, 128), float("nan"), **f32), torch.full((T, h_qk, 128), float("nan"), **f32),
            torch.full((T, h_v, 128), float("nan"), **f32), torch.full((T, h_v), float("nan"), **f32),
            torch.full((T, h_v), float("nan"), **f32), torch.full((N, h_v, 128, 128), float("nan"), **f32)]
    p = lambda t: None if t is None else ctypes.c_void_p(t.data_ptr())
    st = gdn.lib().gdn_chunk_bwd_static(
        p(q), p(dd["k"]), p(v), p(dd["g"]), p(dd["beta"]), p(dd["h0"]), p(dd["cu_seqlens"]), None, p(do), p(dht),
        *[p(t) for t in outs], N, T, h_qk, h_v, 128, 128, gdn.BF16, gdn.BF16, 0.0,
        ctypes.c_void_p(torch.cuda.current_stream().cuda_stream))
    assert st == 0, gdn.lib().gdn_status_string(st)
    torch.cuda.synchronize()
    assert gdn.get_device_error() == 0
    return [t.cpu().numpy() for t in outs]


def _with_workspace(dd, do, dht):
    out = gdn.chunk_bwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], do, dd["h0"], dht, dd["cu_seqlens"])
    torch.cuda.synchronize()
    return [t.cpu().numpy() for t in out]


def test_static_scratch_two_calls_match_workspace_entry_point():
    problems = [_problem(31, [70, 33, 1], 2, 4), _problem(32, [129, 0, 64], 4, 4)]
    for i, (dd, do, dht, oref) in enumerate(problems):
        need = gdn.chunk_bwd_workspace_size(dd["cu_seqlens"].numel() - 1, dd["q"].shape[0],
                                            dd["q"].shape[1], dd["v"].shape[1])
        assert 0 < need <= SCRATCH_BYTES
        got = _static(dd, do, dht)
        ref = _with_workspace(dd, do, dht)
        for name, x, y in zip(("dq", "dk", "dv", "dg", "dbeta", "dh0"), got, ref):
            assert_parity(x, oref[name], TAU_BWD, f"call {i + 1}: {name} vs oracle")
            assert_parity(x, y, TAU_BWD, f"call {i + 1}: {name}")


def test_static_scratch_refuses_problems_beyond_its_size():
    # 4 sequences x 4096 tokens, 32 value heads: about 1.6 GB of scratch
    assert gdn.chunk_bwd_workspace_size(4, 16384, 16, 32) > SCRATCH_BYTES
    fake = ctypes.c_void_p(0x10000)
    st = gdn.lib().gdn_chunk_bwd_static(fake, fake, fake, fake, fake, None, None, None, fake, None, fake, fake,
                                        fake, fake, fake, None, 4, 16384, 16, 32, 128, 128, gdn.BF16, gdn.BF16,
                                        0.0, None)
    assert st == UNSUPPORTED
