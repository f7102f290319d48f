"""Failure path of the tensor-core prefill: a wait that runs out.

Every mbarrier wait of the kernel is bounded. A call with
GDN_FLAG_TEST_WAIT_TIMEOUT withholds one internal arrival (the decay factors
of chunk 1 of every unit are never announced) and shortens the wait limit,
so the waits on that arrival run out. The test checks what the contract
promises: the kernel gives up instead of hanging, every role unwinds, the
device error word reports GDN_DEVERR_TIMEOUT (and gdn_get_device_error
returns GDN_ERR_TIMEOUT), and the context and stream stay usable: the next
ordinary call on the same stream is exact against the oracle. Nothing here
faults or hangs the GPU: the failure is a flag that nothing sets.
"""
import ctypes

import pytest
import torch

import gdn_inputs
import oracle
import gated_deltanet_recurrence_05_b300 as gdn
from gdn_testutil import TAU_BF16, assert_parity, to_cuda

pytestmark = pytest.mark.gpu


def test_wait_timeout_unwinds_reports_and_leaves_stream_usable():
    d = gdn_inputs.make_prefill(h_qk=2, h_v=4, d_k=128, d_v=128, dtype="bf16",
                                lengths=[200, 70, 130], h0_std=0.02, seed=41)
    dd = to_cuda(d)
    stream = torch.cuda.current_stream()
    assert gdn.get_device_error() == 0
    gdn.chunk_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["h0"], dd["cu_seqlens"],
                  output_dtype=torch.float32, test_wait_timeout=True, stream=stream)
    code = ctypes.c_uint32(0)
    st = gdn.lib().gdn_get_device_error(ctypes.c_void_p(stream.cuda_stream), ctypes.byref(code))
    assert st == 4, gdn.lib().gdn_status_string(st)            # GDN_ERR_TIMEOUT
    assert code.value & gdn.DEVERR_TIMEOUT
    assert gdn.get_device_error() == 0                          # cleared
    # the same stream, the ordinary call: exact
    o, S = gdn.chunk_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["h0"], dd["cu_seqlens"],
                         output_dtype=torch.float32, stream=stream)
    assert gdn.get_device_error() == 0
    o_ref, S_ref = oracle.recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"],
                                    cu_seqlens=d["cu_seqlens"])
    assert_parity(o.cpu().numpy(), o_ref, TAU_BF16, "o after the timed-out call")
    assert_parity(S.cpu().numpy(), S_ref, TAU_BF16, "final state after the timed-out call")



def test_wait_timeout_with_balanced_shares():
    """The same failure path when every CTA holds two pieces of units (an
    equal-length batch cut into balanced shares): the withheld arrival is the
    CTA's second chunk; every CTA gives up, unwinds and leaves the stream
    usable for an exact ordinary call."""
    d = gdn_inputs.make_prefill(h_qk=2, h_v=4, d_k=128, d_v=128, dtype="bf16", batch=2, seqlen=640,
                                h0_std=0.02, seed=42)
    dd = to_cuda(d)
    stream = torch.cuda.current_stream()
    assert gdn.get_device_error() == 0
    gdn.chunk_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["h0"], None, num_seqs=2,
                  output_dtype=torch.float32, test_wait_timeout=True, balance=True, stream=stream)
    code = ctypes.c_uint32(0)
    st = gdn.lib().gdn_get_device_error(ctypes.c_void_p(stream.cuda_stream), ctypes.byref(code))
    assert st == 4, gdn.lib().gdn_status_string(st)
    assert code.value & gdn.DEVERR_TIMEOUT
    o, S = gdn.chunk_fwd(dd["q"], dd["k"], dd["v"], dd["g"], dd["beta"], dd["h0"], None, num_seqs=2,
                         output_dtype=torch.float32, balance=True, stream=stream)
    assert gdn.get_device_error() == 0
    o_ref, S_ref = oracle.recurrent(d["q"], d["k"], d["v"], d["g"], d["beta"], h0=d["h0"],
                                    cu_seqlens=torch.tensor([0, 640, 1280], dtype=torch.int32))
    assert_parity(o.cpu().numpy(), o_ref, TAU_BF16, "o after the timed-out call")
    assert_parity(S.cpu().numpy(), S_ref, TAU_BF16, "final state after the timed-out call")
