"""GPU parity of the input prologue (gdn_short_conv, gdn_short_conv_step)
against the fp64 oracle, through the C ABI.

The filter, silu and L2 norm run in fp32 on exactly the oracle's inputs, so the
outputs are held to tau = 1e-4 x RMS (plus one bf16 ulp when written in bf16).
The conv states are copies of inputs: they must match bit for bit.
"""
import numpy as np
import pytest
import torch

import oracle
import gated_deltanet_recurrence_05_b300 as gdn
from gdn_testutil import TAU_F32, assert_parity

pytestmark = pytest.mark.gpu

_DT = {"f32": torch.float32, "bf16": torch.bfloat16}


def _case(lengths, C, K, dtype, seed, state=True):
    g = torch.Generator().manual_seed(seed)
    T = sum(lengths)
    x = torch.randn(T, C, generator=g).to(_DT[dtype])
    w = torch.randn(C, K, generator=g) * 0.5
    s0 = torch.randn(len(lengths), C, K - 1, generator=g) if state else None
    cu = torch.tensor(np.concatenate([[0], np.cumsum(lengths)]), dtype=torch.int32)
    return x, w, s0, cu


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("K", [1, 2, 3, 4])
@pytest.mark.parametrize("ng", [0, 128, 32])
def test_short_conv_varlen(dtype, K, ng):
    lengths = [5, 1, 0, 2, 37, 64, 3]
    C = 256
    x, w, s0, cu = _case(lengths, C, K, dtype, seed=K * 10 + ng)
    y, fs = gdn.short_conv(x.cuda(), w.cuda(), cu_seqlens=cu.cuda(), conv_state=None if K == 1 else s0.cuda(),
                           return_final_state=True, norm_group=ng)
    assert gdn.get_device_error() == 0
    y_ref, fs_ref = oracle.short_conv(x, w, cu_seqlens=cu.numpy(), state0=None if K == 1 else s0, norm_group=ng)
    assert_parity(y.float().cpu().numpy(), y_ref, TAU_F32, "y", out_bf16=(dtype == "bf16"))
    if K > 1:
        np.testing.assert_array_equal(fs.cpu().numpy(), fs_ref.astype(np.float32))


def test_short_conv_equal_lengths_no_state():
    x, w, _, _ = _case([48] * 4, 128, 4, "bf16", seed=5, state=False)
    y, fs = gdn.short_conv(x.cuda(), w.cuda(), num_seqs=4, return_final_state=True, norm_group=64)
    cu = np.arange(5) * 48
    y_ref, fs_ref = oracle.short_conv(x, w, cu_seqlens=cu, norm_group=64)
    assert_parity(y.float().cpu().numpy(), y_ref, TAU_F32, "y", out_bf16=True)
    np.testing.assert_array_equal(fs.cpu().numpy(), fs_ref.astype(np.float32))


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_short_conv_steps(dtype):
    N, C, K, steps = 5, 384, 4, 6
    g = torch.Generator().manual_seed(9)
    xs = torch.randn(steps, N, C, generator=g).to(_DT[dtype])
    w = torch.randn(C, K, generator=g) * 0.5
    s0 = torch.randn(N, C, K - 1, generator=g)
    st = s0.clone().cuda()
    st_ref = s0.numpy().astype(np.float64)
    for t in range(steps):
        y = gdn.short_conv_step(xs[t].cuda(), w.cuda(), st, norm_group=128)
        y_ref, st_ref = oracle.short_conv_step(xs[t], w, st_ref, norm_group=128)
        assert_parity(y.float().cpu().numpy(), y_ref, TAU_F32, f"y step {t}", out_bf16=(dtype == "bf16"))
        np.testing.assert_array_equal(st.cpu().numpy(), st_ref.astype(np.float32))


def test_short_conv_prefill_shapes():
    """The q/k (2048 channels, heads of 128, L2 norm) and v (4096 channels)
    projections of the B=4 x 4096 prefill workload, K = 4; sampled tokens of
    each sequence (including its first three) against the oracle."""
    B, T = 4, 4096
    cu = np.arange(B + 1) * T
    for C, ng in ((2048, 128), (4096, 0)):
        g = torch.Generator().manual_seed(C)
        x = torch.randn(B * T, C, generator=g).to(torch.bfloat16)
        w = torch.randn(C, 4, generator=g) * 0.5
        y = gdn.short_conv(x.cuda(), w.cuda(), num_seqs=B, norm_group=ng).cpu()
        rows = np.unique(np.concatenate([cu[:-1] + o for o in (0, 1, 2, 3, 100, T - 1)]))
        # the oracle on each sampled token's 4-token window
        for r in rows:
            n = int(np.searchsorted(cu, r, side="right") - 1)
            lo = max(cu[n], r - 3)
            yr, _ = oracle.short_conv(x[lo:r + 1], w, norm_group=ng)
            assert_parity(y[r:r + 1].float().numpy(), yr[-1:], TAU_F32, f"y[{r}]", out_bf16=True)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("ng", [0, 128])
def test_short_conv_many_tiles_two_channel_blocks(dtype, ng):
    """Sequences that span several 64-token tiles of the TMA-fed kernel and
    start or end inside a tile (and inside one warp's 8 tokens), two channel
    blocks, conv states in and out: every output and state element against
    the oracle."""
    lengths = [130, 1, 200, 0, 64, 65, 7]
    C = 512 if dtype == "bf16" else 256
    x, w, s0, cu = _case(lengths, C, 4, dtype, seed=77 + ng)
    y, fs = gdn.short_conv(x.cuda(), w.cuda(), cu_seqlens=cu.cuda(), conv_state=s0.cuda(), return_final_state=True,
                           norm_group=ng)
    assert gdn.get_device_error() == 0
    y_ref, fs_ref = oracle.short_conv(x, w, cu_seqlens=cu.numpy(), state0=s0, norm_group=ng)
    assert_parity(y.float().cpu().numpy(), y_ref, TAU_F32, "y", out_bf16=(dtype == "bf16"))
    np.testing.assert_array_equal(fs.cpu().numpy(), fs_ref.astype(np.float32))


def test_short_conv_tma_and_register_kernels_agree():
    """bf16 with 256 channels goes through the TMA-fed kernel (whole 512-byte
    channel blocks); each half of 128 channels alone goes through the
    register-tiled kernel. Both evaluate every token with the same code, so
    with heads of 128 channels the outputs and states are bit-identical."""
    lengths = [100, 37, 3, 70]
    x, w, s0, cu = _case(lengths, 256, 4, "bf16", seed=91)
    xc, wc, s0c, cuc = x.cuda(), w.cuda(), s0.cuda(), cu.cuda()
    y, fs = gdn.short_conv(xc, wc, cu_seqlens=cuc, conv_state=s0c, return_final_state=True, norm_group=128)
    for h in range(2):
        sl = slice(128 * h, 128 * (h + 1))
        yh, fsh = gdn.short_conv(xc[:, sl].contiguous(), wc[sl].contiguous(), cu_seqlens=cuc,
                                 conv_state=s0c[:, sl].contiguous(), return_final_state=True, norm_group=128)
        assert gdn.get_device_error() == 0
        np.testing.assert_array_equal(yh.float().cpu().numpy(), y[:, sl].float().cpu().numpy())
        np.testing.assert_array_equal(fsh.cpu().numpy(), fs[:, sl].cpu().numpy())
    y_ref, fs_ref = oracle.short_conv(x, w, cu_seqlens=cu.numpy(), state0=s0, norm_group=128)
    assert_parity(y.float().cpu().numpy(), y_ref, TAU_F32, "y", out_bf16=True)
    np.testing.assert_array_equal(fs.cpu().numpy(), fs_ref.astype(np.float32))


def test_short_conv_rejects_bad_seqlens_on_device():
    """A cu_seqlens entry past the end of the tokens is caught by the kernel's
    own check before any access: the affected run is skipped and the error bit
    recorded."""
    x = torch.randn(16, 128, device="cuda")
    w = torch.randn(128, 4, device="cuda")
    cu = torch.tensor([0, 8, 40], dtype=torch.int32, device="cuda")
    gdn.short_conv(x, w, cu_seqlens=cu)
    assert gdn.get_device_error() & 1
