"""Host-side checks of the C ABI (no GPU needed, no kernel launched).

The library must load, export every entry point that include/gdn.h declares,
and reject bad arguments on the host with the documented status before it
touches the device.
"""
import ctypes
import os
import re

import pytest
import torch

import gated_deltanet_recurrence_05_b300 as gdn
from gated_deltanet_recurrence_05_b300 import build as gbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "gdn.h")

OK, INVALID, UNSUPPORTED = 0, 1, 2


@pytest.fixture(scope="module")
def L():
    gbuild.build()
    return gdn.lib()


def declared_functions():
    text = open(HEADER).read()
    text = re.sub(r"/\*.*?\*/", "", text, flags=re.S)
    return sorted(set(re.findall(r"\b(gdn_[a-z0-9_]+)\s*\(", text)))


def test_header_declares_entry_points():
    names = declared_functions()
    for need in ("gdn_chunk_fwd", "gdn_decode_step", "gdn_decode_step_gated", "gdn_gated_rmsnorm",
                 "gdn_short_conv", "gdn_short_conv_step", "gdn_chunk_bwd", "gdn_chunk_bwd_workspace_size",
                 "gdn_chunk_fwd_workspace_size", "gdn_chunk_fwd_gated",
                 "gdn_chunk_bwd_static", "gdn_kda_chunk_fwd", "gdn_kda_decode_step",
                 "gdn_plan_seq_order",
                 "gdn_get_device_error", "gdn_status_string", "gdn_version"):
        assert need in names


def test_library_exports_every_declared_symbol(L):
    missing = [n for n in declared_functions() if not hasattr(L, n)]
    assert not missing, f"not exported: {missing}"


def test_status_strings_and_version(L):
    assert L.gdn_status_string(0) == b"GDN_OK"
    assert L.gdn_status_string(2) == b"GDN_ERR_UNSUPPORTED"
    assert L.gdn_version() >= 100


def test_plan_seq_order_longest_first(L):
    cu = [0, 5, 5, 17, 20, 32]  # lengths 5, 0, 12, 3, 12
    order = gdn.plan_seq_order(cu).tolist()
    assert order == [2, 4, 0, 3, 1]


def test_plan_seq_order_rejects_decreasing(L):
    with pytest.raises(gdn.GdnError):
        gdn.plan_seq_order([0, 4, 3])


FAKE = 0x10000  # 16-byte aligned, never dereferenced: every call below fails validation


def _fwd(L, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, h0=None, cu=None, order=None, o=FAKE,
             hT=None, N=1, T=64, h_qk=2, h_v=4, d_k=64, d_v=64, dq=1, do=1, scale=0.0,
             chunk=0, flags=0)
    a.update(kw)
    return L.gdn_chunk_fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["h0"], a["cu"], a["order"],
                           a["o"], a["hT"], a["N"], a["T"], a["h_qk"], a["h_v"], a["d_k"], a["d_v"],
                           a["dq"], a["do"], a["scale"], a["chunk"], a["flags"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(q=None), INVALID),
    (dict(v=FAKE + 4), INVALID),                 # q/k/v need 16 bytes (TMA)
    (dict(g=FAKE + 2), INVALID),                 # g needs 4 bytes
    (dict(h0=FAKE + 8), INVALID),
    (dict(h_qk=3, h_v=4), INVALID),              # H_v % H_qk != 0
    (dict(h_qk=0), INVALID),
    (dict(N=-1), INVALID),
    (dict(T=-5), INVALID),
    (dict(N=3, T=64), INVALID),                  # equal lengths need T % N == 0
    (dict(dq=7), INVALID),
    (dict(do=2), INVALID),
    (dict(chunk=48), INVALID),
    (dict(flags=32), INVALID),
    (dict(flags=2 | 16), INVALID),               # only documented flag bits
    (dict(d_k=256), UNSUPPORTED),
    (dict(d_v=129), UNSUPPORTED),
    (dict(N=0, T=0), OK),                        # nothing to do
    (dict(N=0, T=5), INVALID),
    (dict(T=0, hT=None), OK),                    # no tokens, no state requested
])
def test_chunk_fwd_host_validation(L, kw, status):
    assert _fwd(L, **kw) == status


def _dec(L, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, S=FAKE, o=FAKE, N=4, h_qk=2, h_v=4,
             d_k=128, d_v=128, dq=1, do=1, scale=0.0)
    a.update(kw)
    return L.gdn_decode_step(a["q"], a["k"], a["v"], a["g"], a["beta"], a["S"], a["o"], a["N"],
                             a["h_qk"], a["h_v"], a["d_k"], a["d_v"], a["dq"], a["do"], a["scale"],
                             None)


@pytest.mark.parametrize("kw,status", [
    (dict(S=None), INVALID),
    (dict(o=FAKE + 1), INVALID),                 # not element-aligned
    (dict(S=FAKE + 4), INVALID),                 # state needs 16 bytes
    (dict(h_qk=3), INVALID),
    (dict(dq=5), INVALID),
    (dict(d_k=200), UNSUPPORTED),
    (dict(N=0), OK),
    (dict(N=-2), INVALID),
])
def test_decode_host_validation(L, kw, status):
    assert _dec(L, **kw) == status


def test_binding_rejects_cpu_tensors():
    x = torch.zeros(4, 1, 8)
    g = torch.zeros(4, 1)
    with pytest.raises(ValueError):
        gdn.chunk_fwd(x, x, x, g, g)
    with pytest.raises(ValueError):
        gdn.decode_step(x[:1], x[:1], x[:1], g[:1], g[:1], torch.zeros(1, 1, 8, 8))


def test_missing_library_fails_loudly(monkeypatch, tmp_path):
    monkeypatch.setattr(gdn, "_lib", None)
    monkeypatch.setattr(gdn, "LIB_PATH", str(tmp_path / "absent.so"))
    with pytest.raises(ImportError):
        gdn.lib()


def _norm(L, **kw):
    a = dict(x=FAKE, z=FAKE, w=None, y=FAKE + 0x1000, rows=8, d=128, dx=1, dy=1, eps=1e-6)
    a.update(kw)
    return L.gdn_gated_rmsnorm(a["x"], a["z"], a["w"], a["y"], a["rows"], a["d"], a["dx"], a["dy"], a["eps"],
                               None)


@pytest.mark.parametrize("kw,status", [
    (dict(x=None), INVALID),
    (dict(z=None), INVALID),
    (dict(y=None), INVALID),
    (dict(x=FAKE + 1), INVALID),                 # bf16 needs 2-byte alignment
    (dict(w=FAKE + 2), INVALID),                 # the fp32 weight needs 4 bytes
    (dict(rows=-1), INVALID),
    (dict(d=0), INVALID),
    (dict(dx=7), INVALID),
    (dict(eps=-1.0), INVALID),
    (dict(eps=float("nan")), INVALID),
    (dict(y=FAKE, dy=0), INVALID),               # in place needs equal dtypes
    (dict(d=1025), UNSUPPORTED),
    (dict(rows=0), OK),                          # nothing to do, nothing launched
])
def test_gated_rmsnorm_host_validation(L, kw, status):
    assert _norm(L, **kw) == status


def _dec_gated(L, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, S=FAKE, o=FAKE, z=FAKE, w=None, eps=1e-6, N=2, h_qk=1,
             h_v=2, d_k=128, d_v=128, dq=1, do=1, scale=0.0)
    a.update(kw)
    return L.gdn_decode_step_gated(a["q"], a["k"], a["v"], a["g"], a["beta"], a["S"], a["o"], a["z"], a["w"],
                                   a["eps"], a["N"], a["h_qk"], a["h_v"], a["d_k"], a["d_v"], a["dq"], a["do"],
                                   a["scale"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(z=FAKE + 1), INVALID),                 # the gate takes the q/k/v dtype alignment
    (dict(z=None, w=FAKE), INVALID),             # a weight without a gate
    (dict(eps=-0.5), INVALID),
    (dict(d_v=129), UNSUPPORTED),
    (dict(N=0), OK),
])
def test_decode_gated_host_validation(L, kw, status):
    assert _dec_gated(L, **kw) == status


def _conv(L, **kw):
    a = dict(x=FAKE, w=FAKE, y=FAKE + 0x1000, cu=None, s_in=None, s_out=None, N=2, T=64, C=256, K=4, ng=128,
             eps=1e-6, dt=1)
    a.update(kw)
    return L.gdn_short_conv(a["x"], a["w"], a["y"], a["cu"], a["s_in"], a["s_out"], a["N"], a["T"], a["C"], a["K"],
                            a["ng"], a["eps"], a["dt"], None)


@pytest.mark.parametrize("kw,status", [
    (dict(x=None), INVALID),
    (dict(w=FAKE + 2), INVALID),
    (dict(y=FAKE), INVALID),                     # no in-place: the taps read neighbours
    (dict(C=130), INVALID),                      # C % 4
    (dict(ng=48), INVALID),                      # not a power-of-two divisor of 128
    (dict(C=192, ng=128), INVALID),              # C % norm_group
    (dict(T=63), INVALID),                       # equal lengths need T % N == 0
    (dict(N=0, T=64), INVALID),
    (dict(K=0), INVALID),
    (dict(K=5), UNSUPPORTED),
    (dict(eps=-1.0), INVALID),
    (dict(N=0, T=0), OK),
])
def test_short_conv_host_validation(L, kw, status):
    assert _conv(L, **kw) == status


def test_short_conv_step_host_validation(L):
    call = lambda **kw: L.gdn_short_conv_step(kw.get("x", FAKE), kw.get("w", FAKE), kw.get("s", FAKE),
                                              kw.get("y", FAKE + 0x1000), kw.get("N", 2), kw.get("C", 256),
                                              kw.get("K", 4), kw.get("ng", 0), kw.get("eps", 1e-6), 1, None)
    assert call(s=None) == INVALID
    assert call(y=FAKE) == INVALID
    assert call(K=5) == UNSUPPORTED
    assert call(N=0) == OK


def _bwd(L, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, h0=None, cu=None, order=None, do=FAKE, dht=None,
             dq=FAKE, dk=FAKE, dv=FAKE, dg=FAKE, db=FAKE, dh0=None, N=2, T=64, h_qk=2, h_v=4, d_k=128,
             d_v=128, dtq=1, dtd=1, scale=0.0, ws=FAKE, ws_bytes=None)
    a.update(kw)
    if a["ws_bytes"] is None:
        a["ws_bytes"] = L.gdn_chunk_bwd_workspace_size(a["N"], a["T"], a["h_qk"], a["h_v"], a["d_k"], a["d_v"])
    return L.gdn_chunk_bwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["h0"], a["cu"], a["order"], a["do"],
                           a["dht"], a["dq"], a["dk"], a["dv"], a["dg"], a["db"], a["dh0"], a["N"], a["T"],
                           a["h_qk"], a["h_v"], a["d_k"], a["d_v"], a["dtq"], a["dtd"], a["scale"], a["ws"],
                           a["ws_bytes"], None)


# Every case below has at least one invalid argument, so nothing is launched.
@pytest.mark.parametrize("kw,status", [
    (dict(ws_bytes=0), INVALID),                 # workspace too small
    (dict(ws=None), INVALID),
    (dict(ws=FAKE + 16), INVALID),               # workspace needs 256 bytes
    (dict(q=None), INVALID),
    (dict(do=FAKE + 8), INVALID),
    (dict(dq=FAKE + 4), INVALID),                # gradients need 16 bytes
    (dict(dg=FAKE + 2), INVALID),
    (dict(dh0=FAKE + 8), INVALID),
    (dict(dht=FAKE + 4), INVALID),
    (dict(h_qk=3), INVALID),
    (dict(dtd=2), INVALID),
    (dict(N=3, T=64), INVALID),                  # equal lengths need T % N == 0
    (dict(d_k=64, d_v=64), UNSUPPORTED),         # only d = 128 is compiled
    (dict(d_v=96), UNSUPPORTED),
    (dict(N=0, T=0), OK),                        # nothing to do
    (dict(N=0, T=4), INVALID),
])
def test_chunk_bwd_host_validation(L, kw, status):
    assert _bwd(L, **kw) == status


def test_chunk_bwd_workspace_size(L):
    f = L.gdn_chunk_bwd_workspace_size
    st = 128 * 128 * 4
    up = lambda x: (x + 255) // 256 * 256
    # checkpoints: H_v * (T/32 + N + 1) states; per token and value head the error
    # vector and one scalar; grouped heads add two [T, H_v, 128] fp32 parts
    assert f(4, 16384, 16, 32, 128, 128) == (32 * (512 + 5) * st + 2 * 16384 * 32 * 128 * 4
                                             + 16384 * 32 * 128 * 4 + 16384 * 32 * 4)
    assert f(1, 100, 4, 4, 128, 128) == 4 * (3 + 2) * st + 100 * 4 * 128 * 4 + up(100 * 4 * 4)
    assert f(0, 0, 1, 1, 128, 128) == 1 * st
    assert f(-1, 0, 1, 1, 128, 128) == 0 and f(1, 10, 3, 4, 128, 128) == 0
    assert gdn.chunk_bwd_workspace_size(4, 16384, 16, 32) == f(4, 16384, 16, 32, 128, 128)


@pytest.mark.parametrize("gate,nw,eps,status", [
    (None, None, 1e-6, INVALID),                 # the gated call needs a gate
    (FAKE + 8, None, 1e-6, INVALID),             # gate read 16 bytes at a time
    (FAKE, FAKE + 4, 1e-6, INVALID),             # norm weight too
    (FAKE, None, -1.0, INVALID),                 # eps >= 0
    (FAKE, None, float("nan"), INVALID),
])
def test_chunk_fwd_gated_host_validation(L, gate, nw, eps, status):
    st = L.gdn_chunk_fwd_gated(FAKE, FAKE, FAKE, FAKE, FAKE, None, None, None, FAKE, gate, nw, eps, None, 1, 64, 2, 4,
                               128, 128, 1, 1, 0.0, 0, 0, None)
    assert st == status


def test_chunk_fwd_workspace_size_is_zero(L):
    """The prefill keeps every intermediate on chip: no workspace for any size
    (the prefill, long and varlen workloads, a tiny fp32 case, invalid sizes)."""
    f = L.gdn_chunk_fwd_workspace_size
    assert f(4, 16384, 16, 32, 128, 128, 1) == 0
    assert f(1, 65536, 16, 32, 128, 128, 1) == 0
    assert f(64, 243613, 16, 32, 128, 128, 1) == 0
    assert f(1, 64, 2, 2, 16, 16, 0) == 0
    assert f(-1, 0, 1, 1, 128, 128, 1) == 0
    assert gdn.chunk_fwd_workspace_size(4, 16384, 16, 32) == 0


@pytest.mark.parametrize("kw,status", [
    (dict(T=1 << 31, N=1), UNSUPPORTED),         # more tokens than int32 cu_seqlens can index
    (dict(h_qk=3), INVALID),
    (dict(N=-1), INVALID),
    (dict(dq=5), INVALID),
    (dict(d_k=64), UNSUPPORTED),
    (dict(N=3, T=100), INVALID),                 # equal lengths need T % N == 0
    (dict(g=FAKE + 2), INVALID),
    (dict(N=0, T=0), OK),
    (dict(N=0, T=4), INVALID),
])
def test_chunk_bwd_static_refuses_like_chunk_bwd(L, kw, status):
    """The allocation-free gradient entry point runs the same host checks as
    gdn_chunk_bwd, in the same order, so both give one status for one bad
    argument (nothing reaches the device in any case below)."""
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, h0=None, cu=None, order=None, do=FAKE, dht=None,
             dq_=FAKE, dk_=FAKE, dv_=FAKE, dg_=FAKE, db_=FAKE, dh0=None, N=1, T=100, h_qk=4, h_v=4, d_k=128,
             d_v=128, dq=1, ddo=1, scale=0.0)
    a.update(kw)
    args = [a[n] for n in ("q", "k", "v", "g", "beta", "h0", "cu", "order", "do", "dht", "dq_", "dk_", "dv_",
                           "dg_", "db_", "dh0", "N", "T", "h_qk", "h_v", "d_k", "d_v", "dq", "ddo", "scale")]
    assert L.gdn_chunk_bwd_static(*args, None) == status
    assert L.gdn_chunk_bwd(*args, None, 0, None) == status


def _kda(L, **kw):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, h0=None, cu=None, order=None, o=FAKE, hT=FAKE, N=2,
             T=64, h_qk=2, h_v=4, d_k=128, d_v=128, dq=1, do=1, scale=0.0)
    a.update(kw)
    return L.gdn_kda_chunk_fwd(a["q"], a["k"], a["v"], a["g"], a["beta"], a["h0"], a["cu"], a["order"], a["o"],
                               a["hT"], a["N"], a["T"], a["h_qk"], a["h_v"], a["d_k"], a["d_v"], a["dq"], a["do"],
                               a["scale"], None)


# Every case below has at least one invalid argument, so nothing is launched.
@pytest.mark.parametrize("kw,status", [
    (dict(g=FAKE + 4), INVALID),                 # per-channel g is read 16 bytes at a time
    (dict(q=None), INVALID),
    (dict(hT=FAKE + 8), INVALID),
    (dict(h_qk=3), INVALID),
    (dict(dq=2), INVALID),
    (dict(N=3, T=64), INVALID),
    (dict(d_k=64, d_v=64), UNSUPPORTED),
    (dict(N=0, T=0), OK),
])
def test_kda_chunk_fwd_host_validation(L, kw, status):
    assert _kda(L, **kw) == status


@pytest.mark.parametrize("kw,status", [
    (dict(state=FAKE + 4), INVALID),
    (dict(q=FAKE + 2), INVALID),                 # q, k are read 4 elements at a time
    (dict(d_v=64), UNSUPPORTED),
    (dict(N=0), OK),
])
def test_kda_decode_host_validation(L, kw, status):
    a = dict(q=FAKE, k=FAKE, v=FAKE, g=FAKE, beta=FAKE, state=FAKE, o=FAKE, N=4, h_qk=2, h_v=4, d_k=128,
             d_v=128, dq=1, do=1, scale=0.0)
    a.update(kw)
    assert L.gdn_kda_decode_step(a["q"], a["k"], a["v"], a["g"], a["beta"], a["state"], a["o"], a["N"], a["h_qk"],
                                 a["h_v"], a["d_k"], a["d_v"], a["dq"], a["do"], a["scale"], None) == status


def test_binding_rejects_bad_shapes():
    """Shapes are checked in the binding before anything reaches the C ABI
    (which only sees pointers): a too-small tensor raises ValueError."""
    T, hq, hv, d = 6, 1, 2, 8
    q = torch.zeros(T, hq, d)
    v = torch.zeros(T, hv, d)
    g = torch.zeros(T, hv)
    with pytest.raises(ValueError, match="g must"):
        gdn.chunk_fwd(q, q, v, g[:, :1], g)
    with pytest.raises(ValueError, match="initial_state"):
        gdn.chunk_fwd(q, q, v, g, g, torch.zeros(1, hv, d, d - 1))
    with pytest.raises(ValueError, match="d_o"):
        gdn.chunk_bwd(q, q, v, g, g, v[:5])
    with pytest.raises(ValueError, match="d_final_state"):
        gdn.chunk_bwd(q, q, v, g, g, v, None, torch.zeros(2, hv, d, d))
    with pytest.raises(ValueError, match="g must"):
        gdn.kda_chunk_fwd(q, q, v, g, g)
    with pytest.raises(ValueError, match="g must"):
        gdn.kda_decode_step(q[:2], q[:2], v[:2], torch.zeros(2, hv, d - 1), g[:2], torch.zeros(2, hv, d, d))
    with pytest.raises(ValueError, match="state must"):
        gdn.decode_step(q[:2], q[:2], v[:2], g[:2], g[:2], torch.zeros(3, hv, d, d))
    with pytest.raises(ValueError, match="k must"):
        gdn.chunk_fwd(q, q[:, :, :4], v, g, g)


C_PROGRAM = r"""
#include <stdio.h>
#include "gdn.h"
int main(void) {
    int32_t order[3];
    const int32_t cu[4] = {0, 5, 17, 20};
    gdn_status st = gdn_plan_seq_order(cu, 3, order);
    printf("%d %s %zu %d %d %d %d %zu\n", (int)gdn_version(), gdn_status_string(GDN_ERR_UNSUPPORTED),
           gdn_chunk_bwd_workspace_size(1, 100, 4, 4, 128, 128), (int)st, order[0], order[1], order[2],
           gdn_chunk_fwd_workspace_size(4, 16384, 16, 32, 128, 128, GDN_BF16));
    return st == GDN_OK ? 0 : 1;
}
"""


def test_header_is_plain_c_and_links(L, tmp_path):
    """include/gdn.h compiles as strict C11 (no C++ or torch types in the
    boundary) and a C program links libgdn.so and calls its host-only entry
    points."""
    import shutil
    import subprocess
    if shutil.which("gcc") is None:
        pytest.skip("gcc not available")
    src = tmp_path / "t.c"
    src.write_text(C_PROGRAM)
    exe = tmp_path / "t"
    libdir = os.path.dirname(gbuild.LIB)
    subprocess.run(["gcc", "-std=c11", "-Wall", "-Wextra", "-pedantic", "-Werror", "-I", os.path.join(ROOT, "include"),
                    "-o", str(exe), str(src), "-L", libdir, "-lgdn", f"-Wl,-rpath,{libdir}"], check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    assert int(out[0]) == L.gdn_version()
    assert out[1] == "GDN_ERR_UNSUPPORTED"
    assert int(out[2]) == L.gdn_chunk_bwd_workspace_size(1, 100, 4, 4, 128, 128)
    assert out[3:7] == ["0", "1", "0", "2"]   # lengths 5, 12, 3: longest first
    assert out[7] == "0"                       # the prefill needs no workspace
