"""B300-native Gated DeltaNet forward recurrence: Python binding of libgdn.so.

The operation (see include/gdn.h for the full contract): per sequence and value
head, with the fp32 state S of shape d_k x d_v,

    S_t = exp(g_t) (I - beta_t k_t k_t^T) S_{t-1} + beta_t k_t v_t^T
    o_t = scale S_t^T q_t

This module only marshals arguments: it allocates outputs with torch (device
memory and streams are torch's job here) and passes raw device pointers to the
C ABI. Every step of the computation runs in the library's CUDA kernels; there
is no CPU or PyTorch fallback, and a missing or unloadable library raises.

Entry points (same names as the C ABI, without the ``gdn_`` prefix):
  chunk_fwd(q, k, v, g, beta, ...)          prefill -> (o, final_state)
  decode_step(q, k, v, g, beta, state, ...) one token, state updated in place
  plan_seq_order(cu_seqlens)                longest-first schedule (host)
  get_device_error(stream=None)             device-side error bits
"""
from __future__ import annotations

import ctypes
import os
from typing import Optional

import torch

__all__ = ["chunk_fwd", "decode_step", "plan_seq_order", "get_device_error", "lib",
           "GdnError", "LIB_PATH", "F32", "BF16", "FLAG_FORCE_SIMT", "FLAG_TEST_WAIT_TIMEOUT", "FLAG_NO_SPLIT",
           "FLAG_BALANCE", "DEVERR_SEQLENS", "DEVERR_TIMEOUT", "DEVERR_RANGE"]

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libgdn.so")
F32, BF16 = 0, 1
FLAG_FORCE_SIMT = 1
FLAG_TEST_WAIT_TIMEOUT = 2   # failure-path tests only (see include/gdn.h)
FLAG_NO_SPLIT = 4            # one CTA per (sequence, value head): no sequence segments
FLAG_BALANCE = 8             # balanced shares of chunks for any equal-length batch (tests of the share logic)
DEVERR_SEQLENS, DEVERR_TIMEOUT, DEVERR_RANGE = 1, 2, 4
_STATUS = {0: "GDN_OK", 1: "GDN_ERR_INVALID_ARG", 2: "GDN_ERR_UNSUPPORTED", 3: "GDN_ERR_CUDA",
           4: "GDN_ERR_TIMEOUT"}
_lib = None


class GdnError(RuntimeError):
    def __init__(self, fn: str, status: int):
        super().__init__(f"{fn} returned {_STATUS.get(status, status)}")
        self.status = status


def lib():
    """Load libgdn.so (built in-tree by ``build.py``); raises if it is missing."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise ImportError(f"libgdn.so not found at {LIB_PATH}; run "
                              "`python gated_deltanet_recurrence_05_b300/build.py`")
        L = ctypes.CDLL(LIB_PATH)
        P, I32, I64, F = ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float
        L.gdn_chunk_fwd.argtypes = [P, P, P, P, P, P, P, P, P, P, I32, I64, I32, I32, I32, I32,
                                    I32, I32, F, I32, I32, P]
        L.gdn_chunk_fwd.restype = ctypes.c_int
        L.gdn_chunk_fwd_gated.argtypes = [P, P, P, P, P, P, P, P, P, P, P, F, P, I32, I64, I32, I32, I32, I32,
                                          I32, I32, F, I32, I32, P]
        L.gdn_chunk_fwd_gated.restype = ctypes.c_int
        L.gdn_decode_step.argtypes = [P, P, P, P, P, P, P, I32, I32, I32, I32, I32, I32, I32, F, P]
        L.gdn_decode_step.restype = ctypes.c_int
        L.gdn_decode_step_gated.argtypes = [P, P, P, P, P, P, P, P, P, F, I32, I32, I32, I32, I32, I32,
                                            I32, F, P]
        L.gdn_decode_step_gated.restype = ctypes.c_int
        L.gdn_gated_rmsnorm.argtypes = [P, P, P, P, I64, I32, I32, I32, F, P]
        L.gdn_gated_rmsnorm.restype = ctypes.c_int
        L.gdn_short_conv.argtypes = [P, P, P, P, P, P, I32, I64, I32, I32, I32, F, I32, P]
        L.gdn_short_conv.restype = ctypes.c_int
        L.gdn_short_conv_step.argtypes = [P, P, P, P, I32, I32, I32, I32, F, I32, P]
        L.gdn_short_conv_step.restype = ctypes.c_int
        L.gdn_chunk_bwd.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, I32, I64, I32, I32,
                                    I32, I32, I32, I32, F, P, ctypes.c_size_t, P]
        L.gdn_chunk_bwd.restype = ctypes.c_int
        L.gdn_chunk_bwd_static.argtypes = [P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, P, I32, I64, I32,
                                           I32, I32, I32, I32, I32, F, P]
        L.gdn_chunk_bwd_static.restype = ctypes.c_int
        L.gdn_chunk_bwd_workspace_size.argtypes = [I32, I64, I32, I32, I32, I32]
        L.gdn_chunk_fwd_workspace_size.argtypes = [I32, I64, I32, I32, I32, I32, I32]
        L.gdn_chunk_fwd_workspace_size.restype = ctypes.c_size_t
        L.gdn_kda_chunk_fwd.argtypes = [P, P, P, P, P, P, P, P, P, P, I32, I64, I32, I32, I32, I32, I32, I32,
                                        F, P]
        L.gdn_kda_chunk_fwd.restype = ctypes.c_int
        L.gdn_kda_decode_step.argtypes = [P, P, P, P, P, P, P, I32, I32, I32, I32, I32, I32, I32, F, P]
        L.gdn_kda_decode_step.restype = ctypes.c_int
        L.gdn_chunk_bwd_workspace_size.restype = ctypes.c_size_t
        L.gdn_plan_seq_order.argtypes = [P, I32, P]
        L.gdn_plan_seq_order.restype = ctypes.c_int
        L.gdn_get_device_error.argtypes = [P, P]
        L.gdn_get_device_error.restype = ctypes.c_int
        L.gdn_status_string.argtypes = [ctypes.c_int]
        L.gdn_status_string.restype = ctypes.c_char_p
        L.gdn_version.restype = I32
        _lib = L
    return _lib


def _code(t: torch.Tensor) -> int:
    if t.dtype == torch.bfloat16:
        return BF16
    if t.dtype == torch.float32:
        return F32
    raise TypeError(f"unsupported dtype {t.dtype}; expected float32 or bfloat16")


def _ptr(t: Optional[torch.Tensor]):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _dev(t: torch.Tensor, name: str):
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")


def _shape(t: Optional[torch.Tensor], shape, name: str):
    """Raise unless t (when given) has exactly this shape: the C ABI takes bare
    pointers and sizes, so a tensor smaller than the sizes imply would be read
    past its end."""
    if t is not None and tuple(t.shape) != tuple(int(x) for x in shape):
        raise ValueError(f"{name} must have shape {tuple(int(x) for x in shape)}, got {tuple(t.shape)}")


def _shapes_prefill(q, k, v, g, beta, N, h0=None, g_per_channel=False, h0_name="initial_state"):
    """Shape checks shared by the prefill-style calls: q, k [T, H_qk, d_k];
    v [T, H_v, d_v]; g [T, H_v] (or [T, H_v, d_k] per channel); beta [T, H_v];
    h0 [N, H_v, d_k, d_v]. Returns (T, h_qk, h_v, d_k, d_v)."""
    if q.dim() != 3 or v.dim() != 3:
        raise ValueError("q, k must be [T, H_qk, d_k] and v [T, H_v, d_v]")
    T, h_qk, d_k = q.shape
    h_v, d_v = v.shape[1], v.shape[2]
    _shape(k, q.shape, "k")
    _shape(v, (T, h_v, d_v), "v")
    _shape(g, (T, h_v, d_k) if g_per_channel else (T, h_v), "g")
    _shape(beta, (T, h_v), "beta")
    _shape(h0, (N, h_v, d_k, d_v), h0_name)
    return T, h_qk, h_v, d_k, d_v


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _check(fn: str, status: int):
    if status != 0:
        raise GdnError(fn, status)


def chunk_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
              beta: torch.Tensor, initial_state: Optional[torch.Tensor] = None,
              cu_seqlens: Optional[torch.Tensor] = None, *, num_seqs: Optional[int] = None,
              seq_order: Optional[torch.Tensor] = None, output_dtype: Optional[torch.dtype] = None,
              scale: float = 0.0, chunk_size: int = 0, output_final_state: bool = True,
              out: Optional[torch.Tensor] = None, final_state_out: Optional[torch.Tensor] = None,
              force_simt: bool = False, test_wait_timeout: bool = False, split: bool = True,
              balance: bool = False, gate: Optional[torch.Tensor] = None, norm_weight: Optional[torch.Tensor] = None,
              eps: float = 1e-6, stream=None):
    """Prefill of the recurrence over packed tokens (see include/gdn.h).

    q, k: [T, H_qk, d_k]; v: [T, H_v, d_v] (fp32 or bf16, one dtype); g, beta:
    [T, H_v] fp32; initial_state: [N, H_v, d_k, d_v] fp32 or None; cu_seqlens:
    [N+1] int32 CUDA tensor or None (then ``num_seqs`` equal-length sequences,
    default 1). Returns (o [T, H_v, d_v], final_state or None). With ``gate``
    ([T, H_v, d_v], the dtype of q/k/v) the output goes through the layer's
    epilogue (gdn_chunk_fwd_gated: zero-centred RMSNorm with ``norm_weight``
    [d_v] fp32 or None, times sigmoid(gate)).
    """
    N = cu_seqlens.numel() - 1 if cu_seqlens is not None else (1 if num_seqs is None else int(num_seqs))
    T, h_qk, h_v, d_k, d_v = _shapes_prefill(q, k, v, g, beta, N, initial_state)
    _shape(seq_order, (N,), "seq_order")
    _shape(out, (T, h_v, d_v), "out")
    _shape(final_state_out, (N, h_v, d_k, d_v), "final_state_out")
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta)):
        _dev(t, name)
    if cu_seqlens is not None:
        _dev(cu_seqlens, "cu_seqlens")
        if cu_seqlens.dtype != torch.int32:
            raise TypeError("cu_seqlens must be int32")
    if seq_order is not None:
        _dev(seq_order, "seq_order")
    if initial_state is not None:
        _dev(initial_state, "initial_state")
    if g.dtype != torch.float32 or beta.dtype != torch.float32:
        raise TypeError("g and beta must be float32")
    odt = output_dtype or v.dtype
    o = out if out is not None else torch.empty((T, h_v, d_v), dtype=odt, device=v.device)
    fs = None
    if output_final_state:
        fs = final_state_out if final_state_out is not None else torch.empty(
            (N, h_v, d_k, d_v), dtype=torch.float32, device=v.device)
    flags = ((FLAG_FORCE_SIMT if force_simt else 0) | (FLAG_TEST_WAIT_TIMEOUT if test_wait_timeout else 0) |
             (0 if split else FLAG_NO_SPLIT) | (FLAG_BALANCE if balance else 0))
    if gate is None:
        if norm_weight is not None:
            raise ValueError("norm_weight needs a gate")
        st = lib().gdn_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state),
                                 _ptr(cu_seqlens), _ptr(seq_order), _ptr(o), _ptr(fs), N, T, h_qk, h_v,
                                 d_k, d_v, _code(q), _code(o), float(scale), int(chunk_size), flags,
                                 _stream(stream))
        _check("gdn_chunk_fwd", st)
        return o, fs
    _shape(gate, (T, h_v, d_v), "gate")
    _shape(norm_weight, (d_v,), "norm_weight")
    _dev(gate, "gate")
    if gate.dtype != q.dtype:
        raise TypeError("gate must have the dtype of q, k, v")
    if norm_weight is not None:
        _dev(norm_weight, "norm_weight")
        if norm_weight.dtype != torch.float32:
            raise TypeError("norm_weight must be float32")
    st = lib().gdn_chunk_fwd_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state),
                                   _ptr(cu_seqlens), _ptr(seq_order), _ptr(o), _ptr(gate), _ptr(norm_weight),
                                   float(eps), _ptr(fs), N, T, h_qk, h_v, d_k, d_v, _code(q), _code(o),
                                   float(scale), int(chunk_size), flags, _stream(stream))
    _check("gdn_chunk_fwd_gated", st)
    return o, fs


def chunk_fwd_workspace_size(num_seqs: int, total_tokens: int, h_qk: int, h_v: int, d_k: int = 128,
                             d_v: int = 128, dtype: torch.dtype = torch.bfloat16) -> int:
    """Bytes of device workspace ``chunk_fwd`` needs for these sizes (0: the
    prefill keeps every intermediate on chip)."""
    return int(lib().gdn_chunk_fwd_workspace_size(int(num_seqs), int(total_tokens), int(h_qk), int(h_v),
                                                  int(d_k), int(d_v), BF16 if dtype == torch.bfloat16 else F32))


def chunk_bwd_workspace_size(num_seqs: int, total_tokens: int, h_qk: int, h_v: int, d_k: int = 128,
                             d_v: int = 128) -> int:
    """Bytes of device workspace ``chunk_bwd`` needs for these sizes."""
    return int(lib().gdn_chunk_bwd_workspace_size(int(num_seqs), int(total_tokens), int(h_qk), int(h_v),
                                                  int(d_k), int(d_v)))


def chunk_bwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
              d_o: torch.Tensor, initial_state: Optional[torch.Tensor] = None,
              d_final_state: Optional[torch.Tensor] = None, cu_seqlens: Optional[torch.Tensor] = None, *,
              num_seqs: Optional[int] = None, seq_order: Optional[torch.Tensor] = None, scale: float = 0.0,
              need_d_initial_state: bool = True, workspace: Optional[torch.Tensor] = None, out=None,
              stream=None):
    """Gradient of the recurrence (see include/gdn.h, gdn_chunk_bwd).

    Forward inputs as for ``chunk_fwd``; d_o: [T, H_v, d_v] (fp32 or bf16);
    d_final_state: [N, H_v, d_k, d_v] fp32 or None. ``workspace`` is a CUDA
    uint8 tensor of at least ``chunk_bwd_workspace_size`` bytes (allocated
    here when None). ``out`` may give the six output tensors. Returns
    (dq, dk, dv, dg, dbeta, d_initial_state or None), all fp32.
    """
    N = cu_seqlens.numel() - 1 if cu_seqlens is not None else (1 if num_seqs is None else int(num_seqs))
    T, h_qk, h_v, d_k, d_v = _shapes_prefill(q, k, v, g, beta, N, initial_state)
    _shape(d_o, (T, h_v, d_v), "d_o")
    _shape(d_final_state, (N, h_v, d_k, d_v), "d_final_state")
    _shape(seq_order, (N,), "seq_order")
    if out is not None:
        for t, shp, name in zip(out, ((T, h_qk, d_k), (T, h_qk, d_k), (T, h_v, d_v), (T, h_v), (T, h_v),
                                      (N, h_v, d_k, d_v)), ("dq", "dk", "dv", "dg", "dbeta", "d_initial_state")):
            _shape(t, shp, f"out {name}")
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("d_o", d_o)):
        _dev(t, name)
    if cu_seqlens is not None:
        _dev(cu_seqlens, "cu_seqlens")
        if cu_seqlens.dtype != torch.int32:
            raise TypeError("cu_seqlens must be int32")
    for name, t in (("seq_order", seq_order), ("initial_state", initial_state),
                    ("d_final_state", d_final_state)):
        if t is not None:
            _dev(t, name)
    if g.dtype != torch.float32 or beta.dtype != torch.float32:
        raise TypeError("g and beta must be float32")
    if q.dtype != k.dtype or q.dtype != v.dtype:
        raise TypeError("q, k and v must share one dtype")
    dev = v.device
    f32 = dict(dtype=torch.float32, device=dev)
    if out is not None:
        dq, dk, dv, dg, db, dh0 = out
    else:
        dq = torch.empty((T, h_qk, d_k), **f32)
        dk = torch.empty((T, h_qk, d_k), **f32)
        dv = torch.empty((T, h_v, d_v), **f32)
        dg = torch.empty((T, h_v), **f32)
        db = torch.empty((T, h_v), **f32)
        dh0 = torch.empty((N, h_v, d_k, d_v), **f32) if need_d_initial_state else None
    need = chunk_bwd_workspace_size(N, T, h_qk, h_v, d_k, d_v)
    if workspace is None:
        workspace = torch.empty(max(need, 256), dtype=torch.uint8, device=dev)
    _dev(workspace, "workspace")
    st = lib().gdn_chunk_bwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state),
                             _ptr(cu_seqlens), _ptr(seq_order), _ptr(d_o), _ptr(d_final_state), _ptr(dq),
                             _ptr(dk), _ptr(dv), _ptr(dg), _ptr(db), _ptr(dh0), N, T, h_qk, h_v, d_k, d_v,
                             _code(q), _code(d_o), float(scale), _ptr(workspace),
                             workspace.numel() * workspace.element_size(), _stream(stream))
    _check("gdn_chunk_bwd", st)
    return dq, dk, dv, dg, db, dh0


def kda_chunk_fwd(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
                  initial_state: Optional[torch.Tensor] = None, cu_seqlens: Optional[torch.Tensor] = None, *,
                  num_seqs: Optional[int] = None, seq_order: Optional[torch.Tensor] = None,
                  output_dtype: Optional[torch.dtype] = None, scale: float = 0.0, output_final_state: bool = True,
                  out: Optional[torch.Tensor] = None, final_state_out: Optional[torch.Tensor] = None, stream=None):
    """Prefill of the per-channel-decay rule (KDA; see include/gdn.h). As
    ``chunk_fwd`` except g: [T, H_v, d_k] fp32 (one log-decay per key channel)."""
    N = cu_seqlens.numel() - 1 if cu_seqlens is not None else (1 if num_seqs is None else int(num_seqs))
    T, h_qk, h_v, d_k, d_v = _shapes_prefill(q, k, v, g, beta, N, initial_state, g_per_channel=True)
    _shape(seq_order, (N,), "seq_order")
    _shape(out, (T, h_v, d_v), "out")
    _shape(final_state_out, (N, h_v, d_k, d_v), "final_state_out")
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta)):
        _dev(t, name)
    if cu_seqlens is not None:
        _dev(cu_seqlens, "cu_seqlens")
        if cu_seqlens.dtype != torch.int32:
            raise TypeError("cu_seqlens must be int32")
    for name, t in (("seq_order", seq_order), ("initial_state", initial_state)):
        if t is not None:
            _dev(t, name)
    if g.dtype != torch.float32 or beta.dtype != torch.float32:
        raise TypeError("g and beta must be float32")
    odt = output_dtype or v.dtype
    o = out if out is not None else torch.empty((T, h_v, d_v), dtype=odt, device=v.device)
    fs = None
    if output_final_state:
        fs = final_state_out if final_state_out is not None else torch.empty(
            (N, h_v, d_k, d_v), dtype=torch.float32, device=v.device)
    st = lib().gdn_kda_chunk_fwd(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(initial_state),
                                 _ptr(cu_seqlens), _ptr(seq_order), _ptr(o), _ptr(fs), N, T, h_qk, h_v, d_k,
                                 d_v, _code(q), _code(o), float(scale), _stream(stream))
    _check("gdn_kda_chunk_fwd", st)
    return o, fs


def kda_decode_step(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor, beta: torch.Tensor,
                    state: torch.Tensor, *, output_dtype: Optional[torch.dtype] = None, scale: float = 0.0,
                    out: Optional[torch.Tensor] = None, stream=None):
    """One token of KDA for N sequences, state updated in place. q, k
    [N, H_qk, d_k]; v [N, H_v, d_v]; g [N, H_v, d_k] fp32; beta [N, H_v];
    state [N, H_v, d_k, d_v] fp32. Returns o [N, H_v, d_v]."""
    N, h_qk, h_v, d_k, d_v = _shapes_prefill(q, k, v, g, beta, q.shape[0], state, g_per_channel=True,
                                             h0_name="state")
    _shape(out, (N, h_v, d_v), "out")
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("state", state)):
        _dev(t, name)
    o = out if out is not None else torch.empty((N, h_v, d_v), dtype=output_dtype or v.dtype, device=v.device)
    st = lib().gdn_kda_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state), _ptr(o), N,
                                   h_qk, h_v, d_k, d_v, _code(q), _code(o), float(scale), _stream(stream))
    _check("gdn_kda_decode_step", st)
    return o


def decode_step(q: torch.Tensor, k: torch.Tensor, v: torch.Tensor, g: torch.Tensor,
                beta: torch.Tensor, state: torch.Tensor, *, output_dtype: Optional[torch.dtype] = None,
                scale: float = 0.0, out: Optional[torch.Tensor] = None, gate: Optional[torch.Tensor] = None,
                norm_weight: Optional[torch.Tensor] = None, eps: float = 1e-6, stream=None) -> torch.Tensor:
    """One token for N sequences; ``state`` [N, H_v, d_k, d_v] is updated in place.

    q, k: [N, H_qk, d_k]; v: [N, H_v, d_v]; g, beta: [N, H_v] fp32. Returns o [N, H_v, d_v].
    With ``gate`` ([N, H_v, d_v], dtype of q) the output goes through the gated
    RMSNorm epilogue (``gated_rmsnorm``), fused into the decode kernel for
    d_k = d_v = 128; ``norm_weight`` [d_v] fp32 is its zero-centred weight.
    """
    N, h_qk, h_v, d_k, d_v = _shapes_prefill(q, k, v, g, beta, q.shape[0], state, h0_name="state")
    _shape(out, (N, h_v, d_v), "out")
    for name, t in (("q", q), ("k", k), ("v", v), ("g", g), ("beta", beta), ("state", state)):
        _dev(t, name)
    odt = output_dtype or v.dtype
    o = out if out is not None else torch.empty((N, h_v, d_v), dtype=odt, device=v.device)
    if gate is None:
        if norm_weight is not None:
            raise ValueError("norm_weight needs a gate")
        st = lib().gdn_decode_step(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state), _ptr(o),
                                   N, h_qk, h_v, d_k, d_v, _code(q), _code(o), float(scale),
                                   _stream(stream))
        _check("gdn_decode_step", st)
        return o
    _dev(gate, "gate")
    if gate.dtype != q.dtype or tuple(gate.shape) != (N, h_v, d_v):
        raise ValueError("gate must be [N, H_v, d_v] in the dtype of q")
    if norm_weight is not None:
        _dev(norm_weight, "norm_weight")
    st = lib().gdn_decode_step_gated(_ptr(q), _ptr(k), _ptr(v), _ptr(g), _ptr(beta), _ptr(state), _ptr(o),
                                     _ptr(gate), _ptr(norm_weight), float(eps), N, h_qk, h_v, d_k, d_v,
                                     _code(q), _code(o), float(scale), _stream(stream))
    _check("gdn_decode_step_gated", st)
    return o


def gated_rmsnorm(x: torch.Tensor, gate: torch.Tensor, norm_weight: Optional[torch.Tensor] = None, *,
                  eps: float = 1e-6, out: Optional[torch.Tensor] = None,
                  output_dtype: Optional[torch.dtype] = None, stream=None) -> torch.Tensor:
    """GDN output epilogue over the last axis: x / rms(x) * (1 + norm_weight) * sigmoid(gate).

    x, gate: [..., d] (same shape and dtype; e.g. the prefill output [T, H_v, d_v]);
    norm_weight: [d] fp32 or None. ``out`` may be ``x`` itself (in place).
    """
    _dev(x, "x")
    _dev(gate, "gate")
    if gate.dtype != x.dtype or gate.shape != x.shape:
        raise ValueError("gate must match x in shape and dtype")
    if norm_weight is not None:
        _dev(norm_weight, "norm_weight")
    d = x.shape[-1]
    rows = x.numel() // d if d else 0
    y = out if out is not None else torch.empty(x.shape, dtype=output_dtype or x.dtype, device=x.device)
    st = lib().gdn_gated_rmsnorm(_ptr(x), _ptr(gate), _ptr(norm_weight), _ptr(y), rows, d, _code(x), _code(y),
                                 float(eps), _stream(stream))
    _check("gdn_gated_rmsnorm", st)
    return y


def plan_seq_order(cu_seqlens) -> torch.Tensor:
    """Longest-first schedule of the sequences (host computation in the library).

    Accepts a CPU tensor / list of N+1 offsets; returns an int32 CPU tensor [N]."""
    cu = torch.as_tensor(cu_seqlens, dtype=torch.int32).cpu().contiguous()
    N = cu.numel() - 1
    order = torch.empty(max(N, 0), dtype=torch.int32)
    _check("gdn_plan_seq_order", lib().gdn_plan_seq_order(_ptr(cu), N, _ptr(order)))
    return order


def get_device_error(stream=None) -> int:
    """Synchronise the stream and return (and clear) the GDN_DEVERR_* bits.
    (The C call's GDN_ERR_TIMEOUT status mirrors the DEVERR_TIMEOUT bit, which
    is returned here like the other bits.)"""
    code = ctypes.c_uint32(0)
    st = lib().gdn_get_device_error(_stream(stream), ctypes.byref(code))
    if st != 4:
        _check("gdn_get_device_error", st)
    return int(code.value)


def short_conv(x: torch.Tensor, w: torch.Tensor, *, cu_seqlens: Optional[torch.Tensor] = None,
               num_seqs: Optional[int] = None, conv_state: Optional[torch.Tensor] = None,
               return_final_state: bool = False, norm_group: int = 0, eps: float = 1e-6,
               out: Optional[torch.Tensor] = None, stream=None):
    """GDN input prologue on one projected tensor: causal depthwise conv over the
    tokens of each sequence, silu, and (norm_group > 0) an L2 norm per head.

    x: [T, C] or [T, H, d] (C = H d); w: [C, K] fp32, K <= 4; cu_seqlens: [N + 1]
    int32 (CUDA) or None with ``num_seqs`` equal-length sequences (default 1);
    conv_state: [N, C, K - 1] fp32, the inputs preceding each sequence. Returns y
    (shape of x) and, with ``return_final_state``, the [N, C, K - 1] final state.
    """
    _dev(x, "x")
    _dev(w, "w")
    T = x.shape[0]
    C = x.numel() // T if T else int(w.shape[0])
    K = int(w.shape[1])
    if cu_seqlens is not None:
        _dev(cu_seqlens, "cu_seqlens")
        N = cu_seqlens.numel() - 1
    else:
        N = 1 if num_seqs is None else int(num_seqs)
    if conv_state is not None:
        _dev(conv_state, "conv_state")
    y = out if out is not None else torch.empty_like(x)
    fs = torch.empty(N, C, K - 1, dtype=torch.float32, device=x.device) if return_final_state else None
    st = lib().gdn_short_conv(_ptr(x), _ptr(w), _ptr(y), _ptr(cu_seqlens), _ptr(conv_state), _ptr(fs), N, T, C, K,
                              int(norm_group), float(eps), _code(x), _stream(stream))
    _check("gdn_short_conv", st)
    return (y, fs) if return_final_state else y


def short_conv_step(x: torch.Tensor, w: torch.Tensor, conv_state: torch.Tensor, *, norm_group: int = 0,
                    eps: float = 1e-6, out: Optional[torch.Tensor] = None, stream=None) -> torch.Tensor:
    """The prologue for one token per sequence (decode): x [N, C] or [N, H, d];
    ``conv_state`` [N, C, K - 1] fp32 is shifted in place. Returns y (shape of x)."""
    _dev(x, "x")
    _dev(w, "w")
    _dev(conv_state, "conv_state")
    N = x.shape[0]
    C = x.numel() // N if N else int(w.shape[0])
    y = out if out is not None else torch.empty_like(x)
    st = lib().gdn_short_conv_step(_ptr(x), _ptr(w), _ptr(conv_state), _ptr(y), N, C, int(w.shape[1]),
                                   int(norm_group), float(eps), _code(x), _stream(stream))
    _check("gdn_short_conv_step", st)
    return y

