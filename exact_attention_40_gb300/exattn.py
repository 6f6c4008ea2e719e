"""Thin ctypes binding of libexattn.so (C ABI in include/exattn.h).

Argument marshalling only: every step of the computation runs in the CUDA
kernels behind the C ABI.  PyTorch supplies device memory and the stream.
Importing this module loads the library and raises if it has not been
built (``python -m exact_attention_40_gb300.build``) -- there is no
fallback path.

The functions carry the C names.  ``attn_fwd`` and ``attn_decode_paged``
take torch tensors, allocate outputs when none are given, and raise
``ExattnError`` on a non-zero status.  ``lib`` is the raw ctypes handle for
callers (and tests) that pass pointers themselves.
"""
from __future__ import annotations

import contextlib
import ctypes
import math
import os

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "libexattn.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        "libexattn.so is not built (%s); run `python -m exact_attention_40_gb300.build`" % LIB_PATH)

lib = ctypes.CDLL(LIB_PATH)

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float
_SZ = ctypes.c_size_t

lib.attn_fwd.argtypes = [_P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P]
lib.attn_fwd.restype = _I
lib.attn_decode_workspace_bytes.argtypes = [_I, _I, _I, _I, _I]
lib.attn_decode_workspace_bytes.restype = _SZ
lib.attn_decode_paged.argtypes = [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F, _P,
                                  _SZ, _P]
lib.attn_decode_paged.restype = _I
lib.attn_decode_paged_static.argtypes = [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                                         _F, _P]
lib.attn_decode_paged_static.restype = _I
lib.attn_get_device_status.argtypes = [_P, ctypes.POINTER(ctypes.c_int)]
lib.attn_get_device_status.restype = _I
lib.attn_status_string.argtypes = [_I]
lib.attn_status_string.restype = ctypes.c_char_p
lib.attn_decode_split_tokens.argtypes = []
lib.attn_decode_split_tokens.restype = _I
lib.attn_debug_expire_wait.argtypes = [ctypes.c_ulonglong, _P]
lib.attn_debug_expire_wait.restype = _I
lib.attn_add_rms_norm.argtypes = [_P, _P, _P, _P, _P, _I, _I, _F, _P]
lib.attn_add_rms_norm.restype = _I
lib.attn_rope_cache_write.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I,
                                      _F, _P]
lib.attn_rope_cache_write.restype = _I
lib.attn_decode_graph_capture.argtypes = [_P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _I, _F,
                                          _P, _SZ, ctypes.POINTER(ctypes.c_void_p)]
lib.attn_decode_graph_capture.restype = _I
lib.attn_graph_launch.argtypes = [_P, _P]
lib.attn_graph_launch.restype = _I
lib.attn_graph_destroy.argtypes = [_P]
lib.attn_graph_destroy.restype = _I
lib.attn_bwd_workspace_bytes.argtypes = [_I, _I, _I, _I, _I, _I]
lib.attn_bwd_workspace_bytes.restype = _SZ
lib.attn_bwd.argtypes = [_P, _P, _P, _P, _P, _P, _P, _P, _P, _I, _I, _I, _I, _I, _I, _F, _I, _P, _SZ, _P]
lib.attn_bwd.restype = _I
lib.attn_shutdown.argtypes = []
lib.attn_shutdown.restype = None

EXATTN_OK = 0
DEVICE_TIMEOUT_BIT = 1
DEVICE_BOUNDS_BIT = 2


class ExattnError(RuntimeError):
    def __init__(self, fn, status):
        super().__init__("%s failed: %s" % (fn, attn_status_string(status)))
        self.status = status


def attn_status_string(status: int) -> str:
    return lib.attn_status_string(int(status)).decode()


def attn_decode_split_tokens() -> int:
    return lib.attn_decode_split_tokens()


def attn_decode_workspace_bytes(num_seqs, Hq, d, max_blocks_per_seq, block_size=16) -> int:
    return int(lib.attn_decode_workspace_bytes(num_seqs, Hq, d, max_blocks_per_seq, block_size))


def _stream_handle(stream):
    import torch
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream)


def _on_device(t):
    """Context that makes t's device current for the call; a no-op (no device
    switch and restore) when it already is, as in a single-GPU loop."""
    import torch
    if t.device.index == torch.cuda.current_device():
        return contextlib.nullcontext()
    return torch.cuda.device(t.device)


def _check_tensor(name, t, dtype, ndim):
    import torch
    if not isinstance(t, torch.Tensor):
        raise TypeError("%s must be a torch.Tensor" % name)
    if not t.is_cuda:
        raise ValueError("%s must live on a CUDA device" % name)
    if t.dtype != dtype:
        raise TypeError("%s must be %s, got %s" % (name, dtype, t.dtype))
    if t.dim() != ndim:
        raise ValueError("%s must have %d dimensions, got %d" % (name, ndim, t.dim()))
    if not t.is_contiguous():
        raise ValueError("%s must be contiguous" % name)


def attn_fwd(q, k, v, causal: bool = False, scale: float | None = None, out=None, lse=None,
             return_lse: bool = True, stream=None):
    """Prefill attention.  q [B,Hq,Nq,d], k/v [B,Hkv,Nk,d], bf16, contiguous.

    Returns (out [B,Hq,Nq,d] bf16, lse [B,Hq,Nq] fp32 or None)."""
    import torch
    _check_tensor("q", q, torch.bfloat16, 4)
    _check_tensor("k", k, torch.bfloat16, 4)
    _check_tensor("v", v, torch.bfloat16, 4)
    B, Hq, Nq, d = q.shape
    Bk, Hkv, Nk, dk = k.shape
    if tuple(v.shape) != tuple(k.shape) or Bk != B or dk != d:
        raise ValueError("shape mismatch: q %s k %s v %s" % (tuple(q.shape), tuple(k.shape), tuple(v.shape)))
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    else:
        _check_tensor("out", out, torch.bfloat16, 4)
    if lse is None and return_lse:
        lse = torch.empty((B, Hq, Nq), device=q.device, dtype=torch.float32)
    elif lse is not None:
        _check_tensor("lse", lse, torch.float32, 3)
    with _on_device(q):
        rc = lib.attn_fwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(),
                          lse.data_ptr() if lse is not None else None, B, Hq, Hkv, Nq, Nk, d,
                          float(scale), int(bool(causal)), _stream_handle(stream))
    if rc != EXATTN_OK:
        raise ExattnError("attn_fwd", rc)
    return out, lse


def attn_decode_paged(q, k_cache, v_cache, block_table, ctx_lens, scale: float | None = None,
                      out=None, lse=None, workspace=None, return_lse: bool = True, stream=None):
    """One-token decode.  q [S,Hq,d]; caches [num_blocks,Hkv,16,d] bf16;
    block_table int32 [S,max_blocks]; ctx_lens int32 [S].

    Returns (out [S,Hq,d] bf16, lse [S,Hq] fp32 or None)."""
    import torch
    _check_tensor("q", q, torch.bfloat16, 3)
    _check_tensor("k_cache", k_cache, torch.bfloat16, 4)
    _check_tensor("v_cache", v_cache, torch.bfloat16, 4)
    _check_tensor("block_table", block_table, torch.int32, 2)
    _check_tensor("ctx_lens", ctx_lens, torch.int32, 1)
    S, Hq, d = q.shape
    num_blocks, Hkv, bs, dk = k_cache.shape
    if tuple(v_cache.shape) != tuple(k_cache.shape) or dk != d or block_table.shape[0] != S \
            or ctx_lens.shape[0] != S:
        raise ValueError("shape mismatch")
    max_blocks = block_table.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((S, Hq), device=q.device, dtype=torch.float32)
    if workspace is None:  # (the library checks a given workspace's size)
        need = attn_decode_workspace_bytes(S, Hq, d, max_blocks, bs)
        workspace = torch.empty(max(need, 16), device=q.device, dtype=torch.uint8)
    with _on_device(q):
        rc = lib.attn_decode_paged(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                   block_table.data_ptr(), ctx_lens.data_ptr(), out.data_ptr(),
                                   lse.data_ptr() if lse is not None else None, S, Hq, Hkv, d, bs,
                                   num_blocks, max_blocks, float(scale), workspace.data_ptr(),
                                   workspace.numel() * workspace.element_size(),
                                   _stream_handle(stream))
    if rc != EXATTN_OK:
        raise ExattnError("attn_decode_paged", rc)
    return out, lse


def attn_add_rms_norm(x, residual, weight, eps: float = 1e-6, out=None, residual_out=None,
                      stream=None):
    """Residual add + RMS normalisation.  x, residual [T, D] bf16; weight [D]
    bf16; contiguous.  out / residual_out may be x or residual (in place).

    Returns (out [T, D] bf16, residual_out = x + residual [T, D] bf16)."""
    import torch
    _check_tensor("x", x, torch.bfloat16, 2)
    _check_tensor("residual", residual, torch.bfloat16, 2)
    _check_tensor("weight", weight, torch.bfloat16, 1)
    T, D = x.shape
    if tuple(residual.shape) != (T, D) or tuple(weight.shape) != (D,):
        raise ValueError("shape mismatch: x %s residual %s weight %s"
                         % (tuple(x.shape), tuple(residual.shape), tuple(weight.shape)))
    if out is None:
        out = torch.empty_like(x)
    else:
        _check_tensor("out", out, torch.bfloat16, 2)
    if residual_out is None:
        residual_out = torch.empty_like(x)
    else:
        _check_tensor("residual_out", residual_out, torch.bfloat16, 2)
    if tuple(out.shape) != (T, D) or tuple(residual_out.shape) != (T, D):
        raise ValueError("output shape mismatch")
    with _on_device(x):
        rc = lib.attn_add_rms_norm(x.data_ptr(), residual.data_ptr(), weight.data_ptr(),
                                   out.data_ptr(), residual_out.data_ptr(), T, D, float(eps),
                                   _stream_handle(stream))
    if rc != EXATTN_OK:
        raise ExattnError("attn_add_rms_norm", rc)
    return out, residual_out


def attn_rope_cache_write(q, k, v, seq_ids, positions, block_table, k_cache, v_cache,
                          base: float = 500000.0, stream=None):
    """Rotary embedding of q (in place) and k at each token's position, then
    the rotated k and v stored into the paged caches.  q [T,Hq,d], k/v
    [T,Hkv,d] bf16; seq_ids, positions int32 [T]; block_table int32
    [S,max_blocks]; caches [num_blocks,Hkv,16,d] bf16.  Returns q."""
    import torch
    _check_tensor("q", q, torch.bfloat16, 3)
    _check_tensor("k", k, torch.bfloat16, 3)
    _check_tensor("v", v, torch.bfloat16, 3)
    _check_tensor("seq_ids", seq_ids, torch.int32, 1)
    _check_tensor("positions", positions, torch.int32, 1)
    _check_tensor("block_table", block_table, torch.int32, 2)
    _check_tensor("k_cache", k_cache, torch.bfloat16, 4)
    _check_tensor("v_cache", v_cache, torch.bfloat16, 4)
    T, Hq, d = q.shape
    num_blocks, Hkv, bs, dk = k_cache.shape
    if tuple(k.shape) != (T, Hkv, d) or tuple(v.shape) != (T, Hkv, d) or dk != d or bs != 16 \
            or tuple(v_cache.shape) != tuple(k_cache.shape) or seq_ids.shape[0] != T \
            or positions.shape[0] != T:
        raise ValueError("shape mismatch")
    S, max_blocks = block_table.shape
    with _on_device(q):
        rc = lib.attn_rope_cache_write(q.data_ptr(), k.data_ptr(), v.data_ptr(), seq_ids.data_ptr(),
                                       positions.data_ptr(), block_table.data_ptr(),
                                       k_cache.data_ptr(), v_cache.data_ptr(), T, Hq, Hkv, d, S,
                                       num_blocks, max_blocks, float(base), _stream_handle(stream))
    if rc != EXATTN_OK:
        raise ExattnError("attn_rope_cache_write", rc)
    return q


class DecodeGraph:
    """A captured decode step (split kernel + merge).  It holds references to
    the tensors it was captured with; change their contents in place and
    call launch() to replay.  close() frees it (no replay may be pending)."""

    def __init__(self, handle, tensors):
        self._h = handle
        self._tensors = tensors

    def launch(self, stream=None):
        if self._h is None:
            raise ValueError("graph already closed")
        rc = lib.attn_graph_launch(self._h, _stream_handle(stream))
        if rc != EXATTN_OK:
            raise ExattnError("attn_graph_launch", rc)

    def close(self):
        if self._h is not None:
            rc = lib.attn_graph_destroy(self._h)
            self._h = None
            self._tensors = None
            if rc != EXATTN_OK:
                raise ExattnError("attn_graph_destroy", rc)

    def __enter__(self):
        return self

    def __exit__(self, *exc):
        self.close()


def attn_decode_graph_capture(q, k_cache, v_cache, block_table, ctx_lens, scale: float | None = None,
                              out=None, lse=None, workspace=None, return_lse: bool = True):
    """Capture one attn_decode_paged step (same arguments) into a CUDA graph.

    Returns (DecodeGraph, out, lse); nothing runs until graph.launch()."""
    import torch
    _check_tensor("q", q, torch.bfloat16, 3)
    _check_tensor("k_cache", k_cache, torch.bfloat16, 4)
    _check_tensor("v_cache", v_cache, torch.bfloat16, 4)
    _check_tensor("block_table", block_table, torch.int32, 2)
    _check_tensor("ctx_lens", ctx_lens, torch.int32, 1)
    S, Hq, d = q.shape
    num_blocks, Hkv, bs, dk = k_cache.shape
    if tuple(v_cache.shape) != tuple(k_cache.shape) or dk != d or block_table.shape[0] != S \
            or ctx_lens.shape[0] != S:
        raise ValueError("shape mismatch")
    max_blocks = block_table.shape[1]
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    if out is None:
        out = torch.empty_like(q)
    if lse is None and return_lse:
        lse = torch.empty((S, Hq), device=q.device, dtype=torch.float32)
    need = attn_decode_workspace_bytes(S, Hq, d, max_blocks, bs)
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=q.device, dtype=torch.uint8)
    h = ctypes.c_void_p()
    with _on_device(q):
        rc = lib.attn_decode_graph_capture(q.data_ptr(), k_cache.data_ptr(), v_cache.data_ptr(),
                                           block_table.data_ptr(), ctx_lens.data_ptr(), out.data_ptr(),
                                           lse.data_ptr() if lse is not None else None, S, Hq, Hkv, d,
                                           bs, num_blocks, max_blocks, float(scale),
                                           workspace.data_ptr(),
                                           workspace.numel() * workspace.element_size(),
                                           ctypes.byref(h))
    if rc != EXATTN_OK:
        raise ExattnError("attn_decode_graph_capture", rc)
    g = DecodeGraph(h, (q, k_cache, v_cache, block_table, ctx_lens, out, lse, workspace))
    return g, out, lse


def attn_bwd(q, k, v, out, dout, lse, causal: bool = False, scale: float | None = None, dq=None,
             dk=None, dv=None, workspace=None, stream=None):
    """Attention backward.  q, out, dout [B,Hq,Nq,d], k/v [B,Hkv,Nk,d] bf16;
    lse [B,Hq,Nq] fp32 from attn_fwd.  Returns (dq, dk, dv), bf16."""
    import torch
    for name, t in (("q", q), ("k", k), ("v", v), ("out", out), ("dout", dout)):
        _check_tensor(name, t, torch.bfloat16, 4)
    _check_tensor("lse", lse, torch.float32, 3)
    B, Hq, Nq, d = q.shape
    Bk, Hkv, Nk, dk_ = k.shape
    if tuple(v.shape) != tuple(k.shape) or Bk != B or dk_ != d or tuple(out.shape) != tuple(q.shape) \
            or tuple(dout.shape) != tuple(q.shape) or tuple(lse.shape) != (B, Hq, Nq):
        raise ValueError("shape mismatch")
    if scale is None:
        scale = 1.0 / math.sqrt(d)
    dq = torch.empty_like(q) if dq is None else dq
    dk = torch.empty_like(k) if dk is None else dk
    dv = torch.empty_like(v) if dv is None else dv
    need = int(lib.attn_bwd_workspace_bytes(B, Hq, Hkv, Nq, Nk, d))
    if workspace is None:
        workspace = torch.empty(max(need, 16), device=q.device, dtype=torch.uint8)
    with _on_device(q):
        rc = lib.attn_bwd(q.data_ptr(), k.data_ptr(), v.data_ptr(), out.data_ptr(), dout.data_ptr(),
                          lse.data_ptr(), dq.data_ptr(), dk.data_ptr(), dv.data_ptr(), B, Hq, Hkv, Nq,
                          Nk, d, float(scale), int(bool(causal)), workspace.data_ptr(),
                          workspace.numel() * workspace.element_size(), _stream_handle(stream))
    if rc != EXATTN_OK:
        raise ExattnError("attn_bwd", rc)
    return dq, dk, dv


def attn_get_device_status(stream=None) -> int:
    """Synchronise the stream, then read and clear the device status word."""
    v = ctypes.c_int(0)
    rc = lib.attn_get_device_status(_stream_handle(stream), ctypes.byref(v))
    if rc != EXATTN_OK:
        raise ExattnError("attn_get_device_status", rc)
    return int(v.value)


def attn_debug_expire_wait(budget_ns: int, stream=None) -> None:
    """Launch the diagnostic kernel whose bounded wait must run out."""
    rc = lib.attn_debug_expire_wait(int(budget_ns), _stream_handle(stream))
    if rc != EXATTN_OK:
        raise ExattnError("attn_debug_expire_wait", rc)


def attn_shutdown() -> None:
    lib.attn_shutdown()
