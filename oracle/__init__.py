"""fp64 CPU oracle for exact scaled-dot-product attention.

TEST INFRASTRUCTURE ONLY.  The tests, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline leg are the only callers; the CUDA library and its
Python binding never import, link or run anything here, and this package
shares no code with them.

The arithmetic lives in ``oracle.c`` (plain C, fp64, OpenMP over query
rows); this module compiles it (``build()``) and marshals numpy arrays into
it.  Every function states the passage of the pages it follows in the C
source.  Inputs are bf16 bit patterns held as ``numpy.uint16``.
"""
from __future__ import annotations

import ctypes
import os
import subprocess

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.c")
_LIB_PATH = os.path.join(_HERE, "liboracle.so")
_lib = None


def build(force: bool = False) -> str:
    """Compile ``oracle.c`` into ``liboracle.so`` (gcc, -O2, OpenMP when available)."""
    if not force and os.path.exists(_LIB_PATH) and os.path.getmtime(_LIB_PATH) >= os.path.getmtime(_SRC):
        return _LIB_PATH
    tmp = _LIB_PATH + ".tmp%d" % os.getpid()
    base = ["gcc", "-O2", "-std=c99", "-shared", "-fPIC", _SRC, "-o", tmp, "-lm"]
    try:
        subprocess.run(base[:1] + ["-fopenmp"] + base[1:], check=True, capture_output=True)
    except subprocess.CalledProcessError:
        subprocess.run(base, check=True, capture_output=True)  # serial fallback
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    if _lib is not None:
        return _lib
    lib = ctypes.CDLL(build())
    P = ctypes.c_void_p
    I = ctypes.c_int
    L = ctypes.c_long
    D = ctypes.c_double
    lib.oracle_attn_f64.argtypes = [P, P, P, I, I, I, L, L, I, D, I, P, P]
    lib.oracle_attn_f64.restype = I
    lib.oracle_attn_rows_f64.argtypes = [P, P, P, P, L, I, I, I, L, L, I, D, I, P, P]
    lib.oracle_attn_rows_f64.restype = I
    lib.oracle_decode_paged_f64.argtypes = [P, P, P, P, P, I, I, I, I, I, L, I, D, P, P]
    lib.oracle_decode_paged_f64.restype = I
    lib.oracle_softmax_f64.argtypes = [P, L, P]
    lib.oracle_softmax_f64.restype = None
    lib.oracle_online_softmax_f64.argtypes = [P, L, P]
    lib.oracle_online_softmax_f64.restype = None
    lib.oracle_add_rms_norm_f64.argtypes = [P, P, P, L, L, D, P, P]
    lib.oracle_add_rms_norm_f64.restype = I
    lib.oracle_rope_cache_write_f64.argtypes = [P, P, P, P, P, I, I, I, I, I, I, I, D, P, P, P]
    lib.oracle_rope_cache_write_f64.restype = I
    lib.oracle_attn_bwd_f64.argtypes = [P, P, P, P, I, I, I, L, L, I, D, I, P, P, P]
    lib.oracle_attn_bwd_f64.restype = I
    lib.oracle_num_threads.argtypes = []
    lib.oracle_num_threads.restype = I
    lib.oracle_set_num_threads.argtypes = [I]
    lib.oracle_set_num_threads.restype = None
    _lib = lib
    return lib


def _ptr(a: np.ndarray):
    return a.ctypes.data_as(ctypes.c_void_p)


def _u16(a) -> np.ndarray:
    a = np.ascontiguousarray(a)
    if a.dtype != np.uint16:
        raise TypeError("oracle inputs are bf16 bit patterns (numpy.uint16), got %s" % a.dtype)
    return a


def num_threads() -> int:
    return _load().oracle_num_threads()


def set_num_threads(n: int) -> None:
    _load().oracle_set_num_threads(int(n))


def attn(q, k, v, scale: float, causal: bool):
    """Prefill attention.  q [B,Hq,Nq,d], k/v [B,Hkv,Nk,d] (uint16 bf16 bits).

    Returns (out fp64 [B,Hq,Nq,d], lse fp64 [B,Hq,Nq])."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    B, Hq, Nq, d = q.shape
    Bk, Hkv, Nk, dk = k.shape
    if k.shape != v.shape or Bk != B or dk != d:
        raise ValueError("shape mismatch")
    out = np.zeros((B, Hq, Nq, d), np.float64)
    lse = np.zeros((B, Hq, Nq), np.float64)
    rc = _load().oracle_attn_f64(_ptr(q), _ptr(k), _ptr(v), B, Hq, Hkv, Nq, Nk, d,
                                 float(scale), int(bool(causal)), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_attn_f64 rejected its arguments")
    return out, lse


def attn_rows(q, k, v, rows, scale: float, causal: bool):
    """Attention for selected query rows; rows is int64 [n, 3] of (b, hq, i).

    Returns (out fp64 [n, d], lse fp64 [n])."""
    q, k, v = _u16(q), _u16(k), _u16(v)
    rows = np.ascontiguousarray(rows, dtype=np.int64).reshape(-1, 3)
    B, Hq, Nq, d = q.shape
    _, Hkv, Nk, _ = k.shape
    n = rows.shape[0]
    out = np.zeros((n, d), np.float64)
    lse = np.zeros((n,), np.float64)
    rc = _load().oracle_attn_rows_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(rows), n, B, Hq, Hkv, Nq,
                                      Nk, d, float(scale), int(bool(causal)), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_attn_rows_f64 rejected its arguments")
    return out, lse


def decode_paged(q, k_cache, v_cache, block_table, ctx_lens, scale: float):
    """One-token decode.  q [S,Hq,d]; caches [num_blocks,Hkv,block_size,d];
    block_table int32 [S, max_blocks]; ctx_lens int32 [S].

    Returns (out fp64 [S,Hq,d], lse fp64 [S,Hq])."""
    q, k_cache, v_cache = _u16(q), _u16(k_cache), _u16(v_cache)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    cl = np.ascontiguousarray(ctx_lens, dtype=np.int32)
    S, Hq, d = q.shape
    nb, Hkv, bs, dk = k_cache.shape
    if k_cache.shape != v_cache.shape or dk != d or bt.shape[0] != S or cl.shape != (S,):
        raise ValueError("shape mismatch")
    out = np.zeros((S, Hq, d), np.float64)
    lse = np.zeros((S, Hq), np.float64)
    rc = _load().oracle_decode_paged_f64(_ptr(q), _ptr(k_cache), _ptr(v_cache), _ptr(bt),
                                         _ptr(cl), S, Hq, Hkv, d, bs, nb, bt.shape[1],
                                         float(scale), _ptr(out), _ptr(lse))
    if rc != 0:
        raise ValueError("oracle_decode_paged_f64 rejected its arguments")
    return out, lse


def softmax(x):
    """Two-pass safe softmax of a 1-D fp64 row."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    _load().oracle_softmax_f64(_ptr(x), x.size, _ptr(y))
    return y


def online_softmax(x):
    """Single-sweep running softmax of a 1-D fp64 row (pins the two-pass form)."""
    x = np.ascontiguousarray(x, dtype=np.float64)
    y = np.empty_like(x)
    _load().oracle_online_softmax_f64(_ptr(x), x.size, _ptr(y))
    return y


def add_rms_norm(x, residual, weight, eps: float):
    """Residual add + RMS normalisation.  x, residual [T, D], weight [D]
    (uint16 bf16 bits).

    Returns (out fp64 [T, D], new residual h = x + residual fp64 [T, D])."""
    x, residual, weight = _u16(x), _u16(residual), _u16(weight)
    if x.ndim != 2 or residual.shape != x.shape or weight.shape != (x.shape[1],):
        raise ValueError("shape mismatch")
    T, D = x.shape
    out = np.zeros((T, D), np.float64)
    h = np.zeros((T, D), np.float64)
    rc = _load().oracle_add_rms_norm_f64(_ptr(x), _ptr(residual), _ptr(weight), T, D, float(eps),
                                         _ptr(out), _ptr(h))
    if rc != 0:
        raise ValueError("oracle_add_rms_norm_f64 rejected its arguments")
    return out, h


def rope_cache_write(q, k, seq_ids, positions, block_table, num_blocks: int, base: float):
    """Rotary embedding of q [T, Hq, d] and k [T, Hkv, d] (uint16 bf16 bits)
    at positions[t], and the cache slot each token's key and value go to.

    Returns (q_out fp64 [T, Hq, d], k_out fp64 [T, Hkv, d], slot int64 [T]:
    physical block * 16 + slot, -1 when outside the table or the cache)."""
    q, k = _u16(q), _u16(k)
    sid = np.ascontiguousarray(seq_ids, dtype=np.int32)
    pos = np.ascontiguousarray(positions, dtype=np.int32)
    bt = np.ascontiguousarray(block_table, dtype=np.int32)
    T, Hq, d = q.shape
    Tk, Hkv, dk = k.shape
    if Tk != T or dk != d or sid.shape != (T,) or pos.shape != (T,) or bt.ndim != 2:
        raise ValueError("shape mismatch")
    q_out = np.zeros((T, Hq, d), np.float64)
    k_out = np.zeros((T, Hkv, d), np.float64)
    slot = np.zeros((T,), np.int64)
    rc = _load().oracle_rope_cache_write_f64(_ptr(q), _ptr(k), _ptr(sid), _ptr(pos), _ptr(bt), T, Hq,
                                             Hkv, d, bt.shape[0], int(num_blocks), bt.shape[1],
                                             float(base), _ptr(q_out), _ptr(k_out), _ptr(slot))
    if rc != 0:
        raise ValueError("oracle_rope_cache_write_f64 rejected its arguments")
    return q_out, k_out, slot


def attn_bwd(q, k, v, dout, scale: float, causal: bool):
    """Gradients of attention.  q, dout [B,Hq,Nq,d], k/v [B,Hkv,Nk,d] (uint16
    bf16 bits).  Returns (dq [B,Hq,Nq,d], dk, dv [B,Hkv,Nk,d]) in fp64."""
    q, k, v, dout = _u16(q), _u16(k), _u16(v), _u16(dout)
    B, Hq, Nq, d = q.shape
    Bk, Hkv, Nk, dk_ = k.shape
    if k.shape != v.shape or Bk != B or dk_ != d or dout.shape != q.shape:
        raise ValueError("shape mismatch")
    dq = np.zeros(q.shape, np.float64)
    dk = np.zeros(k.shape, np.float64)
    dv = np.zeros(k.shape, np.float64)
    rc = _load().oracle_attn_bwd_f64(_ptr(q), _ptr(k), _ptr(v), _ptr(dout), B, Hq, Hkv, Nq, Nk, d,
                                     float(scale), int(bool(causal)), _ptr(dq), _ptr(dk), _ptr(dv))
    if rc != 0:
        raise ValueError("oracle_attn_bwd_f64 rejected its arguments")
    return dq, dk, dv
