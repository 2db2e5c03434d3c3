"""CPU oracle for libbeamnorm -- TEST INFRASTRUCTURE ONLY.

A plain, single-threaded C definition of the fused tensor-parallel all-reduce
epilogue (rank-ordered FP32 sum of R BF16 shards, optional per-shard MoE top-k
finalize rounded to BF16, then post-RMSNorm, residual add and the next layer's
input RMSNorm), wrapped here for numpy.  Only the tests, ``__graft_entry__.smoke``
and the CPU-baseline leg of ``bench.py`` may import this package; the product
path never does, and it shares no code with the CUDA library.

BF16 arrays are numpy ``uint16`` bit patterns.  Every function takes an
optional ``rows`` list of token indices; outputs are compact (row ``i`` of an
output belongs to token ``rows[i]``).

Sources: "Fuse Beam's TP all-reduce with its sandwich norms" (vLLM pull request
62366), sections "Claims" and "Details"; sglang pull request 34134 ("cute-dsl"
MNNVL all-reduce fusion backend), description and "Motivation".
"""
from __future__ import annotations

import ctypes
import os
import threading

import numpy as np

from . import build as _build

SINGLE_NORM = 1
PRENORM_FROM_BF16_RESIDUAL = 2

_lib = None
_lock = threading.Lock()

_u16p = ctypes.POINTER(ctypes.c_uint16)
_f32p = ctypes.POINTER(ctypes.c_float)
_i32p = ctypes.POINTER(ctypes.c_int32)
_int = ctypes.c_int
_f32 = ctypes.c_float


def lib() -> ctypes.CDLL:
    """Load (building first if needed) the oracle's shared library."""
    global _lib
    with _lock:
        if _lib is None:
            # A test may point the wrapper at a deliberately broken copy of the
            # oracle (tests/test_oracle_mutations.py); otherwise build and load
            # the real one.
            path = os.environ.get("BEAMNORM_ORACLE_LIB") or _build.build()
            L = ctypes.CDLL(path)
            L.oracle_reduce_norm.argtypes = [_u16p, _int, _int, _int, _u16p, _f32p, _f32p, _f32,
                                             _int, _i32p, _int, _u16p, _u16p, _f32p, _f32p]
            L.oracle_reduce_norm.restype = _int
            L.oracle_finalize_reduce_norm.argtypes = [_u16p, _i32p, _f32p, _u16p, _int, _int, _int,
                                                      _int, _u16p, _f32p, _f32p, _f32, _int, _i32p,
                                                      _int, _u16p, _u16p, _f32p, _f32p, _u16p]
            L.oracle_finalize_reduce_norm.restype = _int
            L.oracle_norm.argtypes = [_f32p, _int, _int, _u16p, _f32p, _f32p, _f32, _int, _i32p,
                                      _int, _u16p, _u16p, _f32p]
            L.oracle_norm.restype = _int
            L.oracle_bf16_from_f32.argtypes = [_f32]
            L.oracle_bf16_from_f32.restype = ctypes.c_uint16
            L.oracle_f32_from_bf16.argtypes = [ctypes.c_uint16]
            L.oracle_f32_from_bf16.restype = _f32
            _lib = L
    return _lib


def _arr(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a


def _p(a, ptype):
    return None if a is None else a.ctypes.data_as(ptype)


def _rows(rows, T):
    if rows is None:
        return None, T
    r = np.ascontiguousarray(rows, dtype=np.int32)
    return r, int(r.size)


def bf16_from_f32(x) -> np.ndarray:
    """Round FP32 values to BF16 bit patterns with the oracle's own rounding."""
    L = lib()
    x = np.asarray(x, dtype=np.float32)
    return np.array([L.oracle_bf16_from_f32(float(v)) for v in x.ravel()], dtype=np.uint16).reshape(x.shape)


def reduce_norm(partials, residual, gamma_post, gamma_pre, eps, *, rows=None, flags=0,
                want_norm=True):
    """Oracle of ``reduce_norm``.

    partials: uint16 [R, T, H]; residual: uint16 [T, H]; gammas: float32 [H].
    Returns a dict with ``sum`` float32 [n, H], ``ss`` float32 [n, 2],
    ``residual_out`` and ``out`` uint16 [n, H] (the last three only when
    ``want_norm``), n = number of selected rows.
    """
    partials = _arr(partials, np.uint16)
    R, T, H = partials.shape
    rws, n = _rows(rows, T)
    res = _arr(residual, np.uint16).reshape(T, H) if want_norm else None
    gp = _arr(gamma_post, np.float32) if want_norm else None
    gq = _arr(gamma_pre, np.float32) if want_norm else None
    s = np.empty((n, H), np.float32)
    ss = np.zeros((n, 2), np.float32)
    ro = np.empty((n, H), np.uint16) if want_norm else None
    out = np.empty((n, H), np.uint16) if want_norm else None
    st = lib().oracle_reduce_norm(_p(partials, _u16p), R, T, H, _p(res, _u16p), _p(gp, _f32p),
                                  _p(gq, _f32p), float(eps), int(flags), _p(rws, _i32p), n,
                                  _p(ro, _u16p), _p(out, _u16p), _p(s, _f32p), _p(ss, _f32p))
    if st != 0:
        raise ValueError(f"oracle_reduce_norm failed with status {st}")
    d = {"sum": s}
    if want_norm:
        d.update(ss=ss, residual_out=ro, out=out)
    return d


def finalize_reduce_norm(expert_out, perm, w, shared, residual, gamma_post, gamma_pre, eps, *,
                         rows=None, flags=0, want_norm=True, want_z=False):
    """Oracle of ``finalize_reduce_norm``.

    expert_out: uint16 [R, T*k, H]; perm: int32 [R, T, k]; w: float32 [R, T, k];
    shared: uint16 [R, T, H] or None (zeros); residual: uint16 [T, H].
    Returns ``sum``, and when asked ``ss``, ``residual_out``, ``out`` and
    ``z`` (uint16 [R, n, H], the per-shard BF16 finalize results).
    """
    perm = _arr(perm, np.int32)
    R, T, k = perm.shape
    expert_out = _arr(expert_out, np.uint16)
    H = expert_out.shape[-1]
    assert expert_out.shape == (R, T * k, H), expert_out.shape
    w = _arr(w, np.float32).reshape(R, T, k)
    sh = None if shared is None else _arr(shared, np.uint16).reshape(R, T, H)
    rws, n = _rows(rows, T)
    res = _arr(residual, np.uint16).reshape(T, H) if want_norm else None
    gp = _arr(gamma_post, np.float32) if want_norm else None
    gq = _arr(gamma_pre, np.float32) if want_norm else None
    s = np.empty((n, H), np.float32)
    ss = np.zeros((n, 2), np.float32)
    ro = np.empty((n, H), np.uint16) if want_norm else None
    out = np.empty((n, H), np.uint16) if want_norm else None
    z = np.empty((R, n, H), np.uint16) if want_z else None
    st = lib().oracle_finalize_reduce_norm(
        _p(expert_out, _u16p), _p(perm, _i32p), _p(w, _f32p), _p(sh, _u16p), R, T, k, H,
        _p(res, _u16p), _p(gp, _f32p), _p(gq, _f32p), float(eps), int(flags), _p(rws, _i32p), n,
        _p(ro, _u16p), _p(out, _u16p), _p(s, _f32p), _p(ss, _f32p), _p(z, _u16p))
    if st != 0:
        raise ValueError(f"oracle_finalize_reduce_norm failed with status {st}")
    d = {"sum": s}
    if want_norm:
        d.update(ss=ss, residual_out=ro, out=out)
    if want_z:
        d["z"] = z
    return d


def norm(sum_, residual, gamma_post, gamma_pre, eps, *, rows=None, flags=0):
    """Oracle of the epilogue alone, given the FP32 reduced sum [T, H]."""
    sum_ = _arr(sum_, np.float32)
    T, H = sum_.shape
    rws, n = _rows(rows, T)
    res = _arr(residual, np.uint16).reshape(T, H)
    gp = _arr(gamma_post, np.float32)
    gq = _arr(gamma_pre, np.float32)
    ss = np.zeros((n, 2), np.float32)
    ro = np.empty((n, H), np.uint16)
    out = np.empty((n, H), np.uint16)
    st = lib().oracle_norm(_p(sum_, _f32p), T, H, _p(res, _u16p), _p(gp, _f32p), _p(gq, _f32p),
                           float(eps), int(flags), _p(rws, _i32p), n, _p(ro, _u16p),
                           _p(out, _u16p), _p(ss, _f32p))
    if st != 0:
        raise ValueError(f"oracle_norm failed with status {st}")
    return {"ss": ss, "residual_out": ro, "out": out}


def library_path() -> str:
    return os.path.abspath(_build.LIB)
