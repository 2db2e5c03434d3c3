"""Python binding of libbeamnorm (argument marshalling only).

Every function here checks dtypes, shapes, devices and contiguity, then calls
the C entry point of the same name with raw device pointers and the current
CUDA stream.  All arithmetic runs in the library's CUDA kernels; there is no
fallback.  If the library is missing the call raises.

BF16 tensors are ``torch.bfloat16``; perm is ``torch.int32``; w, gammas and
FP32 sums are ``torch.float32``.  Shapes: partials [R,T,H], expert_out
[R,T*k,H], perm and w [R,T,k], shared [R,T,H] (or None), residual and out
[T,H], gammas [H].  The residual is updated in place.
"""
from __future__ import annotations

import ctypes
import os
import threading
from dataclasses import dataclass
from typing import Optional

import torch

HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(HERE, "_build", "libbeamnorm.so")

OK, ERR_INVALID, ERR_UNSUPPORTED, ERR_CUDA, ERR_DEVICE = 0, 1, 2, 3, 4
DEVERR_PERM_RANGE, DEVERR_TIMEOUT = 1, 2

# Every symbol declared in include/beamnorm.h.
EXPORTS = (
    "bn_reduce_norm", "bn_finalize_reduce_norm", "bn_reduce_residual_norm",
    "bn_finalize_reduce_residual_norm", "bn_reduce_only", "bn_finalize_reduce_only",
    "bn_norm_only", "bn_finalize_only", "bn_supports", "bn_check_device_error",
    "bn_last_error", "bn_status_string", "bn_version", "bn_set_tuning", "bn_query_launch",
    "bn_finalize_workspace_bytes", "bn_finalize_reduce_norm_ws",
    "bn_finalize_reduce_residual_norm_ws", "bn_finalize_reduce_norm_noalloc",
    "bn_residual_norm_only", "bn_supports_op", "bn_shutdown",
)

# bn_op values of the entry points, for launch_info()
OPS = ("reduce_norm", "finalize_reduce_norm", "reduce_residual_norm",
       "finalize_reduce_residual_norm", "reduce_only", "finalize_reduce_only", "norm_only",
       "finalize_only", "residual_norm_only")


class BeamNormError(RuntimeError):
    def __init__(self, status: int, message: str):
        super().__init__(f"{_STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


_STATUS_NAMES = {OK: "BN_OK", ERR_INVALID: "BN_ERR_INVALID", ERR_UNSUPPORTED: "BN_ERR_UNSUPPORTED",
                 ERR_CUDA: "BN_ERR_CUDA", ERR_DEVICE: "BN_ERR_DEVICE"}


class _Tuning(ctypes.Structure):
    _fields_ = [("cluster_size", ctypes.c_int), ("stages", ctypes.c_int), ("threads", ctypes.c_int),
                ("ctas_per_sm", ctypes.c_int), ("wait_mode", ctypes.c_int), ("group", ctypes.c_int),
                ("split", ctypes.c_int), ("dependent_launch", ctypes.c_int),
                ("wait_limit_polls", ctypes.c_int), ("tiny_pass", ctypes.c_int)]


class _LaunchInfo(ctypes.Structure):
    _fields_ = [(n, ctypes.c_int) for n in (
        "split", "cluster_size", "threads", "chunks_per_thread", "grid", "resident_ctas",
        "stages", "stage_bytes", "group", "smem_bytes")]


class _Debug(ctypes.Structure):
    _fields_ = [("sum", ctypes.c_void_p), ("ss", ctypes.c_void_p), ("z", ctypes.c_void_p)]


@dataclass
class Debug:
    """Optional intermediate outputs: sum [T,H] FP32, ss [T,2] FP32, z [R,T,H] BF16."""
    sum: Optional[torch.Tensor] = None
    ss: Optional[torch.Tensor] = None
    z: Optional[torch.Tensor] = None


_lib = None
_lock = threading.Lock()

_P = ctypes.c_void_p
_I = ctypes.c_int
_F = ctypes.c_float


def load() -> ctypes.CDLL:
    """Load libbeamnorm.so (built by ``tp_reduce_residual_gb300.build``)."""
    global _lib
    with _lock:
        if _lib is not None:
            return _lib
        if not os.path.exists(LIB_PATH):
            raise RuntimeError(f"libbeamnorm is not built ({LIB_PATH} missing); run "
                               "`python -m tp_reduce_residual_gb300.build`")
        L = ctypes.CDLL(LIB_PATH)
        dbgp = ctypes.POINTER(_Debug)
        sig = {
            "bn_reduce_norm": [_P, _I, _I, _I, _P, _P, _P, _F, _P, dbgp, _P],
            "bn_finalize_reduce_norm": [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _F, _P, dbgp, _P],
            "bn_reduce_residual_norm": [_P, _I, _I, _I, _P, _P, _F, _P, dbgp, _P],
            "bn_finalize_reduce_residual_norm": [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _F, _P,
                                                 dbgp, _P],
            "bn_reduce_only": [_P, _I, _I, _I, _P, _P],
            "bn_finalize_reduce_only": [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P],
            "bn_norm_only": [_P, _I, _I, _P, _P, _P, _F, _P, dbgp, _P],
            "bn_residual_norm_only": [_P, _I, _I, _P, _P, _F, _P, dbgp, _P],
            "bn_supports_op": [_I, _I, _I, _I, _I],
            "bn_finalize_only": [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P],
            "bn_supports": [_I, _I, _I, _I],
            "bn_check_device_error": [_P, ctypes.POINTER(ctypes.c_uint)],
            "bn_last_error": [],
            "bn_status_string": [_I],
            "bn_version": [],
            "bn_set_tuning": [ctypes.POINTER(_Tuning)],
            "bn_query_launch": [_I, _I, _I, _I, _I, _I, ctypes.POINTER(_LaunchInfo)],
            "bn_finalize_workspace_bytes": [_I, _I, _I, _I],
            "bn_finalize_reduce_norm_ws": [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _F, _P,
                                           dbgp, _P, ctypes.c_size_t, _P],
            "bn_finalize_reduce_residual_norm_ws": [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _F,
                                                    _P, dbgp, _P, ctypes.c_size_t, _P],
            "bn_finalize_reduce_norm_noalloc": [_P, _P, _P, _P, _I, _I, _I, _I, _P, _P, _P, _F, _P,
                                                dbgp, _P],
        }
        for name, args in sig.items():
            fn = getattr(L, name)
            fn.argtypes = args
            fn.restype = _I
        L.bn_shutdown.argtypes = []
        L.bn_shutdown.restype = None
        L.bn_finalize_workspace_bytes.restype = ctypes.c_size_t
        L.bn_last_error.restype = ctypes.c_char_p
        L.bn_status_string.restype = ctypes.c_char_p
        _lib = L
        return L


def _check(status: int):
    if status != OK:
        msg = load().bn_last_error().decode(errors="replace")
        raise BeamNormError(status, msg)


def _stream(t: torch.Tensor, stream) -> int:
    if stream is None:
        stream = torch.cuda.current_stream(t.device)
    return int(stream.cuda_stream) if hasattr(stream, "cuda_stream") else int(stream)


def _need(t: Optional[torch.Tensor], name: str, dtype, shape, device) -> int:
    if t is None:
        raise ValueError(f"{name} is required")
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch.Tensor")
    if t.device.type != "cuda":
        raise ValueError(f"{name} must be a CUDA tensor (got {t.device})")
    if device is not None and t.device != device:
        raise ValueError(f"{name} is on {t.device}, expected {device}")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype} (got {t.dtype})")
    if tuple(t.shape) != tuple(shape):
        raise ValueError(f"{name} has shape {tuple(t.shape)}, expected {tuple(shape)}")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    return t.data_ptr()


def _opt(t, name, dtype, shape, device) -> Optional[int]:
    return None if t is None else _need(t, name, dtype, shape, device)


def _debug(dbg: Optional[Debug], R, T, H, device, fin: bool):
    if dbg is None:
        return None
    s = _Debug(_opt(dbg.sum, "debug.sum", torch.float32, (T, H), device),
               _opt(dbg.ss, "debug.ss", torch.float32, (T, 2), device),
               _opt(dbg.z, "debug.z", torch.bfloat16, (R, T, H), device) if fin else None)
    return ctypes.byref(s), s


def _with_device(t: torch.Tensor):
    return torch.cuda.device(t.device)


# ---- the decline and its fallback ----------------------------------------------------
#
# A fused entry point that does not serve a shape declines: it returns
# BN_ERR_UNSUPPORTED and enqueues nothing, so the whole reduction is still
# owed.  With on_decline="fallback" the wrappers below then run the unfused
# pieces, which serve larger rows: the deferred finalize is materialised
# (finalize_only), the shards are summed (reduce_only), and the epilogue runs
# on the FP32 sum (norm_only, or residual_norm_only for the single norm).  The
# bits are those the fused call would give.  The temporaries (z, the FP32 sum)
# are allocated here, on the call's stream.

def _fallback_allowed(err: "BeamNormError", on_decline: str) -> bool:
    if on_decline not in ("raise", "fallback"):
        raise ValueError(f"on_decline must be 'raise' or 'fallback' (got {on_decline!r})")
    return on_decline == "fallback" and err.status == ERR_UNSUPPORTED


def _fallback(partials, z_inputs, residual, gamma_post, gamma_pre, eps, out, debug, stream,
              single: bool):
    ctx = torch.cuda.stream(stream) if hasattr(stream, "cuda_stream") else _nullctx()
    with ctx:
        if z_inputs is not None:
            expert_out, perm, w, shared = z_inputs
            partials = finalize_only(expert_out, perm, w, shared, stream=stream)
            if debug is not None and debug.z is not None:
                debug.z.copy_(partials)
        s = reduce_only(partials, stream=stream)
        if debug is not None and debug.sum is not None:
            debug.sum.copy_(s)
        dbg = Debug(ss=debug.ss) if debug is not None and debug.ss is not None else None
        if single:
            residual_norm_only(s, residual, gamma_pre, eps, out=out, debug=dbg, stream=stream)
        else:
            norm_only(s, residual, gamma_post, gamma_pre, eps, out=out, debug=dbg, stream=stream)
    return out


class _nullctx:
    def __enter__(self):
        return self

    def __exit__(self, *exc):
        return False


def reduce_norm(partials, residual, gamma_post, gamma_pre, eps: float, out=None,
                debug: Optional[Debug] = None, stream=None,
                on_decline: str = "raise") -> torch.Tensor:
    """Rank-ordered FP32 sum of the shards, post-RMSNorm, residual add (in
    place), pre-RMSNorm.  Returns ``out`` (BF16 [T,H]).  ``on_decline="fallback"``:
    a shape the fused kernel declines runs as the unfused pieces instead."""
    L = load()
    R, T, H = partials.shape
    dev = partials.device
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    args = (_need(partials, "partials", torch.bfloat16, (R, T, H), dev), R, T, H,
            _need(residual, "residual", torch.bfloat16, (T, H), dev),
            _need(gamma_post, "gamma_post", torch.float32, (H,), dev),
            _need(gamma_pre, "gamma_pre", torch.float32, (H,), dev), float(eps),
            _need(out, "out", torch.bfloat16, (T, H), dev))
    d = _debug(debug, R, T, H, dev, False)
    with _with_device(partials):
        try:
            _check(L.bn_reduce_norm(*args, d[0] if d else None, _stream(partials, stream)))
        except BeamNormError as e:
            if not _fallback_allowed(e, on_decline):
                raise
            return _fallback(partials, None, residual, gamma_post, gamma_pre, eps, out, debug,
                             stream, single=False)
    return out


def finalize_workspace_bytes(R: int, T: int, k: int, H: int) -> int:
    """Workspace bytes with which the finalize entries spread each token row
    over many CTAs (0: that path does not serve the shape)."""
    return int(load().bn_finalize_workspace_bytes(R, T, k, H))


def finalize_workspace(R: int, T: int, k: int, H: int, device=None) -> Optional[torch.Tensor]:
    """A zero-filled workspace for ``finalize_reduce_norm(..., workspace=)``
    (uint8, on ``device``), or None when the shape does not use one.  Calls
    leave it zeroed; one workspace serves one call at a time."""
    n = finalize_workspace_bytes(R, T, k, H)
    if n == 0:
        return None
    return torch.zeros(n, dtype=torch.uint8, device=device if device is not None else "cuda")


def _workspace(ws, dev):
    if ws is None:
        return None, 0
    if not isinstance(ws, torch.Tensor) or ws.dtype != torch.uint8 or ws.dim() != 1:
        raise TypeError("workspace must be a 1-D torch.uint8 tensor")
    if ws.device != dev or not ws.is_contiguous():
        raise ValueError(f"workspace must be contiguous on {dev}")
    return ws.data_ptr(), ws.numel()


def finalize_reduce_norm(expert_out, perm, w, shared, residual, gamma_post, gamma_pre, eps: float,
                         out=None, debug: Optional[Debug] = None, stream=None,
                         workspace: Optional[torch.Tensor] = None,
                         on_decline: str = "raise") -> torch.Tensor:
    """Per-shard MoE top-k finalize (rounded to BF16), rank-ordered FP32 sum,
    post-RMSNorm, residual add (in place), pre-RMSNorm.  Returns ``out``.
    With a ``workspace`` (see ``finalize_workspace``) few token rows are each
    spread over many CTAs; the results are the same.  ``on_decline="fallback"``:
    a declined shape materialises the finalize and runs the unfused pieces."""
    L = load()
    R, T, k = perm.shape
    H = expert_out.shape[-1]
    dev = expert_out.device
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    args = (_need(expert_out, "expert_out", torch.bfloat16, (R, T * k, H), dev),
            _need(perm, "perm", torch.int32, (R, T, k), dev),
            _need(w, "w", torch.float32, (R, T, k), dev),
            _opt(shared, "shared", torch.bfloat16, (R, T, H), dev), R, T, k, H,
            _need(residual, "residual", torch.bfloat16, (T, H), dev),
            _need(gamma_post, "gamma_post", torch.float32, (H,), dev),
            _need(gamma_pre, "gamma_pre", torch.float32, (H,), dev), float(eps),
            _need(out, "out", torch.bfloat16, (T, H), dev))
    d = _debug(debug, R, T, H, dev, True)
    with _with_device(expert_out):
        try:
            if workspace is None:
                _check(L.bn_finalize_reduce_norm(*args, d[0] if d else None,
                                                 _stream(expert_out, stream)))
            else:
                wp, wn = _workspace(workspace, dev)
                _check(L.bn_finalize_reduce_norm_ws(*args, d[0] if d else None, wp, wn,
                                                    _stream(expert_out, stream)))
        except BeamNormError as e:
            if not _fallback_allowed(e, on_decline):
                raise
            return _fallback(None, (expert_out, perm, w, shared), residual, gamma_post, gamma_pre,
                             eps, out, debug, stream, single=False)
    return out


def finalize_reduce_norm_noalloc(expert_out, perm, w, shared, residual, gamma_post, gamma_pre,
                                 eps: float, out=None, debug: Optional[Debug] = None,
                                 stream=None) -> torch.Tensor:
    """``finalize_reduce_norm`` with each token row spread over many CTAs,
    using the library's own static scratch instead of a caller workspace.

    For callers that are handed only the op's tensors and may not allocate
    device memory (an engine whose pool owns all of HBM, a plugin hook with no
    workspace slot).  The library call allocates nothing; ``out`` is allocated
    here only when it is not given.  It serves 1 <= T <= 8 and H <= 8192 with
    at most 2 MiB of scratch and raises BN_ERR_UNSUPPORTED otherwise.  The
    first call on a device looks up the scratch's address: make it before any
    stream capture.  Calls that may overlap on the GPU share the scratch and
    race; order them."""
    L = load()
    R, T, k = perm.shape
    H = expert_out.shape[-1]
    dev = expert_out.device
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    args = (_need(expert_out, "expert_out", torch.bfloat16, (R, T * k, H), dev),
            _need(perm, "perm", torch.int32, (R, T, k), dev),
            _need(w, "w", torch.float32, (R, T, k), dev),
            _opt(shared, "shared", torch.bfloat16, (R, T, H), dev), R, T, k, H,
            _need(residual, "residual", torch.bfloat16, (T, H), dev),
            _need(gamma_post, "gamma_post", torch.float32, (H,), dev),
            _need(gamma_pre, "gamma_pre", torch.float32, (H,), dev), float(eps),
            _need(out, "out", torch.bfloat16, (T, H), dev))
    d = _debug(debug, R, T, H, dev, True)
    with _with_device(expert_out):
        _check(L.bn_finalize_reduce_norm_noalloc(*args, d[0] if d else None,
                                                 _stream(expert_out, stream)))
    return out


def reduce_residual_norm(partials, residual, gamma, eps: float, out=None,
                         debug: Optional[Debug] = None, stream=None,
                         on_decline: str = "raise") -> torch.Tensor:
    """Rank-ordered sum, residual add (in place), RMSNorm; no post-norm.
    ``on_decline`` as for ``reduce_norm``."""
    L = load()
    R, T, H = partials.shape
    dev = partials.device
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    args = (_need(partials, "partials", torch.bfloat16, (R, T, H), dev), R, T, H,
            _need(residual, "residual", torch.bfloat16, (T, H), dev),
            _need(gamma, "gamma", torch.float32, (H,), dev), float(eps),
            _need(out, "out", torch.bfloat16, (T, H), dev))
    d = _debug(debug, R, T, H, dev, False)
    with _with_device(partials):
        try:
            _check(L.bn_reduce_residual_norm(*args, d[0] if d else None,
                                             _stream(partials, stream)))
        except BeamNormError as e:
            if not _fallback_allowed(e, on_decline):
                raise
            return _fallback(partials, None, residual, None, gamma, eps, out, debug, stream,
                             single=True)
    return out


def finalize_reduce_residual_norm(expert_out, perm, w, shared, residual, gamma, eps: float,
                                  out=None, debug: Optional[Debug] = None,
                                  stream=None, workspace: Optional[torch.Tensor] = None,
                                  on_decline: str = "raise") -> torch.Tensor:
    """Per-shard finalize, rank-ordered sum, residual add (in place), RMSNorm.
    ``workspace`` and ``on_decline`` as for ``finalize_reduce_norm``."""
    L = load()
    R, T, k = perm.shape
    H = expert_out.shape[-1]
    dev = expert_out.device
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    args = (_need(expert_out, "expert_out", torch.bfloat16, (R, T * k, H), dev),
            _need(perm, "perm", torch.int32, (R, T, k), dev),
            _need(w, "w", torch.float32, (R, T, k), dev),
            _opt(shared, "shared", torch.bfloat16, (R, T, H), dev), R, T, k, H,
            _need(residual, "residual", torch.bfloat16, (T, H), dev),
            _need(gamma, "gamma", torch.float32, (H,), dev), float(eps),
            _need(out, "out", torch.bfloat16, (T, H), dev))
    d = _debug(debug, R, T, H, dev, True)
    with _with_device(expert_out):
        try:
            if workspace is None:
                _check(L.bn_finalize_reduce_residual_norm(*args, d[0] if d else None,
                                                          _stream(expert_out, stream)))
            else:
                wp, wn = _workspace(workspace, dev)
                _check(L.bn_finalize_reduce_residual_norm_ws(*args, d[0] if d else None, wp, wn,
                                                             _stream(expert_out, stream)))
        except BeamNormError as e:
            if not _fallback_allowed(e, on_decline):
                raise
            return _fallback(None, (expert_out, perm, w, shared), residual, None, gamma, eps,
                             out, debug, stream, single=True)
    return out


def reduce_only(partials, sum_out=None, stream=None) -> torch.Tensor:
    """Rank-ordered FP32 sum only (first half of the unfused split)."""
    L = load()
    R, T, H = partials.shape
    dev = partials.device
    if sum_out is None:
        sum_out = torch.empty((T, H), dtype=torch.float32, device=dev)
    with _with_device(partials):
        _check(L.bn_reduce_only(_need(partials, "partials", torch.bfloat16, (R, T, H), dev), R, T, H,
                                _need(sum_out, "sum_out", torch.float32, (T, H), dev),
                                _stream(partials, stream)))
    return sum_out


def finalize_reduce_only(expert_out, perm, w, shared, sum_out=None, stream=None) -> torch.Tensor:
    """Per-shard finalize rounded to BF16, then the rank-ordered FP32 sum only."""
    L = load()
    R, T, k = perm.shape
    H = expert_out.shape[-1]
    dev = expert_out.device
    if sum_out is None:
        sum_out = torch.empty((T, H), dtype=torch.float32, device=dev)
    with _with_device(expert_out):
        _check(L.bn_finalize_reduce_only(
            _need(expert_out, "expert_out", torch.bfloat16, (R, T * k, H), dev),
            _need(perm, "perm", torch.int32, (R, T, k), dev),
            _need(w, "w", torch.float32, (R, T, k), dev),
            _opt(shared, "shared", torch.bfloat16, (R, T, H), dev), R, T, k, H,
            _need(sum_out, "sum_out", torch.float32, (T, H), dev), _stream(expert_out, stream)))
    return sum_out


def norm_only(sum_, residual, gamma_post, gamma_pre, eps: float, out=None,
              debug: Optional[Debug] = None, stream=None) -> torch.Tensor:
    """The sandwich epilogue given the FP32 sum [T,H] (second half of the split)."""
    L = load()
    T, H = sum_.shape
    dev = sum_.device
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    args = (_need(sum_, "sum", torch.float32, (T, H), dev), T, H,
            _need(residual, "residual", torch.bfloat16, (T, H), dev),
            _need(gamma_post, "gamma_post", torch.float32, (H,), dev),
            _need(gamma_pre, "gamma_pre", torch.float32, (H,), dev), float(eps),
            _need(out, "out", torch.bfloat16, (T, H), dev))
    d = _debug(debug, 1, T, H, dev, False)
    with _with_device(sum_):
        _check(L.bn_norm_only(*args, d[0] if d else None, _stream(sum_, stream)))
    return out


def residual_norm_only(sum_, residual, gamma, eps: float, out=None,
                       debug: Optional[Debug] = None, stream=None) -> torch.Tensor:
    """The single-norm epilogue given the FP32 sum [T,H]: residual add (in
    place) and RMSNorm."""
    L = load()
    T, H = sum_.shape
    dev = sum_.device
    if out is None:
        out = torch.empty((T, H), dtype=torch.bfloat16, device=dev)
    args = (_need(sum_, "sum", torch.float32, (T, H), dev), T, H,
            _need(residual, "residual", torch.bfloat16, (T, H), dev),
            _need(gamma, "gamma", torch.float32, (H,), dev), float(eps),
            _need(out, "out", torch.bfloat16, (T, H), dev))
    d = _debug(debug, 1, T, H, dev, False)
    with _with_device(sum_):
        _check(L.bn_residual_norm_only(*args, d[0] if d else None, _stream(sum_, stream)))
    return out


def finalize_only(expert_out, perm, w, shared, z_out=None, stream=None) -> torch.Tensor:
    """The deferred finalize materialised: z [R,T,H] BF16 per shard, no reduction."""
    L = load()
    R, T, k = perm.shape
    H = expert_out.shape[-1]
    dev = expert_out.device
    if z_out is None:
        z_out = torch.empty((R, T, H), dtype=torch.bfloat16, device=dev)
    with _with_device(expert_out):
        _check(L.bn_finalize_only(
            _need(expert_out, "expert_out", torch.bfloat16, (R, T * k, H), dev),
            _need(perm, "perm", torch.int32, (R, T, k), dev),
            _need(w, "w", torch.float32, (R, T, k), dev),
            _opt(shared, "shared", torch.bfloat16, (R, T, H), dev), R, T, k, H,
            _need(z_out, "z_out", torch.bfloat16, (R, T, H), dev), _stream(expert_out, stream)))
    return z_out


def supports(R: int, T: int, k: int, H: int) -> bool:
    """True if the fused entry points serve this shape (k = 0: reduce entries)."""
    return bool(load().bn_supports(int(R), int(T), int(k), int(H)))


def supports_op(op: str, R: int, T: int, H: int, k: int = 0) -> bool:
    """True if entry point ``op`` (a name of OPS) serves this shape."""
    return bool(load().bn_supports_op(OPS.index(op), int(R), int(T), int(k), int(H)))


def check_device_error(stream=None, raise_on_error: bool = True) -> int:
    """Synchronise ``stream``, read and clear the device error bits."""
    L = load()
    bits = ctypes.c_uint(0)
    if stream is None:
        stream = torch.cuda.current_stream()
    st = L.bn_check_device_error(int(stream.cuda_stream) if hasattr(stream, "cuda_stream")
                                 else int(stream), ctypes.byref(bits))
    if st not in (OK, ERR_DEVICE) or (raise_on_error and st != OK):
        _check(st)
    return int(bits.value)


def set_tuning(cluster_size: int = 0, stages: int = 0, threads: int = 0, ctas_per_sm: int = 0,
               wait_mode: int = 0, group: int = 0, split: int = 0, dependent_launch: int = 0,
               wait_limit_polls: int = 0, tiny_pass: int = 0) -> None:
    """Override the launch shape for measurement sweeps (0 = automatic);
    ``wait_limit_polls`` shortens the pipeline waits' limit, for tests of the
    timeout path; ``tiny_pass`` (1 never, 2 always) overrides the choice of
    the kernels with the second pass over rows of tiny values."""
    t = _Tuning(int(cluster_size), int(stages), int(threads), int(ctas_per_sm), int(wait_mode),
                int(group), int(split), int(dependent_launch), int(wait_limit_polls),
                int(tiny_pass))
    _check(load().bn_set_tuning(ctypes.byref(t)))


def launch_info(op: str, R: int, T: int, H: int, k: int = 0, has_shared: bool = True) -> dict:
    """The launch shape ``op`` would use for this shape on the current device."""
    info = _LaunchInfo()
    _check(load().bn_query_launch(OPS.index(op), int(R), int(T), int(k), int(H),
                                  1 if has_shared else 0, ctypes.byref(info)))
    return {name: int(getattr(info, name)) for name, _ in _LaunchInfo._fields_}


def version() -> int:
    return int(load().bn_version())
