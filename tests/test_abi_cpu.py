"""Host-side tests of the C ABI (no GPU needed, no compute call made).

The library is loaded on a machine without a GPU; every call here is rejected
by host-side validation before any CUDA runtime call, or is pure host logic.
"""
import ctypes
import os
import re

import pytest
import torch

from tp_reduce_residual_gb300 import beamnorm as bn
from tp_reduce_residual_gb300 import build as nbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "beamnorm.h")

A16 = 0x10000      # a 16-byte aligned fake device address (never dereferenced)
MIS = 0x10004      # 4-byte aligned, not 16-byte aligned


@pytest.fixture(scope="module")
def L():
    nbuild.build()
    return bn.load()


def declared_symbols():
    text = open(HEADER).read()
    return sorted(set(re.findall(r"BN_API\s+[\w\s\*]+?\b(bn_\w+)\s*\(", text)))


def test_every_declared_symbol_is_exported(L):
    names = declared_symbols()
    assert len(names) == len(bn.EXPORTS) and set(names) == set(bn.EXPORTS), names
    for name in names:
        assert hasattr(L, name), name


def test_every_declaration_cites_its_passage():
    """Each entry point's comment names the passage that defines it, or says
    that none does ("no passage: library utility", "no counterpart")."""
    text = open(HEADER).read()
    for m in re.finditer(r"/\*((?:(?!\*/).)*)\*/\s*BN_API\s+[\w\s\*]+?\b(bn_\w+)\s*\(", text, re.S):
        comment, name = " ".join(m.group(1).replace("*", " ").split()), m.group(2)
        assert re.search(r"Sources?:", comment), f"{name}: no Source line"
        assert ("pull request" in comment or "sandwich norms" in comment
                or "no passage" in comment or "no counterpart" in comment), \
            f"{name}: the Source line names no page"
    cited = set(re.findall(r"\*/\s*BN_API\s+[\w\s\*]+?\b(bn_\w+)\s*\(", text))
    assert cited == set(declared_symbols()), set(declared_symbols()) - cited


def test_library_is_built_for_sm103a():
    # the build passes exactly one -gencode, for sm_103a
    assert nbuild.ARCH == ["-gencode", "arch=compute_103a,code=sm_103a"]
    assert "-fmad=false" in nbuild.NVCC_FLAGS


def test_version_and_status_strings(L):
    assert L.bn_version() == 10200
    assert L.bn_status_string(0) == b"BN_OK"
    assert L.bn_status_string(2) == b"BN_ERR_UNSUPPORTED"
    assert L.bn_status_string(99) == b"unknown status"


@pytest.mark.parametrize("R,T,k,H,expect", [
    (2, 8, 0, 256, 1), (4, 4096, 0, 5120, 1), (8, 4096, 0, 8192, 1), (8, 1024, 8, 6144, 1),
    (8, 4096, 10, 8192, 1), (16, 1, 16, 32768, 1), (1, 0, 0, 8, 1),
    (0, 8, 0, 256, 0), (17, 8, 0, 256, 0), (2, -1, 0, 256, 0), (2, 8, 0, 0, 0), (2, 8, 0, 100, 0),
    (2, 8, 0, 32776, 0), (16, 8, 17, 256, 0), (8, 2 ** 28, 10, 256, 0),
])
def test_supports(L, R, T, k, H, expect):
    assert L.bn_supports(R, T, k, H) == expect


def _reduce(L, partials=A16, R=2, T=8, H=256, residual=A16 * 2, gp=A16 * 3, gq=A16 * 4,
            eps=1e-6, out=A16 * 5):
    return L.bn_reduce_norm(partials, R, T, H, residual, gp, gq, eps, out, None, None)


@pytest.mark.parametrize("kw,needle", [
    (dict(partials=None), "partials is NULL"),
    (dict(residual=None), "residual is NULL"),
    (dict(out=None), "out is NULL"),
    (dict(gp=None), "gamma_post is NULL"),
    (dict(R=0), "R=0"),
    (dict(R=17), "R=17"),
    (dict(T=-3), "T=-3"),
    (dict(H=250), "multiple of 8"),
    (dict(H=0), "H=0"),
    (dict(partials=MIS), "partials is not 16-byte aligned"),
    (dict(out=MIS), "out is not 16-byte aligned"),
    (dict(eps=-1.0), "eps"),
    (dict(eps=float("nan")), "eps"),
    (dict(eps=float("inf")), "eps"),
    (dict(out=A16 * 2), "overlaps"),           # out == residual
    (dict(out=A16 + 64), "overlaps"),          # out inside partials
    (dict(residual=A16 + 16), "overlaps"),     # residual inside partials
])
def test_reduce_norm_rejects_bad_arguments(L, kw, needle):
    assert _reduce(L, **kw) == bn.ERR_INVALID
    assert needle in L.bn_last_error().decode()


def test_unsupported_shape_is_declined_before_any_work(L):
    # valid arguments, H above the served maximum: declined, nothing enqueued
    st = _reduce(L, H=40960, residual=A16 * 1000, gp=A16 * 2000, gq=A16 * 2100, out=A16 * 3000)
    assert st == bn.ERR_UNSUPPORTED
    assert "H=40960" in L.bn_last_error().decode()


def test_zero_tokens_is_a_no_op(L):
    assert _reduce(L, T=0) == bn.OK
    assert L.bn_last_error() == b""


def test_finalize_rejects_bad_arguments(L):
    f = L.bn_finalize_reduce_norm
    args = dict(x=A16, perm=A16 * 10, w=A16 * 20, sh=A16 * 30, R=2, T=4, k=3, H=64,
                res=A16 * 40, gp=A16 * 50, gq=A16 * 60, eps=1e-6, out=A16 * 70)

    def call(**kw):
        a = dict(args, **kw)
        return f(a["x"], a["perm"], a["w"], a["sh"], a["R"], a["T"], a["k"], a["H"], a["res"],
                 a["gp"], a["gq"], a["eps"], a["out"], None, None)

    assert call(k=0) == bn.ERR_INVALID
    assert call(k=17) == bn.ERR_INVALID
    assert call(perm=None) == bn.ERR_INVALID
    assert call(perm=A16 * 10 + 2) == bn.ERR_INVALID       # perm needs 4-byte alignment
    assert call(w=None) == bn.ERR_INVALID
    assert call(sh=A16 * 30 + 8) == bn.ERR_INVALID         # shared misaligned
    assert call(out=A16 * 10) == bn.ERR_INVALID            # out overlaps perm
    assert call(R=16, k=16, T=0) == bn.OK                  # nothing to do
    assert call(T=0) == bn.OK


def test_finalize_workspace_size(L):
    # the counters (T words, padded to 256 bytes), then z [T, R, H] BF16
    assert L.bn_finalize_workspace_bytes(8, 1, 10, 8192) == 256 + 8 * 8192 * 2
    assert L.bn_finalize_workspace_bytes(8, 8, 10, 8192) == 256 + 8 * 8 * 8192 * 2
    assert L.bn_finalize_workspace_bytes(2, 9, 3, 64) == 0        # above the served T
    assert L.bn_finalize_workspace_bytes(3, 7, 5, 6144) == 256 + 7 * 3 * 6144 * 2
    for R, T, k, H in ((8, 0, 10, 8192), (8, 4, 10, 8200), (0, 4, 1, 64), (17, 4, 1, 64),
                       (2, 4, 0, 64), (2, 4, 17, 64), (2, 4, 3, 60)):
        assert L.bn_finalize_workspace_bytes(R, T, k, H) == 0, (R, T, k, H)
    assert bn.finalize_workspace_bytes(8, 4, 10, 8192) == 256 + 4 * 8 * 8192 * 2


def test_finalize_with_workspace_rejects_bad_arguments(L):
    f = L.bn_finalize_reduce_norm_ws
    need = L.bn_finalize_workspace_bytes(2, 4, 3, 64)
    args = dict(x=A16, perm=A16 * 10, w=A16 * 20, sh=A16 * 30, R=2, T=4, k=3, H=64,
                res=A16 * 40, gp=A16 * 50, gq=A16 * 60, eps=1e-6, out=A16 * 70, ws=A16 * 80,
                wsb=need)

    def call(**kw):
        a = dict(args, **kw)
        return f(a["x"], a["perm"], a["w"], a["sh"], a["R"], a["T"], a["k"], a["H"], a["res"],
                 a["gp"], a["gq"], a["eps"], a["out"], None, a["ws"], a["wsb"], None)

    assert call(ws=A16 * 80 + 8) == bn.ERR_INVALID          # workspace misaligned
    assert call(ws=A16 * 10) == bn.ERR_INVALID              # workspace overlaps perm
    assert call(ws=A16 * 70) == bn.ERR_INVALID              # workspace overlaps out
    assert call(k=0) == bn.ERR_INVALID
    assert call(perm=None) == bn.ERR_INVALID
    assert call(T=0) == bn.OK
    g = L.bn_finalize_reduce_residual_norm_ws
    assert g(A16, A16 * 10, A16 * 20, None, 2, 4, 3, 64, A16 * 40, A16 * 50, 1e-6, A16 * 70, None,
             A16 * 40, need, None) == bn.ERR_INVALID         # workspace overlaps the residual


def test_split_and_finalize_only_reject_bad_arguments(L):
    assert L.bn_reduce_only(A16, 2, 4, 64, None, None) == bn.ERR_INVALID
    assert L.bn_reduce_only(A16, 2, 4, 64, A16 + 32, None) == bn.ERR_INVALID   # sum overlaps
    assert L.bn_norm_only(None, 4, 64, A16, A16 * 2, A16 * 3, 1e-6, A16 * 4, None, None) == bn.ERR_INVALID
    assert L.bn_finalize_only(A16, A16 * 10, A16 * 20, None, 2, 4, 3, 64, None, None) == bn.ERR_INVALID
    assert L.bn_finalize_reduce_only(A16, A16 * 10, A16 * 20, None, 2, 4, 3, 63, A16 * 40,
                                     None) == bn.ERR_INVALID


def test_set_tuning_validates(L):
    def st(*fields):
        return L.bn_set_tuning(ctypes.byref(bn._Tuning(*fields)))
    assert st(17, 0, 0, 0, 0, 0) == bn.ERR_INVALID
    assert st(-1, 0, 0, 0, 0, 0) == bn.ERR_INVALID
    assert st(0, 1, 0, 0, 0, 0) == bn.ERR_INVALID
    assert st(0, 65, 0, 0, 0, 0) == bn.ERR_INVALID
    assert st(0, 0, 48, 0, 0, 0) == bn.ERR_INVALID
    assert st(0, 0, 0, 9, 0, 0) == bn.ERR_INVALID
    assert st(0, 0, 0, 0, 3, 0) == bn.ERR_INVALID
    assert st(0, 0, 0, 0, 0, 65) == bn.ERR_INVALID
    assert st(0, 0, 0, 0, 0, 0, 4) == bn.ERR_INVALID
    assert st(0, 0, 0, 0, 0, 0, 0, 3) == bn.ERR_INVALID
    assert st(0, 0, 0, 0, 0, 0, 0, 0, -1) == bn.ERR_INVALID
    assert st(0, 0, 0, 0, 0, 0, 0, 0, 0, 3) == bn.ERR_INVALID
    assert st(0, 0, 0, 0, 0, 0, 0, 0, 0, -1) == bn.ERR_INVALID
    assert st(16, 8, 256, 2, 2, 4, 2, 1) == bn.OK
    assert st(0, 0, 0, 0, 0, 0, 0, 0, 3) == bn.OK
    assert st(0, 0, 0, 0, 0, 0, 0, 0, 0, 2) == bn.OK
    assert L.bn_set_tuning(None) == bn.OK


def test_python_binding_checks_before_calling(L):
    cpu = torch.zeros(2, 8, 256, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA tensor"):
        bn.reduce_norm(cpu, torch.zeros(8, 256, dtype=torch.bfloat16), torch.zeros(256),
                       torch.zeros(256), 1e-6)


def test_binding_fails_loudly_without_library(monkeypatch):
    monkeypatch.setattr(bn, "_lib", None)
    monkeypatch.setattr(bn, "LIB_PATH", "/nonexistent/libbeamnorm.so")
    with pytest.raises(RuntimeError, match="not built"):
        bn.load()


def test_query_launch_validates_on_the_host(L):
    info = bn._LaunchInfo()
    q = lambda *a: L.bn_query_launch(*a, ctypes.byref(info))
    assert L.bn_query_launch(0, 2, 8, 0, 256, 0, None) == bn.ERR_INVALID
    assert q(9, 2, 8, 0, 256, 0) == bn.ERR_INVALID          # no such operation
    assert q(-1, 2, 8, 0, 256, 0) == bn.ERR_INVALID
    assert q(0, 0, 8, 0, 256, 0) == bn.ERR_INVALID          # R outside [1, 16]
    assert q(1, 8, 8, 0, 256, 1) == bn.ERR_INVALID          # finalize needs k >= 1
    assert q(0, 2, 8, 0, 260, 0) == bn.ERR_INVALID          # H % 8 != 0
    assert q(0, 2, 8, 0, 40000, 0) == bn.ERR_UNSUPPORTED    # declined: H above the maximum
    info.grid = 7
    assert q(3, 8, 0, 10, 8192, 1) == bn.OK                 # T == 0: no launch, all zero
    assert info.grid == 0 and info.stages == 0
    assert bn.OPS.index("finalize_only") == 7 and bn.OPS.index("residual_norm_only") == 8


@pytest.mark.parametrize("op,R,T,k,H,expect", [
    # fused entry points: rows up to 32768
    ("reduce_norm", 4, 8, 0, 32768, 1), ("reduce_norm", 4, 8, 0, 40960, 0),
    ("finalize_reduce_norm", 2, 3, 2, 40960, 0), ("reduce_residual_norm", 2, 3, 0, 65536, 0),
    ("finalize_reduce_residual_norm", 8, 1, 10, 8192, 1),
    # the unfused pieces, the fallback: rows up to 131072
    ("reduce_only", 4, 8, 0, 40960, 1), ("reduce_only", 4, 8, 0, 131072, 1),
    ("reduce_only", 4, 8, 0, 131080, 0), ("finalize_reduce_only", 2, 3, 2, 65536, 1),
    ("finalize_only", 2, 3, 2, 40960, 1), ("norm_only", 1, 3, 0, 131072, 1),
    ("norm_only", 9, 3, 0, 131072, 1),            # R is ignored by the epilogue pieces
    ("residual_norm_only", 1, 3, 0, 98304, 1), ("residual_norm_only", 1, 3, 0, 262144, 0),
    # invalid arguments are not served either
    ("finalize_only", 2, 3, 0, 64, 0), ("reduce_only", 17, 3, 0, 64, 0),
    ("finalize_only", 2, 2 ** 28, 16, 64, 0),      # T * k >= 2^31
])
def test_supports_op(L, op, R, T, k, H, expect):
    assert L.bn_supports_op(bn.OPS.index(op), R, T, k, H) == expect
    if op in ("reduce_norm", "finalize_reduce_norm") and expect == 0:
        assert L.bn_supports(R, T, k, H) == 0


def test_supports_op_rejects_unknown_operations(L):
    assert L.bn_supports_op(len(bn.OPS), 2, 8, 0, 256) == 0
    assert L.bn_supports_op(-1, 2, 8, 0, 256) == 0


def test_residual_norm_only_validates_on_the_host(L):
    f = L.bn_residual_norm_only
    assert f(None, 4, 64, A16 * 10, A16 * 20, 1e-6, A16 * 30, None, None) == bn.ERR_INVALID
    assert f(A16, 4, 64, None, A16 * 20, 1e-6, A16 * 30, None, None) == bn.ERR_INVALID
    assert f(A16, 4, 60, A16 * 10, A16 * 20, 1e-6, A16 * 30, None, None) == bn.ERR_INVALID
    assert f(A16, 4, 64, A16 * 10, A16 * 20, -1.0, A16 * 30, None, None) == bn.ERR_INVALID
    assert f(A16, 4, 64, A16 * 10, A16 * 20, 1e-6, A16 + 16, None, None) == bn.ERR_INVALID
    assert "overlaps" in L.bn_last_error().decode()
    assert f(A16, 0, 64, None, None, 1e-6, None, None, None) == bn.OK
    big = 262144
    assert f(A16, 1, big, A16 * 100000, A16 * 200000, 1e-6, A16 * 300000, None,
             None) == bn.ERR_UNSUPPORTED
    assert "unfused pieces" in L.bn_last_error().decode()


def test_binding_rejects_an_unknown_decline_policy():
    err = bn.BeamNormError(bn.ERR_UNSUPPORTED, "declined")
    with pytest.raises(ValueError, match="on_decline"):
        bn._fallback_allowed(err, "ignore")
    assert bn._fallback_allowed(err, "fallback")
    assert not bn._fallback_allowed(err, "raise")
    assert not bn._fallback_allowed(bn.BeamNormError(bn.ERR_INVALID, "bad"), "fallback")

