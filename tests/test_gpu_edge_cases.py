"""The method's edge cases through the CUDA path, against the oracle (GB300).

Each input set puts one edge case per token row (tp_reduce_residual_gb300.inputs
.edge_inputs): signed zeros, negated shard pairs that sum to +0, the
rank-order witness (1, 2^-24, 2^-24) that sums to 1 only in rank order, BF16
subnormals, constant rows, rows whose sums of squares leave the FP32 range,
shards holding +-inf and NaN, a finalize whose weighted products cancel
exactly (a guard against any fused multiply-add in the finalize), and rows of
tiny values whose squares are FP32 subnormals (their sums of squares normal,
or subnormal).  Every
entry point that runs these rows is compared with the oracle element by
element, with the bar of the other parity tests (sum and z bit-exact, NaN ==
NaN; sums of squares within 1e-5 relative, identical infinities; outputs within
1 BF16 ulp).  Outputs are prefilled with a finite sentinel, so a NaN result
is one the kernel wrote.

Sources: "Fuse Beam's TP all-reduce with its sandwich norms" (vLLM pull request
62366), section Claims (FP32 epilogue, finalize before the reduction keeping
the local BF16 rounding) and section Details (no FMA contraction).
"""
import numpy as np
import pytest
import torch

from tests import parity
from tests.helpers import SUBNORMAL_STEP, assert_bits_equal, f32_from_bf16
from tp_reduce_residual_gb300 import beamnorm as bn
from tp_reduce_residual_gb300 import build as nbuild
from tp_reduce_residual_gb300 import inputs

pytestmark = pytest.mark.gpu

KINDS = inputs.EDGE_KINDS
# the many-CTA finalize serves at most 8 token rows
WS_KINDS = ("neg_zero", "neg_pairs", "witness", "subnormal", "overflow_post", "overflow_pre",
            "inf_nan", "cancel")
EPS0_KINDS = ("normal", "constant", "zero", "neg_pairs")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    nbuild.build()
    bn.load()
    bn.set_tuning()
    yield
    bn.set_tuning()


def _check_known_values(d, g, kinds, single):
    """What the method fixes exactly, asserted on the GPU results themselves."""
    R, H = d["R"], d["H"]
    fin = d["op"] == "finalize_reduce_norm"
    shared = fin and d.get("shared") is not None
    res_in = inputs.u16(d["residual"])
    lanes = np.arange(H)
    for t, kind in enumerate(kinds):
        sb = g["sum"][t].view(np.uint32)
        zero_sum = False
        if kind == "witness":
            want = np.where(lanes % 2 == 0, 1.0, -1.0).astype(np.float32)
            assert_bits_equal(g["sum"][t], want, f"row {t}: rank-order witness sum")
        elif kind == "neg_zero":
            # -0 + -0 stays -0; a +0 anywhere (another shard, the shared row) makes +0
            neg = np.where(lanes % 2 == 0, not shared, R == 1 and not shared)
            assert np.all(sb == np.where(neg, 0x80000000, 0)), f"row {t}: signed zeros"
            zero_sum = True
        elif kind == "neg_pairs" or (kind == "cancel" and fin and d["k"] >= 2):
            assert np.all(sb == 0), f"row {t} ({kind}): the sum is not +0"
            zero_sum = True
            if kind == "cancel":
                assert np.all(g["z"][:, t] == 0), f"row {t}: the cancelling finalize is not +0"
        elif kind == "constant" and not single:
            assert np.all(g["sum"][t] == 1024.0)
            assert g["ss"][t, 0] == np.float32(H * 2.0 ** 20), g["ss"][t]
        elif kind == "overflow_post" and not single:
            assert np.isinf(g["ss"][t, 0]), f"row {t}: post-norm sum of squares {g['ss'][t, 0]}"
            assert np.all(np.isfinite(f32_from_bf16(g["out"][t])))
            assert np.all(np.isfinite(f32_from_bf16(g["residual_out"][t])))
        elif kind == "overflow_pre":
            assert np.isinf(g["ss"][t, 1]), f"row {t}: pre-norm sum of squares {g['ss'][t, 1]}"
            assert np.all(np.isfinite(f32_from_bf16(g["residual_out"][t])))
        if zero_sum:
            # y (or s itself) is a signed zero: the residual comes back unchanged
            assert np.all((g["residual_out"][t] & 0x7FFF) == (res_in[t] & 0x7FFF)), kind
    if single:
        assert np.all(g["ss"][:, 0] == 0.0)


REDUCE = [
    # (R, H, single)
    (1, 1000, False), (1, 1000, True), (3, 256, False), (4, 5120, False), (4, 5120, True),
    (8, 8192, False), (8, 8192, True), (2, 32768, False),
]


@pytest.mark.parametrize("R,H,single", REDUCE)
def test_reduce_edge_cases_match_oracle(R, H, single):
    d = inputs.edge_inputs("reduce_norm", R, H, KINDS, seed=100 + R + H)
    g = parity.run_fused(d, single=single, prefill="sentinel")
    parity.compare(g, parity.run_oracle(d, single=single), what=f"edge reduce R={R} H={H}")
    _check_known_values(d, g, KINDS, single)


FINALIZE = [
    # (R, k, H, with_shared, single)
    (1, 1, 1000, False, False), (2, 2, 256, True, False), (4, 4, 5120, False, False),
    (4, 4, 5120, True, True), (8, 4, 8192, True, False), (8, 8, 6144, False, True),
]


@pytest.mark.parametrize("R,k,H,with_shared,single", FINALIZE)
def test_finalize_edge_cases_match_oracle(R, k, H, with_shared, single):
    d = inputs.edge_inputs("finalize_reduce_norm", R, H, KINDS, k=k, seed=200 + R + H,
                           with_shared=with_shared)
    g = parity.run_fused(d, single=single, prefill="sentinel")
    parity.compare(g, parity.run_oracle(d, single=single), what=f"edge finalize R={R} k={k} H={H}")
    _check_known_values(d, g, KINDS, single)


@pytest.mark.parametrize("tuning", [dict(split=1, cluster_size=1), dict(split=1, cluster_size=4),
                                    dict(split=2, cluster_size=2), dict(cluster_size=8),
                                    dict(split=3, cluster_size=16), dict(split=3, cluster_size=2)],
                         ids=["one-CTA", "columns-x4", "shards-x2", "cluster-x8", "tasks-x16",
                              "tasks-x2"])
def test_edge_cases_on_every_row_split(tuning):
    """The same rows through the column split (1 or 4 CTAs a row), the shard
    split and an 8-CTA cluster: the cluster exchanges carry infinite and NaN
    partial sums of squares too."""
    for op in ("reduce_norm", "finalize_reduce_norm"):
        d = inputs.edge_inputs(op, 4, 5120, KINDS, k=2, seed=300, with_shared=True)
        try:
            bn.set_tuning(**(tuning if op.startswith("finalize") else
                             {"cluster_size": tuning.get("cluster_size", 0),
                              "split": tuning.get("split", 0) if tuning.get("split") != 2 else 0}))
            g = parity.run_fused(d, prefill="sentinel")
        finally:
            bn.set_tuning()
        parity.compare(g, parity.run_oracle(d), what=f"edge {op} {tuning}")
        _check_known_values(d, g, KINDS, False)


@pytest.mark.parametrize("single", [False, True])
@pytest.mark.parametrize("R,k,H", [(8, 4, 8192), (3, 2, 1000), (8, 8, 6144)])
def test_workspace_finalize_edge_cases(R, k, H, single):
    d = inputs.edge_inputs("finalize_reduce_norm", R, H, WS_KINDS, k=k, seed=400 + R + H,
                           with_shared=True)
    ws = bn.finalize_workspace(R, len(WS_KINDS), k, H, device="cuda")
    assert ws is not None
    g = parity.run_fused(d, single=single, workspace=ws, prefill="sentinel")
    parity.compare(g, parity.run_oracle(d, single=single), what=f"edge workspace R={R} H={H}")
    _check_known_values(d, g, WS_KINDS, single)


@pytest.mark.parametrize("op", ["reduce_norm", "finalize_reduce_norm"])
def test_split_and_materialised_finalize_edge_cases(op):
    """The unfused pieces on the same rows: the FP32 sum, then the epilogue;
    and the materialised per-shard finalize."""
    d = inputs.edge_inputs(op, 4, 1000, KINDS, k=4, seed=500, with_shared=True)
    ref = parity.run_oracle(d)
    if op == "reduce_norm":
        s = bn.reduce_only(d["partials"])
    else:
        s = bn.finalize_reduce_only(d["expert_out"], d["perm"], d["w"], d["shared"])
        z = bn.finalize_only(d["expert_out"], d["perm"], d["w"], d["shared"])
        torch.cuda.synchronize()
        assert_bits_equal(inputs.u16(z), ref["z"], "materialised z")
    res = d["residual"].clone()
    ss = parity._sentinel_like((d["T"], 2), torch.float32)
    out = bn.norm_only(s, res, d["gamma_post"], d["gamma_pre"], d["eps"], debug=bn.Debug(ss=ss))
    assert bn.check_device_error() == 0
    g = {"sum": s.cpu().numpy(), "ss": ss.cpu().numpy(), "out": inputs.u16(out),
         "residual_out": inputs.u16(res)}
    parity.compare(g, ref, what=f"edge split {op}")


@pytest.mark.parametrize("op,single", [("reduce_norm", False), ("reduce_norm", True),
                                       ("finalize_reduce_norm", False)])
def test_eps_zero_with_an_all_zero_row(op, single):
    """eps = 0: an all-zero row (and a row of negated pairs) has a zero sum of
    squares, so its RMS factor is 1/0 = inf and 0 * inf gives NaN on both
    sides; the other rows are unaffected."""
    d = inputs.edge_inputs(op, 4, 5120, EPS0_KINDS, k=2, seed=600, eps=0.0)
    g = parity.run_fused(d, single=single, prefill="sentinel")
    ref = parity.run_oracle(d, single=single)
    parity.compare(g, ref, what=f"eps=0 {op}")
    if not single:
        zero_row = EPS0_KINDS.index("zero")
        assert np.all(np.isnan(f32_from_bf16(g["out"][zero_row])))
        normal_row = EPS0_KINDS.index("normal")
        assert np.all(np.isfinite(f32_from_bf16(g["out"][normal_row])))


TINY_KINDS = ("normal", "tiny", "tiny_sub", "tiny")


@pytest.mark.parametrize("tuning", [{}, dict(split=1, cluster_size=1), dict(split=1, cluster_size=4),
                                    dict(split=3, cluster_size=4)],
                         ids=["planner", "one-CTA", "columns-x4", "tasks-x4"])
@pytest.mark.parametrize("op,single", [("reduce_norm", False), ("reduce_norm", True),
                                       ("finalize_reduce_norm", False),
                                       ("finalize_reduce_norm", True)])
def test_tiny_rows_with_eps_zero(op, single, tuning):
    """eps = 0: the RMS factor is the sum of squares' alone, so an inexact sum
    of squares shows in every output.  Rows of values near 2^-66 and 2^-76 have
    subnormal squares; the kernels sum such a row again with its values scaled
    by a power of two, and must match the oracle's exactly accumulated sums
    (rounded once to FP32) within 1e-5 relative or one subnormal step."""
    d = inputs.edge_inputs(op, 4, 5120, TINY_KINDS, k=2, seed=700, eps=0.0, with_shared=True)
    try:
        if op == "finalize_reduce_norm":
            bn.set_tuning(**tuning)
        else:
            bn.set_tuning(**{k: v for k, v in tuning.items() if k == "cluster_size"})
        g = parity.run_fused(d, single=single, prefill="sentinel")
    finally:
        bn.set_tuning()
    ref = parity.run_oracle(d, single=single)
    # eps = 0 < 2^-50: the kernels with the second pass, within one subnormal step
    parity.compare(g, ref, what=f"tiny eps=0 {op} single={single} {tuning}",
                   ss_floor=SUBNORMAL_STEP)
    for t, kind in enumerate(TINY_KINDS):
        if kind == "tiny":
            assert np.all(np.isfinite(f32_from_bf16(g["residual_out"][t]))), kind
            # a normal sum of squares whose squares are all subnormal
            col = 1 if single else 0
            assert 2.0 ** -126 <= ref["ss"][t, col] < 2.0 ** -80, ref["ss"][t]
            assert np.all(np.isfinite(f32_from_bf16(g["out"][t])))
        if kind == "tiny_sub":
            assert 0 < ref["ss"][t, 1 if single else 0] < 2.0 ** -126, ref["ss"][t]


@pytest.mark.parametrize("single", [False, True])
def test_workspace_finalize_tiny_rows(single):
    """The many-CTA finalize (caller workspace) on the same rows, eps = 0 and
    eps = 1e-6 (where the residual sum of squares is tiny too)."""
    for eps in (0.0, 1e-6):
        d = inputs.edge_inputs("finalize_reduce_norm", 8, 8192, TINY_KINDS, k=4, seed=710,
                               eps=eps, with_shared=True)
        ws = bn.finalize_workspace(8, len(TINY_KINDS), 4, 8192, device="cuda")
        assert ws is not None
        g = parity.run_fused(d, single=single, workspace=ws, prefill="sentinel")
        parity.compare(g, parity.run_oracle(d, single=single), what=f"tiny workspace eps={eps}",
                       ss_floor=SUBNORMAL_STEP if eps == 0.0 else None)


@pytest.mark.parametrize("eps", [2.0 ** -50, 1e-6])
@pytest.mark.parametrize("path", ["planner", "one-CTA", "workspace"])
def test_tiny_pass_changes_no_output_for_eps_from_2_pow_minus_50(eps, path):
    """For eps >= 2^-50 the planner runs the kernels without the second pass:
    a sum of squares below 2^-80 then cannot reach the RMS factor, whose sum
    fl(fl(ss / H) + eps) rounds to eps either way.  The same rows with the
    pass forced on and off give bit-identical outputs and residuals; the sums
    of squares meet 2^-149 with the pass and H * 2^-149 without it."""
    d = inputs.edge_inputs("finalize_reduce_norm", 8, 8192, TINY_KINDS, k=4, seed=720, eps=eps,
                           with_shared=True)
    ref = parity.run_oracle(d)
    kw = {}
    if path == "workspace":
        kw["workspace"] = bn.finalize_workspace(8, len(TINY_KINDS), 4, 8192, device="cuda")
    runs = {}
    for tiny_pass in (1, 2):
        try:
            bn.set_tuning(tiny_pass=tiny_pass, **({"split": 1} if path == "one-CTA" else {}))
            runs[tiny_pass] = parity.run_fused(d, prefill="sentinel", **kw)
        finally:
            bn.set_tuning()
    parity.compare(runs[1], ref, what=f"tiny pass off eps={eps} {path}")
    parity.compare(runs[2], ref, what=f"tiny pass on eps={eps} {path}", ss_floor=SUBNORMAL_STEP)
    for key in ("out", "residual_out", "sum"):
        assert np.array_equal(runs[1][key].view(np.uint8), runs[2][key].view(np.uint8)), key
    # the automatic choice is the kernel without the pass: its results exactly
    g = parity.run_fused(d, prefill="sentinel", **kw)
    for key in ("out", "residual_out", "ss"):
        assert np.array_equal(g[key].view(np.uint8), runs[1][key].view(np.uint8)), key


@pytest.mark.parametrize("single", [False, True])
def test_tiny_rows_with_eps_zero_through_the_pieces(single):
    """The epilogue pieces (norm_only, residual_norm_only) on the FP32 sum of
    rows of tiny values at eps = 0: their kernels with the second pass meet the
    oracle within one subnormal step, as the fused entry points do."""
    d = inputs.edge_inputs("reduce_norm", 4, 5120, TINY_KINDS, seed=730, eps=0.0)
    ref = parity.run_oracle(d, single=single)
    s = bn.reduce_only(d["partials"])
    res = d["residual"].clone()
    ss = parity._sentinel_like((d["T"], 2), torch.float32)
    if single:
        out = bn.residual_norm_only(s, res, d["gamma_pre"], d["eps"], debug=bn.Debug(ss=ss))
    else:
        out = bn.norm_only(s, res, d["gamma_post"], d["gamma_pre"], d["eps"], debug=bn.Debug(ss=ss))
    assert bn.check_device_error() == 0
    g = {"sum": s.cpu().numpy(), "ss": ss.cpu().numpy(), "out": inputs.u16(out),
         "residual_out": inputs.u16(res)}
    parity.compare(g, ref, what=f"tiny eps=0 pieces single={single}", ss_floor=SUBNORMAL_STEP)
