"""GPU parity of libbeamnorm's kernels against the CPU oracle (GB300, sm_103a).

Every call goes through the C ABI (via the ctypes binding).  The bar: the FP32
reduced sum and the per-shard BF16 finalize bit-exact; sums of squares within
1e-5 relative; BF16 outputs and the updated residual within 1 BF16 ulp.
"""
import numpy as np
import pytest
import torch

import oracle
from tests import parity
from tests.helpers import assert_bf16_close, assert_bits_equal
from tp_reduce_residual_gb300 import beamnorm as bn
from tp_reduce_residual_gb300 import build as nbuild
from tp_reduce_residual_gb300 import inputs

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    nbuild.build()
    bn.load()
    bn.set_tuning()
    yield
    bn.set_tuning()
    torch.cuda.empty_cache()


def _free():
    torch.cuda.synchronize()
    torch.cuda.empty_cache()


# ---- small shapes: several tiles, ragged tails, extremes ----------------------------

REDUCE_SMALL = [
    # (R, T, H, row_scale, partial_std)
    (2, 8, 256, False, 1.0),
    (4, 37, 5120, False, 0.5),
    (8, 70, 8192, True, 0.5),
    (3, 5, 1000, False, 0.5),      # 125 chunks: ragged against 32-thread warps
    (1, 3, 8, False, 0.5),         # one chunk per row
    (16, 2, 32768, False, 0.5),    # largest served R and H
    (5, 153, 6144, True, 0.5),     # more rows than SMs
    (4, 300, 32768, False, 0.5),   # largest H with many rows: the row needs a cluster
]


@pytest.mark.parametrize("R,T,H,row_scale,std", REDUCE_SMALL)
def test_reduce_norm_small(R, T, H, row_scale, std):
    wl = inputs.custom("reduce_norm", R, H, partial_std=std, row_scale=row_scale)
    d = parity.gpu_inputs(wl, T, seed=1000 + R * 7 + T)
    g = parity.run_fused(d)
    parity.compare(g, parity.run_oracle(d), what=f"reduce R={R} T={T} H={H}")


FIN_SMALL = [
    # (R, T, k, H)
    (8, 19, 8, 6144),
    (8, 13, 10, 8192),
    (2, 7, 3, 1000),
    (1, 5, 1, 64),
    (16, 3, 16, 4096),             # R*k = 256, the served maximum
    (2, 200, 2, 32768),            # largest H with many rows
]


@pytest.mark.parametrize("with_shared", [True, False])
@pytest.mark.parametrize("R,T,k,H", FIN_SMALL)
def test_finalize_reduce_norm_small(R, T, k, H, with_shared):
    wl = inputs.custom("finalize_reduce_norm", R, H, k, partial_std=0.3, shared_std=0.3)
    d = parity.gpu_inputs(wl, T, seed=2000 + R * 11 + T, with_shared=with_shared)
    g = parity.run_fused(d)
    parity.compare(g, parity.run_oracle(d), what=f"finalize R={R} T={T} k={k} H={H}")


@pytest.mark.parametrize("op", ["reduce_norm", "finalize_reduce_norm"])
def test_single_norm_variants(op):
    if op == "reduce_norm":
        wl = inputs.custom(op, 4, 5120)
        d = parity.gpu_inputs(wl, 29, seed=31)
    else:
        wl = inputs.custom(op, 8, 6144, 8, partial_std=0.3)
        d = parity.gpu_inputs(wl, 11, seed=32)
    g = parity.run_fused(d, single=True)
    ref = parity.run_oracle(d, single=True)
    parity.compare(g, ref, what=f"{op} single norm")
    assert np.all(g["ss"][:, 0] == 0.0)


# ---- the five workloads at their full sizes ------------------------------------------

SWEEP = [(wl.index, T) for wl in inputs.WORKLOADS for T in wl.tokens]


@pytest.mark.parametrize("idx,T", SWEEP, ids=[f"C{i}-T{T}" for i, T in SWEEP])
def test_workload_parity(idx, T):
    """Every token row of every workload at its full size, in the launch shape
    the benchmark times, against the oracle."""
    wl = inputs.WORKLOADS[idx]
    d = parity.gpu_inputs(wl, T)
    g = parity.run_fused(d)
    stats = parity.compare(g, parity.run_oracle_all_rows(d), what=wl.describe(T))
    # the compensated sums of squares are the correctly rounded exact sums:
    # nearly all match the oracle's double accumulation bit for bit
    assert stats["ss_exact"] >= 0.99, stats
    del d, g
    _free()


# ---- unfused split and the materialised finalize ---------------------------------------

def test_reduce_split_equals_fused():
    wl = inputs.WORKLOADS[2]
    d = parity.gpu_inputs(wl, 64)
    fused = parity.run_fused(d)
    s = bn.reduce_only(d["partials"])
    res = d["residual"].clone()
    ss = torch.zeros(64, 2, device="cuda")
    out = bn.norm_only(s, res, d["gamma_post"], d["gamma_pre"], d["eps"], debug=bn.Debug(ss=ss))
    torch.cuda.synchronize()
    assert_bits_equal(s.cpu().numpy(), fused["sum"], "sum")
    assert_bits_equal(inputs.u16(res), fused["residual_out"], "residual_out")
    assert_bits_equal(inputs.u16(out), fused["out"], "out")
    assert_bits_equal(ss.cpu().numpy(), fused["ss"], "ss")


@pytest.mark.parametrize("op", ["reduce_norm", "finalize_reduce_norm"])
def test_single_norm_split_equals_fused(op):
    """The single-norm pattern unfused: the FP32 sum, then residual_norm_only."""
    wl = inputs.custom(op, 4, 5120, 3 if op != "reduce_norm" else 0, partial_std=0.3)
    d = parity.gpu_inputs(wl, 29, seed=41)
    fused = parity.run_fused(d, single=True)
    if op == "reduce_norm":
        s = bn.reduce_only(d["partials"])
    else:
        s = bn.finalize_reduce_only(d["expert_out"], d["perm"], d["w"], d["shared"])
    res = d["residual"].clone()
    ss = torch.full((29, 2), float("nan"), device="cuda")
    out = bn.residual_norm_only(s, res, d["gamma_pre"], d["eps"], debug=bn.Debug(ss=ss))
    torch.cuda.synchronize()
    assert_bits_equal(s.cpu().numpy(), fused["sum"], "sum")
    assert_bits_equal(inputs.u16(res), fused["residual_out"], "residual_out")
    assert_bits_equal(inputs.u16(out), fused["out"], "out")
    assert_bits_equal(ss.cpu().numpy(), fused["ss"], "ss")


@pytest.mark.parametrize("with_shared", [True, False])
def test_finalize_split_equals_fused(with_shared):
    wl = inputs.WORKLOADS[4]
    d = parity.gpu_inputs(wl, 16, with_shared=with_shared)
    fused = parity.run_fused(d)
    s = bn.finalize_reduce_only(d["expert_out"], d["perm"], d["w"], d["shared"])
    res = d["residual"].clone()
    out = bn.norm_only(s, res, d["gamma_post"], d["gamma_pre"], d["eps"])
    torch.cuda.synchronize()
    assert_bits_equal(s.cpu().numpy(), fused["sum"], "sum")
    assert_bits_equal(inputs.u16(res), fused["residual_out"], "residual_out")
    assert_bits_equal(inputs.u16(out), fused["out"], "out")


def test_finalize_only_matches_oracle():
    wl = inputs.WORKLOADS[3]
    d = parity.gpu_inputs(wl, 16)
    z = bn.finalize_only(d["expert_out"], d["perm"], d["w"], d["shared"])
    torch.cuda.synchronize()
    ref = parity.run_oracle(d)
    assert_bits_equal(inputs.u16(z), ref["z"], "z")


# ---- the finalize with a workspace: token rows spread over many CTAs ----------------

WIDE = [
    # (R, T, k, H, with_shared)
    (8, 1, 10, 8192, True),
    (8, 4, 10, 8192, True),
    (8, 8, 10, 8192, False),       # the largest T the path serves
    (8, 5, 8, 6144, True),         # 768 chunks: ragged epilogue slices
    (2, 7, 3, 1000, True),         # 125 chunks: one CTA per row, ragged warps
    (16, 3, 16, 4096, True),       # R*k = 256; 16 z rows in two batches
    (1, 5, 1, 64, False),          # one shard, one slot
    (3, 8, 5, 8192, True),         # tasks of a CTA span two shards
    (5, 2, 7, 2048, True),         # 1280 tasks: the third CTA of a row half busy
]


def _counters_zero(ws, T):
    return int(ws[: ((T * 4 + 255) // 256) * 256].count_nonzero().item()) == 0


@pytest.mark.parametrize("R,T,k,H,with_shared", WIDE)
def test_wide_finalize_matches_oracle(R, T, k, H, with_shared):
    wl = inputs.custom("finalize_reduce_norm", R, H, k, partial_std=0.3, shared_std=0.3)
    d = parity.gpu_inputs(wl, T, seed=3000 + R * 13 + T, with_shared=with_shared)
    ws = bn.finalize_workspace(R, T, k, H, device="cuda")
    assert ws is not None and ws.numel() == bn.finalize_workspace_bytes(R, T, k, H)
    g = parity.run_fused(d, workspace=ws)
    parity.compare(g, parity.run_oracle(d), what=f"wide finalize R={R} T={T} k={k} H={H}")
    # the per-shard rounding and the rank-ordered sum are those of the
    # one-CTA-per-row path, bit for bit
    base = parity.run_fused(d)
    assert_bits_equal(g["z"], base["z"], "z")
    assert_bits_equal(g["sum"], base["sum"], "sum")
    torch.cuda.synchronize()
    assert _counters_zero(ws, T)
    # the same workspace serves the next call unchanged
    g2 = parity.run_fused(d, workspace=ws)
    for key in ("sum", "ss", "z", "out", "residual_out"):
        assert_bits_equal(g2[key], g[key], key)


def test_wide_single_norm_variant():
    wl = inputs.custom("finalize_reduce_norm", 8, 6144, 8, partial_std=0.3)
    d = parity.gpu_inputs(wl, 7, seed=33)
    ws = bn.finalize_workspace(8, 7, 8, 6144, device="cuda")
    g = parity.run_fused(d, single=True, workspace=ws)
    parity.compare(g, parity.run_oracle(d, single=True), what="wide single norm")
    assert np.all(g["ss"][:, 0] == 0.0)


def test_wide_workspace_too_small_or_unserved_takes_the_plain_path():
    wl = inputs.custom("finalize_reduce_norm", 8, 8192, 10, partial_std=0.3)
    d = parity.gpu_inputs(wl, 4, seed=34)
    need = bn.finalize_workspace_bytes(8, 4, 10, 8192)
    small = torch.full((need - 16,), 7, dtype=torch.uint8, device="cuda")
    g = parity.run_fused(d, workspace=small)
    base = parity.run_fused(d)
    for key in ("sum", "ss", "z", "out", "residual_out"):
        assert_bits_equal(g[key], base[key], key)
    assert int((small != 7).sum().item()) == 0          # not touched
    assert bn.finalize_workspace_bytes(8, 9, 10, 8192) == 0    # above the served T
    assert bn.finalize_workspace_bytes(8, 4, 10, 16384) == 0   # above the served H


def test_wide_perm_out_of_range_sets_the_device_flag():
    wl = inputs.custom("finalize_reduce_norm", 2, 256, 4, partial_std=0.3)
    d = parity.gpu_inputs(wl, 6, seed=9)
    bad = d["perm"].clone()
    bad[1, 2, 3] = 6 * 4 + 5
    bad[0, 0, 0] = -1
    ws = bn.finalize_workspace(2, 6, 4, 256, device="cuda")
    res = d["residual"].clone()
    bn.finalize_reduce_norm(d["expert_out"], bad, d["w"], d["shared"], res, d["gamma_post"],
                            d["gamma_pre"], d["eps"], workspace=ws)
    assert bn.check_device_error(raise_on_error=False) == bn.DEVERR_PERM_RANGE
    assert _counters_zero(ws, 6)
    g = parity.run_fused(d, workspace=ws)
    parity.compare(g, parity.run_oracle(d), what="wide, after the flagged call")


def test_wide_path_in_a_graph_on_a_side_stream():
    wl = inputs.WORKLOADS[4]
    d = parity.gpu_inputs(wl, 4)
    ws = bn.finalize_workspace(8, 4, 10, 8192, device="cuda")
    res = d["residual"].clone()
    out = torch.empty_like(res)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=s):
            for _ in range(3):  # three dependent calls on one workspace
                bn.finalize_reduce_norm(d["expert_out"], d["perm"], d["w"], d["shared"], res,
                                        d["gamma_post"], d["gamma_pre"], d["eps"], out=out,
                                        workspace=ws)
    res.copy_(d["residual"])
    graph.replay()
    torch.cuda.synchronize()
    # three calls chained through the residual: the same as three plain calls
    res2 = d["residual"].clone()
    out2 = torch.empty_like(res2)
    for _ in range(3):
        bn.finalize_reduce_norm(d["expert_out"], d["perm"], d["w"], d["shared"], res2,
                                d["gamma_post"], d["gamma_pre"], d["eps"], out=out2)
    torch.cuda.synchronize()
    assert_bits_equal(inputs.u16(res), inputs.u16(res2), "residual after 3 calls")
    assert_bits_equal(inputs.u16(out), inputs.u16(out2), "out after 3 calls")
    assert _counters_zero(ws, 4)


def test_decline_then_fallback_gives_the_same_bits():
    """When the fused op declines, a caller that materialises the finalize and
    then reduces and normalises gets exactly the fused result: nothing owed is
    dropped on the fallback path."""
    wl = inputs.WORKLOADS[4]
    d = parity.gpu_inputs(wl, 8)
    fused = parity.run_fused(d)
    z = bn.finalize_only(d["expert_out"], d["perm"], d["w"], d["shared"])
    res = d["residual"].clone()
    out = bn.reduce_norm(z, res, d["gamma_post"], d["gamma_pre"], d["eps"])
    torch.cuda.synchronize()
    assert_bits_equal(inputs.u16(res), fused["residual_out"], "residual_out")
    assert_bits_equal(inputs.u16(out), fused["out"], "out")


DECLINED = [
    # (op, R, T, k, H, with_shared, single): shapes the fused entry points decline
    ("finalize_reduce_norm", 2, 3, 2, 40960, True, False),
    ("finalize_reduce_norm", 3, 2, 4, 65536, False, True),
    ("reduce_norm", 4, 5, 0, 40960, False, False),
    ("reduce_norm", 2, 3, 0, 131072, False, True),
    ("finalize_reduce_norm", 1, 2, 1, 131072, True, False),
]


@pytest.mark.parametrize("op,R,T,k,H,with_shared,single", DECLINED)
def test_declined_shape_falls_back_to_the_unfused_pieces(op, R, T, k, H, with_shared, single):
    """A fused call declines a row it does not serve: it enqueues nothing, so
    the reduction is still owed.  The caller's fallback (the binding's
    on_decline="fallback") materialises the finalize, sums the shards and runs
    the epilogue on the FP32 sum, with the oracle's results."""
    assert not bn.supports(R, T, k, H)
    pieces = (["finalize_only"] if k else []) + ["reduce_only"] + \
        ["residual_norm_only" if single else "norm_only"]
    for piece in pieces:
        assert bn.supports_op(piece, R, T, H, k), piece
    wl = inputs.custom(op, R, H, k, partial_std=0.3, shared_std=0.3)
    d = parity.gpu_inputs(wl, T, seed=700 + R + T, with_shared=with_shared)
    with pytest.raises(bn.BeamNormError) as e:
        parity.run_fused(d, single=single)
    assert e.value.status == bn.ERR_UNSUPPORTED
    g = parity.run_fused(d, single=single, on_decline="fallback")
    ref = parity.run_oracle(d, single=single)
    parity.compare(g, ref, what=f"fallback {op} R={R} T={T} k={k} H={H}")
    assert bn.check_device_error() == 0


# ---- launch shapes, streams, graphs ------------------------------------------------------

@pytest.mark.parametrize("cluster,stages,threads,ctas,wait,group", [
    (1, 0, 0, 0, 0, 0), (2, 0, 0, 0, 0, 1), (4, 3, 0, 0, 2, 0), (8, 0, 0, 0, 0, 7),
    (16, 2, 0, 0, 2, 0), (1, 2, 0, 0, 1, 1), (1, 7, 0, 0, 2, 3), (1, 0, 256, 0, 0, 11),
    (1, 0, 128, 0, 2, 0), (2, 5, 64, 0, 0, 64), (1, 0, 128, 3, 0, 2), (1, 4, 64, 4, 2, 5),
])
def test_launch_shapes_give_identical_bits(cluster, stages, threads, ctas, wait, group):
    wl = inputs.custom("finalize_reduce_norm", 8, 8192, 10, partial_std=0.3)
    d = parity.gpu_inputs(wl, 21, seed=77)
    try:
        bn.set_tuning(cluster, stages, threads, ctas, wait, group)
        g = parity.run_fused(d)
    finally:
        bn.set_tuning()
    base = parity.run_fused(d)
    for key in ("sum", "ss", "z", "out", "residual_out"):
        assert_bits_equal(g[key], base[key], key)
    parity.compare(g, parity.run_oracle(d), what=f"cluster={cluster} stages={stages} ctas={ctas} group={group}")


@pytest.mark.gpu
@pytest.mark.parametrize("op,R,T,k,H", [
    ("reduce_norm", 4, 1024, 0, 5120), ("reduce_norm", 8, 1, 0, 8192),
    ("finalize_reduce_norm", 8, 1, 10, 8192), ("finalize_reduce_norm", 8, 1024, 10, 8192),
    ("norm_only", 1, 64, 0, 8192), ("finalize_only", 8, 4, 8, 6144),
    ("reduce_residual_norm", 2, 8, 0, 256),
])
def test_launch_query_is_coherent(op, R, T, k, H):
    props = torch.cuda.get_device_properties(0)
    i = bn.launch_info(op, R, T, H, k)
    assert i["threads"] % 32 == 0 and 64 <= i["threads"] <= 512 + 32
    assert i["grid"] > 0 and i["grid"] % i["cluster_size"] == 0
    assert i["grid"] // i["cluster_size"] <= T
    if i["split"] == 2:
        # one cluster per row, one (shard, chunk) task per thread: no pipeline
        assert op in ("reduce_norm", "reduce_residual_norm", "finalize_reduce_norm",
                      "finalize_reduce_residual_norm") and i["grid"] == T * i["cluster_size"]
        assert i["chunks_per_thread"] in (1, 2) and i["stages"] == 0
    else:
        assert i["stages"] >= 2 and i["stage_bytes"] % 128 == 0 and i["group"] >= 1
    assert i["resident_ctas"] >= i["grid"]
    assert i["smem_bytes"] <= props.shared_memory_per_block_optin
    if i["split"] == 1:
        assert op.startswith("finalize") and R % i["cluster_size"] == 0
    try:
        bn.set_tuning(stages=2, split=1)
        j = bn.launch_info(op, R, T, H, k)
    finally:
        bn.set_tuning()
    assert j["stages"] == 2 and j["split"] == 0


@pytest.mark.gpu
def test_reduce_planner_balances_rows_per_sm():
    """One CTA per reduce row: the planner takes 512-thread CTAs for heavy rows
    (R=8, H=8192 at T=1024 and 4096) when an SM then runs at least as many
    consumer threads and takes no more rows, with a gain in one; keeps the
    default where both tie (T=256), where the wide CTA runs fewer threads
    (R=4, H=5120) or would hold one chunk per thread (H=4096); gives light
    rows (R <= 4) 128-thread CTAs with up to 4 chunks each; and sizes the
    ring for the CTAs that actually share an SM when rows are fewer than CTA
    slots."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms != 152:
        pytest.skip("expected shapes are those of a 152-SM GB300")
    for T in (1024, 4096):
        i = bn.launch_info("reduce_norm", 8, T, 8192)
        assert (i["threads"], i["chunks_per_thread"], i["cluster_size"]) == (544, 2, 1)
    i = bn.launch_info("reduce_norm", 8, 256, 8192)
    assert (i["threads"], i["chunks_per_thread"]) == (288, 4)
    # rows wider than 1536 chunks split over a cluster (R=8, H=16384: two CTAs)
    i = bn.launch_info("reduce_norm", 8, 1024, 16384)
    assert (i["threads"], i["chunks_per_thread"], i["cluster_size"]) == (288, 4, 2)
    i = bn.launch_info("reduce_norm", 4, 1024, 12288)
    assert (i["threads"], i["chunks_per_thread"], i["cluster_size"]) == (416, 4, 1)
    i = bn.launch_info("finalize_reduce_norm", 8, 256, 16384, 8)
    assert (i["chunks_per_thread"], i["cluster_size"]) == (2, 2)
    i = bn.launch_info("reduce_norm", 8, 1024, 4096)
    assert (i["threads"], i["chunks_per_thread"]) == (288, 2)
    for T in (1024, 4096):
        i = bn.launch_info("reduce_norm", 4, T, 5120)
        assert (i["threads"], i["chunks_per_thread"], i["resident_ctas"]) == (192, 4, 3 * sms)
    i = bn.launch_info("reduce_norm", 4, 256, 5120)
    assert i["threads"] == 192 and i["resident_ctas"] == 2 * sms and i["grid"] == 256
    # light rows (R <= 4) with more rows than SMs: 128 consumer threads, up to
    # 4 chunks each, up to 4 CTAs per SM; the wider CTA only for heavy rows
    for R, H, want in ((2, 2048, (160, 2)), (4, 4096, (160, 4)), (2, 7168, (256, 4)),
                       (4, 8192, (288, 4))):
        i = bn.launch_info("reduce_norm", R, 4096, H)
        assert (i["threads"], i["chunks_per_thread"], i["cluster_size"]) == (*want, 1), (R, H, i)
    i = bn.launch_info("reduce_norm", 8, 4096, 7168)
    assert (i["threads"], i["chunks_per_thread"]) == (256, 4)
    i = bn.launch_info("reduce_norm", 8, 4096, 2048)
    assert (i["threads"], i["chunks_per_thread"]) == (160, 2)
    # a row with an SM to itself keeps the wider CTA
    i = bn.launch_info("reduce_norm", 4, 64, 5120)
    assert (i["threads"], i["chunks_per_thread"]) == (352, 2)


@pytest.mark.gpu
def test_finalize_planner_shares_sms_between_narrow_rows():
    """Narrow finalize rows take two chunks a thread and several CTAs per SM,
    with the stage bytes split between those CTAs; rows of 1024 chunks and
    more keep one 512-thread CTA per SM (the headline shape)."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms != 152:
        pytest.skip("expected shapes are those of a 152-SM GB300")
    expect = {  # H: (threads, chunks per thread, CTAs per SM)
        1024: (160, 1, 4), 2048: (160, 2, 4), 3072: (224, 2, 2), 4096: (288, 2, 2),
        8192: (544, 2, 1),
    }
    for H, (threads, cpt, per_sm) in expect.items():
        i = bn.launch_info("finalize_reduce_norm", 8, 1024, H, 8)
        got = (i["threads"], i["chunks_per_thread"], i["grid"] // sms)
        assert got == (threads, cpt, per_sm), (H, got)
        assert i["split"] == 0 and i["cluster_size"] == 1
        # about 48 KB of stages per SM, split between its CTAs (copies of 2H bytes)
        per_cta = 48 * 1024 // per_sm
        assert i["stage_bytes"] == max(1, per_cta // (2 * H)) * 2 * H, (H, i["stage_bytes"])


NARROW_FIN = [
    # (R, T, k, H): two chunks a thread, several CTAs per SM; ragged slices too
    (8, 300, 8, 2048), (8, 200, 8, 3072), (4, 333, 8, 4096), (8, 160, 2, 4096),
    (8, 157, 8, 2056), (3, 170, 5, 3000),
]


@pytest.mark.gpu
@pytest.mark.parametrize("single", [False, True])
@pytest.mark.parametrize("R,T,k,H", NARROW_FIN)
def test_narrow_finalize_rows_match_oracle(R, T, k, H, single):
    wl = inputs.custom("finalize_reduce_norm", R, H, k, partial_std=0.3, shared_std=0.3)
    d = parity.gpu_inputs(wl, T, seed=3000 + R * 13 + T + H)
    g = parity.run_fused(d, single=single)
    parity.compare(g, parity.run_oracle(d, single=single), what=f"narrow finalize R={R} T={T} k={k} H={H}")


@pytest.mark.gpu
@pytest.mark.parametrize("op,R,T,k,H", [
    ("reduce_norm", 2, 200_000, 0, 64),            # about 1300 rows per CTA
    ("finalize_reduce_norm", 2, 100_000, 2, 64),   # T * k = 200000 gathered rows per shard
    ("reduce_norm", 3, 50_000, 0, 1000),           # ragged rows, several hundred per CTA
])
def test_many_token_rows_match_oracle(op, R, T, k, H):
    """Long grid-stride loops: every CTA of the persistent grid walks hundreds
    of rows, and the finalize's gather indices reach 200000 rows per shard."""
    wl = inputs.custom(op, R, H, k, partial_std=0.5, shared_std=0.3)
    d = parity.gpu_inputs(wl, T, seed=3200 + R + T)
    g = parity.run_fused(d)
    parity.compare(g, parity.run_oracle(d), what=f"{op} R={R} T={T} H={H}")


LIGHT_REDUCE = [
    # (R, T, H): light rows with more rows than SMs take 128-thread CTAs with up
    # to 4 chunks each; ragged widths leave the last thread's chunks short
    (2, 300, 2048), (4, 333, 4096), (2, 200, 7168), (3, 400, 2056), (4, 170, 3000),
    (1, 257, 8192),
]


@pytest.mark.gpu
@pytest.mark.parametrize("single", [False, True])
@pytest.mark.parametrize("R,T,H", LIGHT_REDUCE)
def test_light_reduce_rows_match_oracle(R, T, H, single):
    wl = inputs.custom("reduce_norm", R, H, partial_std=0.5, row_scale=True)
    d = parity.gpu_inputs(wl, T, seed=3100 + R * 17 + T + H)
    g = parity.run_fused(d, single=single)
    parity.compare(g, parity.run_oracle(d, single=single), what=f"light reduce R={R} T={T} H={H}")


@pytest.mark.gpu
def test_every_piece_has_a_launch_up_to_its_maximum():
    """The unfused pieces serve rows the fused entry points decline: the
    planner finds a launch (clusters of up to 16 CTAs) wherever
    bn_supports_op accepts the shape."""
    for H in (32776, 40960, 65536, 98304, 131072):
        for R, k in ((1, 1), (8, 10), (16, 16)):
            for T in (1, 7, 300, 5000):
                for op in ("reduce_only", "norm_only", "residual_norm_only"):
                    assert bn.supports_op(op, R, T, H)
                    bn.launch_info(op, R, T, H)
                for op in ("finalize_reduce_only", "finalize_only"):
                    assert bn.supports_op(op, R, T, H, k)
                    bn.launch_info(op, R, T, H, k)
                    bn.launch_info(op, R, T, H, k, has_shared=False)


@pytest.mark.gpu
def test_every_supported_shape_has_a_launch():
    """bn_supports promises a launch for every valid shape it accepts: the
    planner finds one (widening the row split where one CTA's shared memory
    cannot hold a slice) for the extremes of R, k, T and H."""
    for H in (8, 256, 5120, 8192, 16384, 24576, 32768):
        for R, k in ((1, 1), (2, 2), (8, 10), (16, 16)):
            for T in (1, 17, 300, 5000):
                assert bn.load().bn_supports(R, T, k, H) == 1
                for op in ("reduce_norm", "reduce_residual_norm", "reduce_only", "norm_only"):
                    bn.launch_info(op, R, T, H)
                for op in ("finalize_reduce_norm", "finalize_reduce_residual_norm",
                           "finalize_reduce_only", "finalize_only"):
                    bn.launch_info(op, R, T, H, k)
                    bn.launch_info(op, R, T, H, k, has_shared=False)


SPLIT_CASES = [
    # (R, T, k, H, with_shared, single_norm)
    (8, 1, 10, 8192, True, False),
    (8, 3, 8, 6144, False, False),
    (3, 5, 4, 1000, True, True),
    (2, 7, 3, 256, True, False),
    (16, 2, 16, 4096, True, False),
    (4, 40, 6, 2048, True, False),   # more rows than one pass of clusters
    (6, 9, 5, 1536, True, False),    # cluster sizes 2, 3 and 6
    (12, 2, 3, 768, True, False),    # cluster sizes 2, 3, 4, 6 and 12
]


@pytest.mark.parametrize("R,T,k,H,with_shared,single", SPLIT_CASES)
def test_shard_split_matches_column_split_and_oracle(R, T, k, H, with_shared, single):
    """A cluster that splits a row by shard (each of its cs CTAs finalizes R/cs
    shards over the whole row and sends every chunk of each z row to the CTA
    owning that column slice, where the R rows are summed in rank order)
    gives the bits of the column split, for every cluster size dividing R."""
    wl = inputs.custom("finalize_reduce_norm", R, H, k, partial_std=0.3, shared_std=0.3)
    d = parity.gpu_inputs(wl, T, seed=500 + R * 13 + T, with_shared=with_shared)
    sizes = [c for c in range(2, R + 1) if R % c == 0]
    runs = {}
    try:
        bn.set_tuning(split=1)
        base = parity.run_fused(d, single=single)
        for c in sizes:
            bn.set_tuning(cluster_size=c, split=2)
            info = bn.launch_info("finalize_reduce_residual_norm" if single else "finalize_reduce_norm",
                                  R, T, H, k, has_shared=with_shared)
            assert info["split"] == 1 and info["cluster_size"] == c, info
            runs[info["cluster_size"]] = parity.run_fused(d, single=single)
    finally:
        bn.set_tuning()
    for c, g in runs.items():
        for key in ("sum", "ss", "z", "out", "residual_out"):
            assert_bits_equal(g[key], base[key], f"cs={c} {key}")
    parity.compare(base, parity.run_oracle(d, single=single), what=f"split R={R} T={T} k={k} H={H}")


CLUSTER_TASKS = [
    # (R, T, k, H, with_shared, single, cluster size)
    (8, 1, 10, 8192, True, False, 16),
    (8, 4, 10, 8192, True, False, 16),
    (8, 8, 10, 8192, False, False, 8),
    (8, 3, 8, 6144, True, True, 16),
    (2, 7, 3, 1000, True, False, 4),      # 125 chunks: slices of 31 and 32 chunks
    (16, 3, 16, 4096, True, False, 8),    # R*k = 256, two tasks per thread
    (1, 5, 1, 64, False, False, 2),
    (3, 40, 5, 2048, True, True, 16),     # more rows than resident clusters
]


@pytest.mark.parametrize("R,T,k,H,with_shared,single,cs", CLUSTER_TASKS)
def test_cluster_task_split_matches_oracle(R, T, k, H, with_shared, single, cs):
    """A cluster of cs CTAs per row, one (shard, chunk) finalize task per
    thread, each CTA's finalize results summed and normalised on its column
    slice, the sums of squares exchanged across the cluster: the bits of the
    other row splits and the oracle's results."""
    wl = inputs.custom("finalize_reduce_norm", R, H, k, partial_std=0.3, shared_std=0.3)
    d = parity.gpu_inputs(wl, T, seed=800 + R * 13 + T, with_shared=with_shared)
    op = "finalize_reduce_residual_norm" if single else "finalize_reduce_norm"
    try:
        bn.set_tuning(split=3, cluster_size=cs)
        info = bn.launch_info(op, R, T, H, k, has_shared=with_shared)
        assert info["split"] == 2 and info["cluster_size"] == cs, info
        assert info["grid"] == T * cs
        g = parity.run_fused(d, single=single)
    finally:
        bn.set_tuning()
    base = parity.run_fused(d, single=single)
    for key in ("sum", "z"):
        assert_bits_equal(g[key], base[key], key)
    parity.compare(g, parity.run_oracle(d, single=single), what=f"cluster tasks R={R} T={T} H={H}")


@pytest.mark.parametrize("k", [1, 3, 4, 5, 7, 8, 9, 10, 11, 15, 16])
def test_cluster_task_unroll_widths_match_oracle(k):
    """The cluster path's finalize tasks are compiled for 4, 8, 10 and 16
    expert slots, and a call takes the smallest that holds k: every k at and
    on either side of those widths gives the finalize and sum bits of the
    forced column split, and the oracle's results."""
    R, T, H = 4, 3, 2048
    wl = inputs.custom("finalize_reduce_norm", R, H, k, partial_std=0.3, shared_std=0.3)
    d = parity.gpu_inputs(wl, T, seed=1200 + k, with_shared=True)
    try:
        bn.set_tuning(split=3, cluster_size=4)
        assert bn.launch_info("finalize_reduce_norm", R, T, H, k)["split"] == 2
        g = parity.run_fused(d)
        bn.set_tuning(split=1)
        base = parity.run_fused(d)
    finally:
        bn.set_tuning()
    for key in ("sum", "z"):  # the row reductions' trees differ between the splits
        assert_bits_equal(g[key], base[key], f"k={k} {key}")
    parity.compare(g, parity.run_oracle(d), what=f"cluster tasks k={k}")


@pytest.mark.parametrize("R,T,k,H,cs", [
    (8, 16, 8, 2048, 4), (8, 32, 8, 2048, 4), (8, 64, 8, 2048, 2), (4, 32, 8, 4096, 4),
    (2, 32, 8, 7168, 4), (8, 16, 10, 8192, 0), (8, 64, 8, 4096, 0), (8, 16, 8, 6144, 0),
    (2, 37, 8, 7168, 2),   # 37 clusters of 4 are more than the device holds at once
])
def test_narrow_finalize_rows_keep_the_cluster_path_past_15_rows(R, T, k, H, cs):
    """Past 15 token rows the finalize keeps the cluster path for narrow rows
    (clusters of at most 4 CTAs, at most two tasks a thread, all T * cs CTAs on
    distinct SMs); wider rows go to the main kernel (cs = 0 here).  The
    cluster path's bits equal the forced column split's, and the oracle's."""
    sms = torch.cuda.get_device_properties(0).multi_processor_count
    if sms != 152:
        pytest.skip("expected shapes are those of a 152-SM GB300")
    info = bn.launch_info("finalize_reduce_norm", R, T, H, k)
    if cs:
        assert info["split"] == 2 and info["cluster_size"] == cs and info["grid"] == T * cs, info
    else:
        assert info["split"] != 2, info
    wl = inputs.custom("finalize_reduce_norm", R, H, k, partial_std=0.3, shared_std=0.3)
    d = parity.gpu_inputs(wl, T, seed=860 + R * 7 + T + H)
    g = parity.run_fused(d)
    try:
        bn.set_tuning(split=1)
        base = parity.run_fused(d)
    finally:
        bn.set_tuning()
    for key in ("sum", "z"):
        assert_bits_equal(g[key], base[key], key)
    parity.compare(g, parity.run_oracle(d), what=f"mid-T finalize R={R} T={T} k={k} H={H}")


CLUSTER_REDUCE = [
    # (R, T, H, single, cluster size)
    (4, 1, 5120, False, 16),
    (8, 3, 8192, True, 16),
    (16, 2, 8192, False, 16),     # two tasks per thread
    (3, 5, 1000, False, 4),       # ragged slices
    (1, 4, 64, True, 2),
    (8, 30, 4096, False, 8),      # more rows than resident clusters
]


@pytest.mark.parametrize("R,T,H,single,cs", CLUSTER_REDUCE)
def test_cluster_split_of_reduce_rows_matches_oracle(R, T, H, single, cs):
    """The reduce entry points on the cluster path: each task loads one
    shard's partial chunk into the slice's shared rows; the rank-ordered sum,
    the norms and the exchanges are those of the finalize flavour."""
    wl = inputs.custom("reduce_norm", R, H, partial_std=0.5, row_scale=True)
    d = parity.gpu_inputs(wl, T, seed=850 + R * 7 + T)
    op = "reduce_residual_norm" if single else "reduce_norm"
    try:
        bn.set_tuning(split=3, cluster_size=cs)
        info = bn.launch_info(op, R, T, H)
        assert info["split"] == 2 and info["cluster_size"] == cs and info["grid"] == T * cs, info
        g = parity.run_fused(d, single=single)
    finally:
        bn.set_tuning()
    base = parity.run_fused(d, single=single)
    assert_bits_equal(g["sum"], base["sum"], "sum")
    parity.compare(g, parity.run_oracle(d, single=single), what=f"cluster reduce R={R} T={T} H={H}")


@pytest.mark.parametrize("R,T,H", [(8, 9, 8192), (8, 16, 8192), (8, 32, 8192), (4, 24, 5120),
                                   (8, 20, 4096), (2, 16, 8192), (8, 33, 8192), (16, 34, 4096)])
def test_reduce_rows_keep_the_cluster_path_to_32_rows(R, T, H):
    """Past 8 token rows the planner keeps heavy reduce rows on the cluster
    path, with clusters of at most 8 CTAs all resident at once (from 33 to 36
    rows, clusters of 8 only, for rows of 8 or more shards): the forced column
    split's sum bits and the oracle's results."""
    wl = inputs.custom("reduce_norm", R, H, partial_std=0.5, row_scale=True)
    d = parity.gpu_inputs(wl, T, seed=870 + R * 7 + T + H)
    info = bn.launch_info("reduce_norm", R, T, H)
    assert info["split"] == 2 and info["cluster_size"] <= 8, info
    if T > 32:
        assert info["cluster_size"] == 8, info
    assert info["resident_ctas"] >= info["grid"] == T * info["cluster_size"], info
    g = parity.run_fused(d)
    try:
        bn.set_tuning(split=1)
        base = parity.run_fused(d)
    finally:
        bn.set_tuning()
    assert_bits_equal(g["sum"], base["sum"], "sum")
    parity.compare(g, parity.run_oracle(d), what=f"cluster reduce R={R} T={T} H={H}")
    # past 32 rows only clusters of 8, all resident, for 8 or more shards
    i33 = bn.launch_info("reduce_norm", R, 33, H)
    assert i33["split"] != 2 or (R >= 8 and i33["cluster_size"] == 8 and
                                 i33["resident_ctas"] >= i33["grid"]), i33
    # and past 36 rows the main kernel again
    assert bn.launch_info("reduce_norm", R, 37, H)["split"] != 2


@pytest.mark.parametrize("T", [1, 4, 12])
def test_light_reduce_rows_take_clusters_of_8_to_12_rows(T):
    """Rows of two shards of 5120 (640 chunks) take clusters of 8 CTAs at 160
    tasks a CTA up to 12 token rows, and clusters of 4 past them: the forced
    column split's sum bits and the oracle's results."""
    R, H = 2, 5120
    wl = inputs.custom("reduce_norm", R, H, partial_std=0.5, row_scale=True)
    d = parity.gpu_inputs(wl, T, seed=910 + T)
    info = bn.launch_info("reduce_norm", R, T, H)
    assert info["split"] == 2 and info["cluster_size"] == 8 and info["grid"] == 8 * T, info
    g = parity.run_fused(d)
    try:
        bn.set_tuning(split=1)
        base = parity.run_fused(d)
    finally:
        bn.set_tuning()
    assert_bits_equal(g["sum"], base["sum"], "sum")
    parity.compare(g, parity.run_oracle(d), what=f"light cluster reduce R={R} T={T} H={H}")
    assert bn.launch_info("reduce_norm", R, 13, H)["cluster_size"] == 4


def test_cluster_task_split_flags_bad_perm_and_stays_in_bounds():
    R, T, k, H = 4, 5, 3, 1000
    wl = inputs.custom("finalize_reduce_norm", R, H, k, partial_std=0.3)
    d = parity.gpu_inputs(wl, T, seed=5)
    bad = d["perm"].clone()
    bad[1, 2, 0] = T * k + 3
    ob, out, og = parity.guarded(T * H, torch.bfloat16)
    sb, s, sg = parity.guarded(T * H, torch.float32)
    qb, ss, qg = parity.guarded(T * 2, torch.float32)
    zb, z, zg = parity.guarded(R * T * H, torch.bfloat16)
    rb, res, rg = parity.guarded(T * H, torch.bfloat16)
    res.copy_(d["residual"].reshape(-1))
    try:
        bn.set_tuning(split=3, cluster_size=8)
        bn.finalize_reduce_norm(d["expert_out"], bad, d["w"], d["shared"], res.view(T, H),
                                d["gamma_post"], d["gamma_pre"], d["eps"], out=out.view(T, H),
                                debug=bn.Debug(sum=s.view(T, H), ss=ss.view(T, 2), z=z.view(R, T, H)))
        assert bn.check_device_error(raise_on_error=False) == bn.DEVERR_PERM_RANGE
    finally:
        bn.set_tuning()
    for buf, gd, n in ((ob, og, T * H), (sb, sg, T * H), (qb, qg, T * 2), (zb, zg, R * T * H),
                       (rb, rg, T * H)):
        assert parity.guard_intact(buf, gd, n)
    assert not torch.isnan(out.float()).any() and not torch.isnan(s).any()
    assert not torch.isnan(z.float()).any() and not torch.isnan(ss).any()


@pytest.mark.parametrize("cs", [8, 4, 2])
def test_shard_split_finalize_only(cs):
    wl = inputs.WORKLOADS[4]
    d = parity.gpu_inputs(wl, 4)
    try:
        bn.set_tuning(cluster_size=cs, split=2)
        assert bn.launch_info("finalize_only", wl.R, 4, wl.H, wl.k)["cluster_size"] == cs
        z = bn.finalize_only(d["expert_out"], d["perm"], d["w"], d["shared"])
        torch.cuda.synchronize()
    finally:
        bn.set_tuning()
    assert bn.check_device_error() == 0
    assert_bits_equal(inputs.u16(z), parity.run_oracle(d)["z"], "z")


def test_reduce_launch_shapes_give_identical_bits():
    wl = inputs.custom("reduce_norm", 8, 5120, row_scale=True)
    d = parity.gpu_inputs(wl, 45, seed=78)
    base = parity.run_fused(d)
    for cluster, threads, ctas, group in ((2, 0, 0, 0), (4, 0, 0, 3), (16, 0, 0, 9), (1, 512, 1, 1),
                                          (1, 64, 4, 2)):
        try:
            bn.set_tuning(cluster, 0, threads, ctas, 0, group)
            g = parity.run_fused(d)
        finally:
            bn.set_tuning()
        for key in ("sum", "ss", "out", "residual_out"):
            assert_bits_equal(g[key], base[key], f"cluster={cluster} threads={threads} {key}")


def test_side_stream_and_graph_replay():
    wl = inputs.WORKLOADS[3]
    d = parity.gpu_inputs(wl, 64)
    eager = parity.run_fused(d, debug=False)
    s = torch.cuda.Stream()
    res = d["residual"].clone()
    res0 = res.clone()
    out = torch.empty_like(res)
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        bn.finalize_reduce_norm(d["expert_out"], d["perm"], d["w"], d["shared"], res,
                                d["gamma_post"], d["gamma_pre"], d["eps"], out=out)
    s.synchronize()
    assert_bits_equal(inputs.u16(out), eager["out"], "side stream out")
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        bn.finalize_reduce_norm(d["expert_out"], d["perm"], d["w"], d["shared"], res,
                                d["gamma_post"], d["gamma_pre"], d["eps"], out=out)
    res.copy_(res0)
    out.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert_bits_equal(inputs.u16(out), eager["out"], "graph out")
    assert_bits_equal(inputs.u16(res), eager["residual_out"], "graph residual")


def _dependent_chain(d, use_graph: bool):
    """Five back-to-back calls where each reads what the previous one wrote:
    the unfused pair (finalize_reduce_only writes the FP32 sum that norm_only
    reads), then fused calls whose residual is the previous call's output."""
    T, H = d["T"], d["H"]
    s = torch.empty(T, H, dtype=torch.float32, device="cuda")
    res = d["residual"].clone()
    outs = [torch.empty_like(res) for _ in range(3)]

    def body():
        bn.finalize_reduce_only(d["expert_out"], d["perm"], d["w"], d["shared"], sum_out=s)
        bn.norm_only(s, res, d["gamma_post"], d["gamma_pre"], d["eps"], out=outs[0])
        for i in (1, 2):
            bn.finalize_reduce_norm(d["expert_out"], d["perm"], d["w"], d["shared"], outs[i - 1],
                                    d["gamma_post"], d["gamma_pre"], d["eps"], out=outs[i])

    if use_graph:
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            body()
        s.fill_(float("nan"))
        res.copy_(d["residual"])
        for o in outs:
            o.fill_(float("nan"))
        g.replay()
    else:
        body()
    torch.cuda.synchronize()
    return [inputs.u16(t) for t in (res, *outs)] + [s.cpu().numpy()]


@pytest.mark.parametrize("wl_index,T", [(4, 4), (3, 16), (4, 64)])
def test_dependent_launch_keeps_stream_order(wl_index, T):
    d = parity.gpu_inputs(inputs.WORKLOADS[wl_index], T)
    runs = {}
    try:
        bn.set_tuning(dependent_launch=1)
        plain = _dependent_chain(d, use_graph=False)
        bn.set_tuning(dependent_launch=2)
        runs["eager"] = _dependent_chain(d, use_graph=False)
        runs["in a graph"] = _dependent_chain(d, use_graph=True)
    finally:
        bn.set_tuning()
    names = ("residual", "out0", "out1", "out2", "sum")
    for what, got in runs.items():
        for a, b, n in zip(plain, got, names):
            assert_bits_equal(b, a, f"programmatic launch, {what}: {n}")
    # the unfused pair's results (out0 is overwritten in place by the next call)
    ref = parity.run_oracle(d)
    assert_bits_equal(plain[4], ref["sum"], "unfused pair sum")
    assert_bf16_close(plain[0], ref["residual_out"], parity.MAX_ULP, "unfused pair residual")


def test_two_calls_update_the_residual_twice():
    wl = inputs.WORKLOADS[1]
    d = parity.gpu_inputs(wl, 8)
    res = d["residual"].clone()
    bn.reduce_norm(d["partials"], res, d["gamma_post"], d["gamma_pre"], d["eps"])
    out2 = bn.reduce_norm(d["partials"], res, d["gamma_post"], d["gamma_pre"], d["eps"])
    torch.cuda.synchronize()
    h = inputs.to_numpy(d)
    r1 = oracle.reduce_norm(h["partials"], h["residual"], h["gamma_post"], h["gamma_pre"], h["eps"])
    r2 = oracle.reduce_norm(h["partials"], r1["residual_out"], h["gamma_post"], h["gamma_pre"],
                            h["eps"])
    parity.compare({"out": inputs.u16(out2), "residual_out": inputs.u16(res)}, r2, what="second call")


# ---- memory safety substitutes (guard bands, NaN prefill) --------------------------------

_guarded = parity.guarded
_guard_intact = parity.guard_intact


@pytest.mark.parametrize("cluster", [1, 16])
def test_outputs_stay_inside_their_buffers(cluster):
    wl = inputs.custom("finalize_reduce_norm", 4, 1000, 3, partial_std=0.3)
    R, T, k, H = 4, 9, 3, 1000
    d = parity.gpu_inputs(wl, T, seed=5)
    ob, out, og = _guarded(T * H, torch.bfloat16)
    sb, s, sg = _guarded(T * H, torch.float32)
    qb, ss, qg = _guarded(T * 2, torch.float32)
    zb, z, zg = _guarded(R * T * H, torch.bfloat16)
    rb, res, rg = _guarded(T * H, torch.bfloat16)
    res.copy_(d["residual"].reshape(-1))
    try:
        bn.set_tuning(cluster)
        bn.finalize_reduce_norm(d["expert_out"], d["perm"], d["w"], d["shared"], res.view(T, H),
                                d["gamma_post"], d["gamma_pre"], d["eps"], out=out.view(T, H),
                                debug=bn.Debug(sum=s.view(T, H), ss=ss.view(T, 2), z=z.view(R, T, H)))
        torch.cuda.synchronize()
    finally:
        bn.set_tuning()
    for buf, g, n in ((ob, og, T * H), (sb, sg, T * H), (qb, qg, T * 2), (zb, zg, R * T * H),
                      (rb, rg, T * H)):
        assert _guard_intact(buf, g, n)
    # every element written (no NaN left from the prefill)
    assert not torch.isnan(out.float()).any() and not torch.isnan(s).any()
    assert not torch.isnan(ss).any() and not torch.isnan(z.float()).any()


# ---- errors --------------------------------------------------------------------------------

def test_perm_out_of_range_sets_the_device_flag_without_trapping():
    wl = inputs.custom("finalize_reduce_norm", 2, 256, 4, partial_std=0.3)
    d = parity.gpu_inputs(wl, 6, seed=9)
    bad = d["perm"].clone()
    bad[1, 2, 3] = 6 * 4 + 5
    bad[0, 0, 0] = -1
    res = d["residual"].clone()
    bn.finalize_reduce_norm(d["expert_out"], bad, d["w"], d["shared"], res, d["gamma_post"],
                            d["gamma_pre"], d["eps"])
    bits = bn.check_device_error(raise_on_error=False)
    assert bits == bn.DEVERR_PERM_RANGE
    assert bn.check_device_error() == 0          # cleared
    # the context is still usable
    g = parity.run_fused(d)
    parity.compare(g, parity.run_oracle(d), what="after the flagged call")


def test_zero_tokens_and_declined_shapes_touch_nothing():
    R, H = 2, 64
    p = torch.randn(R, 0, H, device="cuda").to(torch.bfloat16)
    res = torch.empty(0, H, dtype=torch.bfloat16, device="cuda")
    g = torch.ones(H, device="cuda")
    out = bn.reduce_norm(p, res, g, g, 1e-6)
    assert out.shape == (0, H)
    # a valid but unserved shape is declined before any work
    Hb = 40960
    pb = torch.zeros(1, 1, Hb, dtype=torch.bfloat16, device="cuda")
    rb = torch.zeros(1, Hb, dtype=torch.bfloat16, device="cuda")
    gb = torch.ones(Hb, device="cuda")
    ob = torch.full((1, Hb), 3.0, device="cuda").to(torch.bfloat16)
    assert not bn.supports(1, 1, 0, Hb)
    with pytest.raises(bn.BeamNormError) as e:
        bn.reduce_norm(pb, rb, gb, gb, 1e-6, out=ob)
    assert e.value.status == bn.ERR_UNSUPPORTED
    torch.cuda.synchronize()
    assert bool((ob.float() == 3.0).all())
