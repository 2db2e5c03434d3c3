"""Pins of the CPU oracle against what the pages and the mathematics fix.

Each test checks the oracle against something other than itself: a hand-worked
example, a closed form, an invariant, a case that reduces to a library routine
(PyTorch's BF16 rounding, numpy float64 / math.fsum), or a brute-force double
recomputation.  The comment on each test names the mistakes it catches.

Sources: "Fuse Beam's TP all-reduce with its sandwich norms" (vLLM pull request
62366), "Claims" and "Details"; sglang pull request 34134, description.
"""
import math

import numpy as np
import pytest
import torch

import oracle
from tests import golden
from tests.helpers import (assert_bf16_close, assert_bits_equal, bf16_bits, bf16_torch,
                           f32_from_bf16)
from tp_reduce_residual_gb300 import inputs


def _rng(seed):
    return np.random.default_rng(seed)


def _bf16_random(shape, std, seed):
    return bf16_torch(_rng(seed).normal(0.0, std, size=shape).astype(np.float32))


def _rmsnorm64(x, gamma, eps):
    x = np.asarray(x, np.float64)
    return x / np.sqrt(np.mean(x * x, axis=-1, keepdims=True) + eps) * np.asarray(gamma, np.float64)


# ---- hand-worked examples ----------------------------------------------------

def test_golden_reduce_norm_handworked():
    """Catches: wrong residual add, swapped gammas, wrong mean or eps placement,
    (1 + gamma) instead of gamma, wrong sign handling of -0."""
    g = golden.load("reduce_norm_handworked.txt")
    R, T, H = int(g["R"]), int(g["T"]), int(g["H"])
    p = bf16_bits(golden.stack(g, "partials", (R, T, H)))
    res = bf16_bits(golden.stack(g, "residual", (T, H)))
    r = oracle.reduce_norm(p, res, g["gamma_post"], g["gamma_pre"], g["eps"])
    assert_bits_equal(r["sum"], golden.stack(g, "expect_sum", (T, H)).astype(np.float32), "sum")
    assert_bits_equal(r["ss"], golden.stack(g, "expect_ss", (T, 2)).astype(np.float32), "ss")
    assert_bits_equal(r["residual_out"], bf16_bits(golden.stack(g, "expect_residual_out", (T, H))),
                      "residual_out")
    assert_bits_equal(r["out"], bf16_bits(golden.stack(g, "expect_out", (T, H))), "out")


def test_golden_finalize_handworked():
    """Catches: no local BF16 rounding of the finalize, truncation instead of
    round-to-nearest-even, scatter instead of gather, weights of the wrong slot."""
    g = golden.load("finalize_handworked.txt")
    R, T, k, H = int(g["R"]), int(g["T"]), int(g["k"]), int(g["H"])
    x = bf16_bits(golden.stack(g, "expert_out", (R, T * k, H)))
    perm = golden.stack(g, "perm", (R, k)).astype(np.int32).reshape(R, T, k)
    w = golden.stack(g, "w", (R, k)).astype(np.float32).reshape(R, T, k)
    sh = bf16_bits(golden.stack(g, "shared", (R, H))).reshape(R, T, H)
    res = bf16_bits(golden.stack(g, "residual", (T, H)))
    r = oracle.finalize_reduce_norm(x, perm, w, sh, res, g["gamma_post"], g["gamma_pre"], g["eps"],
                                    want_z=True)
    assert_bits_equal(r["z"], bf16_bits(golden.stack(g, "expect_z", (R, H))).reshape(R, T, H), "z")
    assert_bits_equal(r["sum"], golden.stack(g, "expect_sum", (T, H)).astype(np.float32), "sum")
    assert_bits_equal(r["ss"], golden.stack(g, "expect_ss", (T, 2)).astype(np.float32), "ss")
    assert_bits_equal(r["residual_out"], bf16_bits(golden.stack(g, "expect_residual_out", (T, H))),
                      "residual_out")
    assert_bits_equal(r["out"], bf16_bits(golden.stack(g, "expect_out", (T, H))), "out")


# ---- the rank-ordered reduction ----------------------------------------------

def test_single_shard_reduction_is_identity():
    """R = 1: the reduced sum is the widened shard bit for bit, -0 included.
    Catches: a reduction that starts from +0 (0 + p0 turns -0 into +0)."""
    p = _bf16_random((1, 5, 64), 1.0, 1)
    p[0, 0, :8] = 0x8000  # -0.0
    r = oracle.reduce_norm(p, None, None, None, 1e-6, want_norm=False)
    assert_bits_equal(r["sum"], f32_from_bf16(p[0]), "sum")
    assert np.all(r["sum"][0, :8].view(np.uint32) == 0x80000000)


@pytest.mark.parametrize("R", [2, 4])
def test_negated_pairs_sum_to_zero(R):
    """Shards [p, -p] (and [p0,-p0,p1,-p1]) sum to +0 exactly; the post-norm then
    adds nothing, the residual comes back unchanged and the output is a textbook
    RMSNorm of the residual.  Catches: a dropped shard, a sign error, a residual
    written from the wrong tensor."""
    T, H = 6, 128
    base = _bf16_random((R // 2, T, H), 0.7, 2)
    p = np.empty((R, T, H), np.uint16)
    p[0::2] = base
    p[1::2] = base ^ np.uint16(0x8000)
    res = _bf16_random((T, H), 1.0, 3)
    gp = _rng(4).normal(1, 0.1, H).astype(np.float32)
    gq = _rng(5).normal(1, 0.1, H).astype(np.float32)
    r = oracle.reduce_norm(p, res, gp, gq, 1e-6)
    assert np.all(r["sum"].view(np.uint32) == 0)
    assert_bits_equal(r["residual_out"], res, "residual_out")
    expect = bf16_torch(_rmsnorm64(f32_from_bf16(res), gq, 1e-6).astype(np.float32))
    assert_bf16_close(r["out"], expect, 1, "out vs textbook RMSNorm")


def test_rank_order_witness():
    """Shards (1, 2^-24, 2^-24) in rank order give exactly 1 (each half-ulp add
    ties to even); the reverse order gives 1 + 2^-23.  Catches: any other order
    (reverse, pairwise) and accumulation in a wider type."""
    one, tiny = np.float32(1.0), np.float32(2.0 ** -24)
    fwd = bf16_bits(np.array([one, tiny, tiny], np.float32)).reshape(3, 1, 1).repeat(8, axis=2)
    rev = fwd[::-1].copy()
    s_fwd = oracle.reduce_norm(fwd, None, None, None, 0.0, want_norm=False)["sum"]
    s_rev = oracle.reduce_norm(rev, None, None, None, 0.0, want_norm=False)["sum"]
    assert np.all(s_fwd == np.float32(1.0))
    assert np.all(s_rev == np.float32(1.0 + 2.0 ** -23))


def test_two_shard_sum_is_correctly_rounded():
    """With R = 2 the FP32 sum is one rounding of the exact sum.  Catches: a
    transposed [T,R,H] layout, a wrong token offset."""
    d = inputs.to_numpy(inputs.make_inputs(inputs.WORKLOADS[0], 8))
    p = d["partials"]
    r = oracle.reduce_norm(p, None, None, None, 1e-6, want_norm=False)
    exact = f32_from_bf16(p[0]).astype(np.float64) + f32_from_bf16(p[1]).astype(np.float64)
    assert_bits_equal(r["sum"], exact.astype(np.float32), "sum")


def test_many_shard_sum_matches_sequential_numpy():
    """R = 8: the sum equals numpy's FP32 adds in rank order (numpy's own
    float32 addition), on the C2 value distribution."""
    wl = inputs.WORKLOADS[2]
    d = inputs.to_numpy(inputs.make_inputs(inputs.custom("reduce_norm", 8, 512, row_scale=True), 5))
    p = d["partials"]
    s = f32_from_bf16(p[0]).copy()
    for r in range(1, 8):
        s = s + f32_from_bf16(p[r])
    out = oracle.reduce_norm(p, None, None, None, wl.eps, want_norm=False)
    assert_bits_equal(out["sum"], s, "sum")


# ---- the norms -------------------------------------------------------------

@pytest.mark.parametrize("c", [1024.0, -1024.0])
def test_constant_row_gives_sign_times_gamma(c):
    """RMSNorm of a constant row c = +-2^10 is sign(c) * gamma exactly (eps
    vanishes next to c^2).  Catches: mean over H - 1, (1 + gamma), a missing
    gamma, a norm that is not scale free."""
    H, T = 256, 3
    p = np.full((1, T, H), bf16_bits(np.float32(c)), np.uint16)
    res = np.zeros((T, H), np.uint16)
    gp = _rng(6).normal(1, 0.1, H).astype(np.float32)
    gq = _rng(7).normal(1, 0.1, H).astype(np.float32)
    r = oracle.reduce_norm(p, res, gp, gq, 1e-6)
    assert np.all(r["ss"][:, 0] == np.float32(H * c * c))
    expect = bf16_torch(np.sign(c) * gp)
    for t in range(T):
        assert_bits_equal(r["residual_out"][t], expect, "residual_out")


def test_eps_is_inside_the_square_root():
    """A constant row of ones with eps = 1: mean + eps = 2, so y = gamma / sqrt(2).
    Catches: eps added outside the square root (that would give gamma / 2)."""
    H = 64
    p = np.full((1, 1, H), bf16_bits(np.float32(1.0)), np.uint16)
    res = np.zeros((1, H), np.uint16)
    gp = _rng(8).normal(1, 0.1, H).astype(np.float32)
    r = oracle.reduce_norm(p, res, gp, gp, 1.0)
    assert_bf16_close(r["residual_out"][0], bf16_torch(gp / math.sqrt(2.0)), 1, "y")


def test_post_norm_is_scale_free():
    """eps = 0: scaling a shard row by 2^m leaves the post-norm output and
    everything after it unchanged bit for bit (each step scales exactly)."""
    H, T = 512, 4
    p = _bf16_random((1, T, H), 1.0, 9)
    res = _bf16_random((T, H), 1.0, 10)
    gp = _rng(11).normal(1, 0.1, H).astype(np.float32)
    gq = _rng(12).normal(1, 0.1, H).astype(np.float32)
    base = oracle.reduce_norm(p, res, gp, gq, 0.0)
    for m in (-7, 5):
        ps = bf16_torch(f32_from_bf16(p) * np.float32(2.0 ** m))
        r = oracle.reduce_norm(ps, res, gp, gq, 0.0)
        assert_bits_equal(r["residual_out"], base["residual_out"], f"residual_out 2^{m}")
        assert_bits_equal(r["out"], base["out"], f"out 2^{m}")


def test_sums_of_squares_are_correctly_rounded():
    """ss1 is the FP32 rounding of the exact sum of s^2 (math.fsum), on long
    rows with a 100x spread of row scales.  Catches: FP32 accumulation."""
    d = inputs.to_numpy(inputs.make_inputs(inputs.custom("reduce_norm", 4, 8192, row_scale=True), 6))
    r = oracle.reduce_norm(d["partials"], d["residual"], d["gamma_post"], d["gamma_pre"], 1e-6)
    s = r["sum"].astype(np.float64)
    for t in range(s.shape[0]):
        exact = np.float32(math.fsum((s[t] * s[t]).tolist()))
        assert r["ss"][t, 0] == exact, (t, r["ss"][t, 0], exact)


def test_double_recomputation_of_the_whole_chain():
    """Workload C0: a float64 recomputation of sum -> post-norm -> residual add
    -> pre-norm agrees within 1 BF16 ulp on both outputs.  Catches: a missing
    step, swapped gammas, a norm over the wrong axis."""
    d = inputs.to_numpy(inputs.make_inputs(inputs.WORKLOADS[0], 8))
    p, res, gp, gq, eps = d["partials"], d["residual"], d["gamma_post"], d["gamma_pre"], d["eps"]
    r = oracle.reduce_norm(p, res, gp, gq, eps)
    s = f32_from_bf16(p).astype(np.float64).sum(axis=0)
    h = f32_from_bf16(res).astype(np.float64) + _rmsnorm64(s, gp, eps)
    out = _rmsnorm64(h, gq, eps)
    assert_bf16_close(r["residual_out"], bf16_torch(h.astype(np.float32)), 1, "residual_out")
    assert_bf16_close(r["out"], bf16_torch(out.astype(np.float32)), 1, "out")


def test_single_norm_variant_matches_double():
    """AllReduce + residual + RMSNorm (no post-norm): h = residual + s."""
    d = inputs.to_numpy(inputs.make_inputs(inputs.WORKLOADS[0], 8))
    p, res, gq, eps = d["partials"], d["residual"], d["gamma_pre"], d["eps"]
    r = oracle.reduce_norm(p, res, d["gamma_post"], gq, eps, flags=oracle.SINGLE_NORM)
    h = f32_from_bf16(res).astype(np.float64) + f32_from_bf16(p).astype(np.float64).sum(axis=0)
    assert_bf16_close(r["residual_out"], bf16_torch(h.astype(np.float32)), 1, "residual_out")
    assert_bf16_close(r["out"], bf16_torch(_rmsnorm64(h, gq, eps).astype(np.float32)), 1, "out")


def test_prenorm_reading_switch_stays_close():
    """The alternative reading (pre-norm of the BF16 residual) differs from the
    chosen one by at most a few ulps; the switch exists for sensitivity reports."""
    d = inputs.to_numpy(inputs.make_inputs(inputs.WORKLOADS[0], 8))
    a = oracle.reduce_norm(d["partials"], d["residual"], d["gamma_post"], d["gamma_pre"], 1e-6)
    b = oracle.reduce_norm(d["partials"], d["residual"], d["gamma_post"], d["gamma_pre"], 1e-6,
                           flags=oracle.PRENORM_FROM_BF16_RESIDUAL)
    assert_bits_equal(a["residual_out"], b["residual_out"], "residual_out")
    assert_bf16_close(a["out"], b["out"], 2, "out")


def test_split_epilogue_equals_fused():
    """norm(sum) of the oracle equals its fused reduce_norm bit for bit."""
    d = inputs.to_numpy(inputs.make_inputs(inputs.custom("reduce_norm", 4, 640), 7))
    a = oracle.reduce_norm(d["partials"], d["residual"], d["gamma_post"], d["gamma_pre"], 1e-6)
    b = oracle.norm(a["sum"], d["residual"], d["gamma_post"], d["gamma_pre"], 1e-6)
    for key in ("ss", "residual_out", "out"):
        assert_bits_equal(b[key], a[key], key)


def test_row_selection_matches_full_run():
    d = inputs.to_numpy(inputs.make_inputs(inputs.custom("reduce_norm", 3, 256), 9))
    full = oracle.reduce_norm(d["partials"], d["residual"], d["gamma_post"], d["gamma_pre"], 1e-6)
    rows = [8, 0, 3]
    part = oracle.reduce_norm(d["partials"], d["residual"], d["gamma_post"], d["gamma_pre"], 1e-6,
                              rows=rows)
    for key in ("sum", "ss", "residual_out", "out"):
        assert_bits_equal(part[key], full[key][rows], key)


# ---- the MoE finalize --------------------------------------------------------

def _finalize_case(R, T, k, H, seed):
    wl = inputs.custom("finalize_reduce_norm", R, H, k, partial_std=0.3, shared_std=0.3)
    return inputs.to_numpy(inputs.make_inputs(wl, T, seed=seed))


def test_one_hot_weights_make_the_finalize_a_row_gather():
    """One-hot w and no shared term: z[r,t] is row perm[r,t,j*] of shard r's
    expert outputs, bit for bit.  Catches: scatter for gather, the wrong shard's
    perm or rows, a wrong slot stride."""
    R, T, k, H = 3, 5, 4, 64
    d = _finalize_case(R, T, k, H, 11)
    rng = _rng(12)
    jstar = rng.integers(0, k, size=(R, T))
    w = np.zeros((R, T, k), np.float32)
    for r in range(R):
        for t in range(T):
            w[r, t, jstar[r, t]] = 1.0
    out = oracle.finalize_reduce_norm(d["expert_out"], d["perm"], w, None, d["residual"],
                                      d["gamma_post"], d["gamma_pre"], 1e-6, want_z=True)
    for r in range(R):
        for t in range(T):
            row = d["perm"][r, t, jstar[r, t]]
            assert_bits_equal(out["z"][r, t], d["expert_out"][r, row], f"z[{r},{t}]")


def test_top1_finalize_is_a_bf16_add():
    """k = 1, w = 1: z = BF16(x + shared), checked against PyTorch's rounding of
    the exact sum (exact in FP32 for these values)."""
    R, T, k, H = 2, 6, 1, 128
    d = _finalize_case(R, T, k, H, 13)
    w = np.ones((R, T, k), np.float32)
    out = oracle.finalize_reduce_norm(d["expert_out"], d["perm"], w, d["shared"], d["residual"],
                                      d["gamma_post"], d["gamma_pre"], 1e-6, want_z=True)
    x = f32_from_bf16(d["expert_out"]).astype(np.float64)
    sh = f32_from_bf16(d["shared"]).astype(np.float64)
    for r in range(R):
        for t in range(T):
            exact = x[r, d["perm"][r, t, 0]] + sh[r, t]
            assert np.all(exact.astype(np.float32).astype(np.float64) == exact)
            assert_bits_equal(out["z"][r, t], bf16_torch(exact.astype(np.float32)), f"z[{r},{t}]")


def test_identity_perm_finalize_matches_float64_einsum():
    """perm = identity: z is within 1 BF16 ulp of BF16(einsum('tkh,tk->th') +
    shared) computed in float64.  Catches: a weight applied to the wrong slot."""
    R, T, k, H = 2, 4, 6, 256
    d = _finalize_case(R, T, k, H, 14)
    perm = np.tile(np.arange(T * k, dtype=np.int32).reshape(1, T, k), (R, 1, 1))
    out = oracle.finalize_reduce_norm(d["expert_out"], perm, d["w"], d["shared"], d["residual"],
                                      d["gamma_post"], d["gamma_pre"], 1e-6, want_z=True)
    x = f32_from_bf16(d["expert_out"]).astype(np.float64).reshape(R, T, k, H)
    ref = np.einsum("rtkh,rtk->rth", x, d["w"].astype(np.float64))
    ref += f32_from_bf16(d["shared"]).astype(np.float64)
    assert_bf16_close(out["z"], bf16_torch(ref.astype(np.float32)), 1, "z")


def test_finalize_sum_is_rank_ordered_sum_of_z():
    R, T, k, H = 4, 3, 5, 96
    d = _finalize_case(R, T, k, H, 15)
    out = oracle.finalize_reduce_norm(d["expert_out"], d["perm"], d["w"], d["shared"],
                                      d["residual"], d["gamma_post"], d["gamma_pre"], 1e-6,
                                      want_z=True)
    s = f32_from_bf16(out["z"][0]).copy()
    for r in range(1, R):
        s = s + f32_from_bf16(out["z"][r])
    assert_bits_equal(out["sum"], s, "sum")
    # and the epilogue of that sum is the reduce_norm epilogue
    ref = oracle.norm(s, d["residual"], d["gamma_post"], d["gamma_pre"], 1e-6)
    for key in ("ss", "residual_out", "out"):
        assert_bits_equal(out[key], ref[key], key)


def test_perm_out_of_range_is_rejected():
    R, T, k, H = 1, 2, 2, 8
    d = _finalize_case(R, T, k, H, 16)
    bad = d["perm"].copy()
    bad[0, 1, 1] = T * k
    with pytest.raises(ValueError):
        oracle.finalize_reduce_norm(d["expert_out"], bad, d["w"], d["shared"], d["residual"],
                                    d["gamma_post"], d["gamma_pre"], 1e-6)


# ---- the oracle's own BF16 rounding -------------------------------------------

def test_bf16_rounding_matches_pytorch():
    """The oracle's round-to-nearest-even (written from the format's definition)
    agrees with PyTorch's conversion on ties, carries, subnormals, the overflow
    boundary and random values."""
    specials = np.array([0.0, -0.0, 1.0, 1.00390625, 1.01171875, -1.00390625, 3.0e38, 3.4e38,
                         np.float32(3.3961776e38), 1e-40, -1e-40, 2.0 ** -133, np.inf, -np.inf,
                         65504.0, 0.1], dtype=np.float32)
    rnd = _rng(17).normal(0, 1, 20000).astype(np.float32) * np.float32(2.0) ** _rng(18).integers(
        -30, 30, 20000).astype(np.float32)
    x = np.concatenate([specials, rnd]).astype(np.float32)
    assert_bits_equal(oracle.bf16_from_f32(x), bf16_torch(x), "bf16 rounding")
    assert np.isnan(f32_from_bf16(oracle.bf16_from_f32(np.array([np.nan], np.float32))))[0]
