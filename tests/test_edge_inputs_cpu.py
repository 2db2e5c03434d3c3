"""The edge-case inputs and the oracle on them (CPU, no GPU needed).

The GPU edge-case tests compare the kernels with the oracle on these rows.
Here the oracle's own results on them are pinned to what the method fixes
exactly -- the rank-order witness, negated pairs, the cancelling finalize,
constant rows, sums of squares beyond the FP32 range, subnormals kept -- and
the all-rows runner is checked to give the single call's result.
"""
import numpy as np
import pytest

from tests import parity
from tests.helpers import f32_from_bf16
from tp_reduce_residual_gb300 import inputs

KINDS = inputs.EDGE_KINDS


def _oracle(d):
    return parity.run_oracle(d)


@pytest.mark.parametrize("op,R,k,with_shared", [("reduce_norm", 4, 0, False),
                                                ("reduce_norm", 1, 0, False),
                                                ("finalize_reduce_norm", 3, 4, True),
                                                ("finalize_reduce_norm", 2, 2, False)])
def test_edge_rows_give_the_values_the_method_fixes(op, R, k, with_shared):
    H = 200
    d = inputs.edge_inputs(op, R, H, KINDS, k=k or 4, seed=7, with_shared=with_shared,
                           device="cpu")
    r = _oracle(d)
    res = inputs.u16(d["residual"])
    lanes = np.arange(H)
    row = {kind: t for t, kind in enumerate(KINDS)}
    # rank order: 1 + 2^-24 + 2^-24 -> 1 (ties to even); reversed it would be 1 + 2^-23
    sign = np.where(lanes % 2 == 0, 1.0, -1.0)
    assert np.array_equal(r["sum"][row["witness"]], sign.astype(np.float32))
    # negated pairs sum to +0 and leave the residual as it was
    t = row["neg_pairs"]
    assert np.all(r["sum"][t].view(np.uint32) == 0)
    assert np.array_equal(r["residual_out"][t] & 0x7FFF, res[t] & 0x7FFF)
    # a constant row: s = 2^10, ss = H * 2^20 exactly
    t = row["constant"]
    assert np.all(r["sum"][t] == 1024.0) and r["ss"][t, 0] == np.float32(H * 2.0 ** 20)
    # sums of squares beyond the FP32 range: +inf, outputs still finite
    t = row["overflow_post"]
    assert np.isinf(r["ss"][t, 0]) and np.all(np.isfinite(f32_from_bf16(r["out"][t])))
    t = row["overflow_pre"]
    assert np.isinf(r["ss"][t, 1]) and np.all(np.isfinite(f32_from_bf16(r["residual_out"][t])))
    # subnormal shards are summed exactly (nothing flushed to zero)
    t = row["subnormal"]
    if op == "reduce_norm":
        p = f32_from_bf16(inputs.u16(d["partials"]))[:, t].astype(np.float64)
        assert np.any(r["sum"][t] != 0)
        assert np.array_equal(r["sum"][t].astype(np.float64), p.sum(axis=0))
    # inf and NaN in a shard make the whole row NaN
    t = row["inf_nan"]
    assert np.all(np.isnan(f32_from_bf16(r["out"][t])))
    if op == "finalize_reduce_norm" and (k or 4) >= 2:
        # the weighted products (w, -w) cancel exactly: z = +0 on every shard
        assert np.all(r["z"][:, row["cancel"]] == 0)


def test_edge_inputs_are_exact_bf16_and_perm_is_a_permutation():
    d = inputs.edge_inputs("finalize_reduce_norm", 4, 64, KINDS, k=4, seed=3, device="cpu")
    perm = d["perm"].numpy().reshape(4, -1)
    for r in range(4):
        assert sorted(perm[r].tolist()) == list(range(perm.shape[1]))
    w = d["w"].numpy()
    assert np.all(w[:, [t for t, kind in enumerate(KINDS) if kind != "cancel"]] == 0.25)


@pytest.mark.parametrize("op", ["reduce_norm", "finalize_reduce_norm"])
def test_all_rows_runner_equals_one_call(op):
    wl = inputs.custom(op, 3, 256, 2 if op != "reduce_norm" else 0, partial_std=0.3)
    d = inputs.make_inputs(wl, 37, device="cpu", seed=11)
    one = parity.run_oracle(d)
    blocks = parity.run_oracle_all_rows(d, block=5, workers=3)
    assert set(one) == set(blocks)
    for key in one:
        assert np.array_equal(one[key].view(np.uint8), blocks[key].view(np.uint8)), key
