"""The edge-case inputs and the oracle on them (CPU, no GPU needed).

The GPU edge-case tests compare the kernels with the oracle on these rows.
Here the oracle's own results on them are pinned to what the method fixes
exactly -- the rank-order witness, negated pairs, the cancelling finalize,
constant rows, sums of squares beyond the FP32 range, subnormals kept, the
sums of squares of rows of tiny values equal to the exact sums rounded once
-- and the all-rows runner is checked to give the single call's result.
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


def _round_f32(x) -> np.float32:
    """A non-negative exact rational rounded once to FP32 (to nearest, ties
    to even; subnormal below 2^-126, +inf at 2^128 and above)."""
    from fractions import Fraction
    x = Fraction(x)
    if x == 0:
        return np.float32(0.0)
    e = x.numerator.bit_length() - x.denominator.bit_length()
    if Fraction(2) ** e > x:
        e -= 1                                   # now 2^e <= x < 2^(e+1)
    quantum = Fraction(2) ** (max(e, -126) - 23)
    q, rem = divmod(x, quantum)
    if rem * 2 > quantum or (rem * 2 == quantum and q % 2 == 1):
        q += 1
    v = q * quantum
    return np.float32(np.inf) if v >= Fraction(2) ** 128 else np.float32(float(v))


def _exact_ss_rounded(values: np.ndarray) -> np.float32:
    """The exact sum of squares of FP32 ``values`` (rational arithmetic),
    rounded once to FP32."""
    from fractions import Fraction
    return _round_f32(sum(Fraction(float(v)) ** 2 for v in values.astype(np.float64)))


def test_round_f32_matches_numpy_on_doubles():
    """The rounding helper against numpy's FP32 conversion, which rounds a
    double once (exact for these: each is a double within FP32's range)."""
    rng = np.random.default_rng(5)
    xs = np.abs(rng.standard_normal(2000)) * np.exp2(rng.integers(-160, 120, 2000))
    xs = np.concatenate([xs, [2.0 ** -149, 2.0 ** -150, 3 * 2.0 ** -151, 2.0 ** -126,
                              (1 + 2.0 ** -24) * 2.0 ** -126, 1.0 + 2.0 ** -24]])
    for x in xs:
        assert _round_f32(float(x)) == np.float32(x), x


@pytest.mark.parametrize("op,single", [("reduce_norm", False), ("reduce_norm", True),
                                       ("finalize_reduce_norm", False)])
def test_oracle_sums_tiny_rows_exactly(op, single):
    """Rows of values near 2^-66 and 2^-76 (squares below FP32's normal
    range): the oracle's sums of squares are the exact sums rounded once, in
    the normal range ("tiny") and the subnormal one ("tiny_sub") -- nothing
    flushed to zero, no square rounded on its own."""
    kinds = ("tiny", "tiny_sub", "normal")
    H = 512
    d = inputs.edge_inputs(op, 4, H, kinds, k=2, seed=21, eps=0.0, with_shared=True,
                           device="cpu")
    r = parity.run_oracle(d, single=single)
    res = f32_from_bf16(inputs.u16(d["residual"]))
    for t, kind in enumerate(kinds[:2]):
        s = r["sum"][t].astype(np.float32)
        if single:
            vals = (res[t] + s).astype(np.float32)  # h = residual + s, one FP32 add each
            got = r["ss"][t, 1]
        else:
            vals = s
            got = r["ss"][t, 0]
        want = _exact_ss_rounded(vals)
        assert got == want, (kind, got, want)
        if kind == "tiny":
            assert 2.0 ** -126 <= got < 2.0 ** -80
            assert np.all(np.isfinite(f32_from_bf16(r["out"][t])))
        else:
            assert 0.0 < got < 2.0 ** -126
