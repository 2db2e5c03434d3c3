"""Seeded random shapes through the CUDA path, against the oracle (GB300).

Each case draws an entry point (the sandwich or the single pre-norm, reduce
or finalize), R, k, H (any multiple of 8 up to the fused maximum), T, the
value scale, eps, the shared-expert row and the launch path (the planner's
choice, the forced column split, or the many-CTA finalize with a workspace).
The planner then picks among its shapes -- cluster sizes, chunks per thread,
shard or column splits, the cluster-task path at few rows -- as it would for
a caller, so the draws reach combinations that the hand-picked cases do not.
Every token row is compared with the oracle at the usual bar.  The draws are
fixed by the seed; a failure names its case.

Sources: "Fuse Beam's TP all-reduce with its sandwich norms" (vLLM pull
request 62366), sections Claims and Details (the fused op, its served shapes
and its FP32 epilogue); sglang pull request 34134, description (the
finalize, with and without the shared expert, before the reduction).
"""
import numpy as np
import pytest
import torch

from tests import parity
from tp_reduce_residual_gb300 import beamnorm as bn
from tp_reduce_residual_gb300 import build as nbuild
from tp_reduce_residual_gb300 import inputs

pytestmark = pytest.mark.gpu

N_CASES = 160
MAX_BYTES = 48 << 20  # operand bytes per case, so that the oracle stays quick


def _draw(i: int) -> dict:
    rng = np.random.default_rng(90_000 + i)
    fin = bool(rng.integers(0, 2))
    single = bool(rng.integers(0, 4) == 0)
    R = int(rng.choice([1, 2, 3, 4, 5, 8, 12, 16]))
    k = int(rng.choice([1, 2, 3, 4, 8, 10, 16])) if fin else 0
    # H: a multiple of 8, log-uniform over [8, 32768]
    H = 8 * int(np.clip(np.exp(rng.uniform(0.0, np.log(4096.0))), 1, 4096))
    per_row = H * 2 * (R * (k + 1) + 2 if fin else R + 2)
    T_max = max(1, min(640, MAX_BYTES // per_row))  # past one wave of SMs too
    std = float(rng.choice([0.01, 0.3, 1.0, 30.0]))
    eps = float(rng.choice([1e-6, 1e-5, 1e-3]))
    with_shared = fin and bool(rng.integers(0, 2))
    path = str(rng.choice(["planner", "planner", "columns", "workspace"]))
    if path == "workspace" and not fin:
        path = "planner"
    if path == "workspace":
        T_max = min(T_max, 8)  # the many-CTA finalize serves at most 8 rows
    # T log-uniform over [1, T_max]: the few-row paths are drawn as often as the rest
    T = int(np.clip(np.exp(rng.uniform(0.0, np.log(T_max + 1.0))), 1, T_max))
    return dict(fin=fin, single=single, R=R, k=k, H=H, T=T, std=std, eps=eps,
                with_shared=with_shared, path=path)


CASES = [_draw(i) for i in range(N_CASES)]


def _id(c: dict) -> str:
    op = "fin" if c["fin"] else "red"
    return (f"{op}{'-single' if c['single'] else ''}-R{c['R']}-k{c['k']}-H{c['H']}-T{c['T']}"
            f"-{c['path']}{'-shared' if c['with_shared'] else ''}")


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    nbuild.build()
    bn.load()
    bn.set_tuning()
    yield
    bn.set_tuning()
    torch.cuda.empty_cache()


def test_draws_cover_the_paths():
    """The fixed draws reach every entry point and launch path."""
    seen = {(c["fin"], c["single"]) for c in CASES}
    assert seen == {(False, False), (False, True), (True, False), (True, True)}
    assert {c["path"] for c in CASES} == {"planner", "columns", "workspace"}
    assert any(c["with_shared"] for c in CASES) and any(c["fin"] and not c["with_shared"] for c in CASES)
    assert any(c["H"] % 64 for c in CASES)          # ragged against whole warps of chunks
    assert any(c["T"] > 152 for c in CASES) and any(c["T"] <= 8 for c in CASES)


@pytest.mark.parametrize("case", CASES, ids=[_id(c) for c in CASES])
def test_random_shape_matches_oracle(case):
    c = case
    op = "finalize_reduce_norm" if c["fin"] else "reduce_norm"
    wl = inputs.custom(op, c["R"], c["H"], c["k"], partial_std=c["std"], shared_std=c["std"],
                       eps=c["eps"])
    d = parity.gpu_inputs(wl, c["T"], seed=7_000 + c["R"] * 131 + c["T"] * 17 + c["H"],
                          with_shared=c["with_shared"])
    if not bn.supports(c["R"], c["T"], c["k"] if c["fin"] else 1, c["H"]):
        pytest.skip("shape declined by the fused entry points")
    ws = None
    if c["path"] == "workspace":
        ws = bn.finalize_workspace(c["R"], c["T"], c["k"], c["H"], device="cuda")
    try:
        if c["path"] == "columns":
            bn.set_tuning(split=1)
        g = parity.run_fused(d, single=c["single"], workspace=ws)
    finally:
        bn.set_tuning()
    assert bn.check_device_error() == 0
    parity.compare(g, parity.run_oracle(d, single=c["single"]), what=_id(c))


# ---- the unfused pieces (the fallback of a declined fused call) -------------------------

N_PIECE_CASES = 40
MAX_PIECE_H = 131072


def _draw_piece(i: int) -> dict:
    rng = np.random.default_rng(95_000 + i)
    fin = bool(rng.integers(0, 2))
    single = bool(rng.integers(0, 3) == 0)
    R = int(rng.choice([1, 2, 4, 8, 16]))
    k = int(rng.choice([1, 2, 4, 8])) if fin else 0
    # H log-uniform over [8, 131072]: a third of the draws above the fused maximum
    H = 8 * int(np.clip(np.exp(rng.uniform(0.0, np.log(MAX_PIECE_H / 8))), 1, MAX_PIECE_H // 8))
    per_row = H * 2 * (R * (k + 1) + 2 if fin else R + 2) + 8 * H
    T_max = max(1, min(64, MAX_BYTES // per_row))
    T = int(np.clip(np.exp(rng.uniform(0.0, np.log(T_max + 1.0))), 1, T_max))
    with_shared = fin and bool(rng.integers(0, 2))
    return dict(fin=fin, single=single, R=R, k=k, H=H, T=T, with_shared=with_shared)


PIECE_CASES = [_draw_piece(i) for i in range(N_PIECE_CASES)]


def _piece_id(c: dict) -> str:
    return (f"{'fin' if c['fin'] else 'red'}{'-single' if c['single'] else ''}-R{c['R']}-k{c['k']}"
            f"-H{c['H']}-T{c['T']}{'-shared' if c['with_shared'] else ''}")


def test_piece_draws_reach_beyond_the_fused_maximum():
    assert any(c["H"] > 32768 for c in PIECE_CASES) and any(c["H"] <= 32768 for c in PIECE_CASES)
    assert {(c["fin"], c["single"]) for c in PIECE_CASES} == {(False, False), (False, True),
                                                               (True, False), (True, True)}


@pytest.mark.parametrize("case", PIECE_CASES, ids=[_piece_id(c) for c in PIECE_CASES])
def test_random_shape_through_the_pieces_matches_oracle(case):
    """The unfused chain on a random shape: the materialised finalize (z), the
    rank-ordered FP32 sum, then the epilogue on that sum; each against the
    oracle's fused results (z and the sum bit for bit)."""
    c = case
    op = "finalize_reduce_norm" if c["fin"] else "reduce_norm"
    wl = inputs.custom(op, c["R"], c["H"], c["k"], partial_std=0.3, shared_std=0.3)
    d = parity.gpu_inputs(wl, c["T"], seed=8_000 + c["R"] * 7 + c["T"] * 3 + c["H"],
                          with_shared=c["with_shared"])
    for piece in ((["finalize_only", "finalize_reduce_only"] if c["fin"] else ["reduce_only"]) +
                  ["residual_norm_only" if c["single"] else "norm_only"]):
        assert bn.supports_op(piece, c["R"], c["T"], c["H"], c["k"]), piece
    ref = parity.run_oracle(d, single=c["single"])
    g = {}
    if c["fin"]:
        z = bn.finalize_only(d["expert_out"], d["perm"], d["w"], d["shared"])
        s = bn.finalize_reduce_only(d["expert_out"], d["perm"], d["w"], d["shared"])
        g["z"] = inputs.u16(z)
    else:
        s = bn.reduce_only(d["partials"])
    res = d["residual"].clone()
    if c["single"]:
        out = bn.residual_norm_only(s, res, d["gamma_pre"], d["eps"])
    else:
        out = bn.norm_only(s, res, d["gamma_post"], d["gamma_pre"], d["eps"])
    torch.cuda.synchronize()
    assert bn.check_device_error() == 0
    g.update({"sum": s.cpu().numpy(), "out": inputs.u16(out), "residual_out": inputs.u16(res)})
    parity.compare(g, ref, what=_piece_id(c))
