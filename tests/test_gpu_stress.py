"""Repetition under back-to-back launches: the same bits every time (GB300).

A substitute for a race detector (compute-sanitizer is not available): each
launch path runs many calls back to back on one stream, with programmatic
dependent launch overlapping each call's setup with the previous call, on the
same inputs but each with its own copy of the residual and its own outputs.
A race between warps, CTAs of a cluster or consecutive kernels would show as
a call whose outputs differ from the others'.  The first call is also checked
against the oracle.

Paths: the main kernel with one CTA per row (several rows per CTA, the
128-thread light-row CTAs), its shard split and column split over clusters,
the cluster path at few rows (finalize and reduce, narrow rows past 15
tokens), and the many-CTA finalize with a workspace.

Source for the fixed order that makes every call reproducible: "Fuse Beam's
TP all-reduce with its sandwich norms" (vLLM pull request 62366), section
Claims (rank-ordered FP32 sum, no FMA contraction).
"""
import numpy as np
import pytest
import torch

from tests import parity
from tp_reduce_residual_gb300 import beamnorm as bn
from tp_reduce_residual_gb300 import build as nbuild
from tp_reduce_residual_gb300 import inputs

pytestmark = pytest.mark.gpu

REPEATS = 48

CASES = [
    # (id, op, R, T, k, H, tuning, with workspace)
    ("main-one-cta-per-row", "reduce_norm", 8, 400, 0, 8192, {}, False),
    ("main-light-rows", "reduce_norm", 2, 500, 0, 4096, {}, False),
    ("main-finalize", "finalize_reduce_norm", 8, 300, 8, 4096, {}, False),
    ("shard-split", "finalize_reduce_norm", 8, 24, 10, 8192, {"split": 2}, False),
    ("column-split-x4", "reduce_norm", 4, 40, 0, 5120, {"split": 1, "cluster_size": 4}, False),
    ("cluster-path-finalize", "finalize_reduce_norm", 8, 4, 10, 8192, {}, False),
    ("cluster-path-reduce", "reduce_norm", 8, 6, 0, 8192, {}, False),
    ("cluster-path-narrow-32", "finalize_reduce_norm", 8, 32, 8, 2048, {}, False),
    ("workspace", "finalize_reduce_norm", 8, 4, 10, 8192, {}, True),
]


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    nbuild.build()
    bn.load()
    bn.set_tuning()
    yield
    bn.set_tuning()
    torch.cuda.empty_cache()


def _call(d, residual, out, ws):
    if d["op"] == "reduce_norm":
        bn.reduce_norm(d["partials"], residual, d["gamma_post"], d["gamma_pre"], d["eps"], out=out)
    else:
        bn.finalize_reduce_norm(d["expert_out"], d["perm"], d["w"], d["shared"], residual,
                                d["gamma_post"], d["gamma_pre"], d["eps"], out=out, workspace=ws)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_back_to_back_calls_give_the_same_bits(case):
    _, op, R, T, k, H, tuning, with_ws = case
    wl = inputs.custom(op, R, H, k, partial_std=0.3, shared_std=0.3)
    d = parity.gpu_inputs(wl, T, seed=4000 + R + T + H)
    ws = bn.finalize_workspace(R, T, k, H, device="cuda") if with_ws else None
    if with_ws:
        assert ws is not None
    residuals = [d["residual"].clone() for _ in range(REPEATS)]
    outs = [torch.empty_like(d["residual"]) for _ in range(REPEATS)]
    try:
        bn.set_tuning(**tuning)
        stream = torch.cuda.Stream()
        stream.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(stream):
            for i in range(REPEATS):
                # one workspace serves one call at a time: calls on one stream
                # run in order, and each leaves it zeroed for the next
                _call(d, residuals[i], outs[i], ws)
        torch.cuda.synchronize()
    finally:
        bn.set_tuning()
    assert bn.check_device_error() == 0
    out0 = inputs.u16(outs[0])
    res0 = inputs.u16(residuals[0])
    for i in range(1, REPEATS):
        assert np.array_equal(inputs.u16(outs[i]), out0), f"call {i}: out differs"
        assert np.array_equal(inputs.u16(residuals[i]), res0), f"call {i}: residual differs"
    ref = parity.run_oracle(d)
    g = {"out": out0, "residual_out": res0}
    parity.compare(g, ref, what=f"repeated {case[0]}")
