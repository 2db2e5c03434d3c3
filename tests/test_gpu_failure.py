"""The failure path of the bounded waits, made to happen on purpose (GB300).

Every wait of the kernels is bounded.  A test-only tuning field,
``wait_limit_polls``, makes the copy-pipeline waits give up after one poll, so
an ordinary call's first wait for data still in flight expires.  The kernel
must then record BN_DEVERR_TIMEOUT, stop storing, let every bulk copy it
issued land, keep waiting for the cluster exchanges the other CTAs still feed,
and return.  Checked here, in the launch shapes that wait the most (small
rings, clusters of 8 splitting rows by column or by shard, several rows per
CTA): the call returns, the error word holds the timeout bit, nothing was
written outside the outputs (NaN guard bands), and the next call with the
default limit matches the oracle.  Nothing here hangs or faults the GPU: the
waits that time out are ordinary polls of barriers whose copies are in flight.

Source for failing loudly instead of silently: sglang pull request 34134,
NextN follow-up (a marked partial without a residual fails loudly).
"""
import numpy as np
import pytest
import torch

import oracle
from tests import parity
from tp_reduce_residual_gb300 import beamnorm as bn
from tp_reduce_residual_gb300 import build as nbuild
from tp_reduce_residual_gb300 import inputs

pytestmark = pytest.mark.gpu

ATTEMPTS = 5


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    nbuild.build()
    bn.load()
    bn.set_tuning()
    bn.check_device_error(raise_on_error=False)
    yield
    bn.set_tuning()
    bn.check_device_error(raise_on_error=False)


def _call(op, d, bufs):
    """One call of ``op`` writing into the (guarded) buffers ``bufs``."""
    T, H, R = d["T"], d["H"], d["R"]
    if op == "reduce_norm":
        bn.reduce_norm(d["partials"], bufs["residual"], d["gamma_post"], d["gamma_pre"], d["eps"],
                       out=bufs["out"], debug=bn.Debug(sum=bufs["sum"], ss=bufs["ss"]))
    elif op == "finalize_reduce_norm":
        bn.finalize_reduce_norm(d["expert_out"], d["perm"], d["w"], d["shared"], bufs["residual"],
                                d["gamma_post"], d["gamma_pre"], d["eps"], out=bufs["out"],
                                debug=bn.Debug(sum=bufs["sum"], ss=bufs["ss"], z=bufs["z"]))
    elif op == "finalize_only":
        bn.finalize_only(d["expert_out"], d["perm"], d["w"], d["shared"], z_out=bufs["z"])
    elif op == "norm_only":
        bn.norm_only(d["sum_in"], bufs["residual"], d["gamma_post"], d["gamma_pre"], d["eps"],
                     out=bufs["out"], debug=bn.Debug(ss=bufs["ss"]))
    else:
        raise ValueError(op)


def _guarded_outputs(op, d):
    T, H, R = d["T"], d["H"], d["R"]
    shapes = {"out": ((T, H), torch.bfloat16), "residual": ((T, H), torch.bfloat16),
              "sum": ((T, H), torch.float32), "ss": ((T, 2), torch.float32),
              "z": ((R, T, H), torch.bfloat16)}
    used = {"reduce_norm": ("out", "residual", "sum", "ss"),
            "finalize_reduce_norm": ("out", "residual", "sum", "ss", "z"),
            "finalize_only": ("z",), "norm_only": ("out", "residual", "ss")}[op]
    bufs, guards = {}, []
    for name in used:
        shape, dtype = shapes[name]
        n = int(np.prod(shape))
        buf, t, g = parity.guarded(n, dtype)
        bufs[name] = t.view(shape)
        guards.append((name, buf, g, n))
    if "residual" in bufs:
        bufs["residual"].copy_(d["residual"])
    return bufs, guards


# Rings of two stages (one copy each where rows are few) make the consumers
# wait for copies in flight, and the waits probe with the non-suspending
# test_wait (wait_mode 2): a suspending first probe may sleep until the copy
# lands, so that a one-poll limit would expire only when the copies are slow.
CASES = [
    # (id, op, R, T, k, H, tuning)
    ("finalize-columns", "finalize_reduce_norm", 8, 40, 10, 8192, dict(split=1, cluster_size=1)),
    ("finalize-shards-x8", "finalize_reduce_norm", 8, 16, 10, 8192,
     dict(split=2, cluster_size=8, stages=2, group=1)),
    ("finalize-columns-x4", "finalize_reduce_norm", 8, 6, 8, 6144,
     dict(split=1, cluster_size=4, stages=2, group=1)),
    ("reduce-columns-x8", "reduce_norm", 8, 16, 0, 8192, dict(split=1, cluster_size=8, stages=2)),
    ("reduce-rows-per-cta", "reduce_norm", 4, 1024, 0, 5120, dict(stages=2)),
    ("finalize-only-shards-x4", "finalize_only", 8, 4, 10, 8192,
     dict(split=2, cluster_size=4, stages=2, group=1)),
    ("norm-only", "norm_only", 1, 1024, 0, 8192, dict(stages=2)),
]


def _inputs(op, R, T, k, H):
    if op in ("reduce_norm", "norm_only"):
        d = parity.gpu_inputs(inputs.custom("reduce_norm", max(R, 2), H, partial_std=0.5), T,
                              seed=900 + T)
        if op == "norm_only":
            d["sum_in"] = bn.reduce_only(d["partials"])
            d["R"] = 1
        return d
    return parity.gpu_inputs(inputs.custom("finalize_reduce_norm", R, H, k, partial_std=0.3,
                                           shared_std=0.3), T, seed=900 + T)


def _oracle(op, d):
    if op == "norm_only":
        h = inputs.to_numpy(d)
        return oracle.norm(h["sum_in"], h["residual"], h["gamma_post"], h["gamma_pre"], h["eps"])
    return parity.run_oracle(d)


@pytest.mark.parametrize("case", CASES, ids=[c[0] for c in CASES])
def test_expired_waits_report_a_timeout_and_leave_the_context_usable(case):
    _, op, R, T, k, H, tuning = case
    d = _inputs(op, R, T, k, H)
    torch.cuda.synchronize()
    bits = 0
    try:
        bn.set_tuning(wait_limit_polls=1, wait_mode=2, **tuning)
        for _ in range(ATTEMPTS):
            bufs, guards = _guarded_outputs(op, d)
            _call(op, d, bufs)
            bits = bn.check_device_error(raise_on_error=False)   # the call returned
            for name, buf, g, n in guards:
                assert parity.guard_intact(buf, g, n), f"{name}: written outside its buffer"
            if bits & bn.DEVERR_TIMEOUT:
                break
    finally:
        bn.set_tuning()
    assert bits == bn.DEVERR_TIMEOUT, bits
    assert bn.check_device_error() == 0                          # cleared, nothing new

    # the same shape with the default limit: complete and correct
    try:
        bn.set_tuning(**tuning)
        bufs, guards = _guarded_outputs(op, d)
        _call(op, d, bufs)
        assert bn.check_device_error() == 0
    finally:
        bn.set_tuning()
    for name, buf, g, n in guards:
        assert parity.guard_intact(buf, g, n), name
    ref = _oracle(op, d)
    if op == "finalize_only":
        from tests.helpers import assert_bits_equal
        assert_bits_equal(inputs.u16(bufs["z"]), ref["z"], "z after the timeout")
        return
    g = {"out": inputs.u16(bufs["out"]), "residual_out": inputs.u16(bufs["residual"]),
         "ss": bufs["ss"].cpu().numpy()}
    if "sum" in bufs:
        g["sum"] = bufs["sum"].cpu().numpy()
    if "z" in bufs:
        g["z"] = inputs.u16(bufs["z"])
    parity.compare(g, ref, what=f"{case[0]} after the timeout")
