"""The many-CTA finalize for callers that cannot allocate device memory.

Some callers of this epilogue are handed only the op's input and output
tensors and may not allocate: an engine whose memory pool owns all of HBM, or
a plugin hook of an inference runtime with no workspace slot.
bn_finalize_reduce_norm_noalloc serves them with the library's own static
scratch.  This file checks, through the C ABI, that two calls in a row give
what bn_finalize_reduce_norm_ws gives with a caller workspace (the same
tolerances as every parity test: sum and z bit-exact, sums of squares within
1e-5 relative, outputs within 1 BF16 ulp), and that a shape whose scratch would
exceed the static maximum is declined without touching anything.

The file name sorts last, so a run that stops at the first failure has run
every other test first; it also passes on its own in a fresh process.
"""
import pytest
import torch

from tests import parity
from tp_reduce_residual_gb300 import beamnorm as bn
from tp_reduce_residual_gb300 import build as nbuild
from tp_reduce_residual_gb300 import inputs

pytestmark = pytest.mark.gpu

SCRATCH_BYTES = 2 << 20


@pytest.fixture(scope="module", autouse=True)
def _gpu():
    assert torch.cuda.is_available(), "the GPU tests need a CUDA device"
    nbuild.build()
    bn.load()
    bn.set_tuning()
    bn.check_device_error(raise_on_error=False)  # a clean error word to start from
    yield
    bn.set_tuning()


def _run_noalloc(d) -> dict:
    """One no-allocation call on a copy of the residual, NaN-prefilled outputs."""
    T, H, R = d["T"], d["H"], d["R"]
    res = d["residual"].clone()
    out = parity._nan_like((T, H), torch.bfloat16)
    dbg = bn.Debug(sum=parity._nan_like((T, H), torch.float32),
                   ss=parity._nan_like((T, 2), torch.float32),
                   z=parity._nan_like((R, T, H), torch.bfloat16))
    bn.finalize_reduce_norm_noalloc(d["expert_out"], d["perm"], d["w"], d["shared"], res,
                                    d["gamma_post"], d["gamma_pre"], d["eps"], out=out, debug=dbg)
    assert bn.check_device_error() == 0
    return {"out": inputs.u16(out), "residual_out": inputs.u16(res), "sum": dbg.sum.cpu().numpy(),
            "ss": dbg.ss.cpu().numpy(), "z": inputs.u16(dbg.z)}


# two shapes, so that the second call meets the first call's leftovers in the
# scratch: different T (counter words) and R * H (z rows)
CASES = [
    # (R, T, k, H, with_shared, seed)
    (8, 4, 10, 8192, True, 61),
    (3, 7, 5, 1000, False, 62),
]


def test_two_calls_in_a_row_match_the_workspace_entry_point():
    for R, T, k, H, with_shared, seed in CASES:
        assert bn.finalize_workspace_bytes(R, T, k, H) <= SCRATCH_BYTES
        wl = inputs.custom("finalize_reduce_norm", R, H, k, partial_std=0.3, shared_std=0.3)
        d = parity.gpu_inputs(wl, T, seed=seed, with_shared=with_shared)
        ws = bn.finalize_workspace(R, T, k, H, device="cuda")
        ref = parity.run_fused(d, workspace=ws)      # the existing entry, caller workspace
        got = parity.compare(_run_noalloc(d), ref, what=f"no-alloc R={R} T={T} k={k} H={H}")
        assert got["out_exact"] == 1.0 and got["residual_exact"] == 1.0, got


def test_scratch_beyond_the_maximum_is_declined():
    R, T, k, H = 16, 8, 2, 8192                        # needs 2 MiB + 256 bytes
    assert bn.finalize_workspace_bytes(R, T, k, H) > SCRATCH_BYTES
    wl = inputs.custom("finalize_reduce_norm", R, H, k, partial_std=0.3)
    d = parity.gpu_inputs(wl, T, seed=63)
    res = d["residual"].clone()
    out = torch.full((T, H), 3.0, device="cuda").to(torch.bfloat16)
    with pytest.raises(bn.BeamNormError) as e:
        bn.finalize_reduce_norm_noalloc(d["expert_out"], d["perm"], d["w"], d["shared"], res,
                                        d["gamma_post"], d["gamma_pre"], d["eps"], out=out)
    assert e.value.status == bn.ERR_UNSUPPORTED and "scratch" in str(e.value)
    torch.cuda.synchronize()
    assert bool((out.float() == 3.0).all())
    assert torch.equal(res, d["residual"])
    # and the scratch still serves the next call
    wl = inputs.custom("finalize_reduce_norm", 8, 6144, 8, partial_std=0.3, shared_std=0.3)
    d = parity.gpu_inputs(wl, 2, seed=64)
    ws = bn.finalize_workspace(8, 2, 8, 6144, device="cuda")
    parity.compare(_run_noalloc(d), parity.run_fused(d, workspace=ws), what="after the decline")
