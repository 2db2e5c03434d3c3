"""GPU-vs-oracle comparison helpers for the parity tests and the smoke check.

Inputs come from the seeded generator (on the GPU for large cases); the
oracle gets host copies of the same bytes.  A block of token rows can be
handed to the oracle on its own: the rows' operands (their shard rows, or
their gathered expert rows with the perm renumbered) are copied into a
compact input set, which the oracle processes exactly as it would the full
one, since every token row depends only on its own operands.  Large cases
run the oracle on every row this way, in blocks on a pool of host threads.

Acceptance (per element): the FP32 reduced sum and the per-shard BF16
finalize results bit-exact; the sums of squares within 1e-5 relative, or
within H * 2^-149 absolute where that is larger (the one-pass compensated sum
over squares in FP32's subnormal range, which the kernels run for eps >=
2^-50; the kernels for smaller eps meet 2^-149); the BF16 output and updated
residual within 1 BF16 ulp (+0 == -0, NaN == NaN).
"""
from __future__ import annotations

from typing import Optional, Sequence

import numpy as np
import torch

import oracle
from tests.helpers import (SUBNORMAL_STEP, assert_bf16_close, assert_bits_equal, assert_rel_close,
                           bf16_ulp_diff)
from tp_reduce_residual_gb300 import beamnorm as bn
from tp_reduce_residual_gb300 import inputs

SS_RTOL = 1e-5
MAX_ULP = 1
NAN_BF16 = 0x7FC0


def gpu_inputs(wl, T, seed=None, with_shared=True):
    return inputs.make_inputs(wl, T, device="cuda", seed=seed, with_shared=with_shared)


SENTINEL_BF16 = 0x4049      # 3.140625: a finite prefill for outputs that may be NaN
SENTINEL_F32 = 1234.5


def _nan_like(shape, dtype):
    if dtype == torch.bfloat16:
        return torch.full(shape, NAN_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    return torch.full(shape, float("nan"), dtype=dtype, device="cuda")


def _sentinel_like(shape, dtype):
    if dtype == torch.bfloat16:
        return torch.full(shape, SENTINEL_BF16, dtype=torch.int16, device="cuda").view(torch.bfloat16)
    return torch.full(shape, SENTINEL_F32, dtype=dtype, device="cuda")


def run_fused(d, single: bool = False, debug: bool = True, stream=None, workspace=None,
              prefill: str = "nan", on_decline: str = "raise") -> dict:
    """One fused call on a copy of the residual; outputs prefilled with NaN
    (``prefill="sentinel"``: a finite value, for inputs whose results may be
    NaN).  ``workspace`` goes to the finalize entries (their many-CTA path)."""
    op, R, T, H, k = d["op"], d["R"], d["T"], d["H"], d["k"]
    fin = op == "finalize_reduce_norm"
    fill = _nan_like if prefill == "nan" else _sentinel_like
    res = d["residual"].clone()
    out = fill((T, H), torch.bfloat16)
    dbg = None
    if debug:
        dbg = bn.Debug(sum=fill((T, H), torch.float32), ss=fill((T, 2), torch.float32),
                       z=fill((R, T, H), torch.bfloat16) if fin else None)
    if not fin:
        if single:
            bn.reduce_residual_norm(d["partials"], res, d["gamma_pre"], d["eps"], out=out, debug=dbg,
                                    stream=stream, on_decline=on_decline)
        else:
            bn.reduce_norm(d["partials"], res, d["gamma_post"], d["gamma_pre"], d["eps"], out=out,
                           debug=dbg, stream=stream, on_decline=on_decline)
    else:
        if single:
            bn.finalize_reduce_residual_norm(d["expert_out"], d["perm"], d["w"], d["shared"], res,
                                             d["gamma_pre"], d["eps"], out=out, debug=dbg,
                                             stream=stream, workspace=workspace,
                                             on_decline=on_decline)
        else:
            bn.finalize_reduce_norm(d["expert_out"], d["perm"], d["w"], d["shared"], res,
                                    d["gamma_post"], d["gamma_pre"], d["eps"], out=out, debug=dbg,
                                    stream=stream, workspace=workspace, on_decline=on_decline)
    bits = bn.check_device_error(stream=stream)
    assert bits == 0, bits
    r = {"out": inputs.u16(out), "residual_out": inputs.u16(res)}
    if debug:
        r["sum"] = dbg.sum.cpu().numpy()
        r["ss"] = dbg.ss.cpu().numpy()
        if fin:
            r["z"] = inputs.u16(dbg.z)
    return r


def compact(d, rows: Sequence[int]) -> dict:
    """The operands of the selected token rows as a self-contained input set."""
    return inputs.select_rows(d, rows)


def run_oracle(d, rows: Optional[Sequence[int]] = None, single: bool = False) -> dict:
    """Oracle results for all rows, or for ``rows`` (in that order)."""
    src = d if rows is None else compact(d, rows)
    h = inputs.to_numpy(src)
    flags = oracle.SINGLE_NORM if single else 0
    if h["op"] == "reduce_norm":
        return oracle.reduce_norm(h["partials"], h["residual"], h["gamma_post"], h["gamma_pre"],
                                  h["eps"], flags=flags)
    return oracle.finalize_reduce_norm(h["expert_out"], h["perm"], h["w"], h.get("shared"),
                                       h["residual"], h["gamma_post"], h["gamma_pre"], h["eps"],
                                       flags=flags, want_z=True)


def _oracle_host(h: dict, single: bool) -> dict:
    flags = oracle.SINGLE_NORM if single else 0
    if h["op"] == "reduce_norm":
        return oracle.reduce_norm(h["partials"], h["residual"], h["gamma_post"], h["gamma_pre"],
                                  h["eps"], flags=flags)
    return oracle.finalize_reduce_norm(h["expert_out"], h["perm"], h["w"], h.get("shared"),
                                       h["residual"], h["gamma_post"], h["gamma_pre"], h["eps"],
                                       flags=flags, want_z=True)


def run_oracle_all_rows(d, single: bool = False, block: int = 64, workers: int = 0) -> dict:
    """Oracle results for every token row, computed in blocks of rows on a
    pool of host threads.  Each block is a self-contained input set (the
    rows' own operands, see ``compact``) and each oracle call is the plain
    single-threaded C code; the ctypes call releases the interpreter lock, so
    blocks run side by side.  Same result as ``run_oracle(d)``."""
    import concurrent.futures as cf
    import os

    T = d["T"]
    workers = workers or max(1, min(16, os.cpu_count() or 1))
    blocks = [list(range(i, min(T, i + block))) for i in range(0, T, block)]
    parts = [None] * len(blocks)
    with cf.ThreadPoolExecutor(max_workers=workers) as ex:
        pending = {}
        for i, rows in enumerate(blocks):
            h = inputs.to_numpy(compact(d, rows))
            pending[ex.submit(_oracle_host, h, single)] = i
            if len(pending) >= 2 * workers:   # bound the host copies in flight
                done, _ = cf.wait(pending, return_when=cf.FIRST_COMPLETED)
                for f in done:
                    parts[pending.pop(f)] = f.result()
        for f in cf.as_completed(pending):
            parts[pending[f]] = f.result()
    return {key: np.concatenate([p[key] for p in parts], axis=1 if key == "z" else 0)
            for key in parts[0]}


def compare(g: dict, ref: dict, rows: Optional[Sequence[int]] = None, what: str = "",
            ss_floor: Optional[float] = None) -> dict:
    """Assert the acceptance bar; return exact-match statistics.  ``ss_floor``
    replaces the sums of squares' absolute floor H * 2^-149 (2^-149 for the
    calls that run the second pass over rows of tiny values)."""
    sel = slice(None) if rows is None else np.asarray(rows)
    stats = {}
    if "sum" in g:
        assert_bits_equal(g["sum"][sel], ref["sum"], f"{what} sum")
    if "z" in g and "z" in ref:
        assert_bits_equal(g["z"][:, sel], ref["z"], f"{what} z")
    if "ss" in g:
        H = ref["out"].shape[-1]
        floor = H * SUBNORMAL_STEP if ss_floor is None else ss_floor
        assert_rel_close(g["ss"][sel], ref["ss"], SS_RTOL, f"{what} ss", floor=floor)
        stats["ss_exact"] = float(np.mean(g["ss"][sel].view(np.uint32) == ref["ss"].view(np.uint32)))
    assert_bf16_close(g["residual_out"][sel], ref["residual_out"], MAX_ULP, f"{what} residual_out")
    assert_bf16_close(g["out"][sel], ref["out"], MAX_ULP, f"{what} out")
    stats["out_exact"] = float(np.mean(bf16_ulp_diff(g["out"][sel], ref["out"]) == 0))
    stats["residual_exact"] = float(np.mean(bf16_ulp_diff(g["residual_out"][sel], ref["residual_out"]) == 0))
    return stats


# ---- memory-safety substitutes: outputs inside NaN-filled guard bands -----------------

def guarded(n, dtype, guard=4096):
    """A tensor of n elements inside a NaN-filled buffer with guard bands of
    ``guard`` bytes on each side: (buffer, tensor, guard elements)."""
    esz = torch.tensor([], dtype=dtype).element_size()
    g = guard // esz
    buf = _nan_like((g + n + g,), dtype)
    return buf, buf[g:g + n], g


def guard_intact(buf, g, n) -> bool:
    """True if the guard bands around the n elements are still all NaN."""
    if buf.dtype == torch.bfloat16:
        bits = buf.view(torch.int16)
        return bool((bits[:g] == NAN_BF16).all() and (bits[g + n:] == NAN_BF16).all())
    return bool(torch.isnan(buf[:g]).all() and torch.isnan(buf[g + n:]).all())

