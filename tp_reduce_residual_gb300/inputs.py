"""Seeded synthetic inputs for the tensor-parallel reduce / norm epilogue.

This module only draws random numbers and lays them out; it holds none of the
epilogue's arithmetic.  Both the CUDA path (tests, benchmark) and the CPU
oracle's tests take their inputs from here.

The pages measure on model shapes, not on a dataset: Beam at TP4/TP8 with
hidden 5120 and 8192 ("Fuse Beam's TP all-reduce with its sandwich norms",
kernel microbenchmark table) and the GLM MoE layer with hidden 6144 and
GB300-profile hidden 8192 / top-k 10 (sglang pull request 34134, description).
The five workloads below stand in for them with synthetic values.

Recipe (every tensor is drawn in FP32 from a seeded ``torch.Generator`` on the
requested device, then rounded to BF16 where the tensor is BF16):

  draw order: partials or expert_out, perm, logits, shared, residual,
              gamma_post, gamma_pre, row scales
  N(mu, sigma): sigma is the standard deviation
  seed: 0 for the tiny case, 1000 * workload index + T otherwise

A CPU generator and a CUDA generator give different numbers for one seed; each
is deterministic.
"""
from __future__ import annotations

import dataclasses
import math
from typing import Optional, Sequence

import numpy as np
import torch


@dataclasses.dataclass(frozen=True)
class Workload:
    index: int
    op: str                 # "reduce_norm" or "finalize_reduce_norm"
    R: int
    H: int
    k: int                  # top-k (0 for reduce_norm)
    experts: int            # routed experts (sets nothing on the path; recorded only)
    tokens: Sequence[int]
    partial_std: float      # partials or expert_out standard deviation
    shared_std: float
    row_scale: bool         # per-token log-uniform [0.1, 10] row scaling
    eps: float = 1e-6
    name: str = ""

    def seed(self, T: int) -> int:
        return 0 if self.index == 0 else 1000 * self.index + T

    def describe(self, T: int) -> str:
        if self.op == "reduce_norm":
            return f"reduce_norm R={self.R} H={self.H} T={T}"
        return f"finalize_reduce_norm R={self.R} H={self.H} k={self.k} T={T}"


WORKLOADS = [
    Workload(0, "reduce_norm", R=2, H=256, k=0, experts=0, tokens=(8,), partial_std=1.0,
             shared_std=0.0, row_scale=False, name="tiny reduce_norm"),
    Workload(1, "reduce_norm", R=4, H=5120, k=0, experts=0, tokens=(1, 8, 64, 256, 1024, 4096),
             partial_std=0.5, shared_std=0.0, row_scale=False, name="reduce_norm R=4 H=5120"),
    Workload(2, "reduce_norm", R=8, H=8192, k=0, experts=0, tokens=(1, 8, 64, 256, 1024, 4096),
             partial_std=0.5, shared_std=0.0, row_scale=True, name="reduce_norm R=8 H=8192"),
    Workload(3, "finalize_reduce_norm", R=8, H=6144, k=8, experts=256,
             tokens=(1, 16, 64, 256, 1024), partial_std=0.3, shared_std=0.3, row_scale=False,
             name="finalize_reduce_norm R=8 H=6144 k=8"),
    Workload(4, "finalize_reduce_norm", R=8, H=8192, k=10, experts=256,
             tokens=(1, 4, 16, 64, 256, 1024, 4096), partial_std=0.3, shared_std=0.3,
             row_scale=False, name="finalize_reduce_norm R=8 H=8192 k=10"),
]


def custom(op: str, R: int, H: int, k: int = 0, *, partial_std: float = 0.5,
           shared_std: float = 0.3, row_scale: bool = False, eps: float = 1e-6,
           index: int = 99) -> Workload:
    """A workload of arbitrary shape with the same value recipe."""
    return Workload(index, op, R=R, H=H, k=k, experts=0, tokens=(), partial_std=partial_std,
                    shared_std=shared_std, row_scale=row_scale, eps=eps, name="custom")


def _gen(device, seed: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


def _normal(shape, mean, std, g, device) -> torch.Tensor:
    x = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    if mean != 0.0:
        x.add_(mean)
    return x


def _log_uniform(n, lo, hi, g, device) -> torch.Tensor:
    u = torch.rand(n, generator=g, device=device, dtype=torch.float32)
    return torch.exp(math.log(lo) + u * (math.log(hi) - math.log(lo)))


def make_inputs(wl: Workload, T: int, device="cpu", seed: Optional[int] = None,
                with_shared: bool = True) -> dict:
    """Draw one input set for workload ``wl`` at ``T`` tokens.

    Returns a dict of torch tensors on ``device``: ``partials`` (BF16 [R,T,H]) or
    ``expert_out`` (BF16 [R,T*k,H]), ``perm`` (int32 [R,T,k]), ``w`` (FP32
    [R,T,k]), ``shared`` (BF16 [R,T,H] or None), ``residual`` (BF16 [T,H]),
    ``gamma_post`` / ``gamma_pre`` (FP32 [H]) and ``eps``.
    """
    seed = wl.seed(T) if seed is None else seed
    g = _gen(device, seed)
    R, H, k = wl.R, wl.H, wl.k
    d: dict = {"R": R, "T": T, "H": H, "k": k, "eps": wl.eps, "op": wl.op, "seed": seed}
    if wl.op == "reduce_norm":
        p = _normal((R, T, H), 0.0, wl.partial_std, g, device)
        d["partials_f32"] = p
    else:
        x = _normal((R, T * k, H), 0.0, wl.partial_std, g, device)
        d["expert_out"] = x.to(torch.bfloat16)
        del x
        perm = torch.stack([torch.randperm(T * k, generator=g, device=device)
                            for _ in range(R)]).to(torch.int32).reshape(R, T, k)
        d["perm"] = perm.contiguous()
        logits = _normal((R, T, k), 0.0, 1.0, g, device)
        d["w"] = torch.softmax(logits, dim=-1).contiguous()
        sh = _normal((R, T, H), 0.0, wl.shared_std, g, device)
        d["shared"] = sh.to(torch.bfloat16) if with_shared else None
        del sh
    res = _normal((T, H), 0.0, 1.0, g, device)
    d["gamma_post"] = _normal((H,), 1.0, 0.1, g, device)
    d["gamma_pre"] = _normal((H,), 1.0, 0.1, g, device)
    if wl.row_scale:
        f = _log_uniform(T, 0.1, 10.0, g, device)
        gs = _log_uniform(T, 0.1, 10.0, g, device)
        if wl.op == "reduce_norm":
            d["partials_f32"].mul_(f.view(1, T, 1))
        res.mul_(gs.view(T, 1))
    if wl.op == "reduce_norm":
        d["partials"] = d.pop("partials_f32").to(torch.bfloat16)
    d["residual"] = res.to(torch.bfloat16)
    return d


def select_rows(d: dict, rows: Sequence[int]) -> dict:
    """The operands of the selected token rows as a self-contained input set.

    Every token row depends only on its own operands: its shard rows, or its
    gathered expert rows, weights and shared-expert rows.  Those are copied
    into a compact set whose perm is renumbered to the copied rows, so the set
    gives, row for row, the results of the selected rows of the full one.
    """
    idx = torch.as_tensor(list(rows), dtype=torch.long, device=d["residual"].device)
    n = idx.numel()
    c = {key: d[key] for key in ("op", "R", "H", "k", "eps", "gamma_post", "gamma_pre")}
    c["T"] = n
    c["residual"] = d["residual"][idx].contiguous()
    if d["op"] == "reduce_norm":
        c["partials"] = d["partials"][:, idx].contiguous()
    else:
        R, k = d["R"], d["k"]
        rows_used = d["perm"][:, idx, :].long().reshape(R, n * k)
        c["expert_out"] = torch.stack([d["expert_out"][r][rows_used[r]] for r in range(R)]).contiguous()
        c["perm"] = torch.arange(n * k, dtype=torch.int32, device=idx.device).reshape(1, n, k).repeat(R, 1, 1)
        c["w"] = d["w"][:, idx].contiguous()
        c["shared"] = None if d["shared"] is None else d["shared"][:, idx].contiguous()
    return c


def u16(t: torch.Tensor) -> np.ndarray:
    """BF16 torch tensor -> numpy uint16 bit patterns (host copy)."""
    return t.detach().contiguous().view(torch.int16).cpu().numpy().view(np.uint16)


def from_u16(a: np.ndarray, device="cpu") -> torch.Tensor:
    """numpy uint16 bit patterns -> BF16 torch tensor."""
    a = np.ascontiguousarray(a, dtype=np.uint16)
    return torch.from_numpy(a.view(np.int16).copy()).view(torch.bfloat16).to(device)


def to_numpy(d: dict) -> dict:
    """Host numpy copies of an input dict (BF16 as uint16)."""
    out = {}
    for key, v in d.items():
        if isinstance(v, torch.Tensor):
            out[key] = u16(v) if v.dtype == torch.bfloat16 else v.detach().cpu().numpy()
        else:
            out[key] = v
    return out


def algorithmic_bytes(op: str, R: int, T: int, H: int, k: int = 0, split: bool = False,
                      with_shared: bool = True) -> int:
    """Bytes each tensor contributes when read or written exactly once.

    reduce_norm: T*H*(2R + 6) + 8H; finalize_reduce_norm: T*H*(2Rk + 2R + 6)
    + 8RkT + 8H (shared counted when present); the unfused split adds the FP32
    sum written and read back, 8TH.
    """
    if op == "reduce_norm":
        b = T * H * (2 * R + 6) + 8 * H
    else:
        b = T * H * (2 * R * k + (2 * R if with_shared else 0) + 6) + 8 * R * k * T + 8 * H
    if split:
        b += 8 * T * H
    return b


# ---------------------------------------------------------------------------------------
# edge cases of the method: special values and exactly known sums, one kind per token row

EDGE_KINDS = ("normal", "neg_zero", "neg_pairs", "witness", "subnormal", "constant",
              "overflow_post", "overflow_pre", "inf_nan", "cancel", "tiny", "tiny_sub")

# value scales of the rows of tiny values: their squares are FP32 subnormals
# (about 2^-134 and 2^-154), and the row sums of squares, about R*H*2^-134 and
# R*H*2^-154, are normal ("tiny", R*H >= 2^8) or subnormal but nonzero
# ("tiny_sub", 2^5 <= R*H < 2^28)
TINY_SCALE = 2.0 ** -66
TINY_SUB_SCALE = 2.0 ** -76


def _bf16_exact(x: np.ndarray) -> np.ndarray:
    """FP32 values rounded to BF16 (PyTorch's rounding), returned as FP32."""
    t = torch.from_numpy(np.ascontiguousarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.float().numpy()


def _edge_row(kind: str, R: int, H: int, rng: np.random.Generator):
    """Shard values [R, H] and residual [H] (FP32, exact in BF16) of one row."""
    p = np.zeros((R, H), dtype=np.float32)
    res = _bf16_exact(rng.standard_normal(H).astype(np.float32))
    lanes = np.arange(H)
    if kind in ("normal", "cancel"):
        p[:] = _bf16_exact(0.5 * rng.standard_normal((R, H)).astype(np.float32))
    elif kind == "neg_zero":
        # even lanes: every shard -0 (the sum stays -0); odd lanes: shard 0
        # -0 and the others +0 (the sum is +0 once a +0 is added)
        p[:] = 0.0
        p[:, lanes % 2 == 0] = -0.0
        p[0, lanes % 2 == 1] = -0.0
    elif kind == "neg_pairs":
        # shard 2i+1 = -(shard 2i); an odd last shard is +0: the sum is +0
        for r in range(0, R - 1, 2):
            p[r] = _bf16_exact(rng.standard_normal(H).astype(np.float32))
            p[r + 1] = -p[r]
    elif kind == "witness":
        # (1, 2^-24, 2^-24, 0, ...) in rank order sums to 1.0 exactly (each
        # add is a tie to even); any other order gives 1 + 2^-23.  Odd lanes
        # carry the negated values.
        sign = np.where(lanes % 2 == 0, 1.0, -1.0).astype(np.float32)
        p[0] = sign
        for r in (1, 2):
            if r < R:
                p[r] = sign * np.float32(2.0 ** -24)
    elif kind == "subnormal":
        # BF16 subnormals (exponent field 0) with random signs, residual too
        def sub(n):
            bits = rng.integers(1, 0x80, size=n).astype(np.uint32) << 16
            bits |= (rng.integers(0, 2, size=n).astype(np.uint32) << 31)
            return bits.view(np.float32)
        p[:] = sub(R * H).reshape(R, H)
        res = sub(H)
    elif kind == "constant":
        # s = 2^10 on every lane (shard 0 carries it, the rest are +0)
        p[0] = np.float32(1024.0)
    elif kind == "overflow_post":
        # the sum of squares of s leaves the FP32 range
        p[:] = _bf16_exact(1e20 * rng.standard_normal((R, H)).astype(np.float32))
    elif kind == "overflow_pre":
        # the sum of squares of h = residual + y leaves the FP32 range
        p[:] = _bf16_exact(0.5 * rng.standard_normal((R, H)).astype(np.float32))
        res = _bf16_exact(1e20 * rng.standard_normal(H).astype(np.float32))
    elif kind == "inf_nan":
        p[:] = _bf16_exact(0.5 * rng.standard_normal((R, H)).astype(np.float32))
        r = 1 if R > 1 else 0
        p[r, 3 % H] = np.inf
        p[r, 7 % H] = -np.inf
        p[r, 11 % H] = np.nan
    elif kind in ("tiny", "tiny_sub"):
        # shards and residual N(0, 0.5^2) times a power of two (exact in BF16)
        sc = np.float32(TINY_SCALE if kind == "tiny" else TINY_SUB_SCALE)
        p[:] = _bf16_exact(0.5 * rng.standard_normal((R, H)).astype(np.float32)) * sc
        res = _bf16_exact(0.5 * rng.standard_normal(H).astype(np.float32)) * sc
    elif kind == "zero":
        pass
    else:
        raise ValueError(kind)
    return p, res


def edge_inputs(op: str, R: int, H: int, kinds: Sequence[str], k: int = 4, seed: int = 0,
                eps: float = 1e-6, with_shared: bool = False, device="cuda") -> dict:
    """One input set whose token row t is an edge case of kind ``kinds[t]``.

    For reduce_norm the shard rows are the kinds' values.  For
    finalize_reduce_norm each shard's k gathered rows all carry the value
    and every weight is 1/k (k a power of two), so the per-shard finalize
    reproduces the value exactly; the kind "cancel" instead gathers one
    random row twice with weights (w, -w) (w random, its products inexact)
    and zero weights on the other slots, so the finalize is exactly +0
    unless a weighted product is fused into the following addition.  The
    shared-expert rows, when present, are +0 except on "normal" rows.
    Same dict layout as ``make_inputs``.
    """
    rng = np.random.default_rng(seed)
    T = len(kinds)
    P = np.zeros((R, T, H), dtype=np.float32)
    res = np.zeros((T, H), dtype=np.float32)
    for t, kind in enumerate(kinds):
        P[:, t], res[t] = _edge_row(kind, R, H, rng)
    gp = (1.0 + 0.1 * rng.standard_normal(H)).astype(np.float32)
    gq = (1.0 + 0.1 * rng.standard_normal(H)).astype(np.float32)
    d: dict = {"R": R, "T": T, "H": H, "k": k if op == "finalize_reduce_norm" else 0,
               "eps": float(eps), "op": op, "seed": seed,
               "residual": from_u16(_f32_bits_to_bf16(res), device),
               "gamma_post": torch.from_numpy(gp).to(device),
               "gamma_pre": torch.from_numpy(gq).to(device)}
    if op == "reduce_norm":
        d["partials"] = from_u16(_f32_bits_to_bf16(P), device)
        return d
    assert k >= 1 and (k & (k - 1)) == 0, "k must be a power of two"
    X = np.repeat(P[:, :, None, :], k, axis=2)              # [R, T, k, H]
    W = np.full((R, T, k), 1.0 / k, dtype=np.float32)
    for t, kind in enumerate(kinds):
        if kind == "cancel" and k >= 2:
            for r in range(R):
                v = _bf16_exact((1.0 + rng.random(H)).astype(np.float32))
                X[r, t, 0] = v
                X[r, t, 1] = v
                w0 = np.float32(rng.uniform(0.1, 0.9))
                W[r, t] = 0.0
                W[r, t, 0] = w0
                W[r, t, 1] = -w0
    perm = np.stack([rng.permutation(T * k) for _ in range(R)]).astype(np.int32).reshape(R, T, k)
    E = np.zeros((R, T * k, H), dtype=np.float32)
    for r in range(R):
        E[r, perm[r].reshape(-1)] = X[r].reshape(T * k, H)
    d["expert_out"] = from_u16(_f32_bits_to_bf16(E), device)
    d["perm"] = torch.from_numpy(perm).to(device)
    d["w"] = torch.from_numpy(W).to(device)
    if with_shared:
        S = np.zeros((R, T, H), dtype=np.float32)
        for t, kind in enumerate(kinds):
            if kind == "normal":
                S[:, t] = _bf16_exact(0.3 * rng.standard_normal((R, H)).astype(np.float32))
        d["shared"] = from_u16(_f32_bits_to_bf16(S), device)
    else:
        d["shared"] = None
    return d


def _f32_bits_to_bf16(x: np.ndarray) -> np.ndarray:
    """BF16 bit patterns of FP32 values that are exact in BF16 (NaN kept as NaN)."""
    b = np.ascontiguousarray(x, dtype=np.float32).view(np.uint32)
    nan = np.isnan(x)
    assert np.all((b[~nan] & 0xFFFF) == 0), "value not exact in BF16"
    return np.where(nan, (b >> 16) | 0x40, b >> 16).astype(np.uint16)
