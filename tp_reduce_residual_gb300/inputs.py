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
