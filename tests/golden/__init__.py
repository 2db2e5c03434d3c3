"""Loader for the hand-worked text fixtures in this folder."""
from __future__ import annotations

import os

import numpy as np

HERE = os.path.dirname(os.path.abspath(__file__))


def load(name: str) -> dict:
    """Parse ``key: v v v`` lines (``#`` starts a comment) into floats / lists."""
    d: dict = {}
    with open(os.path.join(HERE, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, vals = line.split(":", 1)
            nums = [float(v) for v in vals.split()]
            d[key.strip()] = nums[0] if len(nums) == 1 else np.array(nums, dtype=np.float64)
    return d


def stack(d: dict, prefix: str, shape) -> np.ndarray:
    """Gather ``prefix[i,j]`` (or ``prefix[i]``) rows into an array of ``shape``."""
    out = np.zeros(shape, dtype=np.float64)
    for key, v in d.items():
        if not key.startswith(prefix + "["):
            continue
        idx = tuple(int(i) for i in key[len(prefix) + 1:-1].split(","))
        out[idx] = v
    return out
