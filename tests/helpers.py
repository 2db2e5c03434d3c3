"""Comparison helpers shared by the tests (BF16 bits as numpy uint16)."""
from __future__ import annotations

import numpy as np
import torch


def f32_from_bf16(u: np.ndarray) -> np.ndarray:
    """Exact widening of BF16 bit patterns."""
    return (np.asarray(u, dtype=np.uint16).astype(np.uint32) << 16).view(np.float32)


def bf16_torch(x) -> np.ndarray:
    """Round to BF16 with PyTorch's conversion (an independent rounding routine)."""
    t = torch.as_tensor(np.asarray(x, dtype=np.float32)).to(torch.bfloat16)
    return t.view(torch.int16).numpy().view(np.uint16)


def bf16_bits(values) -> np.ndarray:
    """BF16 bit patterns of values that are exactly representable in BF16."""
    x = np.asarray(values, dtype=np.float32)
    bits = x.view(np.uint32)
    assert np.all((bits & 0xFFFF) == 0), "value not exact in BF16"
    return (bits >> 16).astype(np.uint16)


def ulp_key(u: np.ndarray) -> np.ndarray:
    """Monotone integer map of BF16 bits: adjacent values differ by 1, +0 == -0."""
    u = np.asarray(u, dtype=np.uint16).astype(np.int32)
    mag = u & 0x7FFF
    return np.where(u & 0x8000, -mag, mag)


def is_nan_bf16(u: np.ndarray) -> np.ndarray:
    u = np.asarray(u, dtype=np.uint16)
    return ((u & 0x7F80) == 0x7F80) & ((u & 0x007F) != 0)


def bf16_ulp_diff(a: np.ndarray, b: np.ndarray) -> np.ndarray:
    """Per-element distance in BF16 ulps; 0 where both are NaN, large where one is."""
    na, nb = is_nan_bf16(a), is_nan_bf16(b)
    d = np.abs(ulp_key(a) - ulp_key(b))
    d = np.where(na & nb, 0, d)
    d = np.where(na ^ nb, 1 << 20, d)
    return d


def assert_bf16_close(actual: np.ndarray, expected: np.ndarray, max_ulp: int = 1, what: str = ""):
    d = bf16_ulp_diff(actual, expected)
    worst = int(d.max()) if d.size else 0
    if worst > max_ulp:
        idx = np.unravel_index(int(d.argmax()), d.shape)
        raise AssertionError(
            f"{what}: {int((d > max_ulp).sum())} of {d.size} elements beyond {max_ulp} BF16 ulp; "
            f"worst {worst} at {idx}: actual {f32_from_bf16(actual[idx])} "
            f"expected {f32_from_bf16(expected[idx])}")


def assert_bits_equal(actual: np.ndarray, expected: np.ndarray, what: str = ""):
    a = np.ascontiguousarray(actual)
    e = np.ascontiguousarray(expected)
    assert a.shape == e.shape, (what, a.shape, e.shape)
    ai = a.view(np.uint32) if a.dtype == np.float32 else a.view(np.uint16)
    ei = e.view(np.uint32) if e.dtype == np.float32 else e.view(np.uint16)
    bad = ai != ei
    # a NaN equals any NaN (its sign and payload are not part of the result)
    if a.dtype == np.float32:
        bad &= ~(np.isnan(a) & np.isnan(e))
    else:
        bad &= ~(is_nan_bf16(ai) & is_nan_bf16(ei))
    if bad.any():
        idx = np.unravel_index(int(np.argmax(bad)), bad.shape)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements differ; first at "
                             f"{idx}: actual {a[idx]!r} expected {e[idx]!r}")


SUBNORMAL_STEP = 2.0 ** -149  # the FP32 subnormal spacing


def assert_rel_close(actual: np.ndarray, expected: np.ndarray, rtol: float, what: str = "",
                     floor: float = SUBNORMAL_STEP):
    """Within rtol relative where the expected value is finite, or within the
    absolute ``floor`` where that is larger (by default one FP32 subnormal
    step, 2^-149: expected values in or near the subnormal range, whose
    rounding grid is coarser than rtol); identical infinities and NaN == NaN
    elsewhere."""
    a = np.asarray(actual, dtype=np.float64)
    e = np.asarray(expected, dtype=np.float64)
    fin = np.isfinite(e)
    same = (np.isnan(a) & np.isnan(e)) | (np.isinf(e) & (a == e))
    if not np.all(same | fin):
        idx = np.unravel_index(int(np.argmax(~(same | fin))), e.shape)
        raise AssertionError(f"{what}: expected {e[idx]} at {idx}, got {a[idx]}")
    a, e = a[fin], e[fin]
    if not np.all(np.isfinite(a)):
        raise AssertionError(f"{what}: a non-finite value where the expected one is finite")
    err = np.abs(a - e)
    over = err / np.maximum(rtol * np.abs(e), floor)
    if over.size and over.max() > 1.0:
        i = int(over.argmax())
        raise AssertionError(f"{what}: error {err[i]:.3e} (relative {err[i] / max(abs(e[i]), 1e-300):.3e})"
                             f" > max({rtol:.1e} relative, {floor:.3e}) at finite element {i}: "
                             f"{a[i]!r} vs {e[i]!r}")
