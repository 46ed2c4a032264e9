"""Test-side numerics: the bf16 tolerance and bf16 bit handling.

Nothing here computes a GEMM; it only states how close a bf16 result must be
to the fp64 oracle and converts between bf16 bit patterns and fp64.
"""
from __future__ import annotations

import math

import numpy as np


def bf16_bits_to_f64(bits: np.ndarray) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to fp64."""
    u32 = bits.astype(np.uint32) << np.uint32(16)
    return u32.view(np.float32).astype(np.float64)


def f64_to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """Round fp64 -> fp32 -> bf16 (each round-to-nearest-even); returns bits.

    Only used where the values are exact in bf16 (integer-valued tests and the
    hand-worked fixture), so the double rounding never matters there.
    """
    f = np.asarray(x, dtype=np.float32)
    u = f.view(np.uint32).astype(np.uint64)
    lsb = (u >> np.uint64(16)) & np.uint64(1)
    r = (u + np.uint64(0x7FFF) + lsb) >> np.uint64(16)
    return r.astype(np.uint16)


def ulp_bf16(ref: np.ndarray) -> np.ndarray:
    """bf16 unit in the last place at |ref|: 2**(e - 7), e = floor(log2|ref|).

    e is clamped to >= -126 (bf16 shares fp32's exponent range); ref == 0
    gives 2**-133, so only the additive term of the tolerance counts there.
    """
    ref = np.asarray(ref, dtype=np.float64)
    _, e2 = np.frexp(np.abs(ref))          # |ref| = m * 2**e2, m in [0.5, 1)
    e = np.maximum(e2.astype(np.int64) - 1, -126)
    out = np.ldexp(1.0, e - 7)
    return np.where(ref == 0.0, 2.0 ** -133, out)


def gemm_tolerance(ref: np.ndarray, K: int) -> np.ndarray:
    """Per-element bound |d - ref| <= ulp_bf16(ref) + 1e-3 * sqrt(K / 64)."""
    return ulp_bf16(ref) + 1e-3 * math.sqrt(max(K, 0) / 64.0)


def assert_gemm_close(d_bits: np.ndarray, ref: np.ndarray, K: int, what: str = ""):
    """Asserts every element of a bf16 result is within the GEMM tolerance."""
    d = bf16_bits_to_f64(np.asarray(d_bits))
    ref = np.asarray(ref, dtype=np.float64).reshape(d.shape)
    err = np.abs(d - ref)
    tol = gemm_tolerance(ref, K)
    bad = err > tol
    if bad.any():
        idx = np.argwhere(bad)
        first = tuple(idx[0])
        raise AssertionError(
            f"{what}: {int(bad.sum())} of {bad.size} elements outside tolerance; "
            f"first at {first}: got {d[first]!r}, ref {ref[first]!r}, "
            f"tol {tol[first]!r}; max err/tol {float((err / tol).max()):.3g}")
