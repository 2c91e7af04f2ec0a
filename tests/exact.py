"""Exact-arithmetic helpers for pinning the oracle (Python fractions).

Independent of the oracle's C code: fp32 rounding is done here by searching
the neighbouring fp32 values of an exact rational.
"""
from fractions import Fraction

import numpy as np


def f32_rn(x: Fraction) -> np.float32:
    """Nearest fp32 to the exact rational x, ties to even (normal range)."""
    if x == 0:
        return np.float32(0.0)
    c = np.float32(float(x))          # within one ulp of the answer
    cands = [np.nextafter(c, np.float32(-np.inf)), c, np.nextafter(c, np.float32(np.inf))]
    best = None
    for v in cands:
        d = abs(Fraction(float(v)) - x)
        if best is None or d < best[0] or (d == best[0] and (int(np.float32(v).view(np.uint32)) & 1) == 0):
            best = (d, v)
    return np.float32(best[1])


def fma32(a, b, c) -> np.float32:
    """fp32 fused multiply-add with one rounding, by exact arithmetic."""
    r = Fraction(float(np.float32(a))) * Fraction(float(np.float32(b))) + Fraction(float(np.float32(c)))
    if r == 0:
        # IEEE: exact zero sum of opposite signs is +0 in round-to-nearest
        return np.float32(0.0)
    return f32_rn(r)
