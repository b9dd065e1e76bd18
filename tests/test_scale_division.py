"""The per-token scale S = fl32(amax / 2688) is computed on the GPU without a
division: q = fl32(amax r) with r = fl32(1/2688), then S = fl32(q + (amax - q 2688) r)
on fused multiply-adds.  Here that claim is checked for every positive finite bf16
amax with exact rational arithmetic (each step rounded once to binary32, subnormals
included) against numpy's correctly rounded binary32 division.  No GPU involved; the
GPU tests check the device's results against the oracle for the same values."""
from fractions import Fraction

import numpy as np


def _rn32(x: Fraction) -> Fraction:
    """Round to the nearest binary32 value, ties to even (subnormals included)."""
    if x == 0:
        return Fraction(0)
    sign = -1 if x < 0 else 1
    m = abs(x)
    e = m.numerator.bit_length() - m.denominator.bit_length()
    if Fraction(2) ** e > m:
        e -= 1
    elif Fraction(2) ** (e + 1) <= m:
        e += 1
    quantum = Fraction(2) ** (max(e, -126) - 23)
    n = m / quantum
    whole = n.numerator // n.denominator
    rest = n - whole
    if rest > Fraction(1, 2) or (rest == Fraction(1, 2) and whole % 2 == 1):
        whole += 1
    return sign * whole * quantum


def test_scale_without_division_matches_ieee_for_every_bf16_amax():
    bits = np.arange(1 << 16, dtype=np.uint32)
    vals = (bits << 16).astype(np.uint32).view(np.float32)
    amax = vals[np.isfinite(vals) & (vals > 0)]
    r = Fraction(float(np.float32(1.0) / np.float32(2688.0)))
    c = Fraction(2688)
    want = (amax / np.float32(2688.0)).astype(np.float32)
    for a, w in zip(amax, want):
        fa = Fraction(float(a))
        q = _rn32(fa * r)
        res = _rn32(fa - q * c)
        s = _rn32(q + res * r)
        assert float(s) == float(w), (float(a), float(s), float(w))
