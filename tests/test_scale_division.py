"""Division-free quotients in the NVFP4 quantizer, checked on the CPU.

1. The per-token scale S = fl32(amax / 2688) is computed on the GPU without a
   division: q = fl32(amax r) with r = fl32(1/2688), then S = fl32(q + (amax - q 2688) r)
   on fused multiply-adds.  Checked for every positive finite bf16 amax with exact
   rational arithmetic (each step rounded once to binary32, subnormals included)
   against numpy's correctly rounded binary32 division.
2. The element codes E2M1(fl32(x / e)) come from one negated correction step after
   an approximate reciprocal (see ``quotient_check.c``): checked exhaustively over
   every row amax, block scale and bf16 x, for every reciprocal within four ulps of
   1/e, by a C program using the C library's correctly rounded fmaf.

No GPU involved; the GPU tests check the device's results against the oracle."""
import os
import shutil
import subprocess
from fractions import Fraction

import numpy as np
import pytest

_HERE = os.path.dirname(os.path.abspath(__file__))


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


def _build_checker() -> str:
    out_dir = os.path.join(_HERE, "_build")
    os.makedirs(out_dir, exist_ok=True)
    exe = os.path.join(out_dir, "quotient_check")
    src = os.path.join(_HERE, "quotient_check.c")
    base = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math", "-o", exe, src, "-lm"]
    env = dict(os.environ, TMPDIR=out_dir)  # gcc's intermediates stay in the tree
    if subprocess.run(base[:1] + ["-fopenmp"] + base[1:], capture_output=True, env=env).returncode != 0:
        subprocess.run(base, check=True, env=env)  # no OpenMP: one thread, same result
    return exe


@pytest.mark.skipif(shutil.which("gcc") is None, reason="needs gcc")
def test_e2m1_correction_step_is_the_ieee_quotient_exhaustively():
    exe = _build_checker()
    # reciprocals within 4 ulps of 1/e (rcp.approx is documented within 1);
    # every 2999-th row amax also over all small quotients and negative x
    res = subprocess.run([exe, "4", "2999"], capture_output=True, text=True, timeout=900)
    line = res.stdout.strip().splitlines()[-1]
    fields = dict(kv.split("=") for kv in line.split())
    assert int(fields["mismatches"]) == 0, line
    # 32639 amax x ~126 scales x 9 reciprocals x ~600 x in [2^-4, 8]
    assert int(fields["checked"]) > 2_000_000_000, line
    assert res.returncode == 0
