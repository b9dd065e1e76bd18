"""Checks that pin the CPU oracle to things other than itself.

Every ``check_*`` function takes an ``oracle.Oracle`` and raises
``AssertionError`` when the oracle disagrees with the fact it pins.  The pins are
library casts (torch, ml_dtypes), the format definitions' closed forms,
hand-worked examples (``tests/golden``), brute force over all codes, and
invariants the pages fix ("Composer 2 Technical Report", section 6.1: a
token's NVFP4 codes and scales do not depend on the rest of the batch and do not
see later tokens).  ``test_oracle_pins.py`` runs them against the oracle, and
``test_oracle_mutants.py`` runs them against deliberately broken copies of it to
show that each plausible mistake fails at least one of them.
"""
from __future__ import annotations

import numpy as np

from fp8_moe_expert_gb300 import synth
from tests.golden import read_cases

E2M1_GRID = [0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0]


def _all_bf16_finite() -> np.ndarray:
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = synth.bf16_float(bits)
    return bits[np.isfinite(vals)]


def _nearest_even(v: float, mags: list[float]) -> int:
    """Brute force: index of the nearest magnitude, ties to the even index."""
    a = abs(v)
    if a >= mags[-1]:
        return len(mags) - 1
    best = min(range(len(mags)), key=lambda i: (abs(mags[i] - a), i % 2))
    return best


# ---------------------------------------------------------------- tables ----
def check_e2m1_decode(orc):
    """All 16 E2M1 codes: the grid {0, .5, 1, 1.5, 2, 3, 4, 6} with a sign bit."""
    got = orc.e2m1_value(np.arange(16))
    want = np.array(E2M1_GRID + [-g for g in E2M1_GRID])
    assert np.array_equal(got, want) and np.signbit(got[8]), (got, want)


def check_e4m3_decode(orc):
    """All 256 E4M3 codes against torch.float8_e4m3fn."""
    import torch

    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = orc.e4m3_value(codes)
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all(), codes[~same]
    assert np.array_equal(np.signbit(got[~np.isnan(got)]), np.signbit(want[~np.isnan(want)]))


def check_e8m0_decode(orc):
    """All 256 E8M0 codes against torch.float8_e8m0fnu."""
    import torch

    codes = np.arange(256, dtype=np.uint8)
    want = torch.from_numpy(codes).view(torch.float8_e8m0fnu).to(torch.float64).numpy()
    got = orc.e8m0_value(codes)
    same = (got == want) | (np.isnan(got) & np.isnan(want))
    assert same.all(), codes[~same]


def check_e4m3_encode_all_bf16(orc):
    """Every finite bf16 value below 464 in magnitude: oracle E4M3 encode equals
    torch's float -> float8_e4m3fn cast (round to nearest even).  At and above 464
    torch overflows to NaN while the oracle saturates to 448 (0x7e / 0xfe)."""
    import torch

    bits = _all_bf16_finite()
    vals = synth.bf16_float(bits).astype(np.float64)
    got = orc.e4m3_encode(vals)
    inr = np.abs(vals) < 464.0
    want = torch.from_numpy(vals[inr].astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    bad = got[inr] != want
    assert not bad.any(), vals[inr][bad][:8]
    sat = got[~inr]
    assert np.all((sat == 0x7E) | (sat == 0xFE)), np.unique(sat)
    assert np.array_equal(sat >> 7, np.signbit(vals[~inr]).astype(np.uint8))


def check_e2m1_encode_all_bf16(orc):
    """Every finite bf16 value: oracle E2M1 encode equals ml_dtypes' float4_e2m1fn
    cast (nearest even, saturating at 6)."""
    import ml_dtypes

    bits = _all_bf16_finite()
    vals = synth.bf16_float(bits)
    got = orc.e2m1_encode(vals.astype(np.float64))
    want = vals.astype(ml_dtypes.float4_e2m1fn).view(np.uint8) & 0xF
    bad = got != want
    assert not bad.any(), vals[bad][:8]


def check_ties_brute_force(orc):
    """Every midpoint between neighbouring magnitudes goes to the even code, and a
    hair either side goes to the nearer one (brute-force nearest search)."""
    e2 = [float(v) for v in E2M1_GRID]
    e4 = [float(v) for v in orc.e4m3_value(np.arange(127))]
    for mags, enc, sign in ((e2, orc.e2m1_encode, 8), (e4, orc.e4m3_encode, 0x80)):
        mids = [(mags[i] + mags[i + 1]) / 2 for i in range(len(mags) - 1)]
        probes = []
        for m, lo, hi in zip(mids, mags[:-1], mags[1:]):
            eps = (hi - lo) * 1e-6
            probes += [m, m - eps, m + eps, -m, -(m - eps), -(m + eps)]
        probes = np.array(probes)
        got = enc(probes)
        want = np.array([_nearest_even(p, mags) | (sign if np.signbit(p) else 0) for p in probes], np.uint8)
        assert np.array_equal(got, want), probes[got != want][:8]


def check_saturation_and_sign(orc):
    for enc, top, sign in ((orc.e2m1_encode, 7, 8), (orc.e4m3_encode, 0x7E, 0x80)):
        got = enc(np.array([1e30, -1e30, 1e6, -1e6, 0.0, -0.0, 1e-30, -1e-30]))
        want = np.array([top, top | sign, top, top | sign, 0, sign, 0, sign], np.uint8)
        assert np.array_equal(got, want), (got, want)


# --------------------------------------------------------- worked examples ---
def _parse_floats(s):
    return np.array([float(v) for v in s.split()], np.float64)


def check_nvfp4_worked(orc):
    for name, case in read_cases("nvfp4_worked.txt").items():
        x = synth.bf16_bits(_parse_floats(case["x"]).astype(np.float32)).reshape(1, 16)
        codes, sf, scale = orc.quant_nvfp4(x)
        s_bits = int(np.array(scale, np.float32).view(np.uint32)[0])
        assert s_bits == int(case["S_bits"], 16), (name, hex(s_bits))
        assert int(sf[0, 0]) == int(case["sf"], 16), (name, hex(int(sf[0, 0])))
        want_codes = [int(c, 16) for c in case["codes"].split()]
        got_codes = [(int(codes[0, j // 2]) >> (4 * (j % 2))) & 0xF for j in range(16)]
        assert got_codes == want_codes, (name, got_codes, want_codes)
        want_packed = [int(c, 16) for c in case["packed"].split()]
        assert [int(c) for c in codes[0]] == want_packed, (name, codes[0])


def check_mxfp8_worked(orc):
    for name, case in read_cases("mxfp8_worked.txt").items():
        lead = _parse_floats(case["x"]).astype(np.float32)
        x = np.zeros(32, np.float32)
        x[: len(lead)] = lead
        xb = synth.bf16_bits(x).reshape(1, 32)
        assert np.array_equal(synth.bf16_float(xb).reshape(-1)[: len(lead)], lead), name
        codes, sf = orc.quant_mxfp8_rows(xb)
        assert int(sf[0, 0]) == int(case["scale"]), (name, int(sf[0, 0]))
        want = [int(c, 16) for c in case["codes"].split()]
        assert [int(c) for c in codes[0, : len(want)]] == want, (name, codes[0, : len(want)])
        tail = codes[0, len(want):]
        assert np.all(tail == 0), (name, tail)


# ---------------------------------------------------- NVFP4 invariants -------
def _rows_with_outliers(rows=64, k=256, seed=11):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((rows, k), dtype=np.float32)
    x[rng.random((rows, k)) < 0.02] *= 40.0
    x[:: 7] *= np.float32(1e-3)
    x[3, 16:32] = 0.0                  # an all-zero block in a non-zero row
    x[5] = 0.0                         # an all-zero row
    x[9, :16] *= np.float32(1e-6)      # a block far below the row amax
    return synth.bf16_bits(x)


def check_nvfp4_batch_invariance(orc):
    """Per-token scales: a row quantized alone, in a shuffled batch, or ahead of
    appended later rows gets identical codes and scales."""
    x = _rows_with_outliers()
    full = orc.quant_nvfp4(x)
    perm = np.random.default_rng(5).permutation(x.shape[0])
    shuf = orc.quant_nvfp4(x[perm])
    for a, b in zip(full, shuf):
        assert np.array_equal(a[perm], b)
    for t in (0, 3, 9, 40):
        one = orc.quant_nvfp4(x[t:t + 1])
        for a, b in zip(full, one):
            assert np.array_equal(a[t:t + 1], b), t
    later = synth.bf16_bits(np.random.default_rng(6).standard_normal((32, x.shape[1]), dtype=np.float32) * 1e4)
    ext = orc.quant_nvfp4(np.concatenate([x, later]))
    for a, b in zip(full, ext):
        assert np.array_equal(a, b[: x.shape[0]])


def check_nvfp4_sign_symmetry(orc):
    """q(-x) = -q(x): negating a row flips exactly the sign bit of every code in
    blocks with a non-zero scale, and changes nothing else."""
    x = _rows_with_outliers()
    neg = x ^ np.uint16(0x8000)
    c1, s1, t1 = orc.quant_nvfp4(x)
    c2, s2, t2 = orc.quant_nvfp4(neg)
    assert np.array_equal(s1, s2) and np.array_equal(t1, t2)
    lo1, hi1 = c1 & 0xF, c1 >> 4
    lo2, hi2 = c2 & 0xF, c2 >> 4
    nib1 = np.stack([lo1, hi1], -1).reshape(x.shape)
    nib2 = np.stack([lo2, hi2], -1).reshape(x.shape)
    live = np.repeat(s1 != 0, 16, axis=1)
    assert np.array_equal(nib1[live] ^ 8, nib2[live])
    assert np.all(nib1[~live] == 0) and np.all(nib2[~live] == 0)


def check_nvfp4_power_of_two_scaling(orc):
    """Scaling a row by 2^j (no under/overflow) scales S_t by 2^j and leaves every
    code and block scale unchanged: each step is an IEEE operation on scaled
    operands."""
    x = _rows_with_outliers()
    f = synth.bf16_float(x)
    for j in (-3, 5):
        xs = synth.bf16_bits(f * np.float32(2.0 ** j))
        c1, s1, t1 = orc.quant_nvfp4(x)
        c2, s2, t2 = orc.quant_nvfp4(xs)
        rows = np.abs(f).max(axis=1) > 1e-2   # keep S_t and d clear of fp32 subnormals
        assert np.array_equal(c1[rows], c2[rows]) and np.array_equal(s1[rows], s2[rows])
        assert np.array_equal(t1[rows] * np.float32(2.0 ** j), t2[rows])


def check_nvfp4_amax_maps_to_six(orc):
    """The row maximum lands in a block whose scale is 448 (0x7e), and every
    block with a normal E4M3 scale maps its own maximum to |code| = 6."""
    x = _rows_with_outliers()
    f = np.abs(synth.bf16_float(x))
    codes, sf, scale = orc.quant_nvfp4(x)
    nib = np.stack([codes & 0xF, codes >> 4], -1).reshape(x.shape)
    for t in range(x.shape[0]):
        if f[t].max() == 0:
            assert scale[t] == 0 and np.all(sf[t] == 0)
            continue
        j = int(np.argmax(f[t]))
        assert sf[t, j // 16] == 0x7E, (t, hex(int(sf[t, j // 16])))
        for b in range(x.shape[1] // 16):
            if sf[t, b] < 0x08:            # subnormal E4M3 scale: coarser steps
                continue
            blk = f[t, 16 * b: 16 * b + 16]
            jb = int(np.argmax(blk))
            assert (nib[t, 16 * b + jb] & 7) == 7, (t, b)


def check_nvfp4_error_bound(orc):
    """|x - x_hat| is at most half a grid step of the E2M1 value, times the block's
    scale e, plus a relative 2^-22 for the fp32 rounding of x/e; saturated
    elements dequantize to exactly +-6e and, in blocks with a normal E4M3 scale,
    lie within 6.5e."""
    x = _rows_with_outliers()
    f = synth.bf16_float(x).astype(np.float64)
    codes, sf, scale = orc.quant_nvfp4(x)
    xh = orc.dequant_nvfp4(codes, sf, scale)
    e = np.repeat(orc.e4m3_value(sf) * scale[:, None].astype(np.float64), 16, axis=1)
    e32 = (orc.e4m3_value(sf).astype(np.float32) * scale[:, None]).astype(np.float64)
    e32 = np.repeat(e32, 16, axis=1)
    live = e > 0
    q = np.abs(f[live] / e32[live])
    step = np.select([q < 2, q < 4], [0.5, 1.0], 2.0)
    err = np.abs(f[live] - xh[live])
    sat = q >= 6
    bound = 0.5 * step * e32[live] * (1 + 2.0 ** -22) + np.abs(f[live]) * 2.0 ** -22
    assert np.all(err[~sat] <= bound[~sat])
    assert np.all(np.abs(xh[live][sat]) == 6 * e[live][sat])
    # a normal E4M3 block scale is within 2^-4 of amax_b / (6 S), so nothing in
    # such a block lies further out than 6 e (1 + 2^-4) / (1 - 2^-4) < 6.5 e
    normal = np.repeat(sf >= 0x08, 16, axis=1)[live]
    assert np.all(np.abs(f[live][normal]) <= 6.5 * e32[live][normal])
    assert np.all(xh[~live] == 0)


def check_nvfp4_exact_grid(orc):
    """A row whose values all lie on the E2M1 grid with amax 6 (S = fl32(6/2688),
    every block scale 448, e = fl32(448 S) = 1 exactly, so every quotient is exact)
    gets the grid codes back, and dequantizes to x * (448 S) exactly."""
    grid = np.array(E2M1_GRID + [-g for g in E2M1_GRID], np.float32)
    row = np.tile(grid, 4)[:64]
    row[0] = 6.0
    xb = synth.bf16_bits(row).reshape(1, -1)
    codes, sf, scale = orc.quant_nvfp4(xb)
    assert np.all(sf == 0x7E)
    nib = np.stack([codes & 0xF, codes >> 4], -1).reshape(-1)
    assert np.array_equal(orc.e2m1_value(nib), row.astype(np.float64))
    xh = orc.dequant_nvfp4(codes, sf, scale)
    assert np.array_equal(xh.reshape(-1), row.astype(np.float64) * (448.0 * float(scale[0])))


# ---------------------------------------------------------- MXFP8 pins -------
def check_mxfp8_rows(orc):
    """Row-wise MXFP8 on random data with outliers and tiny blocks:
      * the scale rule: for a non-zero block, amax / 2^(code-127) lies in [256, 512);
      * elements: code = torch float8_e4m3fn cast of the exact x / X where that is
        below 448 in magnitude, 0x7e / 0xfe where it is 448 or more;
      * error: |x_hat - x| <= 2^-4 |x| in the E4M3 normal range."""
    import torch

    rng = np.random.default_rng(21)
    f = rng.standard_normal((48, 256), dtype=np.float32)
    f[rng.random(f.shape) < 0.01] *= 1000.0
    f[::5] *= np.float32(1e-30)
    f[7, :32] = 0.0
    x = synth.bf16_bits(f)
    fv = synth.bf16_float(x).astype(np.float64)
    codes, sf = orc.quant_mxfp8_rows(x)
    X = np.repeat(np.ldexp(1.0, sf.astype(np.int64) - 127), 32, axis=1)
    blocks = np.abs(fv).reshape(48, 8, 32).max(axis=2)
    nz = blocks > 0
    ratio = blocks[nz] / np.ldexp(1.0, sf[nz].astype(np.int64) - 127)
    assert np.all((ratio >= 256) & (ratio < 512)), ratio.min()
    assert np.all(sf[~nz] == 0)
    q = fv / X
    small = np.abs(q) < 448
    want = torch.from_numpy(q[small].astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes[small], want)
    big = codes[~small]
    assert np.all((big == 0x7E) | (big == 0xFE))
    xh = orc.dequant_mxfp8(codes, sf)
    normal = small & (np.abs(q) >= 2.0 ** -6)
    assert np.all(np.abs(xh[normal] - fv[normal]) <= 2.0 ** -4 * np.abs(fv[normal]))


def check_mxfp8_cols(orc):
    """Column-wise MXFP8 equals row-wise MXFP8 of each group's transposed rows,
    zero-padded to a multiple of 128 positions; padded offsets are the running
    sum of the rounded-up group sizes."""
    rng = np.random.default_rng(31)
    counts = np.array([0, 37, 128, 1, 0, 200, 95])
    off = synth.offsets_from_counts(counts)
    rows = int(off[-1])
    x = synth.bf16_bits(rng.standard_normal((rows, 64), dtype=np.float32) * 3)
    ct, st, poff = orc.quant_mxfp8_cols(x, off)
    want_poff = np.concatenate([[0], np.cumsum((counts + 127) // 128 * 128)])
    assert np.array_equal(poff, want_poff)
    for g in range(len(counts)):
        n = counts[g]
        pad = (n + 127) // 128 * 128
        seg = np.zeros((pad, 64), np.uint16)
        seg[:n] = x[off[g]: off[g] + n]
        rc, rs = orc.quant_mxfp8_rows(np.ascontiguousarray(seg.T))
        assert np.array_equal(ct[:, poff[g]: poff[g] + pad], rc), g
        assert np.array_equal(st[:, poff[g] // 32: (poff[g] + pad) // 32], rs), g


def check_mxfp8_single_group_is_transpose(orc):
    """With one group and rows a multiple of 128, column-wise is row-wise of X^T."""
    rng = np.random.default_rng(32)
    x = synth.bf16_bits(rng.standard_normal((256, 96), dtype=np.float32))
    ct, st, _ = orc.quant_mxfp8_cols(x, np.array([0, 256]))
    rc, rs = orc.quant_mxfp8_rows(np.ascontiguousarray(x.T))
    assert np.array_equal(ct, rc) and np.array_equal(st, rs)


# ----------------------------------------------------------------- GEMM ------
def check_gemm_vs_torch(orc):
    """fp64 GEMM on dequantized operands against torch.matmul in float64."""
    import torch

    rng = np.random.default_rng(41)
    a = rng.standard_normal((7, 48))
    b = rng.standard_normal((5, 48))
    got = orc.gemm_abt(a, b)
    want = (torch.from_numpy(a) @ torch.from_numpy(b).T).numpy()
    assert np.allclose(got, want, rtol=1e-13, atol=1e-13)
    assert got.shape == (7, 5)


def check_gemm_identity(orc):
    """B = I gives Y = A exactly (no transposition, no lost term)."""
    rng = np.random.default_rng(42)
    a = rng.standard_normal((6, 32))
    assert np.array_equal(orc.gemm_abt(a, np.eye(32)), a)
    perm = rng.permutation(32)
    assert np.array_equal(orc.gemm_abt(a, np.eye(32)[perm]), a[:, perm])


def check_quantized_gemm_end_to_end(orc):
    """NVFP4 forward on 16-wide rows whose values lie on the E2M1 grid (block
    scales 448, e = 1, so the codes are the values): the closed form is
    y = (x . w) * (448 S_x) * (448 S_w)."""
    grid = np.array(E2M1_GRID, np.float32)
    xa = np.zeros((2, 16), np.float32)
    xa[0, :8] = grid
    xa[1, :8] = -grid[::-1]
    wa = np.zeros((3, 16), np.float32)
    wa[0, :8] = grid
    wa[1, 8:] = grid
    wa[2, 0] = 6.0
    xb, wb = synth.bf16_bits(xa), synth.bf16_bits(wa)
    ca, sa, ta = orc.quant_nvfp4(xb)
    cb, sb, tb = orc.quant_nvfp4(wb)
    y = orc.gemm_abt(orc.dequant_nvfp4(ca, sa, ta), orc.dequant_nvfp4(cb, sb, tb))
    assert np.all(sa == 0x7E) and np.all(sb[sb != 0] == 0x7E)
    want = (xa.astype(np.float64) @ wa.astype(np.float64).T) * (448.0 * ta[:, None].astype(np.float64)) \
        * (448.0 * tb[None, :].astype(np.float64))
    assert np.allclose(y, want, rtol=1e-14, atol=0), (y, want)


def _swiglu_rows(g, u):
    return synth.bf16_bits(np.concatenate([np.asarray(g, np.float32), np.asarray(u, np.float32)], axis=1))


def check_swiglu_closed_forms(orc):
    """silu(0) = 0; silu(v) - silu(-v) = v (sigma(v) + sigma(-v) = 1), so
    h(g, u) - h(-g, u) = g u; silu(v) -> v for large v and -> 0 for very negative
    v; the bf16 gate and up halves are read from the right half of the row."""
    g = np.array([[0.0, 0.5, -1.25, 3.0, -7.0, 20.0, -30.0, 100.0]], np.float32)
    u = np.array([[1.0, -2.0, 0.75, 1.5, -0.5, 2.0, 4.0, -1.0]], np.float32)
    hp = orc.swiglu(_swiglu_rows(g, u))
    hn = orc.swiglu(_swiglu_rows(-g, u))
    gd, ud = g.astype(np.float64), u.astype(np.float64)
    assert hp[0, 0] == 0.0
    assert np.allclose(hp - hn, gd * ud, rtol=1e-14, atol=1e-300)
    assert abs(hp[0, 7] - gd[0, 7] * ud[0, 7]) < 1e-30 * abs(gd[0, 7])
    assert abs(hp[0, 6]) < 1e-10
    big = orc.swiglu(_swiglu_rows(np.full((1, 4), 88.0), np.full((1, 4), 1.0)))
    assert np.allclose(big, 88.0, rtol=1e-30, atol=1e-30)


def check_swiglu_vs_scipy(orc):
    """fp64 silu(g) * u against scipy's logistic function (another implementation
    of e^-v), on bf16 inputs spanning the range that matters."""
    from scipy.special import expit

    rng = np.random.default_rng(17)
    g = synth.bf16_float(synth.bf16_bits(rng.standard_normal((8, 96)) * 4.0))
    u = synth.bf16_float(synth.bf16_bits(rng.standard_normal((8, 96))))
    h = orc.swiglu(_swiglu_rows(g, u))
    want = g.astype(np.float64) * expit(g.astype(np.float64)) * u.astype(np.float64)
    assert np.allclose(h, want, rtol=4e-16, atol=1e-300)


def check_swiglu_f64(orc):
    """The fp64-input activation: equal to the bf16-input one on bf16 values (same
    definition, other entry); against scipy's logistic function on fp64 values with
    full mantissas; h(g, u) - h(-g, u) = g u on those values too; gate and up read
    from the right halves (a swapped pair changes h, since silu is not odd)."""
    from scipy.special import expit

    rng = np.random.default_rng(23)
    g = synth.bf16_float(synth.bf16_bits(rng.standard_normal((6, 64)) * 4.0))
    u = synth.bf16_float(synth.bf16_bits(rng.standard_normal((6, 64))))
    rows = np.concatenate([g, u], axis=1).astype(np.float64)
    assert np.array_equal(orc.swiglu_f64(rows), orc.swiglu(_swiglu_rows(g, u)))
    gf = rng.standard_normal((5, 48)) * 6.0
    uf = rng.standard_normal((5, 48))
    h = orc.swiglu_f64(np.concatenate([gf, uf], axis=1))
    assert np.allclose(h, gf * expit(gf) * uf, rtol=4e-16, atol=1e-300)
    hn = orc.swiglu_f64(np.concatenate([-gf, uf], axis=1))
    assert np.allclose(h - hn, gf * uf, rtol=1e-13, atol=1e-300)


def check_mxfp8_ceil_scale_brute_force(orc):
    """Round-up scale rule on every positive finite bf16 amax (one 32-block per
    value, the amax in the block's first element): the code is the smallest c
    with amax <= 448 * 2^(c - 127), found by search, clamped at 0; no element
    saturates (every E4M3 code decodes to at most 448 in magnitude, exact x / X
    below 448 is the torch float8_e4m3fn cast); the code is the standard rule's or
    one more."""
    import torch

    bits = _all_bf16_finite()
    vals = synth.bf16_float(bits).astype(np.float64)
    pos = bits[vals > 0]
    pv = synth.bf16_float(pos).astype(np.float64)
    x = np.zeros((len(pos), 32), np.uint16)
    x[:, 0] = pos
    x[:, 1] = synth.bf16_bits(-synth.bf16_float(pos) * np.float32(0.75))
    codes, sf = orc.quant_mxfp8_rows(x, ceil_scale=True)
    c = np.zeros(len(pos), np.int64)
    for k in range(256):                     # c ends as the first k with pv <= 448 * 2^(k-127)
        c[pv > 448.0 * 2.0 ** (k - 127)] = k + 1
    assert np.array_equal(sf[:, 0].astype(np.int64), c)
    _, sf_std = orc.quant_mxfp8_rows(x)
    d = sf[:, 0].astype(np.int64) - sf_std[:, 0].astype(np.int64)
    assert np.all((d == 0) | (d == 1))
    q = synth.bf16_float(x[:, :2]).astype(np.float64) / np.ldexp(1.0, sf[:, :1].astype(np.int64) - 127)
    assert np.all(np.abs(q) <= 448.0)
    want = torch.from_numpy(q.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    assert np.array_equal(codes[:, :2], want)


def check_mxfp8_ceil_scale_worked(orc):
    """Worked values: amax 448 -> code 127 (X = 1); 450 -> 128; 3.0 -> 120 (as the
    standard rule); 3.75 -> 121 where the standard rule's 120 saturates 3.75 * 128
    = 480 to 448; the column-wise quantizer follows the same rule along tokens."""
    x = np.zeros((4, 32), np.float32)
    x[0, 3], x[1, 0], x[2, 5], x[3, 31] = 448.0, -450.0, 3.0, 3.75
    xb = synth.bf16_bits(x)
    codes, sf = orc.quant_mxfp8_rows(xb, ceil_scale=True)
    assert sf[:, 0].tolist() == [127, 128, 120, 121]
    assert orc.e4m3_value(codes[3, 31:32])[0] == 240.0
    _, sf_std = orc.quant_mxfp8_rows(xb)
    assert sf_std[3, 0] == 120
    ct, st, _ = orc.quant_mxfp8_cols(np.ascontiguousarray(xb.T), np.array([0, 32]), ceil_scale=True)
    assert st[:, 0].tolist() == [127, 128, 120, 121]


def check_nvfp4_pertensor_special_cases(orc):
    """Standard NVFP4 is the per-token variant when the tensor is one row, or when
    every row has the tensor's amax; its scale is fl32(amax_tensor / 2688) (numpy
    binary32 division) in every row."""
    x, _, _ = synth.quantizer_batch(rows=24, cols=512, seed=41)
    one = x[5:6]
    assert all(np.array_equal(a, b) for a, b in zip(orc.quant_nvfp4_pertensor(one), orc.quant_nvfp4(one)))
    same = x.copy()
    big = synth.bf16_bits(np.float32(-4.0) * np.abs(synth.bf16_float(x)).max())
    same[:, 7] = big
    assert all(np.array_equal(a, b) for a, b in zip(orc.quant_nvfp4_pertensor(same), orc.quant_nvfp4(same)))
    _, _, scale = orc.quant_nvfp4_pertensor(x)
    amax = np.abs(synth.bf16_float(x)).max()
    assert np.all(scale.view(np.uint32) == (np.float32(amax) / np.float32(2688.0)).view(np.uint32))


def check_nvfp4_pertensor_batch_variance(orc):
    """The reason for the per-token variant: with one scale per tensor a row's codes
    change when a row with a larger amax joins the batch (here appended last, so
    a later token changes earlier tokens' codes), while the per-token codes of the
    same rows do not."""
    x, _, small = synth.quantizer_batch(rows=32, cols=256, seed=43)
    loud = synth.bf16_bits(synth.bf16_float(x[:1]) * np.float32(64.0))
    both = np.concatenate([x, loud])
    c0, s0, _ = orc.quant_nvfp4_pertensor(x)
    c1, s1, _ = orc.quant_nvfp4_pertensor(both)
    assert not np.array_equal(c1[:32], c0) and not np.array_equal(s1[:32], s0)
    p0, ps0, _ = orc.quant_nvfp4(x)
    p1, ps1, _ = orc.quant_nvfp4(both)
    assert np.array_equal(p1[:32], p0) and np.array_equal(ps1[:32], ps0)


def check_swiglu_bwd_finite_differences(orc):
    """The backward is the derivative of the forward: dg / (dh u) against central
    differences of silu (scipy's logistic function, fp64, step 1e-5), and
    du / dh against silu itself, on bf16 inputs over the range that matters."""
    from scipy.special import expit

    rng = np.random.default_rng(31)
    g = synth.bf16_float(synth.bf16_bits(rng.standard_normal((4, 64)) * 4.0))
    u = synth.bf16_float(synth.bf16_bits(rng.standard_normal((4, 64))))
    dh = synth.bf16_float(synth.bf16_bits(rng.standard_normal((4, 64))))
    d = orc.swiglu_bwd(_swiglu_rows(g, u), synth.bf16_bits(dh))
    gd, ud, hd = (a.astype(np.float64) for a in (g, u, dh))
    silu = lambda v: v * expit(v)  # noqa: E731
    eps = 1e-5
    dsilu = (silu(gd + eps) - silu(gd - eps)) / (2 * eps)
    assert np.allclose(d[:, :64], hd * ud * dsilu, rtol=1e-7, atol=1e-9)
    assert np.allclose(d[:, 64:], hd * silu(gd), rtol=1e-14, atol=1e-300)


def check_swiglu_bwd_closed_forms(orc):
    """silu'(0) = 1/2 and silu(0) = 0; silu' -> 1 and silu(g) -> g for large g, both
    -> 0 for very negative g; u = 0 gives dg = 0; silu' changes sign between
    g = -1.2734375 and -1.28515625 (its root is near -1.2785); the gate and up
    halves of the gradient are [dg | du]."""
    g = np.array([[0.0, 0.0, 60.0, -60.0, 2.5, -1.2734375, -1.28515625, 1.0]], np.float32)
    u = np.array([[1.5, -2.0, 0.75, 3.0, 0.0, 1.0, 1.0, -1.0]], np.float32)
    dh = np.array([[1.0, 0.5, -2.0, 1.0, 4.0, 1.0, 1.0, 2.0]], np.float32)
    d = orc.swiglu_bwd(_swiglu_rows(g, u), synth.bf16_bits(dh))
    dg, du = d[0, :8], d[0, 8:]
    assert dg[0] == 0.75 and dg[1] == -0.5 and du[0] == 0.0 and du[1] == 0.0
    assert abs(dg[2] - (-1.5)) < 1e-20 and abs(du[2] - (-120.0)) < 1e-20
    assert abs(dg[3]) < 1e-20 and abs(du[3]) < 1e-20
    assert dg[4] == 0.0 and du[4] != 0.0
    assert dg[5] > 0.0 > dg[6] and abs(dg[5]) < 1e-2 and abs(dg[6]) < 1e-2
    assert np.isclose(du[7], 2.0 * 1.0 / (1.0 + np.exp(-1.0)), rtol=1e-15)


# --------------------------------------------------------------- routing ----
def check_route_vs_stable_argsort(orc):
    """Grouping = numpy's stable argsort of the ids (another sort algorithm);
    offsets = the prefix sums of numpy's bincount; row_of inverts src_row."""
    ids, _ = synth.topk_routing(tokens=3000, top_k=6, experts=40, seed=21)
    offsets, row_of, src_row = orc.route(ids, 40)
    flat = ids.ravel()
    want_src = np.argsort(flat, kind="stable")
    assert np.array_equal(src_row, want_src)
    want_off = np.concatenate([[0], np.cumsum(np.bincount(flat, minlength=40))])
    assert np.array_equal(offsets, want_off)
    assert np.array_equal(row_of.ravel()[src_row], np.arange(flat.size))
    assert np.all(flat[src_row][:-1] <= flat[src_row][1:])


def check_route_brute_force(orc):
    """Every id pattern of 2 tokens x top-2 over 3 experts (81 cases): grouped
    row r holds the r-th assignment in the order of the pairs (id, a), found by
    Python's sorted."""
    import itertools

    for pat in itertools.product(range(3), repeat=4):
        ids = np.array(pat, np.int32).reshape(2, 2)
        offsets, row_of, src_row = orc.route(ids, 3)
        want = [a for _, a in sorted((e, a) for a, e in enumerate(pat))]
        assert list(src_row) == want, pat
        assert list(offsets) == [0, pat.count(0), pat.count(0) + pat.count(1), 4]
        for r, a in enumerate(want):
            assert row_of.ravel()[a] == r


def check_route_invalid_and_empty(orc):
    """Ids outside [0, E) take no grouped row and get row_of = -1; experts with no
    assignment have empty ranges; zero tokens give zero offsets."""
    ids = np.array([[3, -1], [0, 7], [3, 0]], np.int32)
    offsets, row_of, src_row = orc.route(ids, 5)
    assert list(offsets) == [0, 2, 2, 2, 4, 4]
    assert row_of.tolist() == [[2, -1], [0, -1], [3, 1]]
    assert list(src_row[:4]) == [2, 5, 0, 4]
    off0, _, _ = orc.route(np.zeros((0, 4), np.int32), 3)
    assert list(off0) == [0, 0, 0, 0]


def _combine(orc, y_vals, row_of, w):
    y = synth.bf16_bits(np.asarray(y_vals, np.float32))
    return synth.bf16_float(orc.combine(y, np.asarray(row_of, np.int32), np.asarray(w, np.float32)))


def check_combine_closed_forms(orc):
    """Hand-worked fp32 cases, one column each, rounded once to bf16 at the end:
    one-hot weight returns the row; the sum is taken in fp32 (exact sum
    1 + 2^-8 + 2^-30 rounds up in bf16, the fp32 running sum sits on the tie and
    goes to even); in k order (1 - 1 + 2^-30 is 2^-30, 1 + 2^-30 - 1 is 0); each
    product rounded before the add ((1 + 2^-23)(1 + 2^-7) loses its 2^-30);
    skipped entries (row_of < 0); the bf16 rounding ties to even."""
    t = 2.0 ** -30
    cases = [
        # (y rows [r x 1], row_of [1 x k], weights [1 x k], expected)
        ([[5.0], [-3.25]], [[1, 0]], [[1.0, 0.0]], -3.25),
        ([[1.0], [2.0 ** -8], [t]], [[0, 1, 2]], [[1.0, 1.0, 1.0]], 1.0),
        ([[1.0], [-1.0], [t]], [[0, 1, 2]], [[1.0, 1.0, 1.0]], t),
        ([[1.0], [t], [-1.0]], [[0, 1, 2]], [[1.0, 1.0, 1.0]], 0.0),
        ([[-(1.0 + 2.0 ** -7)], [1.0 + 2.0 ** -7]], [[0, 1]], [[1.0, 1.0 + 2.0 ** -23]], 2.0 ** -23),
        ([[2.0], [7.0]], [[-1, 1]], [[9.0, 0.5]], 3.5),
        ([[1.0], [3.0 * 2.0 ** -8]], [[0, 1]], [[1.0, 1.0]], 1.0 + 2.0 ** -6),
        ([[1.0], [2.0 ** -8]], [[0, 1]], [[1.0, 1.0]], 1.0),
        ([[1.0 + 2.0 ** -7], [2.0 ** -8]], [[0, 1]], [[1.0, 1.0]], 1.0 + 2.0 ** -6),
    ]
    for y, ro, w, want in cases:
        got = _combine(orc, y, ro, w)
        assert got.shape == (1, 1) and got[0, 0] == np.float32(want), (y, ro, w, got, want)


def check_combine_error_bound(orc):
    """Random routed outputs: the result is within half a bf16 ulp of the fp32
    sum, which is within top_k * 2^-24 * sum |w y| of the exact (fp64) sum."""
    ids, w = synth.topk_routing(tokens=200, top_k=8, experts=16, seed=23)
    offsets, row_of, _ = orc.route(ids, 16)
    y = synth.normal_bits((int(offsets[-1]), 64), 1.0, seed=24)
    out = synth.bf16_float(orc.combine(y, row_of, w)).astype(np.float64)
    yv = synth.bf16_float(y).astype(np.float64)
    gathered = yv[row_of]  # [tokens, top_k, n]
    exact = np.einsum("tk,tkn->tn", w.astype(np.float64), gathered)
    mag = np.einsum("tk,tkn->tn", np.abs(w.astype(np.float64)), np.abs(gathered))
    fp32_err = 8 * 2.0 ** -24 * mag
    half_ulp = np.exp2(np.floor(np.log2(np.maximum(np.abs(exact) + fp32_err, 1e-30))) - 8)
    assert np.all(np.abs(out - exact) <= half_ulp + fp32_err * 1.01 + 1e-30)
    y_rows = yv[row_of[5, 3]]
    single = synth.bf16_float(orc.combine(y, row_of[5:6, 3:4], np.ones((1, 1), np.float32)))
    assert np.array_equal(single[0], y_rows.astype(np.float32))


ALL_CHECKS = [v for k, v in sorted(globals().items()) if k.startswith("check_")]
