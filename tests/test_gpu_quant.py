"""Quantizers on the GPU against the CPU oracle: codes and scales bit-exact.

Workloads: the tiny one-expert case, the 16384 x 7168 heterogeneous quantizer
batch, and edge shapes (ragged groups, empty groups, zero rows and blocks,
subnormal and tiny inputs, saturating outliers).  Invariants from "Composer 2
Technical Report" section 6.1 (per-token scales: no dependence on the rest of
the batch, no leakage from later tokens) are checked on the GPU bit for bit.
"""
import numpy as np
import pytest

from fp8_moe_expert_gb300 import synth
from tests.fmetest import bf16_tensor, to_np, unswizzle
from tests.golden import read_cases

pytestmark = pytest.mark.gpu


def _dev_offsets(offsets):
    import torch

    return None if offsets is None else torch.from_numpy(np.asarray(offsets, np.int32)).cuda()


def _status():
    import torch

    return torch.zeros(1, dtype=torch.int32, device="cuda")


def run_nvfp4(fme, x_bits, offsets=None):
    import torch

    x = bf16_tensor(x_bits)
    st = _status()
    codes, sf, scale = fme.quantize_nvfp4_pertoken(x, _dev_offsets(offsets), status=st)
    code, raw = fme.read_device_status(st)
    assert code == 0, raw
    rows, k = x_bits.shape
    return to_np(codes), unswizzle(to_np(sf), rows, k // 16, offsets), to_np(scale)


def check_nvfp4(fme, orc, x_bits, offsets=None):
    codes, sf, scale = run_nvfp4(fme, x_bits, offsets)
    oc, osf, oscale = orc.quant_nvfp4(x_bits)
    assert np.array_equal(scale.view(np.uint32), oscale.view(np.uint32)), "per-token scales differ"
    assert np.array_equal(sf, osf), f"block scales differ at {np.argwhere(sf != osf)[:5].tolist()}"
    bad = np.argwhere(codes != oc)
    assert bad.size == 0, f"{len(bad)} code bytes differ, first {bad[:5].tolist()}"
    return codes, sf, scale


def run_mx_rows(fme, x_bits, offsets=None):
    x = bf16_tensor(x_bits)
    st = _status()
    codes, sf = fme.quantize_mxfp8(x, fme.ROWWISE, _dev_offsets(offsets), status=st)
    assert fme.read_device_status(st)[0] == 0
    rows, cols = x_bits.shape
    return to_np(codes), unswizzle(to_np(sf), rows, cols // 32, offsets)


def run_mx_cols(fme, x_bits, offsets):
    x = bf16_tensor(x_bits)
    st = _status()
    codes, sf, poff, ld = fme.quantize_mxfp8(x, fme.COLWISE, _dev_offsets(offsets), status=st)
    assert fme.read_device_status(st)[0] == 0
    cols = x_bits.shape[1]
    return to_np(codes), unswizzle(to_np(sf), cols, ld // 32), to_np(poff), ld


def check_mx_rows(fme, orc, x_bits, offsets=None):
    codes, sf = run_mx_rows(fme, x_bits, offsets)
    oc, osf = orc.quant_mxfp8_rows(x_bits)
    assert np.array_equal(sf, osf), f"scales differ at {np.argwhere(sf != osf)[:5].tolist()}"
    bad = np.argwhere(codes != oc)
    assert bad.size == 0, f"{len(bad)} codes differ, first {bad[:5].tolist()}"


def check_mx_cols(fme, orc, x_bits, offsets):
    codes, sf, poff, ld = run_mx_cols(fme, x_bits, offsets)
    oc, osf, opoff = orc.quant_mxfp8_cols(x_bits, offsets, ld=ld)
    assert np.array_equal(poff, opoff)
    p = int(opoff[-1])
    assert np.array_equal(sf[:, : p // 32], osf[:, : p // 32]), "column-wise scales differ"
    bad = np.argwhere(codes[:, :p] != oc[:, :p])
    assert bad.size == 0, f"{len(bad)} codes differ, first {bad[:5].tolist()}"


# ------------------------------------------------------------------- NVFP4 --
def test_nvfp4_worked_examples(fme, orc):
    """The hand-worked rows of tests/golden, each embedded in a 64-wide row of zeros."""
    cases = read_cases("nvfp4_worked.txt")
    rows = []
    for case in cases.values():
        r = np.zeros(64, np.float32)
        r[:16] = [float(v) for v in case["x"].split()]
        rows.append(r)
    x_bits = synth.bf16_bits(np.stack(rows))
    codes, sf, scale = run_nvfp4(fme, x_bits)
    for i, case in enumerate(cases.values()):
        assert int(scale[i:i + 1].view(np.uint32)[0]) == int(case["S_bits"], 16)
        assert int(sf[i, 0]) == int(case["sf"], 16)
        assert [int(c) for c in codes[i, :8]] == [int(c, 16) for c in case["packed"].split()]
        assert np.all(codes[i, 8:] == 0) and np.all(sf[i, 1:] == 0)


def test_nvfp4_tiny(fme, orc):
    x, w = synth.tiny(0)
    check_nvfp4(fme, orc, x)
    check_nvfp4(fme, orc, w)


def test_nvfp4_quantizer_batch(fme, orc):
    x, _, _ = synth.quantizer_batch()
    check_nvfp4(fme, orc, x)


@pytest.mark.parametrize("rows", [1, 31, 32, 33, 127, 128, 129])
@pytest.mark.parametrize("k", [64, 192, 2048, 8192])
def test_nvfp4_edge_shapes(fme, orc, rows, k):
    rng = np.random.default_rng(rows * 1000 + k)
    f = rng.standard_normal((rows, k), dtype=np.float32)
    f[rng.random(f.shape) < 0.01] *= 500.0
    if rows > 3:
        f[1] = 0.0                                # zero row
        f[2] *= np.float32(2.0 ** -140)           # bf16 subnormals
        f[3, : min(k, 48)] = 0.0                  # zero blocks
    check_nvfp4(fme, orc, synth.bf16_bits(f))


def test_nvfp4_groups_pad_scale_rows(fme, orc):
    counts = np.array([0, 1, 127, 128, 129, 0, 300, 0])
    off = synth.offsets_from_counts(counts)
    rng = np.random.default_rng(7)
    x = synth.bf16_bits(rng.standard_normal((int(off[-1]), 256), dtype=np.float32))
    check_nvfp4(fme, orc, x, off)


def test_nvfp4_every_bf16_amax(fme, orc):
    """Row r holds the r-th positive finite bf16 value (subnormals included) and a
    few smaller ones: every per-token scale S = amax/2688, every 6 S and the block
    scale of the amax block, over the whole bf16 range, bit-exact."""
    mags = np.arange(1, 0x7F80, dtype=np.uint32)            # +subnormals .. +max finite
    x = np.zeros((mags.size, 64), np.uint16)
    x[:, 0] = mags
    x[:, 1] = 0x8000 | (mags >> 1)                          # negative, about half the magnitude
    x[:, 17] = mags >> 3                                    # second block
    x[:, 40] = np.maximum(mags, 1) - 1
    check_nvfp4(fme, orc, x)


def test_nvfp4_exact_ties(fme, orc):
    """Quotients exactly on rounding midpoints, where round-to-nearest-even decides:
    amax = 2688 * 2^j makes S = 2^j and 6 S exact; the amax block has scale 448 so
    x = 448 m 2^j sits on the E2M1 midpoint m; a block with amax 6.375 * 2^j
    divides to 1.0625, an E4M3 midpoint."""
    mids = [0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0]
    rows = []
    for j in range(-20, 21, 3):
        r = np.zeros(64, np.float32)
        r[0] = 2688.0 * 2.0 ** j
        for i, m in enumerate(mids):
            r[1 + i] = 448.0 * m * 2.0 ** j * (-1 if i % 2 else 1)
        r[16] = 6.375 * 2.0 ** j
        r[17:24] = [6.375 * 2.0 ** j * v for v in (0.5, 0.25, 0.75, 0.125, -0.375, 0.0625, -1.0)]
        r[32] = 3.1875 * 2.0 ** j                      # 3.1875 / 6 = 0.53125: between E4M3 grid points
        r[33] = -448.0 * 5.0 * 2.0 ** j / 2.0 ** 4
        rows.append(r)
    x = synth.bf16_bits(np.stack(rows))
    assert np.array_equal(synth.bf16_float(x), np.stack(rows)), "the tie values must be exact in bf16"
    check_nvfp4(fme, orc, x)


def near_midpoint_rows():
    """Rows for every normal bf16 row amax (32512 rows, k = 2048): block 0 holds the
    amax, blocks 1..127 a block amax chosen for E4M3 block scales spread over 1..126.
    Every block's other elements are the bf16 values just below and just above m e
    for each E2M1 midpoint m (e the block's decode scale, from the E4M3 rounding of
    fl32(amax_b / fl32(6 S))), signs alternating, plus a -0: quotients as close to
    the E2M1 code boundaries as bf16 inputs get."""
    import torch

    mags = np.arange(0x0080, 0x7F80, dtype=np.uint32)
    amax = (mags << 16).view(np.float32)
    s_t = (amax / np.float32(2688.0)).astype(np.float32)
    d = (np.float32(6.0) * s_t).astype(np.float32)
    nblk = 128
    target = np.round(np.linspace(1, 126, nblk - 1)).astype(np.uint8)
    dec = torch.from_numpy(target).view(torch.float8_e4m3fn).float().numpy().astype(np.float64)
    want_b = np.minimum(dec[None, :] * d[:, None].astype(np.float64), amax[:, None].astype(np.float64))
    amax_b = np.concatenate([amax[:, None], synth.bf16_float(synth.bf16_bits(want_b.astype(np.float32)))], axis=1)
    amax_b = np.minimum(amax_b, amax[:, None])
    q = np.minimum((amax_b / d[:, None]).astype(np.float32), np.float32(448.0))
    sb_val = torch.from_numpy(q).to(torch.float8_e4m3fn).float().numpy()
    e = (sb_val * s_t[:, None]).astype(np.float32)
    mids = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    t = (e[..., None].astype(np.float64) * mids).astype(np.float32)     # [rows, blocks, 7]
    lo = (t.view(np.uint32) >> 16).astype(np.uint16)                   # bf16 at or below
    hi = lo + 1
    blk = np.empty(e.shape + (16,), np.uint16)
    blk[..., 0] = synth.bf16_bits(amax_b)
    blk[..., 1:8] = lo ^ np.array([0, 0x8000] * 3 + [0], np.uint16)
    blk[..., 8:15] = hi ^ np.array([0x8000, 0] * 3 + [0x8000], np.uint16)
    blk[..., 15] = 0x8000
    return blk.reshape(mags.size, nblk * 16)


def test_nvfp4_near_midpoints_every_amax(fme, orc):
    """Element codes, block scales and per-token scales bit-exact on the rows of
    near_midpoint_rows: where the division-free element coding would first go wrong."""
    check_nvfp4(fme, orc, near_midpoint_rows())


def test_near_midpoint_rows_are_hard():
    """The generator does what it says: most blocks have the intended scale and
    elements whose quotients sit within 2^-7 of an E2M1 midpoint (CPU only)."""
    pytest.importorskip("torch")
    x = near_midpoint_rows()
    assert x.shape == (32512, 2048)
    v = synth.bf16_float(x).reshape(32512, 128, 16).astype(np.float64)
    amax_b = np.abs(v).max(axis=2)
    assert np.array_equal(amax_b[:, 0], np.abs(v[:, 0, 0]))
    assert (np.abs(v[..., 1:15]) <= amax_b[..., None]).all()
    assert (x.reshape(32512, 128, 16)[..., 15] == 0x8000).all()


def test_nvfp4_batch_invariance_and_causality(fme, orc):
    """Per-token scales: shuffling, splitting and appending later rows leave every
    row's codes and scales bit-identical."""
    x, _, _ = synth.quantizer_batch(rows=2048)
    full = run_nvfp4(fme, x)
    perm = np.random.default_rng(3).permutation(x.shape[0])
    shuf = run_nvfp4(fme, x[perm])
    for a, b in zip(full, shuf):
        assert np.array_equal(a[perm], b)
    cuts = [0, 1, 700, 701, 1500, 2048]
    for lo, hi in zip(cuts[:-1], cuts[1:]):
        part = run_nvfp4(fme, x[lo:hi])
        for a, b in zip(full, part):
            assert np.array_equal(a[lo:hi], b)
    later = synth.normal_bits((512, x.shape[1]), 1e3, seed=9)
    ext = run_nvfp4(fme, np.concatenate([x, later]))
    for a, b in zip(full, ext):
        assert np.array_equal(a, b[: x.shape[0]])


def test_nvfp4_deterministic(fme):
    x, _, _ = synth.quantizer_batch(rows=1024)
    a = run_nvfp4(fme, x)
    b = run_nvfp4(fme, x)
    for u, v in zip(a, b):
        assert np.array_equal(u, v)


# ------------------------------------------------------------------- MXFP8 --
def test_mxfp8_worked_examples(fme):
    cases = read_cases("mxfp8_worked.txt")
    rows = []
    for case in cases.values():
        r = np.zeros(32, np.float32)
        lead = [float(v) for v in case["x"].split()]
        r[: len(lead)] = lead
        rows.append(r)
    codes, sf = run_mx_rows(fme, synth.bf16_bits(np.stack(rows)))
    for i, case in enumerate(cases.values()):
        want = [int(c, 16) for c in case["codes"].split()]
        assert int(sf[i, 0]) == int(case["scale"]), case
        assert [int(c) for c in codes[i, : len(want)]] == want, case


def test_mxfp8_rows_tiny(fme, orc):
    x, w = synth.tiny(0)
    check_mx_rows(fme, orc, x)
    check_mx_rows(fme, orc, w)


def test_mxfp8_rows_quantizer_batch(fme, orc):
    x, _, _ = synth.quantizer_batch()
    check_mx_rows(fme, orc, x)


@pytest.mark.parametrize("rows,cols", [(1, 32), (33, 96), (129, 1056), (257, 7168)])
def test_mxfp8_rows_edges(fme, orc, rows, cols):
    rng = np.random.default_rng(rows + cols)
    f = rng.standard_normal((rows, cols), dtype=np.float32)
    f[rng.random(f.shape) < 0.02] *= 1e4
    f[0, :32] = 0.0
    if rows > 2:
        f[2] *= np.float32(2.0 ** -135)
    counts = np.array([rows // 3, 0, rows - rows // 3])
    check_mx_rows(fme, orc, synth.bf16_bits(f), synth.offsets_from_counts(counts))


def test_mxfp8_cols_quantizer_batch(fme, orc):
    x, _, _ = synth.quantizer_batch()
    counts = synth.dirichlet_counts(rows=x.shape[0], seed=1)
    check_mx_cols(fme, orc, x, synth.offsets_from_counts(counts))


@pytest.mark.parametrize("counts", [[1], [128], [0, 5, 0], [37, 0, 200, 1, 129], [0, 0, 0]])
def test_mxfp8_cols_edges(fme, orc, counts):
    off = synth.offsets_from_counts(counts)
    rng = np.random.default_rng(len(counts) + int(off[-1]))
    f = rng.standard_normal((int(off[-1]), 256), dtype=np.float32)
    f[rng.random(f.shape) < 0.02] *= 300.0
    x = synth.bf16_bits(f)
    if off[-1] == 0:
        codes, sf, poff, ld = run_mx_cols(fme, x, off)
        assert np.all(poff == 0)
        return
    check_mx_cols(fme, orc, x, off)


@pytest.mark.parametrize("counts", [[16384], [37, 0, 200, 1, 129], [4000, 3000, 0, 9384]])
def test_mxfp8_rowcol_fused_matches_oracle(fme, orc, counts):
    """One-pass row-wise + column-wise quantization equals the oracle both ways."""
    off = synth.offsets_from_counts(counts)
    x, _, _ = synth.quantizer_batch(rows=int(off[-1]), cols=1024, seed=5)
    st = _status()
    (rc, rs), (cc, cs, poff, ld) = fme.quantize_mxfp8_rowcol(bf16_tensor(x), _dev_offsets(off), status=st)
    assert fme.read_device_status(st)[0] == 0
    oc, osf = orc.quant_mxfp8_rows(x)
    assert np.array_equal(to_np(rc), oc)
    assert np.array_equal(unswizzle(to_np(rs), x.shape[0], 1024 // 32, off), osf)
    occ, ocs, opoff = orc.quant_mxfp8_cols(x, off, ld=ld)
    p = int(opoff[-1])
    assert np.array_equal(to_np(poff), opoff)
    assert np.array_equal(to_np(cc)[:, :p], occ[:, :p])
    assert np.array_equal(unswizzle(to_np(cs), 1024, ld // 32)[:, : p // 32], ocs[:, : p // 32])


def test_mxfp8_rows_cols_deterministic(fme):
    x, _, _ = synth.quantizer_batch(rows=512)
    off = synth.offsets_from_counts([100, 0, 412])
    assert all(np.array_equal(a, b) for a, b in zip(run_mx_rows(fme, x, off), run_mx_rows(fme, x, off)))
    a, b = run_mx_cols(fme, x, off), run_mx_cols(fme, x, off)
    p = int(a[2][-1])
    assert np.array_equal(a[0][:, :p], b[0][:, :p]) and np.array_equal(a[1][:, : p // 32], b[1][:, : p // 32])


def test_bad_offsets_set_device_status(fme):
    import torch

    x = bf16_tensor(synth.normal_bits((64, 256), 1.0, seed=1))
    st = _status()
    bad = torch.tensor([0, 40, 30, 64], dtype=torch.int32, device="cuda")
    fme.quantize_nvfp4_pertoken(x, bad, status=st)
    code, raw = fme.read_device_status(st)
    assert raw & fme.DEV_BAD_OFFSETS and code == 7
    st.zero_()
    short = torch.tensor([0, 10, 20], dtype=torch.int32, device="cuda")   # does not reach rows
    fme.quantize_mxfp8(x, fme.COLWISE, short, status=st)
    assert fme.read_device_status(st)[1] & fme.DEV_BAD_OFFSETS


# ------------------------------------------------ standard NVFP4 (per tensor) --
def run_nvfp4_pertensor(fme, x_bits, offsets=None):
    x = bf16_tensor(x_bits)
    st = _status()
    codes, sf, scale, amax = fme.quantize_nvfp4_pertensor(x, _dev_offsets(offsets), status=st)
    code, raw = fme.read_device_status(st)
    assert code == 0, raw
    rows, k = x_bits.shape
    return to_np(codes), unswizzle(to_np(sf), rows, k // 16, offsets), to_np(scale), float(to_np(amax)[0])


@pytest.mark.parametrize("case", ["tiny", "batch", "groups", "one_row", "zeros"])
def test_nvfp4_pertensor_matches_oracle(fme, orc, case):
    off = None
    if case == "tiny":
        x, _ = synth.tiny(0)
    elif case == "batch":
        x, _, _ = synth.quantizer_batch(rows=4096)
    elif case == "groups":
        off = synth.offsets_from_counts([37, 0, 200, 1, 129])
        x, _, _ = synth.quantizer_batch(rows=int(off[-1]), cols=2048, seed=3)
    elif case == "one_row":
        x, _, _ = synth.quantizer_batch(rows=1, cols=7168, seed=4)
    else:
        x = np.zeros((64, 512), np.uint16)
    codes, sf, scale, amax = run_nvfp4_pertensor(fme, x, off)
    oc, osf, oscale = orc.quant_nvfp4_pertensor(x)
    assert amax == float(np.abs(synth.bf16_float(x)).max())
    assert np.array_equal(scale.view(np.uint32), oscale.view(np.uint32))
    assert np.array_equal(sf, osf)
    assert np.array_equal(codes, oc)


def test_nvfp4_pertensor_batch_variance_on_gpu(fme):
    """A louder row joining the batch changes the other rows' standard-NVFP4 codes
    and leaves their per-token codes alone."""
    x, _, _ = synth.quantizer_batch(rows=512, cols=1024, seed=8)
    loud = synth.bf16_bits(synth.bf16_float(x[:1]) * np.float32(64.0))
    both = np.concatenate([x, loud])
    a = run_nvfp4_pertensor(fme, x)
    b = run_nvfp4_pertensor(fme, both)
    assert not np.array_equal(a[0], b[0][:512])
    pa, pb = run_nvfp4(fme, x), run_nvfp4(fme, both)
    assert np.array_equal(pa[0], pb[0][:512]) and np.array_equal(pa[1], pb[1][:512])


# ------------------------------------------------ MXFP8, round-up scale rule --
def test_mxfp8_ceil_rows_and_cols(fme, orc):
    """Both quantizers with FME_MX_SCALE_CEIL against the oracle's round-up rule,
    on the heterogeneous batch (ragged groups for the column-wise one)."""
    off = synth.offsets_from_counts([300, 0, 129, 1, 594])
    x, _, _ = synth.quantizer_batch(rows=int(off[-1]), cols=1024, seed=12)
    st = _status()
    codes, sf = fme.quantize_mxfp8(bf16_tensor(x), fme.ROWWISE | fme.MX_SCALE_CEIL, _dev_offsets(off), status=st)
    ct, cs, poff, ld = fme.quantize_mxfp8(bf16_tensor(x), fme.COLWISE | fme.MX_SCALE_CEIL, _dev_offsets(off),
                                         status=st)
    assert fme.read_device_status(st)[0] == 0
    oc, osf = orc.quant_mxfp8_rows(x, ceil_scale=True)
    assert np.array_equal(to_np(codes), oc)
    assert np.array_equal(unswizzle(to_np(sf), x.shape[0], 1024 // 32, off), osf)
    occ, ocs, opoff = orc.quant_mxfp8_cols(x, off, ld=ld, ceil_scale=True)
    p = int(opoff[-1])
    assert np.array_equal(to_np(poff), opoff)
    assert np.array_equal(to_np(ct)[:, :p], occ[:, :p])
    assert np.array_equal(unswizzle(to_np(cs), 1024, ld // 32)[:, : p // 32], ocs[:, : p // 32])
    # the standard rule differs from it somewhere on this batch
    std, _ = fme.quantize_mxfp8(bf16_tensor(x), fme.ROWWISE, _dev_offsets(off), status=st)
    assert not np.array_equal(to_np(std), to_np(codes))


def test_mxfp8_ceil_every_bf16_amax(fme, orc):
    """Every positive finite bf16 value as a block's amax (with a -0.75x partner)."""
    bits = np.arange(1 << 16, dtype=np.uint32).astype(np.uint16)
    vals = synth.bf16_float(bits)
    pos = bits[np.isfinite(vals) & (vals > 0)]
    x = np.zeros((len(pos), 32), np.uint16)
    x[:, 0] = pos
    x[:, 9] = synth.bf16_bits(-synth.bf16_float(pos) * np.float32(0.75))
    st = _status()
    codes, sf = fme.quantize_mxfp8(bf16_tensor(x), fme.ROWWISE | fme.MX_SCALE_CEIL, status=st)
    assert fme.read_device_status(st)[0] == 0
    oc, osf = orc.quant_mxfp8_rows(x, ceil_scale=True)
    assert np.array_equal(unswizzle(to_np(sf), len(pos), 1), osf)
    assert np.array_equal(to_np(codes), oc)
