"""Every quantizer of the step at the benchmark's full size, in the launch
configuration the benchmark times: bench.MoEStep's own inputs, shapes and calls
(262144 routed rows over 32 experts with Zipf(1.2) loads, hidden 7168,
intermediate 2048).  The outputs are compared bit for bit with the oracle on
sampled rows and, for the column-wise layouts, on sampled channels of sampled
experts, every sampled scale read back through the tiled layouts.

"Composer 2 Technical Report", section 6.1 (NVFP4 per-token forward, MXFP8
backward); "Scaling and Optimizing Frontier Model Training", "MXFP8 expert
kernels" (row-wise and column-wise MXFP8 per expert)."""
import numpy as np
import pytest

from tests.fmetest import bf16_bits_np, padded_rows, sf_index, to_np

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def step(fme):
    import torch

    import bench

    wl = bench.WORKLOADS[bench.DEFAULT_WORKLOAD]
    s = bench.MoEStep(bench.counts_for(wl), wl["seed"], "cuda")
    for call in s.calls():
        call()
    torch.cuda.synchronize()
    code, raw = fme.read_device_status(s.status)
    assert code == 0, raw
    return s


def _sample_rows(off, rng, per_group=3):
    """First, last and a random row of every non-empty expert."""
    rows = []
    for g in range(len(off) - 1):
        lo, hi = int(off[g]), int(off[g + 1])
        if hi > lo:
            rows += [lo, hi - 1, int(rng.integers(lo, hi))][:per_group]
    return np.unique(np.array(rows, np.int64))


def _tiled_rows(sf_flat, prow, c_logical):
    """Logical scale rows [len(prow), c_logical] from the tiled layout."""
    c = np.arange(c_logical)
    return np.asarray(sf_flat)[sf_index(prow[:, None], c[None, :], c_logical)]


def _cols(t, lo, hi, channels):
    """Rows lo..hi-1 of a device tensor restricted to the given columns."""
    import torch

    return t[lo:hi].index_select(1, torch.from_numpy(channels).to(t.device))


def _check_nvfp4(orc, x, q, rows, prow, what):
    import torch

    codes, sf, scale = q
    k = x.shape[1]
    idx = torch.from_numpy(rows).to(x.device)
    xb = bf16_bits_np(x[idx])
    oc, osf, oscale = orc.quant_nvfp4(xb)
    got_codes = to_np(codes[idx])
    got_scale = to_np(scale[idx])
    assert np.array_equal(got_scale.view(np.uint32), oscale.view(np.uint32)), f"{what}: per-token scales differ"
    flat = to_np(sf)
    got_sf = _tiled_rows(flat, prow, k // 16)
    assert np.array_equal(got_sf, osf), f"{what}: block scales differ at {np.argwhere(got_sf != osf)[:5].tolist()}"
    bad = np.argwhere(got_codes != oc)
    assert bad.size == 0, f"{what}: {len(bad)} code bytes differ, first {bad[:5].tolist()}"


def test_full_size_nvfp4_activations(step, orc):
    off = to_np(step.offsets)
    rows = _sample_rows(off, np.random.default_rng(11))
    prow = padded_rows(off)[rows]
    _check_nvfp4(orc, step.x, step.xq, rows, prow, "x")
    _check_nvfp4(orc, step.h, step.hq, rows, prow, "h")


def test_full_size_nvfp4_weights(step, orc):
    rng = np.random.default_rng(12)
    for w, q in ((step.w_gu, step.wguq), (step.w_d, step.wdq)):
        n = w.shape[0]
        # rows at both ends, around a 128-row block boundary in the middle, and random rows
        rows = np.unique(np.concatenate([[0, 1, 31, 32, 127, n - 1], (n // 2) + np.arange(-2, 3),
                                         rng.integers(0, n, size=40)]))
        _check_nvfp4(orc, w, q, rows, rows, f"weights {tuple(w.shape)}")  # one group: padded row = row


def test_full_size_mxfp8_rowwise(step, orc):
    import torch

    off = to_np(step.offsets)
    rows = _sample_rows(off, np.random.default_rng(13))
    idx = torch.from_numpy(rows).to(step.dy.device)
    oc, osf = orc.quant_mxfp8_rows(bf16_bits_np(step.dy[idx]))
    got = to_np(step.dyr[0][idx])
    got_sf = _tiled_rows(to_np(step.dyr[1]), padded_rows(off)[rows], step.H // 32)
    assert np.array_equal(got_sf, osf), "dY row-wise scales differ"
    assert np.array_equal(got, oc), f"dY row-wise codes differ at {np.argwhere(got != oc)[:5].tolist()}"


def _check_cols(orc, x, off, q, ld, channels, groups, what):
    """Column-wise codes and scales of the sampled channels over the sampled groups."""
    import torch

    sel = torch.from_numpy(channels).to(q[0].device)
    codes, sf, poff = to_np(q[0].index_select(0, sel)), to_np(q[1]), to_np(q[2])
    n_ch = x.shape[1]
    expect_poff = np.concatenate([[0], np.cumsum((np.diff(off) + 127) // 128 * 128)])
    assert np.array_equal(poff, expect_poff.astype(np.int32)), f"{what}: padded offsets"
    for g in groups:
        lo, hi = int(off[g]), int(off[g + 1])
        n = hi - lo
        if n == 0:
            continue
        xb = bf16_bits_np(_cols(x, lo, hi, channels))
        oc, osf, opoff = orc.quant_mxfp8_cols(xb, np.array([0, n], np.int32))
        p0, width = int(poff[g]), int(opoff[-1])
        got = codes[:, p0:p0 + width]
        assert np.array_equal(got, oc[:, :width]), f"{what}: expert {g} codes differ"
        blocks = p0 // 32 + np.arange(width // 32)
        got_sf = np.asarray(sf)[sf_index(channels[:, None], blocks[None, :], ld // 32)]
        assert np.array_equal(got_sf, osf[:, : width // 32]), f"{what}: expert {g} scales differ"
    assert channels.max() < n_ch


def test_full_size_mxfp8_columnwise(step, orc):
    off = to_np(step.offsets)
    rng = np.random.default_rng(14)
    counts = np.diff(off)
    live = np.flatnonzero(counts)
    groups = sorted(set([int(live[0]), int(live[-1]), int(np.argmax(counts))] +
                        [int(g) for g in rng.choice(live, size=2, replace=False)]))
    ch_h = np.unique(np.concatenate([[0, 127, 128, step.H - 1], rng.integers(0, step.H, size=4)]))
    _check_cols(orc, step.dy, off, step.dyc, step.ld_r, ch_h, groups, "dY column-wise")
    ch_i = np.unique(np.concatenate([[0, 129, step.I - 1], rng.integers(0, step.I, size=3)]))
    _check_cols(orc, step.h, off, step.hc, step.ld_r, ch_i, groups, "H column-wise")
    # W_down column-wise: one group of E * H rows; 256-row stretches at the first and
    # the last expert's weight block
    import torch

    codes = to_np(step.wdc[0].index_select(0, torch.from_numpy(ch_i).to(step.wdc[0].device)))
    sf = to_np(step.wdc[1])
    for e in (0, step.E - 1):
        lo = e * step.H
        xb = bf16_bits_np(_cols(step.w_d, lo, lo + 256, ch_i))
        oc, osf, _ = orc.quant_mxfp8_cols(xb, np.array([0, 256], np.int32))
        assert np.array_equal(codes[:, lo:lo + 256], oc[:, :256]), f"W_down expert {e} codes differ"
        blocks = lo // 32 + np.arange(8)
        got_sf = sf[sf_index(ch_i[:, None], blocks[None, :], step.ld_w // 32)]
        assert np.array_equal(got_sf, osf[:, :8]), f"W_down expert {e} scales differ"
