"""The per-token formats' invariants at the configurations' own sizes, bit for bit.

"Cursor Composer 2 report deep dive", section 1, and "Composer 2 Technical
Report", section 6.1 (the NVFP4-variant paragraph): scales computed per token
make a token's quantized values independent of the rest of the batch (no batch
variance) and of the tokens after it (no future-token leakage).  Both properties
are checked here end to end on the device:

  * the skewed long batch (262144 routed rows over 32 experts, Zipf(1.2) loads,
    3 empty experts, no count a multiple of 128): future rows are appended to
    every expert -- the empty ones included -- so that each expert's last tile
    gains rows and every later expert's rows and scale tiles move; the original
    rows' NVFP4 codes, block scales and row scales, both forward GEMMs' outputs
    (gate/up, its SwiGLU form's h, and down), and their MXFP8 row-wise codes, scales and dgrad outputs
    must not change by a single bit;
  * the quantizer batch (16384 x 7168, 0.1% hot channels, 1% small rows): a
    seeded permutation and a seeded split into ragged chunks give every row the
    same NVFP4 and MXFP8 row-wise outputs.

Comparisons run on the device (torch.equal on bit views); the oracle parity of
the same calls is covered at these sizes by test_gpu_full_size_quant.py and the
full-size cases of test_gpu_gemm.py."""
import numpy as np
import pytest

from fp8_moe_expert_gb300 import synth
from tests.fmetest import padded_rows

pytestmark = pytest.mark.gpu

FUTURE_ROWS = 4096


def _status():
    import torch

    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _ok(fme, st):
    code, raw = fme.read_device_status(st)
    assert code == 0, f"device status {raw:#x}"


def _logical_sf(sf, prow, c_logical):
    """Tiled scale bytes (device) -> logical [len(prow) x c_logical] (device),
    gathered through the layout formula of include/fme.h."""
    import torch

    pr = torch.as_tensor(prow, dtype=torch.int64, device=sf.device)[:, None]
    c = torch.arange(c_logical, dtype=torch.int64, device=sf.device)[None, :]
    c4 = (c_logical + 3) // 4 * 4
    idx = ((pr // 128) * (c4 // 4) + c // 4) * 512 + (pr % 32) * 16 + ((pr % 128) // 32) * 4 + c % 4
    return sf[idx]


def _same(a, b):
    import torch

    if a.dtype in (torch.bfloat16, torch.float32):
        a, b = a.view(torch.int16 if a.dtype == torch.bfloat16 else torch.int32), \
            b.view(torch.int16 if b.dtype == torch.bfloat16 else torch.int32)
    return torch.equal(a, b)


@pytest.fixture(scope="module")
def extended():
    """The long batch and its extension: counts, future rows per expert, and the
    extended position of every original row."""
    counts = synth.zipf_counts()
    assert (counts == 0).sum() == 3 and sum(counts) == 262144
    rng = np.random.default_rng(44)
    e = len(counts)
    extra = 1 + rng.multinomial(FUTURE_ROWS - e, np.ones(e) / e)   # every expert gains rows
    off = synth.offsets_from_counts(counts)
    off2 = synth.offsets_from_counts(counts + extra)
    pos = np.concatenate([off2[g] + np.arange(counts[g]) for g in range(e)]).astype(np.int64)
    assert len(pos) == off[-1] and off2[-1] == off[-1] + FUTURE_ROWS
    return counts, extra, off, off2, pos


def _extend_rows(x, pos, total_rows, seed, std):
    """x's rows at `pos` of a new [total_rows x k] tensor; the other rows are new
    (loud, so that a leak would show) seeded draws."""
    import torch

    out = synth.torch_normal((total_rows, x.shape[1]), std, seed)
    out[torch.from_numpy(pos).to(x.device)] = x
    return out


def test_future_rows_change_no_earlier_output(fme, extended):
    import torch

    counts, extra, off_np, off2_np, pos_np = extended
    e, hid, inter = len(counts), synth.HIDDEN, synth.INTERMEDIATE
    rows, rows2 = int(off_np[-1]), int(off2_np[-1])
    off = torch.from_numpy(off_np).cuda()
    off2 = torch.from_numpy(off2_np).cuda()
    pos = torch.from_numpy(pos_np).cuda()
    pr1 = padded_rows(off_np)
    pr2 = padded_rows(off2_np)[pos_np]
    st = _status()

    # ---- forward, NVFP4: X -> gate/up
    x = synth.torch_normal((rows, hid), 1.0, 41)
    x2 = _extend_rows(x, pos_np, rows2, 401, 1e3)
    q1 = fme.quantize_nvfp4_pertoken(x, off, status=st)
    q2 = fme.quantize_nvfp4_pertoken(x2, off2, status=st)
    del x, x2
    assert _same(q2[0][pos], q1[0]), "NVFP4 codes of X moved"
    assert _same(q2[2][pos], q1[2]), "NVFP4 row scales of X moved"
    assert torch.equal(_logical_sf(q2[1], pr2, hid // 16), _logical_sf(q1[1], pr1, hid // 16)), \
        "NVFP4 block scales of X moved"
    wgu = fme.quantize_nvfp4_pertoken(synth.torch_normal((e * 2 * inter, hid), 0.02, 42), status=st)
    y1 = fme.grouped_gemm_fwd_nvfp4(*q1, *wgu, off, 2 * inter, hid, status=st)
    y2 = fme.grouped_gemm_fwd_nvfp4(*q2, *wgu, off2, 2 * inter, hid, status=st)
    _ok(fme, st)
    assert _same(y2[pos], y1), "gate/up outputs of the original rows moved"
    del y1, y2
    # the same projection with SwiGLU in the epilogue (h of the original rows)
    h1 = fme.grouped_gemm_fwd_nvfp4_swiglu(*q1, *wgu, off, 2 * inter, hid, status=st)
    h2 = fme.grouped_gemm_fwd_nvfp4_swiglu(*q2, *wgu, off2, 2 * inter, hid, status=st)
    _ok(fme, st)
    assert _same(h2[pos], h1), "SwiGLU outputs of the original rows moved"
    del q1, q2, wgu, h1, h2

    # ---- forward, NVFP4: H -> down
    h = synth.torch_normal((rows, inter), 1.0, 43)
    h2 = _extend_rows(h, pos_np, rows2, 403, 1e3)
    p1 = fme.quantize_nvfp4_pertoken(h, off, status=st)
    p2 = fme.quantize_nvfp4_pertoken(h2, off2, status=st)
    del h, h2
    assert _same(p2[0][pos], p1[0]) and _same(p2[2][pos], p1[2]), "NVFP4 of H moved"
    assert torch.equal(_logical_sf(p2[1], pr2, inter // 16), _logical_sf(p1[1], pr1, inter // 16))
    wd_bf16 = synth.torch_normal((e * hid, inter), 0.02, 44)
    wd = fme.quantize_nvfp4_pertoken(wd_bf16, status=st)
    y1 = fme.grouped_gemm_fwd_nvfp4(*p1, *wd, off, hid, inter, status=st)
    y2 = fme.grouped_gemm_fwd_nvfp4(*p2, *wd, off2, hid, inter, status=st)
    _ok(fme, st)
    assert _same(y2[pos], y1), "down outputs of the original rows moved"
    del p1, p2, wd, y1, y2

    # ---- backward, MXFP8: dY row-wise -> dgrad
    dy = synth.torch_normal((rows, hid), 1e-2, 45)
    dy2 = _extend_rows(dy, pos_np, rows2, 405, 10.0)
    r1 = fme.quantize_mxfp8(dy, fme.ROWWISE, off, status=st)
    r2 = fme.quantize_mxfp8(dy2, fme.ROWWISE, off2, status=st)
    del dy, dy2
    assert _same(r2[0][pos], r1[0]), "MXFP8 codes of dY moved"
    assert torch.equal(_logical_sf(r2[1], pr2, hid // 32), _logical_sf(r1[1], pr1, hid // 32))
    wdc = fme.quantize_mxfp8(wd_bf16, fme.COLWISE, status=st)
    d1 = fme.grouped_gemm_dgrad_mxfp8(r1[0], r1[1], wdc[0], wdc[1], wdc[3], off, inter, hid, status=st)
    d2 = fme.grouped_gemm_dgrad_mxfp8(r2[0], r2[1], wdc[0], wdc[1], wdc[3], off2, inter, hid, status=st)
    _ok(fme, st)
    assert _same(d2[pos], d1), "dgrad outputs of the original rows moved"


@pytest.fixture(scope="module")
def quantizer_batch():
    import torch

    x_bits, _, _ = synth.quantizer_batch()
    assert x_bits.shape == (16384, synth.HIDDEN)
    return torch.from_numpy(x_bits.view(np.int16)).cuda().view(torch.bfloat16)


def _quantize_both(fme, x, st):
    return fme.quantize_nvfp4_pertoken(x, status=st), fme.quantize_mxfp8(x, fme.ROWWISE, status=st)


def _rows_of(q, k, rows_idx, rows_total):
    """codes, row scales and logical scales of the given rows of one call's outputs
    (one group: padded row = row)."""
    (c4, s4, r4), (c8, s8) = q
    return (c4[rows_idx], r4[rows_idx], _logical_sf(s4, rows_idx.cpu().numpy(), k // 16),
            c8[rows_idx], _logical_sf(s8, rows_idx.cpu().numpy(), k // 32))


def test_quantizer_batch_shuffled_and_split(fme, quantizer_batch):
    import torch

    x = quantizer_batch
    rows, k = x.shape
    st = _status()
    ref = _rows_of(_quantize_both(fme, x, st), k, torch.arange(rows, device="cuda"), rows)
    # a seeded permutation
    perm = torch.from_numpy(np.random.default_rng(3).permutation(rows)).cuda()
    got = _rows_of(_quantize_both(fme, x[perm].contiguous(), st), k, torch.arange(rows, device="cuda"), rows)
    for a, b, what in zip(got, ref, ("nvfp4 codes", "row scales", "nvfp4 scales", "mxfp8 codes", "mxfp8 scales")):
        assert _same(a, b[perm]), f"shuffled batch: {what} differ"
    # a seeded split into ragged chunks (sizes 1 .. 3000)
    rng = np.random.default_rng(5)
    cuts = [0]
    while cuts[-1] < rows:
        cuts.append(min(rows, cuts[-1] + int(rng.integers(1, 3000))))
    assert len(cuts) > 8
    for lo, hi in zip(cuts[:-1], cuts[1:]):
        part = _rows_of(_quantize_both(fme, x[lo:hi].contiguous(), st), k, torch.arange(hi - lo, device="cuda"),
                        hi - lo)
        for a, b, what in zip(part, ref, ("nvfp4 codes", "row scales", "nvfp4 scales", "mxfp8 codes",
                                          "mxfp8 scales")):
            assert _same(a, b[lo:hi]), f"chunk [{lo}, {hi}): {what} differ"
    _ok(fme, st)
