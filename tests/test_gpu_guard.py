"""Guard bands around every output of every call: nothing is written outside the
buffers the header describes, and nothing inside them that the header says is
left alone.

Each output is carved out of a larger device buffer whose 4 KiB on either side
and whose own bytes start as a fill pattern (0xA5).  After the call:
  * the 4 KiB on both sides still hold the pattern (no write before or after);
  * in tiled scale buffers, the bytes of padding rows (each group's rows past its
    last real row, up to the 128-row boundary) still hold the pattern, and a
    row's padding columns (C <= c < C4) hold 0 (include/fme.h, "Scale-factor
    layout");
  * column-wise codes and scales of positions at or past the last expert's padded
    end P_G still hold the pattern, and padding positions inside an expert's
    128-position range hold code 0.
Cases: ragged groups with empty experts, 1024 groups (most of them empty), the
smallest and odd widths (MXFP8 row-wise with cols / 32 = 3), one-row inputs.
This stands in for a memory checker on a pool where compute-sanitizer is closed;
no kernel is made to fault."""
import numpy as np
import pytest

from fp8_moe_expert_gb300 import synth
from tests.fmetest import bf16_tensor, padded_rows, sf_index

pytestmark = pytest.mark.gpu

GUARD = 4096
PAT = 0xA5


class Guarded:
    """A device buffer of `nbytes` with GUARD bytes of pattern on both sides."""

    def __init__(self, nbytes):
        import torch

        self.nbytes = int(nbytes)
        self.buf = torch.full((self.nbytes + 2 * GUARD,), PAT, dtype=torch.uint8, device="cuda")

    def view(self, shape, dtype):
        import torch

        t = self.buf[GUARD:GUARD + self.nbytes].view(dtype)
        return t.view(shape) if shape is not None else t

    @property
    def body(self) -> np.ndarray:
        return self.buf[GUARD:GUARD + self.nbytes].cpu().numpy()

    def check_guards(self, what):
        host = self.buf.cpu().numpy()
        lo, hi = host[:GUARD], host[GUARD + self.nbytes:]
        assert (lo == PAT).all(), f"{what}: {int((lo != PAT).sum())} bytes written before the buffer"
        assert (hi == PAT).all(), f"{what}: {int((hi != PAT).sum())} bytes written after the buffer"


def out(shape, dtype):
    import torch

    n = int(np.prod(shape)) * torch.empty((), dtype=dtype).element_size()
    g = Guarded(n)
    return g, g.view(shape, dtype)


def sf_out(nbytes):
    import torch

    g = Guarded(max(nbytes, 16))
    return g, g.view(None, torch.uint8)


def check_tiled(g, offsets, c_logical, what):
    """Guards, then: written exactly the real rows' scale bytes and their padding
    columns (as 0); padding rows untouched."""
    g.check_guards(what)
    body = g.body
    pr = padded_rows(np.asarray(offsets, np.int64))
    c4 = (c_logical + 3) // 4 * 4
    real = sf_index(pr[:, None], np.arange(c_logical)[None, :], c_logical).ravel()
    pad_cols = sf_index(pr[:, None], np.arange(c_logical, c4)[None, :], c_logical).ravel()
    touched = np.zeros(body.size, bool)
    touched[real] = True
    touched[pad_cols] = True
    assert (body[~touched] == PAT).all(), f"{what}: {int((body[~touched] != PAT).sum())} padding-row bytes written"
    if pad_cols.size:
        assert (body[pad_cols] == 0).all(), f"{what}: padding columns not 0"


def check_colwise(gc, gs, counts, cols, ld, what):
    """Column-wise codes [cols x ld] and scales: positions >= P_G untouched, padding
    positions inside each expert's range 0."""
    gc.check_guards(what + " codes")
    gs.check_guards(what + " scales")
    codes = gc.body.reshape(cols, ld)
    pads = (np.asarray(counts) + 127) // 128 * 128
    p_end = int(pads.sum())
    assert (codes[:, p_end:] == PAT).all(), f"{what}: codes written past the last expert"
    start = 0
    for n, p in zip(counts, pads):
        assert (codes[:, start + n:start + p] == 0).all(), f"{what}: padding positions not 0"
        start += p
    # scales: a [cols x ld/32] tiled matrix, one group; columns past P_G / 32 untouched
    c_logical = ld // 32
    pr = np.arange(cols)
    live = sf_index(pr[:, None], np.arange(p_end // 32)[None, :], c_logical).ravel()
    touched = np.zeros(gs.nbytes, bool)
    touched[live] = True
    body = gs.body
    assert (body[~touched] == PAT).all(), f"{what}: scale bytes written past the last expert"


CASES = {
    # name: (counts per group, k)
    "ragged_with_empty": ([0, 130, 0, 1, 169, 0], 448),
    "one_row": ([1], 64),
    "many_groups": ([0] * 500 + [3] * 20 + [0] * 480 + [257] + [0] * 23, 256),
}


def _offsets(counts):
    import torch

    return torch.from_numpy(synth.offsets_from_counts(np.asarray(counts))).cuda()


@pytest.mark.parametrize("case", sorted(CASES))
def test_nvfp4_quantizers_stay_inside(fme, case):
    import torch

    counts, k = CASES[case]
    rows = int(sum(counts))
    g = len(counts)
    off = _offsets(counts)
    x = bf16_tensor(synth.normal_bits((rows, k), 1.0, seed=rows + k))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gc, codes = out((rows, k // 2), torch.uint8)
    gs, sf = sf_out(fme.sf_bytes(rows, k, 16, g))
    gr, rs = out((rows,), torch.float32)
    fme.quantize_nvfp4_pertoken(x, off, codes=codes, sf=sf, row_scale=rs, status=st)
    gc.check_guards("nvfp4 codes")
    gr.check_guards("nvfp4 row scales")
    check_tiled(gs, synth.offsets_from_counts(np.asarray(counts)), k // 16, "nvfp4 scales")
    # standard NVFP4 (per-tensor), with its amax word guarded too
    gc, codes = out((rows, k // 2), torch.uint8)
    gs, sf = sf_out(fme.sf_bytes(rows, k, 16, g))
    gr, rs = out((rows,), torch.float32)
    ga, amax = out((1,), torch.float32)
    fme.quantize_nvfp4_pertensor(x, off, codes=codes, sf=sf, row_scale=rs, tensor_amax=amax, status=st)
    for gg, w in ((gc, "codes"), (gr, "row scales"), (ga, "amax")):
        gg.check_guards("per-tensor " + w)
    check_tiled(gs, synth.offsets_from_counts(np.asarray(counts)), k // 16, "per-tensor scales")
    # fused SwiGLU: gate/up [rows x 2k] -> h [rows x k] and its NVFP4
    gu = bf16_tensor(synth.normal_bits((rows, 2 * k), 1.0, seed=rows + 2 * k))
    gc, codes = out((rows, k // 2), torch.uint8)
    gs, sf = sf_out(fme.sf_bytes(rows, k, 16, g))
    gr, rs = out((rows,), torch.float32)
    gh, h = out((rows, k), torch.bfloat16)
    fme.swiglu_quantize_nvfp4(gu, off, codes=codes, sf=sf, row_scale=rs, h=h, status=st)
    for gg, w in ((gc, "codes"), (gr, "row scales"), (gh, "h")):
        gg.check_guards("swiglu " + w)
    check_tiled(gs, synth.offsets_from_counts(np.asarray(counts)), k // 16, "swiglu scales")
    assert fme.read_device_status(st)[0] == 0


@pytest.mark.parametrize("case,cols", [("ragged_with_empty", 96), ("ragged_with_empty", 256), ("one_row", 32),
                                       ("many_groups", 128)])
def test_mxfp8_quantizers_stay_inside(fme, case, cols):
    import torch

    counts, _ = CASES[case]
    rows = int(sum(counts))
    g = len(counts)
    off = _offsets(counts)
    off_np = synth.offsets_from_counts(np.asarray(counts))
    x = bf16_tensor(synth.normal_bits((rows, cols), 1.0, seed=rows + cols + 1))
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    gc, codes = out((rows, cols), torch.uint8)
    gs, sf = sf_out(fme.sf_bytes(rows, cols, 32, g))
    fme.quantize_mxfp8(x, fme.ROWWISE, off, codes=codes, sf=sf, status=st)
    gc.check_guards("mxfp8 row codes")
    check_tiled(gs, off_np, cols // 32, "mxfp8 row scales")
    if cols % 128 == 0:
        ld = fme.colwise_ld(rows, g)
        gc, ccodes = out((cols, ld), torch.uint8)
        gs, csf = sf_out(fme.sf_bytes(cols, ld, 32, 1))
        gp, poff = out((g + 1,), torch.int32)
        fme.quantize_mxfp8(x, fme.COLWISE, off, codes=ccodes, sf=csf, padded_offsets=poff, status=st)
        gp.check_guards("padded offsets")
        check_colwise(gc, gs, counts, cols, ld, "mxfp8 column-wise")
        # both layouts in one pass
        grc, rcodes = out((rows, cols), torch.uint8)
        grs, rsf = sf_out(fme.sf_bytes(rows, cols, 32, g))
        gc, ccodes = out((cols, ld), torch.uint8)
        gs, csf = sf_out(fme.sf_bytes(cols, ld, 32, 1))
        gp, poff = out((g + 1,), torch.int32)
        fme.quantize_mxfp8_rowcol(x, off, row_codes=rcodes, row_sf=rsf, col_codes=ccodes, col_sf=csf,
                                  padded_offsets=poff, status=st)
        grc.check_guards("rowcol row codes")
        gp.check_guards("rowcol padded offsets")
        check_tiled(grs, off_np, cols // 32, "rowcol row scales")
        check_colwise(gc, gs, counts, cols, ld, "rowcol column-wise")
        # the SwiGLU backward (cols = 2 inter) with its bf16 gradient out
        inter = cols // 2
        if inter % 128 == 0:
            dh = bf16_tensor(synth.normal_bits((rows, inter), 0.05, seed=rows + 7))
            grc, rcodes = out((rows, cols), torch.uint8)
            grs, rsf = sf_out(fme.sf_bytes(rows, cols, 32, g))
            gc, ccodes = out((cols, ld), torch.uint8)
            gs, csf = sf_out(fme.sf_bytes(cols, ld, 32, 1))
            gp, poff = out((g + 1,), torch.int32)
            gd, dgu = out((rows, cols), torch.bfloat16)
            fme.swiglu_backward_quantize_mxfp8(x, dh, off, row_codes=rcodes, row_sf=rsf, col_codes=ccodes,
                                               col_sf=csf, padded_offsets=poff, d_gate_up=dgu, status=st)
            for gg, w in ((grc, "row codes"), (gp, "padded offsets"), (gd, "d(gate/up)")):
                gg.check_guards("swiglu backward " + w)
            check_tiled(grs, off_np, cols // 32, "swiglu backward row scales")
            check_colwise(gc, gs, counts, cols, ld, "swiglu backward column-wise")
    assert fme.read_device_status(st)[0] == 0


@pytest.mark.parametrize("case", ["ragged_with_empty", "one_row", "many_groups"])
def test_gemms_stay_inside(fme, case):
    import torch

    counts, _ = CASES[case]
    rows = int(sum(counts))
    e = len(counts)
    n, k = 256, 256
    off = _offsets(counts)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    x = bf16_tensor(synth.normal_bits((rows, k), 1.0, seed=31))
    w = bf16_tensor(synth.normal_bits((e * n, k), 0.02, seed=32))
    a = fme.quantize_nvfp4_pertoken(x, off, status=st)
    b = fme.quantize_nvfp4_pertoken(w, status=st)
    gy, y = out((rows, n), torch.bfloat16)
    fme.grouped_gemm_fwd_nvfp4(*a, *b, off, n, k, y=y, status=st)
    gy.check_guards("forward NVFP4 y")
    gh, h = out((rows, n // 2), torch.bfloat16)
    fme.grouped_gemm_fwd_nvfp4_swiglu(*a, *b, off, n, k, h=h, status=st)
    gh.check_guards("forward NVFP4 SwiGLU h")
    am = fme.quantize_mxfp8(x, fme.ROWWISE, off, status=st)
    bm = fme.quantize_mxfp8(w, fme.ROWWISE, status=st)
    gy, y = out((rows, n), torch.bfloat16)
    fme.grouped_gemm_fwd_mxfp8(*am, *bm, off, n, k, y=y, status=st)
    gy.check_guards("forward MXFP8 y")
    # dgrad: B = column-wise MXFP8 of the stacked [e k x n] weights
    wt = bf16_tensor(synth.normal_bits((e * k, n), 0.02, seed=33))
    bc = fme.quantize_mxfp8(wt, fme.COLWISE, status=st)
    gy, y = out((rows, k), torch.bfloat16)
    dy = bf16_tensor(synth.normal_bits((rows, n), 0.01, seed=34))
    dyr = fme.quantize_mxfp8(dy, fme.ROWWISE, off, status=st)
    fme.grouped_gemm_dgrad_mxfp8(dyr[0], dyr[1], bc[0], bc[1], bc[3], off, k, n, y=y, status=st)
    gy.check_guards("dgrad y")
    # wgrad (bf16 out and fp32 accumulate): dW_e [n x k] over each expert's rows
    dyc = fme.quantize_mxfp8(dy, fme.COLWISE, off, status=st)
    xc = fme.quantize_mxfp8(x, fme.COLWISE, off, status=st)
    gy, y = out((e, n, k), torch.bfloat16)
    fme.grouped_gemm_wgrad_mxfp8(dyc[0], dyc[1], dyc[3], xc[0], xc[1], xc[3], dyc[2], n, k, y=y, status=st)
    gy.check_guards("wgrad y")
    gy, y = out((e, n, k), torch.float32)
    y.zero_()
    fme.grouped_gemm_wgrad_mxfp8_accumulate(dyc[0], dyc[1], dyc[3], xc[0], xc[1], xc[3], dyc[2], n, k, y, status=st)
    gy.check_guards("wgrad accumulate")
    assert fme.read_device_status(st)[0] == 0


@pytest.mark.parametrize("tokens,top_k,experts", [(1, 1, 1), (300, 8, 32), (2048, 4, 1024)])
def test_routing_stays_inside(fme, tokens, top_k, experts):
    import torch

    ids_np, w_np = synth.topk_routing(tokens=tokens, top_k=top_k, experts=experts, seed=tokens + 5)
    ids = torch.from_numpy(ids_np).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    go, off = out((experts + 1,), torch.int32)
    grw, row_of = out((tokens, top_k), torch.int32)
    gsr, src = out((tokens * top_k,), torch.int32)
    gw, ws = out((fme.route_workspace_bytes(tokens, top_k, experts),), torch.uint8)
    fme.moe_route(ids, experts, offsets=off, row_of=row_of, src_row=src, workspace=ws, status=st)
    for gg, what in ((go, "offsets"), (grw, "row_of"), (gsr, "src_row"), (gw, "workspace")):
        gg.check_guards("moe_route " + what)
    k = 256
    x = bf16_tensor(synth.normal_bits((tokens, k), 1.0, seed=tokens + 6))
    rows = tokens * top_k
    counts = np.diff(off.cpu().numpy())
    gc, codes = out((rows, k // 2), torch.uint8)
    gs, sf = sf_out(fme.sf_bytes(rows, k, 16, experts))
    gr, rs = out((rows,), torch.float32)
    fme.permute_quantize_nvfp4(x, src, top_k, off, codes=codes, sf=sf, row_scale=rs, status=st)
    gc.check_guards("permute nvfp4 codes")
    gr.check_guards("permute nvfp4 row scales")
    check_tiled(gs, synth.offsets_from_counts(counts), k // 16, "permute nvfp4 scales")
    gc, codes = out((rows, k), torch.uint8)
    gs, sf = sf_out(fme.sf_bytes(rows, k, 32, experts))
    fme.permute_quantize_mxfp8(x, src, top_k, off, codes=codes, sf=sf, status=st)
    gc.check_guards("permute mxfp8 codes")
    check_tiled(gs, synth.offsets_from_counts(counts), k // 32, "permute mxfp8 scales")
    y = bf16_tensor(synth.normal_bits((rows, k), 1.0, seed=tokens + 8))
    weights = torch.from_numpy(w_np).cuda()
    gcb, comb = out((tokens, k), torch.bfloat16)
    fme.moe_combine(y, row_of, weights, out=comb, status=st)
    gcb.check_guards("moe_combine out")
    assert fme.read_device_status(st)[0] == 0
