"""Fused SwiGLU backward + MXFP8 row-wise and column-wise quantization on the GPU.

d(gate/up) = [dg | du] is evaluated in fp32 with a hardware exponential and
rounded to bf16, so it is compared with the oracle's fp64 value within half a
bf16 unit plus an fp32 evaluation term (dg's factor 1 + g sigma(-g) cancels near
g = -1.28, so that term is absolute in the size of the summands).  The
quantization of that bf16 gradient is then checked bit for bit against the
oracle's quantizers run on the kernel's own values, and against the GPU's
stand-alone row/column quantizer.
"""
import numpy as np
import pytest

from fp8_moe_expert_gb300 import synth
from tests.fmetest import bf16_tensor, bf16_bits_np, to_np, unswizzle

pytestmark = pytest.mark.gpu


def _i32(a):
    import torch

    return torch.from_numpy(np.asarray(a, np.int32)).cuda()


def _status():
    import torch

    return torch.zeros(1, dtype=torch.int32, device="cuda")


def inputs(rows, inter, seed):
    rng = np.random.default_rng(seed)
    g = rng.standard_normal((rows, inter), dtype=np.float32) * 2.0
    u = rng.standard_normal((rows, inter), dtype=np.float32)
    dh = rng.standard_normal((rows, inter), dtype=np.float32) * 0.05
    g[rng.random(g.shape) < 0.003] *= 40.0           # saturated gates, both signs
    g[rng.random(g.shape) < 0.003] = -1.28125         # next to the root of silu'
    dh[rng.random(dh.shape) < 0.001] *= 300.0         # large gradients
    if rows > 3:
        dh[1] = 0.0                                   # an all-zero row of d(gate/up)
        g[2, : inter // 2] = 0.0
        u[3] = 0.0
    return synth.bf16_bits(np.concatenate([g, u], axis=1)), synth.bf16_bits(dh)


def _sigma(v):
    from scipy.special import expit

    return expit(v)


def check_values(d_bits, y_bits, dh_bits, ref):
    rows, two = y_bits.shape
    inter = two // 2
    g = synth.bf16_float(y_bits[:, :inter]).astype(np.float64)
    u = synth.bf16_float(y_bits[:, inter:]).astype(np.float64)
    dh = synth.bf16_float(dh_bits).astype(np.float64)
    s, sn = _sigma(g), _sigma(-g)
    scale = np.concatenate([np.abs(dh * u) * s * (1.0 + np.abs(g) * sn), np.abs(dh * g) * s], axis=1)
    got = synth.bf16_float(d_bits).astype(np.float64)
    a = np.abs(ref)
    half_ulp = np.ldexp(1.0, (np.floor(np.log2(np.maximum(a, 2.0 ** -126))) - 8).astype(np.int64))
    bound = half_ulp + scale * 2.0 ** -17 + 2.0 ** -133
    bad = np.abs(got - ref) > bound
    assert not bad.any(), f"{int(bad.sum())} values out of bound, e.g. {np.argwhere(bad)[:3].tolist()}"


def check_bwd(fme, orc, y_bits, dh_bits, offsets):
    rows, two = y_bits.shape
    dev_off = None if offsets is None else _i32(offsets)
    off_np = np.array([0, rows], np.int32) if offsets is None else np.asarray(offsets, np.int32)
    st = _status()
    y, dh = bf16_tensor(y_bits), bf16_tensor(dh_bits)
    rc, rs, cc, cs, poff, ld, d = fme.swiglu_backward_quantize_mxfp8(y, dh, dev_off, want_d=True, status=st)
    code, raw = fme.read_device_status(st)
    assert code == 0, raw
    d_bits = bf16_bits_np(d)
    check_values(d_bits, y_bits, dh_bits, orc.swiglu_bwd(y_bits, dh_bits))
    # row-wise: bit for bit against the oracle on the kernel's bf16 gradient
    oc, osf = orc.quant_mxfp8_rows(d_bits)
    assert np.array_equal(to_np(rc), oc)
    assert np.array_equal(unswizzle(to_np(rs), rows, two // 32, off_np), osf)
    # column-wise
    occ, ocs, opoff = orc.quant_mxfp8_cols(d_bits, off_np, ld=ld)
    p = int(opoff[-1])
    assert np.array_equal(to_np(poff), opoff)
    assert np.array_equal(to_np(cc)[:, :p], occ[:, :p])
    assert np.array_equal(unswizzle(to_np(cs), two, ld // 32)[:, : p // 32], ocs[:, : p // 32])
    # the GPU's stand-alone one-pass quantizer gives the same bytes
    (rc2, rs2), (cc2, cs2, _, _) = fme.quantize_mxfp8_rowcol(d, dev_off, status=st)
    assert np.array_equal(to_np(rc2), to_np(rc))
    assert np.array_equal(to_np(cc2)[:, :p], to_np(cc)[:, :p])
    assert np.array_equal(unswizzle(to_np(rs2), rows, two // 32, off_np), unswizzle(to_np(rs), rows, two // 32, off_np))
    # without the bf16 output: the same quantized bytes
    rc3, rs3, cc3, cs3, _, _, d3 = fme.swiglu_backward_quantize_mxfp8(y, dh, dev_off, status=st)
    assert d3 is None
    assert np.array_equal(to_np(rc3), to_np(rc)) and np.array_equal(to_np(cc3)[:, :p], to_np(cc)[:, :p])
    assert fme.read_device_status(st)[0] == 0


@pytest.mark.parametrize("rows,inter", [(1, 128), (130, 256), (200, 2048), (97, 384)])
def test_swiglu_bwd_shapes(fme, orc, rows, inter):
    y, dh = inputs(rows, inter, seed=rows + inter)
    check_bwd(fme, orc, y, dh, None)


def test_swiglu_bwd_groups(fme, orc):
    counts = [37, 0, 200, 1, 129, 0, 128]
    off = synth.offsets_from_counts(counts)
    y, dh = inputs(int(off[-1]), 512, seed=7)
    check_bwd(fme, orc, y, dh, off)


def test_swiglu_bwd_expert_batch(fme, orc):
    """16384 rows over 8 experts at the bench's intermediate width (2048)."""
    counts = synth.dirichlet_counts(rows=16384, experts=8, seed=9)
    off = synth.offsets_from_counts(counts)
    y, dh = inputs(16384, 2048, seed=11)
    check_bwd(fme, orc, y, dh, off)


def test_swiglu_bwd_empty_rows(fme):
    import torch

    y = torch.zeros((0, 256), dtype=torch.bfloat16, device="cuda")
    dh = torch.zeros((0, 128), dtype=torch.bfloat16, device="cuda")
    st = _status()
    off = _i32([0, 0, 0])
    out = fme.swiglu_backward_quantize_mxfp8(y, dh, off, status=st)
    assert fme.read_device_status(st)[0] == 0
    assert to_np(out[4]).tolist() == [0, 0, 0]


def test_swiglu_bwd_full_size_sampled(fme, orc):
    """The bench's rows: 262144 over 32 experts (Zipf loads), inter 2048; the
    gradient in full against the stand-alone quantizer, sampled rows against the
    oracle's values and row-wise codes."""
    import torch

    counts = synth.zipf_counts()
    off = synth.offsets_from_counts(counts)
    R, inter = int(off[-1]), 2048
    y = synth.torch_normal((R, 2 * inter), 1.0, seed=51)
    dh = synth.torch_normal((R, inter), 1e-2, seed=52)
    st = _status()
    dev_off = _i32(off)
    rc, rs, cc, cs, poff, ld, d = fme.swiglu_backward_quantize_mxfp8(y, dh, dev_off, want_d=True, status=st)
    (rc2, _), (cc2, _, _, _) = fme.quantize_mxfp8_rowcol(d, dev_off, status=st)
    assert fme.read_device_status(st)[0] == 0
    assert torch.equal(rc, rc2)
    p = int(to_np(poff)[-1])
    assert torch.equal(cc[:, :p], cc2[:, :p])
    rng = np.random.default_rng(53)
    rows = np.sort(rng.choice(R, size=64, replace=False))
    idx = torch.from_numpy(rows).cuda()
    y_s, dh_s, d_s = bf16_bits_np(y[idx]), bf16_bits_np(dh[idx]), bf16_bits_np(d[idx])
    check_values(d_s, y_s, dh_s, orc.swiglu_bwd(y_s, dh_s))
    oc, _ = orc.quant_mxfp8_rows(d_s)
    assert np.array_equal(to_np(rc[idx]), oc)


def test_gate_up_backward_chain(fme, orc):
    """The gate/up gradients from the fused kernel's outputs: dX_e = dGU_e W_gu,e
    (contraction over 2I) through the dgrad kernel and dW_gu,e = dGU_e^T X_e
    through the wgrad kernel, against the oracle on the kernel's bf16 dGU; an empty
    expert gets dW = 0."""
    from tests.fmetest import bf16_to_f64, check_gemm_tolerance
    from tests.test_gpu_gemm import ref_dgrad_rows, ref_wgrad

    counts = [150, 0, 333]
    off = synth.offsets_from_counts(counts)
    R, inter, H, E = int(off[-1]), 256, 512, 3
    y_bits, dh_bits = inputs(R, inter, seed=61)
    x_bits = synth.normal_bits((R, H), 1.0, seed=62)
    w_bits = synth.normal_bits((E * 2 * inter, H), 0.02, seed=63)
    st = _status()
    dev_off = _i32(off)
    rc, rs, cc, cs, poff, ld, d = fme.swiglu_backward_quantize_mxfp8(bf16_tensor(y_bits), bf16_tensor(dh_bits),
                                                                     dev_off, want_d=True, status=st)
    wc, ws, _, ldw = fme.quantize_mxfp8(bf16_tensor(w_bits), fme.COLWISE, status=st)
    xc, xs, _, ldx = fme.quantize_mxfp8(bf16_tensor(x_bits), fme.COLWISE, dev_off, status=st)
    dx = fme.grouped_gemm_dgrad_mxfp8(rc, rs, wc, ws, ldw, dev_off, H, 2 * inter, status=st)
    dw = fme.grouped_gemm_wgrad_mxfp8(cc, cs, ld, xc, xs, ldx, poff, 2 * inter, H, status=st)
    assert fme.read_device_status(st)[0] == 0
    d_bits = bf16_bits_np(d)
    dx64, dw64 = bf16_to_f64(dx), bf16_to_f64(dw)
    for e in range(E):
        lo, hi = int(off[e]), int(off[e + 1])
        if hi == lo:
            assert not dw64[e].any()
            continue
        w_e = w_bits[e * 2 * inter:(e + 1) * 2 * inter]
        check_gemm_tolerance(dx64[lo:hi], ref_dgrad_rows(orc, d_bits[lo:hi], w_e), what=f"gate/up dgrad e{e}")
        check_gemm_tolerance(dw64[e], ref_wgrad(orc, d_bits[lo:hi], x_bits[lo:hi]), what=f"gate/up wgrad e{e}")
