"""Fused SwiGLU + NVFP4 per-token quantization on the GPU.

h = silu(g) * u is evaluated in fp32 with a hardware exponential and rounded to
bf16, so it is compared with the oracle's fp64 value to within one bf16 unit in
the last place; the quantization of that h is then checked bit for bit against
the oracle run on the kernel's own h, and against the stand-alone quantizer.
"""
import numpy as np
import pytest

from fp8_moe_expert_gb300 import synth
from tests.fmetest import bf16_bits_np, bf16_tensor, to_np, unswizzle

pytestmark = pytest.mark.gpu


def _i32(a):
    import torch

    return torch.from_numpy(np.asarray(a, np.int32)).cuda()


def _status():
    import torch

    return torch.zeros(1, dtype=torch.int32, device="cuda")


def gate_up_bits(rows, inter, seed):
    rng = np.random.default_rng(seed)
    g = rng.standard_normal((rows, inter), dtype=np.float32) * 2.0
    u = rng.standard_normal((rows, inter), dtype=np.float32)
    g[rng.random(g.shape) < 0.002] *= 40.0          # saturated gates, both signs
    if rows > 2:
        g[1] = 0.0                                   # silu(0) = 0: an all-zero row of h
        u[2, : inter // 2] = 0.0
    return synth.bf16_bits(np.concatenate([g, u], axis=1))


def bf16_ulp(v: np.ndarray) -> np.ndarray:
    """Spacing of bf16 values at |v| (normal range; subnormal spacing below)."""
    a = np.abs(v)
    e = np.floor(np.log2(np.maximum(a, 2.0 ** -126)))
    return np.ldexp(1.0, (e - 7).astype(np.int64))


def check_fused(fme, orc, y_bits, offsets):
    rows, two_inter = y_bits.shape
    inter = two_inter // 2
    st = _status()
    codes, sf, scale, h = fme.swiglu_quantize_nvfp4(bf16_tensor(y_bits), None if offsets is None else _i32(offsets),
                                                    status=st)
    code, raw = fme.read_device_status(st)
    assert code == 0, raw
    h_bits = bf16_bits_np(h)
    ref = orc.swiglu(y_bits)
    err = np.abs(synth.bf16_float(h_bits).astype(np.float64) - ref)
    bad = err > bf16_ulp(ref)
    assert not bad.any(), f"{int(bad.sum())} h values off by more than one bf16 ulp, e.g. {np.argwhere(bad)[:3]}"
    oc, osf, oscale = orc.quant_nvfp4(h_bits)
    assert np.array_equal(to_np(codes), oc)
    assert np.array_equal(unswizzle(to_np(sf), rows, inter // 16, offsets), osf)
    assert np.array_equal(to_np(scale).view(np.uint32), oscale.view(np.uint32))
    # the fused quantization is the stand-alone quantizer's, byte for byte
    pc, psf, ps = fme.quantize_nvfp4_pertoken(h, None if offsets is None else _i32(offsets), status=st)
    assert np.array_equal(to_np(pc), to_np(codes)) and np.array_equal(to_np(ps), to_np(scale))
    assert np.array_equal(unswizzle(to_np(psf), rows, inter // 16, offsets), unswizzle(to_np(sf), rows, inter // 16,
                                                                                       offsets))
    return h_bits


@pytest.mark.parametrize("rows,inter", [(1, 64), (130, 2048), (64, 4608)])
def test_swiglu_quantize_shapes(fme, orc, rows, inter):
    check_fused(fme, orc, gate_up_bits(rows, inter, seed=rows + inter), None)


def test_swiglu_quantize_groups(fme, orc):
    counts = [37, 0, 200, 1, 129]
    off = synth.offsets_from_counts(counts)
    check_fused(fme, orc, gate_up_bits(int(off[-1]), 2048, seed=7), off)


def test_swiglu_quantize_without_h_output(fme):
    y = gate_up_bits(96, 2048, seed=3)
    st = _status()
    a = fme.swiglu_quantize_nvfp4(bf16_tensor(y), status=st)
    b = fme.swiglu_quantize_nvfp4(bf16_tensor(y), want_h=False, status=st)
    assert b[3] is None
    assert np.array_equal(to_np(a[0]), to_np(b[0]))
    assert np.array_equal(to_np(a[2]), to_np(b[2]))
    # padding rows of the scale layout are unwritten: compare the logical scales
    assert np.array_equal(unswizzle(to_np(a[1]), 96, 128), unswizzle(to_np(b[1]), 96, 128))


def test_swiglu_quantize_expert_batch(fme, orc):
    """16384 tokens over 8 experts at the bench's intermediate width (2048)."""
    counts = synth.dirichlet_counts(rows=16384, experts=8, seed=9)
    off = synth.offsets_from_counts(counts)
    check_fused(fme, orc, gate_up_bits(16384, 2048, seed=11), off)
