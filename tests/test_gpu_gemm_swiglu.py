"""The NVFP4 gate/up GEMM with SwiGLU in its epilogue, against the oracle.

The oracle quantizes the same inputs itself (its codes equal the GPU's bit for
bit, test_gpu_quant.py), forms the gate/up product in fp64 and then
h = silu(g) * u in fp64 (swiglu_f64 on the unrounded product).  Tolerance,
derived from the GEMM's: each of g and u may be off by dy = 8e-3 |y| + 1e-3
rms(y_gu) (the per-element GEMM bound, rms over the gate/up product), and since
|silu'| <= SILU_SLOPE_MAX everywhere (test_silu_slope_bound),
    |silu(g') u' - silu(g) u| <= SILU_SLOPE_MAX dg (|u| + du) + |silu(g)| du;
the GPU then rounds h to bf16 once (2^-9 relative; 2^-8 allowed).
"""
import numpy as np
import pytest

from fp8_moe_expert_gb300 import synth
from tests.fmetest import bf16_bits_np, bf16_tensor, bf16_to_f64
from tests.test_gpu_gemm import COUNTS, _i32, _ok, _sample_rows, _sampled_experts, _status, ref_fwd_rows

SILU_SLOPE_MAX = 1.0999  # above max over v of d/dv (v sigma(v)) = 1.09984, reached near v = 2.40


def test_silu_slope_bound():
    """sup |silu'| on a dense grid (scipy's logistic function): 1.09984, just under
    the bound used (the slope tends to 1 and 0 at the ends, its minimum is -0.0998)."""
    from scipy.special import expit

    v = np.linspace(-60.0, 60.0, 2_400_001)
    s = expit(v)
    slope = s * (1.0 + v * (1.0 - s))
    assert np.abs(slope).max() <= SILU_SLOPE_MAX
    assert np.abs(slope).max() > SILU_SLOPE_MAX - 1e-4
    assert abs(v[np.argmax(slope)] - 2.3994) < 1e-3


def gpu_fwd_swiglu(fme, x, w, offsets, n, k):
    st = _status()
    off = _i32(offsets)
    a = fme.quantize_nvfp4_pertoken(x, off, status=st)
    b = fme.quantize_nvfp4_pertoken(w, status=st)
    h = fme.grouped_gemm_fwd_nvfp4_swiglu(*a, *b, off, n, k, status=st)
    _ok(fme, st)
    return h


def check_swiglu_tolerance(orc, h, y_gu_ref, rms=None, what=""):
    """h (GPU, any float array [rows x I]) against the oracle's SwiGLU of the fp64
    gate/up product y_gu_ref [rows x 2 I], element by element."""
    y = np.asarray(y_gu_ref, np.float64)
    h = np.asarray(h, np.float64)
    inter = y.shape[1] // 2
    if rms is None:
        rms = float(np.sqrt(np.mean(y ** 2))) if y.size else 0.0
    g, u = y[:, :inter], y[:, inter:]
    h_ref = orc.swiglu_f64(y)
    silu_g = orc.swiglu_f64(np.concatenate([g, np.ones_like(g)], axis=1))
    dg = 8e-3 * np.abs(g) + 1e-3 * rms
    du = 8e-3 * np.abs(u) + 1e-3 * rms
    prop = SILU_SLOPE_MAX * dg * (np.abs(u) + du) + np.abs(silu_g) * du
    bound = prop + 2.0 ** -8 * (np.abs(h_ref) + prop)
    err = np.abs(h - h_ref)
    bad = err > bound
    if bad.any():
        idx = np.argwhere(bad)[:5]
        detail = ", ".join(f"{tuple(i)}: got {h[tuple(i)]:.6g} want {h_ref[tuple(i)]:.6g}" for i in idx)
        raise AssertionError(f"{what}: {int(bad.sum())} of {bad.size} elements out of tolerance; {detail}")


@pytest.mark.gpu
def test_swiglu_gemm_tiny(fme, orc):
    """One expert: X [128 x 256], W_gu [512 x 256] (I = 256: two output tiles)."""
    x_bits = synth.normal_bits((128, 256), 1.0, seed=61)
    w_bits = synth.normal_bits((512, 256), 0.05, seed=62)
    h = gpu_fwd_swiglu(fme, bf16_tensor(x_bits), bf16_tensor(w_bits), [0, 128], 512, 256)
    assert tuple(h.shape) == (128, 256)
    check_swiglu_tolerance(orc, bf16_to_f64(h), ref_fwd_rows(orc, x_bits, w_bits), what="tiny swiglu")


@pytest.mark.gpu
def test_swiglu_gemm_ragged_experts(fme, orc):
    """Empty, single-row, partial and exact 128-row experts; several K stages."""
    off = synth.offsets_from_counts(COUNTS)
    e, n, k = len(COUNTS), 512, 768
    x_bits = synth.normal_bits((int(off[-1]), k), 1.0, seed=63)
    w_bits = synth.normal_bits((e * n, k), 0.04, seed=64)
    h = bf16_to_f64(gpu_fwd_swiglu(fme, bf16_tensor(x_bits), bf16_tensor(w_bits), off, n, k))
    for g in range(e):
        if COUNTS[g]:
            ref = ref_fwd_rows(orc, x_bits[off[g]:off[g + 1]], w_bits[g * n:(g + 1) * n])
            check_swiglu_tolerance(orc, h[off[g]:off[g + 1]], ref, what=f"ragged swiglu expert {g}")


@pytest.mark.gpu
def test_swiglu_gemm_expert_shapes(fme, orc):
    """The gate/up projection of the expert shapes (hidden 7168, I = 2048, 32
    experts, 65536 Dirichlet-loaded rows): sampled rows of sampled experts."""
    import torch

    counts = synth.dirichlet_counts()
    off = synth.offsets_from_counts(counts)
    rows, E, H, I = int(off[-1]), len(counts), synth.HIDDEN, synth.INTERMEDIATE
    x = synth.torch_normal((rows, H), 1.0, seed=71)
    w_gu = synth.torch_normal((E * 2 * I, H), 0.02, seed=72)
    h = gpu_fwd_swiglu(fme, x, w_gu, off, 2 * I, H)
    torch.cuda.synchronize()
    rng = np.random.default_rng(7)
    for g in _sampled_experts(counts, rng, count=3):
        r = _sample_rows(off, g, rng)
        ridx = torch.from_numpy(r).cuda()
        ref = ref_fwd_rows(orc, bf16_bits_np(x[ridx]), bf16_bits_np(w_gu[g * 2 * I:(g + 1) * 2 * I]))
        check_swiglu_tolerance(orc, bf16_to_f64(h[ridx]), ref, what=f"expert-shape swiglu expert {g}")


@pytest.mark.gpu
def test_swiglu_gemm_rows_independent(fme):
    """A row's h is bit-identical with other experts' rows appended, and two runs
    agree bit for bit (no split over K, no M-dependent order)."""
    import torch

    counts = [100, 260]
    off = synth.offsets_from_counts(counts)
    n, k = 512, 512
    x = bf16_tensor(synth.normal_bits((360, k), 1.0, seed=65))
    w = bf16_tensor(synth.normal_bits((3 * n, k), 0.04, seed=66))
    more = bf16_tensor(synth.normal_bits((300, k), 5.0, seed=67))
    h1 = bf16_bits_np(gpu_fwd_swiglu(fme, x, w[: 2 * n], off, n, k))
    h1b = bf16_bits_np(gpu_fwd_swiglu(fme, x, w[: 2 * n], off, n, k))
    h2 = bf16_bits_np(gpu_fwd_swiglu(fme, torch.cat([x, more]), w, synth.offsets_from_counts(counts + [300]), n, k))
    assert np.array_equal(h1, h1b)
    assert np.array_equal(h1, h2[:360])


@pytest.mark.gpu
def test_swiglu_gemm_shapes_checked(fme):
    """n (= 2 I) must be a multiple of 256: 384 is refused before any launch; no
    rows is a no-op."""
    import torch

    st = _status()
    x = bf16_tensor(synth.normal_bits((64, 256), 1.0, seed=68))
    w = bf16_tensor(synth.normal_bits((384, 256), 0.04, seed=69))
    off = _i32([0, 64])
    a = fme.quantize_nvfp4_pertoken(x, off, status=st)
    b = fme.quantize_nvfp4_pertoken(w, status=st)
    with pytest.raises(fme.FmeError) as info:
        fme.grouped_gemm_fwd_nvfp4_swiglu(*a, *b, off, 384, 256, status=st)
    assert info.value.status == fme.ERR_UNSUPPORTED_SHAPE
    # m = 0: nothing to do, and the operand pointers are not read
    ae = (torch.empty((0, 128), dtype=torch.uint8, device="cuda"), torch.zeros(16, dtype=torch.uint8, device="cuda"),
          torch.empty(0, dtype=torch.float32, device="cuda"))
    w2 = bf16_tensor(synth.normal_bits((512, 256), 0.04, seed=70))
    b2 = fme.quantize_nvfp4_pertoken(w2, status=st)
    h = fme.grouped_gemm_fwd_nvfp4_swiglu(*ae, *b2, _i32([0, 0]), 512, 256, status=st)
    assert tuple(h.shape) == (0, 256)
    _ok(fme, st)
