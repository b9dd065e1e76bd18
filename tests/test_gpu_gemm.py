"""Block-scaled grouped GEMMs on the GPU against the CPU oracle's fp64 GEMM.

The GPU quantizes and multiplies; the oracle quantizes the same inputs itself
(its codes equal the GPU's bit for bit, test_gpu_quant.py) and computes
y_ref = sum_k dequant(a) dequant(b) in fp64.  Tolerance per element:
|y - y_ref| <= 8e-3 |y_ref| + 1e-3 rms(y_ref).  Small cases are checked in full;
the expert-shaped workloads (32 experts, hidden 7168, intermediate 2048) on
sampled rows: every sampled expert's first and last row plus random rows.
"""
import numpy as np
import pytest

from fp8_moe_expert_gb300 import synth
from tests.fmetest import bf16_bits_np, bf16_tensor, bf16_to_f64, check_gemm_tolerance, to_np

pytestmark = pytest.mark.gpu


def _i32(a):
    import torch

    return torch.from_numpy(np.asarray(a, np.int32)).cuda()


def _status():
    import torch

    return torch.zeros(1, dtype=torch.int32, device="cuda")


def _ok(fme, st):
    code, raw = fme.read_device_status(st)
    assert code == 0, f"device status {raw:#x}"


# ------------------------------------------------------------ GPU pipelines --
def gpu_fwd(fme, x, w, offsets, n, k):
    st = _status()
    off = _i32(offsets)
    a = fme.quantize_nvfp4_pertoken(x, off, status=st)
    b = fme.quantize_nvfp4_pertoken(w, status=st)
    y = fme.grouped_gemm_fwd_nvfp4(*a, *b, off, n, k, status=st)
    _ok(fme, st)
    return y


def gpu_fwd_mxfp8(fme, x, w, offsets, n, k):
    st = _status()
    off = _i32(offsets)
    a = fme.quantize_mxfp8(x, fme.ROWWISE, off, status=st)
    b = fme.quantize_mxfp8(w, fme.ROWWISE, status=st)
    y = fme.grouped_gemm_fwd_mxfp8(*a, *b, off, n, k, status=st)
    _ok(fme, st)
    return y


def gpu_dgrad(fme, dy, w_stacked, offsets, n, k):
    """dX_e = dY_e W_e with W_e = rows [e k, e k + k) of w_stacked [E k x n]."""
    st = _status()
    off = _i32(offsets)
    a_codes, a_sf = fme.quantize_mxfp8(dy, fme.ROWWISE, off, status=st)
    b_codes, b_sf, _, ldb = fme.quantize_mxfp8(w_stacked, fme.COLWISE, status=st)
    y = fme.grouped_gemm_dgrad_mxfp8(a_codes, a_sf, b_codes, b_sf, ldb, off, n, k, status=st)
    _ok(fme, st)
    return y


def gpu_wgrad(fme, dy, h, offsets):
    st = _status()
    off = _i32(offsets)
    a_codes, a_sf, poff, lda = fme.quantize_mxfp8(dy, fme.COLWISE, off, status=st)
    b_codes, b_sf, _, ldb = fme.quantize_mxfp8(h, fme.COLWISE, off, status=st)
    y = fme.grouped_gemm_wgrad_mxfp8(a_codes, a_sf, lda, b_codes, b_sf, ldb, poff, dy.shape[1], h.shape[1],
                                     status=st)
    _ok(fme, st)
    return y


# ---------------------------------------------------------- oracle references --
def ref_fwd_rows(orc, x_bits_rows, w_bits_e):
    a = orc.dequant_nvfp4(*orc.quant_nvfp4(x_bits_rows))
    b = orc.dequant_nvfp4(*orc.quant_nvfp4(w_bits_e))
    return orc.gemm_abt(a, b)


def ref_fwd_mxfp8_rows(orc, x_bits_rows, w_bits_e):
    a = orc.dequant_mxfp8(*orc.quant_mxfp8_rows(x_bits_rows))
    b = orc.dequant_mxfp8(*orc.quant_mxfp8_rows(w_bits_e))
    return orc.gemm_abt(a, b)


def ref_dgrad_rows(orc, dy_bits_rows, w_bits_e):
    """rows of dY_e W_e with W_e [k x n] quantized column-wise (blocks along k)."""
    a = orc.dequant_mxfp8(*orc.quant_mxfp8_rows(dy_bits_rows))
    k = w_bits_e.shape[0]
    ct, st, _ = orc.quant_mxfp8_cols(w_bits_e, np.array([0, k]))
    b = orc.dequant_mxfp8(ct, st)[:, :k]
    return orc.gemm_abt(a, b)


def ref_wgrad(orc, dy_bits_e, h_bits_e, rows_sel=None):
    n_e = dy_bits_e.shape[0]
    off = np.array([0, n_e])
    ca, sa, _ = orc.quant_mxfp8_cols(dy_bits_e, off)
    cb, sb, _ = orc.quant_mxfp8_cols(h_bits_e, off)
    if rows_sel is not None:
        ca, sa = ca[rows_sel], sa[rows_sel]
    return orc.gemm_abt(orc.dequant_mxfp8(ca, sa), orc.dequant_mxfp8(cb, sb))


# --------------------------------------------------------------- tiny cases --
def test_tiny_fwd_nvfp4(fme, orc):
    """One expert: X [128 x 256] with 1% x30 outliers, W [256 x 256] ~ N(0, 0.02^2)."""
    x_bits, w_bits = synth.tiny(0)
    y = gpu_fwd(fme, bf16_tensor(x_bits), bf16_tensor(w_bits), [0, 128], 256, 256)
    check_gemm_tolerance(bf16_to_f64(y), ref_fwd_rows(orc, x_bits, w_bits), what="tiny fwd")


def test_tiny_mxfp8_gemm(fme, orc):
    """Same tensors, both MXFP8 row-wise along K = 256: Y = X W^T through the
    dgrad kernel (A row-wise, B given row-wise as [n x ldb] with ldb = k)."""
    x_bits, w_bits = synth.tiny(0)
    st = _status()
    off = _i32([0, 128])
    a = fme.quantize_mxfp8(bf16_tensor(x_bits), fme.ROWWISE, off, status=st)
    b = fme.quantize_mxfp8(bf16_tensor(w_bits), fme.ROWWISE, status=st)
    y = fme.grouped_gemm_dgrad_mxfp8(*a, *b, 256, off, 256, 256, status=st)
    _ok(fme, st)
    ya = orc.dequant_mxfp8(*orc.quant_mxfp8_rows(x_bits))
    yb = orc.dequant_mxfp8(*orc.quant_mxfp8_rows(w_bits))
    check_gemm_tolerance(bf16_to_f64(y), orc.gemm_abt(ya, yb), what="tiny mxfp8")


def test_tiny_fwd_mxfp8(fme, orc):
    """The MXFP8 forward on the tiny tensors (one expert, K = 256)."""
    x_bits, w_bits = synth.tiny(0)
    y = gpu_fwd_mxfp8(fme, bf16_tensor(x_bits), bf16_tensor(w_bits), [0, 128], 256, 256)
    check_gemm_tolerance(bf16_to_f64(y), ref_fwd_mxfp8_rows(orc, x_bits, w_bits), what="tiny mxfp8 fwd")


# --------------------------------------------------- small ragged, full check --
COUNTS = [0, 37, 128, 1, 200, 0, 129]


def test_fwd_ragged_experts(fme, orc):
    off = synth.offsets_from_counts(COUNTS)
    e, n, k = len(COUNTS), 512, 768
    x_bits = synth.normal_bits((int(off[-1]), k), 1.0, seed=11)
    w_bits = synth.normal_bits((e * n, k), 0.02, seed=12)
    y = bf16_to_f64(gpu_fwd(fme, bf16_tensor(x_bits), bf16_tensor(w_bits), off, n, k))
    ref = np.zeros_like(y)
    for g in range(e):
        if COUNTS[g]:
            ref[off[g]:off[g + 1]] = ref_fwd_rows(orc, x_bits[off[g]:off[g + 1]], w_bits[g * n:(g + 1) * n])
    check_gemm_tolerance(y, ref, what="ragged fwd")


def test_fwd_mxfp8_ragged_experts(fme, orc):
    off = synth.offsets_from_counts(COUNTS)
    e, n, k = len(COUNTS), 512, 640
    x_bits = synth.normal_bits((int(off[-1]), k), 1.0, seed=13)
    w_bits = synth.normal_bits((e * n, k), 0.02, seed=14)
    y = bf16_to_f64(gpu_fwd_mxfp8(fme, bf16_tensor(x_bits), bf16_tensor(w_bits), off, n, k))
    ref = np.zeros_like(y)
    for g in range(e):
        if COUNTS[g]:
            ref[off[g]:off[g + 1]] = ref_fwd_mxfp8_rows(orc, x_bits[off[g]:off[g + 1]], w_bits[g * n:(g + 1) * n])
    check_gemm_tolerance(y, ref, what="ragged mxfp8 fwd")


def test_dgrad_ragged_experts(fme, orc):
    off = synth.offsets_from_counts(COUNTS)
    e, n, k = len(COUNTS), 512, 384
    dy_bits = synth.normal_bits((int(off[-1]), k), 1e-2, seed=21)
    w_bits = synth.normal_bits((e * k, n), 0.02, seed=22)
    y = bf16_to_f64(gpu_dgrad(fme, bf16_tensor(dy_bits), bf16_tensor(w_bits), off, n, k))
    ref = np.zeros_like(y)
    for g in range(e):
        if COUNTS[g]:
            ref[off[g]:off[g + 1]] = ref_dgrad_rows(orc, dy_bits[off[g]:off[g + 1]], w_bits[g * k:(g + 1) * k])
    check_gemm_tolerance(y, ref, what="ragged dgrad")


def test_wgrad_ragged_experts(fme, orc):
    off = synth.offsets_from_counts(COUNTS)
    m, n = 256, 512
    dy_bits = synth.normal_bits((int(off[-1]), m), 1e-2, seed=31)
    h_bits = synth.normal_bits((int(off[-1]), n), 1.0, seed=32)
    y = bf16_to_f64(gpu_wgrad(fme, bf16_tensor(dy_bits), bf16_tensor(h_bits), off))
    assert y.shape == (len(COUNTS), m, n)
    for g, c in enumerate(COUNTS):
        if c == 0:
            assert np.all(y[g] == 0), f"expert {g} without rows must get zeros"
            continue
        ref = ref_wgrad(orc, dy_bits[off[g]:off[g + 1]], h_bits[off[g]:off[g + 1]])
        check_gemm_tolerance(y[g], ref, what=f"wgrad expert {g}")


def test_wgrad_accumulate_fp32(fme, orc):
    """The fp32-accumulating wgrad: from zero it is the wgrad's fp32 result (its
    bf16 rounding equals the bf16 wgrad bit for bit, and it is within the GEMM
    tolerance of the oracle); a second call doubles it exactly; on a random
    buffer it is that buffer plus the result, one binary32 add per element (numpy);
    empty experts keep their buffer."""
    import torch

    off = synth.offsets_from_counts(COUNTS)
    m, n = 256, 512
    dy_bits = synth.normal_bits((int(off[-1]), m), 1e-2, seed=33)
    h_bits = synth.normal_bits((int(off[-1]), n), 1.0, seed=34)
    st = _status()
    o = _i32(off)
    a_codes, a_sf, poff, lda = fme.quantize_mxfp8(bf16_tensor(dy_bits), fme.COLWISE, o, status=st)
    b_codes, b_sf, _, ldb = fme.quantize_mxfp8(bf16_tensor(h_bits), fme.COLWISE, o, status=st)
    E = len(COUNTS)
    y16 = fme.grouped_gemm_wgrad_mxfp8(a_codes, a_sf, lda, b_codes, b_sf, ldb, poff, m, n, status=st)
    acc = torch.zeros((E, m, n), dtype=torch.float32, device="cuda")
    fme.grouped_gemm_wgrad_mxfp8_accumulate(a_codes, a_sf, lda, b_codes, b_sf, ldb, poff, m, n, acc, status=st)
    first = acc.clone()
    fme.grouped_gemm_wgrad_mxfp8_accumulate(a_codes, a_sf, lda, b_codes, b_sf, ldb, poff, m, n, acc, status=st)
    rng = np.random.default_rng(35)
    init = rng.standard_normal((E, m, n)).astype(np.float32)
    acc2 = torch.from_numpy(init).cuda()
    fme.grouped_gemm_wgrad_mxfp8_accumulate(a_codes, a_sf, lda, b_codes, b_sf, ldb, poff, m, n, acc2, status=st)
    _ok(fme, st)
    f = to_np(first)
    live = np.array([c > 0 for c in COUNTS])
    assert np.array_equal(bf16_bits_np(first.to(torch.bfloat16))[live], bf16_bits_np(y16)[live])
    assert np.array_equal(to_np(acc), 2.0 * f)
    want = init.copy()
    want[live] = (init[live] + f[live]).astype(np.float32)
    assert np.array_equal(to_np(acc2), want)
    assert not f[~live].any()
    for g, c in enumerate(COUNTS):
        if c:
            ref = ref_wgrad(orc, dy_bits[off[g]:off[g + 1]], h_bits[off[g]:off[g + 1]])
            check_gemm_tolerance(f[g].astype(np.float64), ref, what=f"accumulating wgrad expert {g}")


def test_row_invariance_and_determinism(fme):
    """A row's forward and dgrad outputs are bit-identical when other experts'
    rows are appended (no split over K, no M-dependent reduction order), and two
    runs agree bit for bit."""
    counts = [100, 260]
    off = synth.offsets_from_counts(counts)
    n, k = 512, 512
    x = bf16_tensor(synth.normal_bits((360, k), 1.0, seed=41))
    w = bf16_tensor(synth.normal_bits((3 * n, k), 0.02, seed=42))
    more = bf16_tensor(synth.normal_bits((300, k), 5.0, seed=43))
    import torch

    y1 = bf16_bits_np(gpu_fwd(fme, x, w[: 2 * n], off, n, k))
    y1b = bf16_bits_np(gpu_fwd(fme, x, w[: 2 * n], off, n, k))
    y2 = bf16_bits_np(gpu_fwd(fme, torch.cat([x, more]), w, synth.offsets_from_counts(counts + [300]), n, k))
    assert np.array_equal(y1, y1b)
    assert np.array_equal(y1, y2[:360])
    wd = bf16_tensor(synth.normal_bits((3 * k, n), 0.02, seed=44))
    d1 = bf16_bits_np(gpu_dgrad(fme, x, wd[: 2 * k], off, n, k))
    d2 = bf16_bits_np(gpu_dgrad(fme, torch.cat([x, more]), wd, synth.offsets_from_counts(counts + [300]), n, k))
    assert np.array_equal(d1, d2[:360])


def test_gemm_bad_offsets_status(fme):
    import torch

    x = bf16_tensor(synth.normal_bits((64, 256), 1.0, seed=1))
    w = bf16_tensor(synth.normal_bits((512, 256), 0.02, seed=2))
    st = _status()
    a = fme.quantize_nvfp4_pertoken(x, status=st)
    b = fme.quantize_nvfp4_pertoken(w, status=st)
    bad = torch.tensor([0, 50, 40], dtype=torch.int32, device="cuda")
    fme.grouped_gemm_fwd_nvfp4(*a, *b, bad, 256, 256, status=st)
    code, raw = fme.read_device_status(st)
    assert code == 7 and raw & fme.DEV_BAD_OFFSETS


# ------------------------------------------------ expert-shaped workloads --
def _sample_rows(off, g, rng, extra=2):
    lo, hi = int(off[g]), int(off[g + 1])
    picks = {lo, hi - 1}
    picks.update(int(v) for v in rng.integers(lo, hi, size=extra))
    return np.array(sorted(picks))


def _sampled_experts(counts, rng, count=5):
    live = [g for g, c in enumerate(counts) if c > 0]
    chosen = {live[0], live[-1], int(np.argmax(counts))}
    chosen.update(int(g) for g in rng.choice(live, size=min(count, len(live)), replace=False))
    return sorted(chosen)


def _moe_fwd_sampled(fme, orc, counts, seed, label):
    import torch

    off = synth.offsets_from_counts(counts)
    rows = int(off[-1])
    E, H, I = len(counts), synth.HIDDEN, synth.INTERMEDIATE
    x = synth.torch_normal((rows, H), 1.0, seed=seed * 10 + 1)
    w_gu = synth.torch_normal((E * 2 * I, H), 0.02, seed=seed * 10 + 2)
    h = synth.torch_normal((rows, I), 1.0, seed=seed * 10 + 3)
    w_d = synth.torch_normal((E * H, I), 0.02, seed=seed * 10 + 4)
    y_gu = gpu_fwd(fme, x, w_gu, off, 2 * I, H)
    y_d = gpu_fwd(fme, h, w_d, off, H, I)
    torch.cuda.synchronize()
    rng = np.random.default_rng(seed)
    for g in _sampled_experts(counts, rng):
        r = _sample_rows(off, g, rng)
        ridx = torch.from_numpy(r).cuda()
        ref = ref_fwd_rows(orc, bf16_bits_np(x[ridx]), bf16_bits_np(w_gu[g * 2 * I:(g + 1) * 2 * I]))
        check_gemm_tolerance(bf16_to_f64(y_gu[ridx]), ref, what=f"{label} gate/up expert {g}")
        ref = ref_fwd_rows(orc, bf16_bits_np(h[ridx]), bf16_bits_np(w_d[g * H:(g + 1) * H]))
        check_gemm_tolerance(bf16_to_f64(y_d[ridx]), ref, what=f"{label} down expert {g}")


def _moe_bwd_sampled(fme, orc, counts, seed, label):
    import torch

    off = synth.offsets_from_counts(counts)
    rows = int(off[-1])
    E, H, I = len(counts), synth.HIDDEN, synth.INTERMEDIATE
    dy = synth.torch_normal((rows, H), 1e-2, seed=seed * 10 + 5)
    h = synth.torch_normal((rows, I), 1.0, seed=seed * 10 + 3)
    w_d = synth.torch_normal((E * H, I), 0.02, seed=seed * 10 + 4)
    dh = gpu_dgrad(fme, dy, w_d, off, I, H)
    dw = gpu_wgrad(fme, dy, h, off)
    torch.cuda.synchronize()
    rng = np.random.default_rng(seed + 100)
    for g in _sampled_experts(counts, rng, count=3):
        r = _sample_rows(off, g, rng)
        ridx = torch.from_numpy(r).cuda()
        ref = ref_dgrad_rows(orc, bf16_bits_np(dy[ridx]), bf16_bits_np(w_d[g * H:(g + 1) * H]))
        check_gemm_tolerance(bf16_to_f64(dh[ridx]), ref, what=f"{label} dgrad expert {g}")
        chans = np.array(sorted({0, H - 1, *rng.integers(0, H, size=3).tolist()}))
        lo, hi = int(off[g]), int(off[g + 1])
        ref = ref_wgrad(orc, bf16_bits_np(dy[lo:hi]), bf16_bits_np(h[lo:hi]), rows_sel=chans)
        got = bf16_to_f64(dw[g][torch.from_numpy(chans).cuda()])
        check_gemm_tolerance(got, ref, what=f"{label} wgrad expert {g}")
    for g, c in enumerate(counts):
        if c == 0:
            assert bool((dw[g] == 0).all()), f"expert {g} without rows must get zero dW"


def test_moe_forward_dirichlet(fme, orc):
    """MoE forward, NVFP4: 65536 rows over 32 experts (Dirichlet loads)."""
    _moe_fwd_sampled(fme, orc, synth.dirichlet_counts(), seed=2, label="dirichlet")


def test_moe_forward_mxfp8_dirichlet(fme, orc):
    """MoE forward with MXFP8 operands (the continued-pretraining recipe): gate/up
    and down over 65536 rows in 32 experts, sampled rows of sampled experts."""
    import torch

    counts = synth.dirichlet_counts()
    off = synth.offsets_from_counts(counts)
    rows, E, H, I = int(off[-1]), len(counts), synth.HIDDEN, synth.INTERMEDIATE
    x = synth.torch_normal((rows, H), 1.0, seed=51)
    w_gu = synth.torch_normal((E * 2 * I, H), 0.02, seed=52)
    h = synth.torch_normal((rows, I), 1.0, seed=53)
    w_d = synth.torch_normal((E * H, I), 0.02, seed=54)
    y_gu = gpu_fwd_mxfp8(fme, x, w_gu, off, 2 * I, H)
    y_d = gpu_fwd_mxfp8(fme, h, w_d, off, H, I)
    torch.cuda.synchronize()
    rng = np.random.default_rng(5)
    for g in _sampled_experts(counts, rng):
        r = _sample_rows(off, g, rng)
        ridx = torch.from_numpy(r).cuda()
        ref = ref_fwd_mxfp8_rows(orc, bf16_bits_np(x[ridx]), bf16_bits_np(w_gu[g * 2 * I:(g + 1) * 2 * I]))
        check_gemm_tolerance(bf16_to_f64(y_gu[ridx]), ref, what=f"mxfp8 gate/up expert {g}")
        ref = ref_fwd_mxfp8_rows(orc, bf16_bits_np(h[ridx]), bf16_bits_np(w_d[g * H:(g + 1) * H]))
        check_gemm_tolerance(bf16_to_f64(y_d[ridx]), ref, what=f"mxfp8 down expert {g}")


def test_moe_backward_dirichlet(fme, orc):
    """MoE backward, MXFP8: same loads, dY ~ N(0, 0.01^2)."""
    _moe_bwd_sampled(fme, orc, synth.dirichlet_counts(), seed=3, label="dirichlet")


def test_moe_skewed_long_batch(fme, orc):
    """262144 rows, Zipf(1.2) loads with 3 empty experts: forward and backward."""
    counts = synth.zipf_counts()
    _moe_fwd_sampled(fme, orc, counts, seed=4, label="zipf")
    _moe_bwd_sampled(fme, orc, counts, seed=4, label="zipf")


def test_fwd_pertensor_comparator(fme, orc):
    """The forward GEMM on standard-NVFP4 X (one scale for the batch) against the
    oracle, and the reason for the per-token variant ("Composer 2 Technical
    Report", section 6.1): with a louder token appended to the batch, the earlier
    tokens' outputs change under the per-tensor scale and stay bit-identical under
    the per-token one."""
    import torch

    x_bits, _, _ = synth.quantizer_batch(rows=1024, cols=1024, seed=71)
    w_bits = synth.normal_bits((256, 1024), 0.02, seed=72)
    loud = synth.bf16_bits(synth.bf16_float(x_bits[:128]) * np.float32(64.0))
    st = _status()
    w = bf16_tensor(w_bits)
    wq = fme.quantize_nvfp4_pertoken(w, status=st)

    def fwd(xb, per_tensor):
        off = _i32([0, xb.shape[0]])
        x = bf16_tensor(xb)
        q = fme.quantize_nvfp4_pertensor(x, off, status=st)[:3] if per_tensor else \
            fme.quantize_nvfp4_pertoken(x, off, status=st)
        return fme.grouped_gemm_fwd_nvfp4(*q, *wq, off, 256, 1024, status=st)

    y_t = fwd(x_bits, True)
    a = orc.dequant_nvfp4(*orc.quant_nvfp4_pertensor(x_bits))
    b = orc.dequant_nvfp4(*orc.quant_nvfp4(w_bits))
    check_gemm_tolerance(bf16_to_f64(y_t), orc.gemm_abt(a, b), what="fwd per-tensor")
    both = np.concatenate([x_bits, loud])
    y_t2 = fwd(both, True)
    y_p, y_p2 = fwd(x_bits, False), fwd(both, False)
    _ok(fme, st)
    assert not torch.equal(y_t, y_t2[:1024])
    assert torch.equal(y_p, y_p2[:1024])


def test_many_experts_fwd_dgrad_wgrad(fme, orc):
    """1024 experts (the ABI's maximum: the group tables take 12 KB of shared memory
    and may shorten the operand ring), most of them empty, some with a single row;
    checked on a sample of experts."""
    rng = np.random.default_rng(91)
    counts = np.zeros(1024, np.int64)
    live = rng.choice(1024, size=40, replace=False)
    counts[live] = rng.integers(1, 300, size=40)
    counts[live[:3]] = 1
    off = synth.offsets_from_counts(counts)
    R, n, k = int(off[-1]), 256, 256
    x_bits = synth.normal_bits((R, k), 1.0, seed=92)
    w_bits = synth.normal_bits((1024 * n, k), 0.02, seed=93)
    y = bf16_to_f64(gpu_fwd(fme, bf16_tensor(x_bits), bf16_tensor(w_bits), off, n, k))
    wd_bits = synth.normal_bits((1024 * k, n), 0.02, seed=94)
    yd = bf16_to_f64(gpu_dgrad(fme, bf16_tensor(x_bits), bf16_tensor(wd_bits), off, n, k))
    h_bits = synth.normal_bits((R, n), 1.0, seed=95)
    dw = bf16_to_f64(gpu_wgrad(fme, bf16_tensor(x_bits), bf16_tensor(h_bits), off))
    for g in list(live[:6]) + [int(np.argmax(counts))]:
        lo, hi = int(off[g]), int(off[g + 1])
        check_gemm_tolerance(y[lo:hi], ref_fwd_rows(orc, x_bits[lo:hi], w_bits[g * n:(g + 1) * n]),
                             what=f"many-expert fwd {g}")
        check_gemm_tolerance(yd[lo:hi], ref_dgrad_rows(orc, x_bits[lo:hi], wd_bits[g * k:(g + 1) * k]),
                             what=f"many-expert dgrad {g}")
        check_gemm_tolerance(dw[g], ref_wgrad(orc, x_bits[lo:hi], h_bits[lo:hi]), what=f"many-expert wgrad {g}")
    empty = [g for g in range(1024) if counts[g] == 0][:50]
    assert not dw[empty].any()
