"""Routing on the GPU: grouping the routed tokens by expert, quantizing them in
grouped order, and combining the experts' outputs per token.

The grouping is integer work and is compared bit for bit with the oracle's
stable counting sort; the permuted quantizations bit for bit with the oracle's
quantizers on the gathered rows; the combine (fp32 products and sums in k order,
one bf16 rounding) bit for bit with the oracle's combine.
"""
import numpy as np
import pytest

from fp8_moe_expert_gb300 import synth
from tests.fmetest import bf16_bits_np, bf16_tensor, padded_rows, sf_index, to_np, unswizzle

pytestmark = pytest.mark.gpu


def _i32(a):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a, np.int32)).cuda()


def _f32(a):
    import torch

    return torch.from_numpy(np.ascontiguousarray(a, np.float32)).cuda()


def _status():
    import torch

    return torch.zeros(1, dtype=torch.int32, device="cuda")


def run_route(fme, ids, experts):
    st = _status()
    off, row_of, src = fme.moe_route(_i32(ids), experts, status=st)
    code, raw = fme.read_device_status(st)
    return to_np(off), to_np(row_of), to_np(src), code, raw


@pytest.mark.parametrize("tokens,top_k,experts", [
    (1, 1, 1), (1, 8, 32), (1000, 8, 32), (3000, 6, 40), (129, 3, 1024), (8192, 8, 256), (32768, 8, 32),
    (65536, 2, 7),
])
def test_route_matches_oracle(fme, orc, tokens, top_k, experts):
    ids, _ = synth.topk_routing(tokens=tokens, top_k=top_k, experts=experts, seed=tokens + experts)
    off, row_of, src, code, raw = run_route(fme, ids, experts)
    assert code == 0, raw
    o_off, o_row, o_src = orc.route(ids, experts)
    assert np.array_equal(off, o_off)
    assert np.array_equal(row_of, o_row)
    assert np.array_equal(src, o_src)


def test_route_one_hot_expert_and_skew(fme, orc):
    """All assignments to one expert (the others empty), then a load where every
    chunk of assignments sees a different mix."""
    ids = np.full((5000, 4), 17, np.int32)
    off, row_of, src, code, _ = run_route(fme, ids, 32)
    assert code == 0
    assert list(off) == [0] * 18 + [20000] * 15
    assert np.array_equal(src, np.arange(20000))
    rng = np.random.default_rng(5)
    ids = np.sort(rng.integers(0, 64, size=(7000, 5)), axis=0).astype(np.int32)
    off, row_of, src, code, _ = run_route(fme, ids, 64)
    o_off, o_row, o_src = orc.route(ids, 64)
    assert code == 0 and np.array_equal(off, o_off) and np.array_equal(row_of, o_row) and np.array_equal(src, o_src)


def test_route_empty(fme):
    off, row_of, src, code, _ = run_route(fme, np.zeros((0, 8), np.int32), 32)
    assert code == 0 and list(off) == [0] * 33 and row_of.size == 0


def test_route_invalid_ids_reported(fme, orc):
    ids, _ = synth.topk_routing(tokens=2000, top_k=4, experts=16, seed=3)
    ids[7, 1] = -1
    ids[1500, 3] = 16
    ids[1999, 0] = 1 << 30
    off, row_of, src, code, raw = run_route(fme, ids, 16)
    assert code == 8 and raw & fme.DEV_BAD_INDEX
    o_off, o_row, o_src = orc.route(ids, 16)
    assert np.array_equal(off, o_off) and np.array_equal(row_of, o_row)
    assert np.array_equal(src[: int(o_off[-1])], o_src)
    assert row_of[7, 1] == -1 and row_of[1500, 3] == -1 and row_of[1999, 0] == -1


def test_route_deterministic(fme):
    ids, _ = synth.topk_routing(tokens=20000, top_k=8, experts=32, seed=8)
    a = run_route(fme, ids, 32)
    b = run_route(fme, ids, 32)
    assert all(np.array_equal(x, y) for x, y in zip(a[:3], b[:3]))


def test_route_host_checks(fme):
    ids = _i32(np.zeros((4, 2), np.int32))
    with pytest.raises(fme.FmeError):
        fme.moe_route(ids, 0)
    with pytest.raises(fme.FmeError):
        fme.moe_route(ids, 2000)
    import torch

    with pytest.raises(fme.FmeError):   # workspace too small
        fme.moe_route(ids, 4, workspace=torch.empty(0, dtype=torch.uint8, device="cuda"))


# ------------------------------------------------------- permute + quantize --
def _tokens_x(tokens, k, seed):
    rng = np.random.default_rng(seed)
    x = rng.standard_normal((tokens, k), dtype=np.float32)
    x[rng.random(x.shape) < 0.002] *= 60.0
    if tokens > 3:
        x[3] = 0.0
    return synth.bf16_bits(x)


@pytest.mark.parametrize("tokens,top_k,experts,k", [(1, 1, 1, 64), (300, 8, 32, 2048), (97, 4, 9, 7168),
                                                    (2000, 8, 32, 576)])
def test_permute_quantize_nvfp4(fme, orc, tokens, top_k, experts, k):
    ids, _ = synth.topk_routing(tokens=tokens, top_k=top_k, experts=experts, seed=tokens + 1)
    x_bits = _tokens_x(tokens, k, seed=k)
    st = _status()
    off, row_of, src = fme.moe_route(_i32(ids), experts, status=st)
    x = bf16_tensor(x_bits)
    codes, sf, scale = fme.permute_quantize_nvfp4(x, src, top_k, off, status=st)
    code, raw = fme.read_device_status(st)
    assert code == 0, raw
    src_np, off_np = to_np(src), to_np(off)
    gathered = x_bits[src_np // top_k]
    oc, osf, oscale = orc.quant_nvfp4(gathered)
    rows = tokens * top_k
    assert np.array_equal(to_np(codes), oc)
    assert np.array_equal(unswizzle(to_np(sf), rows, k // 16, off_np), osf)
    assert np.array_equal(to_np(scale).view(np.uint32), oscale.view(np.uint32))
    # the same bytes as quantizing the materialised grouped rows
    pc, psf, ps = fme.quantize_nvfp4_pertoken(x[src.long() // top_k].contiguous(), off, status=st)
    assert np.array_equal(to_np(pc), to_np(codes)) and np.array_equal(to_np(ps), to_np(scale))


@pytest.mark.parametrize("tokens,top_k,experts,k", [(1, 1, 1, 32), (300, 8, 32, 7168), (129, 3, 5, 96)])
def test_permute_quantize_mxfp8(fme, orc, tokens, top_k, experts, k):
    ids, _ = synth.topk_routing(tokens=tokens, top_k=top_k, experts=experts, seed=tokens + 2)
    x_bits = _tokens_x(tokens, k, seed=k + 1)
    st = _status()
    off, row_of, src = fme.moe_route(_i32(ids), experts, status=st)
    codes, sf = fme.permute_quantize_mxfp8(bf16_tensor(x_bits), src, top_k, off, status=st)
    code, raw = fme.read_device_status(st)
    assert code == 0, raw
    src_np, off_np = to_np(src), to_np(off)
    oc, osf = orc.quant_mxfp8_rows(x_bits[src_np // top_k])
    assert np.array_equal(to_np(codes), oc)
    assert np.array_equal(unswizzle(to_np(sf), tokens * top_k, k // 32, off_np), osf)


def test_permute_quantize_bad_index_reported(fme):
    import torch

    x = bf16_tensor(_tokens_x(16, 256, seed=1))
    off = _i32([0, 32, 64])
    src = torch.arange(64, dtype=torch.int32, device="cuda")
    src[10] = 64          # 64 // 4 = token 16: past the 16 tokens
    src[20] = -4
    for fn in (fme.permute_quantize_nvfp4, fme.permute_quantize_mxfp8):
        st = _status()
        fn(x, src, 4, off, status=st)
        code, raw = fme.read_device_status(st)
        assert code == 8 and raw & fme.DEV_BAD_INDEX


# ------------------------------------------------------------------ combine --
def run_combine(fme, y_bits, row_of, w):
    st = _status()
    out = fme.moe_combine(bf16_tensor(y_bits), _i32(row_of), _f32(w), status=st)
    code, raw = fme.read_device_status(st)
    return bf16_bits_np(out), code, raw


@pytest.mark.parametrize("tokens,top_k,experts,n", [(1, 1, 1, 8), (700, 8, 32, 7168), (333, 6, 16, 264),
                                                    (64, 64, 64, 256), (5, 3, 4, 2056)])
def test_combine_matches_oracle(fme, orc, tokens, top_k, experts, n):
    ids, w = synth.topk_routing(tokens=tokens, top_k=top_k, experts=experts, seed=n + tokens)
    off, row_of, _ = orc.route(ids, experts)
    y = synth.normal_bits((int(off[-1]), n), 1.5, seed=n)
    out, code, raw = run_combine(fme, y, row_of, w)
    assert code == 0, raw
    assert np.array_equal(out, orc.combine(y, row_of, w))


def test_combine_closed_form_rounding(fme, orc):
    """The fp32 tie case: 1 + 2^-8 + 2^-30 sums to the bf16 tie in fp32 and
    rounds to even (an fp64 or fused sum would round up); products rounded
    before the add; skipped assignments."""
    t = 2.0 ** -30
    y = synth.bf16_bits(np.array([[1.0] * 8, [2.0 ** -8] * 8, [t] * 8, [-(1.0 + 2.0 ** -7)] * 8,
                                  [1.0 + 2.0 ** -7] * 8], np.float32))
    row_of = np.array([[0, 1, 2], [3, 4, -1], [-1, -1, -1]], np.int32)
    w = np.array([[1.0, 1.0, 1.0], [1.0, 1.0 + 2.0 ** -23, 5.0], [1.0, 1.0, 1.0]], np.float32)
    out, code, _ = run_combine(fme, y, row_of, w)
    assert code == 0
    v = synth.bf16_float(out)
    assert np.all(v[0] == 1.0) and np.all(v[1] == np.float32(2.0 ** -23)) and np.all(v[2] == 0.0)
    assert np.array_equal(out, orc.combine(y, row_of, w))


def test_combine_bad_row_reported(fme):
    y = synth.normal_bits((10, 64), 1.0, seed=2)
    row_of = np.array([[0, 3], [10, 1]], np.int32)
    w = np.ones((2, 2), np.float32)
    _, code, raw = run_combine(fme, y, row_of, w)
    assert code == 8 and raw & fme.DEV_BAD_INDEX


def test_combine_empty_tokens(fme):
    import torch

    y = bf16_tensor(synth.normal_bits((4, 64), 1.0, seed=2))
    out = fme.moe_combine(y, _i32(np.zeros((0, 8), np.int32)), torch.zeros((0, 8), device="cuda"))
    assert out.shape == (0, 64)


# ------------------------------------------------------ the bench's workload --
def test_routing_full_size_sampled(fme, orc):
    """32768 tokens x top-8 over 32 experts, hidden 7168: the grouping in full,
    the grouped NVFP4 quantization and the combine on sampled tokens."""
    import torch

    tokens, top_k, experts, k = 32768, 8, 32, 7168
    ids, w = synth.topk_routing(tokens=tokens, top_k=top_k, experts=experts)
    st = _status()
    off, row_of, src = fme.moe_route(_i32(ids), experts, status=st)
    x = synth.torch_normal((tokens, k), 1.0, seed=41)
    codes, sf, scale = fme.permute_quantize_nvfp4(x, src, top_k, off, status=st)
    y = synth.torch_normal((tokens * top_k, k), 0.5, seed=42)
    out = fme.moe_combine(y, row_of, _f32(w), status=st)
    code, raw = fme.read_device_status(st)
    assert code == 0, raw
    o_off, o_row, o_src = orc.route(ids, experts)
    assert np.array_equal(to_np(off), o_off) and np.array_equal(to_np(row_of), o_row)
    assert np.array_equal(to_np(src), o_src)
    rng = np.random.default_rng(43)
    rows = np.sort(rng.choice(tokens * top_k, size=96, replace=False))
    rows_t = torch.from_numpy(rows).cuda()
    gathered = bf16_bits_np(x[torch.from_numpy(o_src[rows] // top_k).cuda().long()])
    oc, osf, oscale = orc.quant_nvfp4(gathered)
    assert np.array_equal(to_np(codes[rows_t]), oc)
    assert np.array_equal(to_np(scale[rows_t]).view(np.uint32), oscale.view(np.uint32))
    pr = padded_rows(o_off)[rows]
    idx = sf_index(pr[:, None], np.arange(k // 16)[None, :], k // 16)
    assert np.array_equal(to_np(sf)[idx], osf)
    toks = np.sort(rng.choice(tokens, size=64, replace=False))
    ro = o_row[toks]
    y_rows = bf16_bits_np(y[torch.from_numpy(ro.ravel()).cuda().long()])
    local = np.arange(ro.size, dtype=np.int32).reshape(ro.shape)
    want = orc.combine(y_rows, local, w[toks])
    assert np.array_equal(bf16_bits_np(out)[toks], want)
