"""moe_route_noalloc: routing whose per-(chunk, expert) counters live in the
library's static device array, so the call allocates nothing.

CPU: the symbol is exported and the host refuses shapes past the static array.
GPU: the outputs equal moe_route's and the oracle's bit for bit, calls ordered
on one stream reuse the array correctly, and repeated calls change neither the
device's free memory nor torch's allocator counters.
"""
import ctypes

import numpy as np
import pytest

import fp8_moe_expert_gb300 as fme
from fp8_moe_expert_gb300 import synth

STATIC_WORDS = 1 << 20   # FME_ROUTE_STATIC_WORDS


def test_noalloc_symbol_and_host_checks():
    fme.ensure_built()
    lib = fme.lib()
    assert hasattr(lib, "moe_route_noalloc") and "moe_route_noalloc" in fme.SYMBOLS
    P = ctypes.c_void_p
    good, odd, s = P(0x100000), P(0x100001), P(0)
    r = lib.moe_route_noalloc
    # 8M assignments = 8192 chunks; x 1024 experts is past the static array
    assert r(good, 1 << 20, 8, 1024, good, good, good, None, s) == 3
    assert r(good, 10, 8, 0, good, good, good, None, s) == 1
    assert r(good, 10, 65, 32, good, good, good, None, s) == 1
    assert r(good, 10, 8, 32, None, good, good, None, s) == 1
    assert r(None, 10, 8, 32, good, good, good, None, s) == 1
    assert r(good, 10, 8, 32, good, good, odd, None, s) == 2


def _outputs(tokens, top_k, experts):
    import torch

    return (torch.empty(experts + 1, dtype=torch.int32, device="cuda"),
            torch.empty((tokens, top_k), dtype=torch.int32, device="cuda"),
            torch.empty(tokens * top_k, dtype=torch.int32, device="cuda"))


@pytest.mark.gpu
@pytest.mark.parametrize("tokens,top_k,experts", [(1, 1, 1), (1000, 8, 32), (32768, 8, 32), (4096, 8, 256),
                                                  (131072, 8, 1024)])
def test_noalloc_matches_route_and_oracle(orc, tokens, top_k, experts):
    import torch

    chunks = (tokens * top_k + 1023) // 1024
    assert chunks * experts <= STATIC_WORDS
    ids_np, _ = synth.topk_routing(tokens=tokens, top_k=top_k, experts=experts, seed=tokens + 3)
    ids = torch.from_numpy(ids_np).cuda()
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = fme.moe_route_noalloc(ids, experts, *_outputs(tokens, top_k, experts), status=st)
    b = fme.moe_route(ids, experts, status=st)
    code, raw = fme.read_device_status(st)
    assert code == 0, raw
    want = orc.route(ids_np, experts)
    for x, y, z in zip(a, b, want):
        assert np.array_equal(x.cpu().numpy(), y.cpu().numpy())
        assert np.array_equal(x.cpu().numpy(), z)


@pytest.mark.gpu
def test_noalloc_largest_static_shape_and_ordered_reuse(orc):
    """The full static array (1024 chunks x 1024 experts), then two calls queued
    back to back on one stream with different ids: each result is its own."""
    import torch

    tokens, top_k, experts = 131072, 8, 1024
    assert ((tokens * top_k + 1023) // 1024) * experts == STATIC_WORDS
    rng = np.random.default_rng(12)
    ids1 = rng.integers(0, experts, size=(tokens, top_k)).astype(np.int32)
    ids2 = np.ascontiguousarray(ids1[::-1])
    o1, o2 = _outputs(tokens, top_k, experts), _outputs(tokens, top_k, experts)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fme.moe_route_noalloc(torch.from_numpy(ids1).cuda(), experts, *o1, status=st)
    fme.moe_route_noalloc(torch.from_numpy(ids2).cuda(), experts, *o2, status=st)
    code, raw = fme.read_device_status(st)
    assert code == 0, raw
    for got, ids in ((o1, ids1), (o2, ids2)):
        for x, z in zip(got, orc.route(ids, experts)):
            assert np.array_equal(x.cpu().numpy(), z)


@pytest.mark.gpu
def test_noalloc_makes_no_allocation():
    import torch

    tokens, top_k, experts = 32768, 8, 32
    ids_np, _ = synth.topk_routing(tokens=tokens, top_k=top_k, experts=experts, seed=9)
    ids = torch.from_numpy(ids_np).cuda()
    outs = _outputs(tokens, top_k, experts)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    fme.moe_route_noalloc(ids, experts, *outs, status=st)     # loads the module once
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    n0 = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
    for _ in range(20):
        fme.moe_route_noalloc(ids, experts, *outs, status=st)
    torch.cuda.synchronize()
    free1, _ = torch.cuda.mem_get_info()
    n1 = torch.cuda.memory_stats().get("allocation.all.allocated", 0)
    # torch's allocator counter is this process's own record: no allocation at all
    assert n1 == n0
    assert fme.read_device_status(st)[0] == 0
    # the device-wide free memory also counts other processes on a shared GPU,
    # so a change there is reported, not failed on
    if free1 != free0:
        import warnings

        warnings.warn(f"device free memory moved by {free0 - free1} bytes during the calls (other processes?)")


def test_noalloc_binding_refuses_host_tensors():
    """The binding checks its buffers before calling the library: host tensors
    (or any buffer that is not a contiguous int32 CUDA tensor of the right size)
    are refused, so an undersized buffer never reaches the kernel."""
    import torch

    ids = torch.zeros((4, 2), dtype=torch.int32)
    outs = (torch.empty(5, dtype=torch.int32), torch.empty((4, 2), dtype=torch.int32),
            torch.empty(8, dtype=torch.int32))
    with pytest.raises(ValueError):
        fme.moe_route_noalloc(ids, 4, *outs)


@pytest.mark.gpu
def test_noalloc_binding_refuses_wrong_buffers():
    import torch

    tokens, top_k, experts = 64, 2, 4
    ids = torch.zeros((tokens, top_k), dtype=torch.int32, device="cuda")
    good = _outputs(tokens, top_k, experts)
    bad_cases = [
        (torch.empty(experts, dtype=torch.int32, device="cuda"), good[1], good[2]),               # offsets short
        (good[0], torch.empty((tokens, top_k - 1), dtype=torch.int32, device="cuda"), good[2]),   # row_of short
        (good[0], good[1], torch.empty(tokens * top_k, dtype=torch.int64, device="cuda")),        # src_row int64
        (good[0], good[1].t(), good[2]),                                                          # not contiguous
    ]
    for outs in bad_cases:
        with pytest.raises(ValueError):
            fme.moe_route_noalloc(ids, experts, *outs)
    with pytest.raises(ValueError):
        fme.moe_route_noalloc(ids.to(torch.int64), experts, *good)
