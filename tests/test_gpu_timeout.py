"""The bounded waits' failure path, exercised by a build whose waits give up
after 1 us and read the clock after every barrier poll
(-DFME_WAIT_LIMIT_NS=1000 -DFME_WAIT_SPINS=1): the grouped GEMMs' roles then
run out of time waiting for copies and MMAs that are merely slow, not missing.

A kernel that gives up must report FME_DEV_TIMEOUT through the status word and
return: the copies and MMAs already issued land first (those drains keep their
own 2 s limit; the leader of each CTA pair waits for both producers' copies,
whose counts may differ after an abort), tensor memory is freed, and the context
stays usable.  Each short-wait run must either report the time-out or give the
normal library's result bit for bit; at least one run of each kernel must time
out (a 65536-deep K keeps every accumulator wait at tens of microseconds).  The
normal library's result after the short runs must equal its result before them.
No wait is made to hang: the short build only changes when a wait stops."""
import ctypes
import os

import pytest

import fp8_moe_expert_gb300 as fme_mod
from fp8_moe_expert_gb300 import build as fme_build
from fp8_moe_expert_gb300 import synth

pytestmark = pytest.mark.gpu

SHORT_LIB = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libfme_short_wait.so")
K_DEEP = 65536
N = 1024
COUNTS = (200, 256)  # two experts: a ragged row block and a full one, 4 column tiles each
RUNS = 4


@pytest.fixture(scope="module")
def short_lib():
    os.makedirs(os.path.dirname(SHORT_LIB), exist_ok=True)
    fme_build.build(output=SHORT_LIB, extra_flags=["-DFME_WAIT_LIMIT_NS=1000ull", "-DFME_WAIT_SPINS=1"])
    return fme_mod._declare(ctypes.CDLL(SHORT_LIB))


def _P(t):
    return ctypes.c_void_p(t.data_ptr())


def _short_runs(fme, call_short, y_ref, st):
    """Launch the short-wait build RUNS times; returns how many runs timed out."""
    import torch

    timeouts = 0
    for _ in range(RUNS):
        st.zero_()
        y = torch.zeros_like(y_ref)
        assert call_short(y) == 0, "the launch itself must succeed"
        code, raw = fme.read_device_status(st)  # synchronises: the kernel has returned
        if code == fme.ERR_DEVICE_TIMEOUT:
            assert raw & fme.DEV_TIMEOUT, hex(raw)
            timeouts += 1
        else:
            assert code == 0, hex(raw)
            assert torch.equal(y.view(torch.int16), y_ref.view(torch.int16)), "a run that did not time out differs"
    return timeouts


def _nvfp4_operand(fme, rows, k, num_groups, seed):
    """A well-formed NVFP4 operand deeper than the quantizer accepts: seeded E2M1
    code bytes (every nibble is a finite value), E4M3 block scales in
    [0.5, 1.875] (bytes 0x30 to 0x3f) and unit row scales, in the sizes of the
    tiled layout.  Only the failure path is under test, so the values need not come
    from a quantization."""
    import torch

    g = torch.Generator(device="cpu").manual_seed(seed)
    codes = torch.randint(0, 256, (rows, k // 2), generator=g, dtype=torch.int32).to(torch.uint8)
    sf = torch.randint(0x30, 0x40, (fme.sf_bytes(rows, k, 16, num_groups),), generator=g,
                       dtype=torch.int32).to(torch.uint8)
    return codes.cuda(), sf.cuda(), torch.ones(rows, dtype=torch.float32, device="cuda")


def test_forward_gemm_times_out_and_leaves_the_gpu_usable(fme, short_lib):
    import torch

    off_list = [0, COUNTS[0], sum(COUNTS)]
    off = torch.tensor(off_list, dtype=torch.int32, device="cuda")
    m, e = off_list[-1], len(COUNTS)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    a = _nvfp4_operand(fme, m, K_DEEP, e, 61)
    b = _nvfp4_operand(fme, e * N, K_DEEP, 1, 62)
    y_before = fme.grouped_gemm_fwd_nvfp4(*a, *b, off, N, K_DEEP, status=st)
    assert fme.read_device_status(st)[0] == 0
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def call_short(y):
        return short_lib.grouped_gemm_fwd_nvfp4(*map(_P, a), *map(_P, b), _P(off), e, m, N, K_DEEP, _P(y), _P(st),
                                                stream)

    assert _short_runs(fme, call_short, y_before, st) > 0, "no short-wait run timed out"
    st.zero_()
    y_after = fme.grouped_gemm_fwd_nvfp4(*a, *b, off, N, K_DEEP, status=st)
    assert fme.read_device_status(st)[0] == 0
    assert torch.equal(y_before.view(torch.int16), y_after.view(torch.int16))
    assert torch.isfinite(y_after.float()).all() and float(y_after.float().abs().max()) > 0


def test_dgrad_gemm_times_out_and_leaves_the_gpu_usable(fme, short_lib):
    import torch

    off_list = [0, COUNTS[0], sum(COUNTS)]
    off = torch.tensor(off_list, dtype=torch.int32, device="cuda")
    m, e = off_list[-1], len(COUNTS)
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    dy = synth.torch_normal((m, K_DEEP), 1e-2, 63)
    w = synth.torch_normal((e * K_DEEP, N), 0.02, 64)  # per expert [K_DEEP x N], reduced over its K_DEEP rows
    a_codes, a_sf = fme.quantize_mxfp8(dy, fme.ROWWISE, off, status=st)
    b_codes, b_sf, _, ldb = fme.quantize_mxfp8(w, fme.COLWISE, status=st)
    del dy, w
    y_before = fme.grouped_gemm_dgrad_mxfp8(a_codes, a_sf, b_codes, b_sf, ldb, off, N, K_DEEP, status=st)
    assert fme.read_device_status(st)[0] == 0
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)

    def call_short(y):
        return short_lib.grouped_gemm_dgrad_mxfp8(_P(a_codes), _P(a_sf), _P(b_codes), _P(b_sf), ldb, _P(off), e, m,
                                                  N, K_DEEP, _P(y), _P(st), stream)

    assert _short_runs(fme, call_short, y_before, st) > 0, "no short-wait run timed out"
    st.zero_()
    y_after = fme.grouped_gemm_dgrad_mxfp8(a_codes, a_sf, b_codes, b_sf, ldb, off, N, K_DEEP, status=st)
    assert fme.read_device_status(st)[0] == 0
    assert torch.equal(y_before.view(torch.int16), y_after.view(torch.int16))
    assert torch.isfinite(y_after.float()).all() and float(y_after.float().abs().max()) > 0
