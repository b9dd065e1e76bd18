"""Positive control for the NVFP4 quantizer's IEEE-division requirement.

"Composer 2 Technical Report", section 6.1, hardware-level math paragraph: the
NVFP4 variant's quantizer must divide with IEEE-compliant (correctly rounded)
division; a fast approximate divide made training diverge.  The library codes
every element as the E2M1 rounding of fl32(x / e), reached without dividing by
one exact correction step after a reciprocal product (checked exhaustively on
the CPU in tests/test_scale_division.py).  This test shows that the bit-exact
parity tests would notice a kernel that divided approximately: a second build of
the library with -DFME_TEST_APPROX_DIVIDE codes the elements from the plain
product x * rcp.approx(e), the quotient of a fast divide.  On a batch shaped like
the quantizer workload, the normal build's codes equal the oracle's; the
approximate build's differ from them on some elements, while its per-token and
block scales (computed the exact way in both builds) agree.  The same holds on the
rows built to put quotients next to every E2M1 midpoint, where the difference
shows on many more elements.
"""
import ctypes
import os

import numpy as np
import pytest

import fp8_moe_expert_gb300 as fme_mod
from fp8_moe_expert_gb300 import build as fme_build
from fp8_moe_expert_gb300 import synth
from tests.fmetest import bf16_tensor, to_np, unswizzle
from tests.test_gpu_quant import near_midpoint_rows

pytestmark = pytest.mark.gpu

APPROX_LIB = os.path.join(os.path.dirname(os.path.abspath(__file__)), "_build", "libfme_approx_divide.so")


@pytest.fixture(scope="module")
def approx_lib():
    os.makedirs(os.path.dirname(APPROX_LIB), exist_ok=True)
    fme_build.build(output=APPROX_LIB, extra_flags=["-DFME_TEST_APPROX_DIVIDE"])
    return fme_mod._declare(ctypes.CDLL(APPROX_LIB))


def _quantize(lib, x_bits):
    """codes, untiled block scales and per-token scales from one library build."""
    import torch

    rows, k = x_bits.shape
    x = bf16_tensor(x_bits)
    codes = torch.empty(rows, k // 2, dtype=torch.uint8, device="cuda")
    sf = torch.empty(fme_mod.sf_bytes(rows, k, 16), dtype=torch.uint8, device="cuda")
    scale = torch.empty(rows, dtype=torch.float32, device="cuda")
    st = torch.zeros(1, dtype=torch.int32, device="cuda")
    stream = ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)
    P = lambda t: ctypes.c_void_p(t.data_ptr())  # noqa: E731
    assert lib.quantize_nvfp4_pertoken(P(x), rows, k, None, 1, P(codes), P(sf), P(scale), P(st), stream) == 0
    code, raw = fme_mod.read_device_status(st)
    assert code == 0, hex(raw)
    return to_np(codes), unswizzle(to_np(sf), rows, k // 16), to_np(scale)


def test_approximate_divide_changes_codes_the_parity_tests_compare(fme, orc, approx_lib):
    x_bits, _, _ = synth.quantizer_batch(rows=2048)  # the quantizer workload's distribution, 2048 rows
    oc, osf, oscale = orc.quant_nvfp4(x_bits)

    codes, sf, scale = _quantize(fme.lib(), x_bits)
    assert np.array_equal(codes, oc) and np.array_equal(sf, osf)
    assert np.array_equal(scale.view(np.uint32), oscale.view(np.uint32))

    a_codes, a_sf, a_scale = _quantize(approx_lib, x_bits)
    assert np.array_equal(a_sf, osf) and np.array_equal(a_scale.view(np.uint32), oscale.view(np.uint32))
    differ = int(np.count_nonzero(a_codes != oc))
    # every differing byte is a near-midpoint quotient rounded the other way
    assert differ > 0, "an approximate divide went unnoticed: the control shows nothing"
    nibbles = int(np.count_nonzero((a_codes ^ oc) & 0x0F) + np.count_nonzero((a_codes ^ oc) & 0xF0))
    print(f"quantizer batch: {nibbles} of {x_bits.size} element codes differ under the approximate divide")
    assert nibbles < x_bits.size // 100, f"{nibbles} codes differ: more than near-midpoint quotients"


def test_approximate_divide_changes_near_midpoint_codes(fme, orc, approx_lib):
    x_bits = near_midpoint_rows()
    oc, osf, _ = orc.quant_nvfp4(x_bits)
    codes, _, _ = _quantize(fme.lib(), x_bits)
    assert np.array_equal(codes, oc)
    a_codes, a_sf, _ = _quantize(approx_lib, x_bits)
    assert np.array_equal(a_sf, osf)
    diff = a_codes ^ oc
    nibbles = int(np.count_nonzero(diff & 0x0F) + np.count_nonzero(diff & 0xF0))
    print(f"near-midpoint rows: {nibbles} of {x_bits.size} element codes differ under the approximate divide")
    assert nibbles > 0, "an approximate divide went unnoticed on near-midpoint rows"
