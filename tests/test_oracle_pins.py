"""The CPU oracle against its pins (no GPU)."""
import pytest

from tests import pins


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(orc, check):
    if check.__name__ in ("check_e2m1_encode_all_bf16",):
        pytest.importorskip("ml_dtypes")
    check(orc)


# ------------------------------------------- the golden fixtures, re-derived --
# The values in tests/golden were worked by hand.  These tests redo each
# derivation from the formulas the fixtures state, with numpy binary32 arithmetic
# (every step one correctly rounded fp32 operation) and the E4M3 / E2M1 roundings
# of torch's float8_e4m3fn and ml_dtypes' float4_e2m1fn casts -- neither the
# oracle nor the CUDA library is involved.
def _e4m3_code(v):
    import numpy as np
    import torch

    return int(torch.tensor([float(np.float32(v))], dtype=torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)[0])


def _e4m3_value(code):
    import torch

    return float(torch.tensor([code], dtype=torch.uint8).view(torch.float8_e4m3fn).to(torch.float32)[0])


def test_nvfp4_golden_rederived():
    import numpy as np

    ml = pytest.importorskip("ml_dtypes")
    from tests.golden import read_cases

    f = np.float32
    for name, case in read_cases("nvfp4_worked.txt").items():
        x = np.array([float(v) for v in case["x"].split()], np.float32)
        amax = f(np.max(np.abs(x)))
        s = f(amax) / f(2688.0)                          # fl32(amax / 2688)
        assert int(np.array([s], np.float32).view(np.uint32)[0]) == int(case["S_bits"], 16), name
        d = f(6.0) * s                                   # fl32(6 S)
        sb = _e4m3_code(f(amax) / d if amax > 0 else f(0.0))
        assert sb == int(case["sf"], 16), (name, hex(sb))
        e = f(_e4m3_value(sb)) * s                       # fl32(dec(sb) S)
        q = (x / e).astype(np.float32) if sb else np.zeros(16, np.float32)
        codes = q.astype(ml.float4_e2m1fn).view(np.uint8) & 0xF
        if sb == 0:
            codes[:] = 0
        want = [int(c, 16) for c in case["codes"].split()]
        assert [int(c) for c in codes] == want, (name, list(codes), want)


def test_mxfp8_golden_rederived():
    import numpy as np
    import torch

    from tests.golden import read_cases

    for name, case in read_cases("mxfp8_worked.txt").items():
        lead = np.array([float(v) for v in case["x"].split()], np.float32)
        amax = float(np.max(np.abs(lead)))
        if amax == 0.0:
            code = 0
        else:
            _, ex = np.frexp(amax)                        # amax = m 2^ex, 0.5 <= m < 1
            code = int(np.clip((ex - 1) - 8 + 127, 0, 254))
        assert code == int(case["scale"]), (name, code)
        scaled = lead.astype(np.float64) * 2.0 ** (127 - code)   # exact: a power-of-two scale
        got = torch.from_numpy(scaled.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
        # torch's cast does not saturate: values past 448 go to 448 (0x7e) by the format's satfinite rule
        big = np.abs(scaled) > 464.0
        got = np.where(big, np.where(scaled > 0, 0x7E, 0xFE), got)
        want = [int(c, 16) for c in case["codes"].split()]
        assert [int(c) for c in got] == want, (name, list(got), want)
