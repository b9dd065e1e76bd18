"""The CPU oracle against its pins (no GPU)."""
import pytest

from tests import pins


@pytest.mark.parametrize("check", pins.ALL_CHECKS, ids=lambda f: f.__name__)
def test_pin(orc, check):
    if check.__name__ in ("check_e2m1_encode_all_bf16",):
        pytest.importorskip("ml_dtypes")
    check(orc)
