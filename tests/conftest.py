import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) and the CUDA library")
    # temporary files of the tests (tmp_path) stay inside the repository, git-ignored;
    # pytest empties this directory at the start of each session
    if not config.option.basetemp:
        config.option.basetemp = os.path.join(ROOT, "tests", "_tmp")


@pytest.fixture(scope="session")
def orc():
    import oracle

    return oracle.Oracle()


@pytest.fixture(scope="session")
def fme():
    """The CUDA library's Python binding; built on first use, never a fallback."""
    import torch

    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without a GPU")
    import fp8_moe_expert_gb300 as fme_mod

    fme_mod.ensure_built()
    return fme_mod
