import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: large CPU oracle case")


@pytest.fixture(scope="session")
def lib():
    """The C-ABI library through its Python binding (GPU tests only).  Every
    call that takes a device status word and is not given one by the test
    runs with a fresh word that must read MOE_OK afterwards."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from unpermute_moe_permute_gb300 import binding
    from gpu_util import StatusChecked
    return StatusChecked(binding)
