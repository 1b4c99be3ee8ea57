import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: longer CPU case")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built CUDA library on a GPU; GPU tests fail (not skip) when it cannot load."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    from transformer_decode_step_ns_gb300 import _lib
    return _lib.lib()
