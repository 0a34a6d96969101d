import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built CUDA library on a GPU machine; GPU tests fail (not skip) when it
    is missing, so a silent fallback can never pass them."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but torch.cuda.is_available() is False")
    import mamba_mimo_chunked_gb300 as mm
    mm.load_library()
    return mm
