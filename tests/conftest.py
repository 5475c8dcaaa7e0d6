import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (sm_103a) and the built library")


@pytest.fixture(scope="session")
def cuda_lib():
    """The product library on cuda:0; the test fails loudly when it is missing."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a gpu-marked test ran without a CUDA device")
    import exact_io_aware_26_gb300 as fa
    fa.load()
    return fa
