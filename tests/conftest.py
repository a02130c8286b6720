import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA device (GB300, sm_103a); run with -m gpu")


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA extension, built in-tree; GPU tests fail loudly without it."""
    import torch

    if not torch.cuda.is_available():
        pytest.fail("GPU test collected without a CUDA device")
    import exact_attention_90_gb300 as fa

    fa.load_library()  # raises if the shared library is missing
    return fa
