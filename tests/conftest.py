import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the compiled CUDA library")


@pytest.fixture(scope="session")
def oracle():
    import oracle as _oracle
    _oracle.build()
    return _oracle.Oracle()


@pytest.fixture(scope="session")
def sgemm_lib():
    """The compiled C-ABI library (built on demand); no GPU needed to load it."""
    import dense_fp32_matrix_07_gb300 as pkg
    return pkg.load()


@pytest.fixture(scope="session")
def cuda_device():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without a CUDA device")
    torch.cuda.init()
    return torch.device("cuda:0")
