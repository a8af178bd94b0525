import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a); runs the CUDA library")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    return oracle.default()


@pytest.fixture(scope="session")
def tgemm():
    """The CUDA library's Python binding, loaded for a GPU test."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import tiled_matrix_multiplication_sm_gb300 as t
    t.load()            # raises if the compiled library is missing
    return t
