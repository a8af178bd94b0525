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


@pytest.fixture(scope="session")
def workload_reference():
    """The oracle's full product (C_ref, absAB) of a named workload, computed
    once per session and shared by the tests of every path that run it.

    Returns a function name -> (A, B, C_ref, absAB) with A and B the host
    operands the CUDA path receives."""
    cache = {}

    def get(name):
        if name not in cache:
            import oracle
            from tiled_matrix_multiplication_sm_gb300 import inputs
            w = inputs.WORKLOADS[name]
            A, B = inputs.operands(w)
            C_ref, absAB = oracle.gemm(A, B)
            cache[name] = (A, B, C_ref, absAB)
        return cache[name]

    return get
