import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

# Tolerances for the CUDA path against the fp64 oracle (bf16 inputs, fp32
# accumulation, bf16 output): max |dO|, mean |dO|, max |dLSE|.
TOL_O_MAX = 2e-2
TOL_O_MEAN = 2e-3
TOL_LSE_MAX = 1e-3


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a GB300 (sm_103) GPU and the built CUDA library")
    config.addinivalue_line(
        "markers", "slow: full-size workloads (minutes)")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def tk_lib():
    """The built C library through its Python binding (builds it if needed)."""
    from attention_forward_tk_gb300 import api
    from attention_forward_tk_gb300.build import build_library
    build_library()
    api.library()
    return api


@pytest.fixture(scope="session")
def cuda_dev():
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a gpu-marked test ran without a CUDA device")
    return torch.device("cuda", 0)
