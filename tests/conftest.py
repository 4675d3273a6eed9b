import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def cuda():
    import torch
    if not torch.cuda.is_available():
        pytest.skip("CUDA GPU required")
    return torch.device("cuda:0")


def pytest_sessionstart(session):
    # (Re)build the CUDA library and the CPU oracle when their sources are
    # newer than the binaries; a no-op when they are current.
    from gemv_w4a16_gemm_gb300 import build as libbuild
    import oracle
    libbuild.build()
    oracle.build()
