import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def golden(name):
    import json

    with open(os.path.join(ROOT, "tests", "golden", name)) as f:
        return json.load(f)


def _build_libraries():
    """Build the oracle (gcc) and the CUDA library (nvcc, sm_103a) if stale."""
    import __graft_entry__

    __graft_entry__.build()


_build_libraries()


@pytest.fixture(scope="session")
def cuda_device():
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    return torch.device("cuda", 0)
