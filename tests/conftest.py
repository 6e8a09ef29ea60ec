import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


import pytest


@pytest.fixture(scope="session")
def cplib():
    """Build (if stale) and load libcpattn.so."""
    from context_causal_attention_gb300 import build as _build
    from context_causal_attention_gb300 import _lib
    _build.build()
    return _lib.lib()


@pytest.fixture(scope="session")
def cuda_dev(cplib):
    import torch
    if not torch.cuda.is_available():
        pytest.fail("a GPU test was selected but no CUDA device is visible")
    return torch.device("cuda:0")
