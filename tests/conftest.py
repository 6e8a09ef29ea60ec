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


@pytest.fixture(autouse=True)
def _no_kernel_gave_up(request):
    """After every test that used the GPU, no kernel may have given up a bounded
    wait: such a kernel leaves its outputs unwritten, which a value check would
    report only as a mismatch.  The failure self-tests read (and so clear) the
    status word themselves."""
    yield
    if "cuda_dev" not in request.fixturenames:
        return
    from context_causal_attention_gb300 import ops as F
    code = F.cp_device_status()
    assert code == 0, "a kernel gave up a bounded wait during this test (device status %d)" % code
