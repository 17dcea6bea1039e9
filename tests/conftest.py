import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


@pytest.fixture(scope="session")
def cuda_available():
    import torch
    return torch.cuda.is_available()


@pytest.fixture(autouse=True)
def device_error_word_clear(request):
    """After every GPU test: the library's device error word must read 0.

    Kernels record skipped bad slots or copy triples and timed-out waits there;
    a test that provokes one on purpose reads (and so clears) the word itself.
    An error left behind means a kernel returned early and its output is not
    defined, whatever the test compared.
    """
    yield
    if request.node.get_closest_marker("gpu") is None:
        return
    import torch
    if not torch.cuda.is_available():
        return
    from paged_kv_cache_kvcache_gb300 import pagedattn as pa
    code = pa.pa_read_device_error()
    assert code == 0, f"device error word {code:#x} left set by {request.node.name}"
