import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def gpu_available():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def cuda_lib():
    """The built CUDA library; GPU tests fail (not skip) when it is missing."""
    if not gpu_available():
        pytest.skip("no CUDA device")
    from paged_kv_decode_10_gb300 import binding
    return binding.load()


@pytest.fixture(scope="session")
def host_lib():
    """The library built in-tree (compiled here if needed) for host-only calls."""
    from paged_kv_decode_10_gb300 import binding, build
    build.build()
    return binding.load()
