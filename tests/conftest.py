import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GB300 (sm_103) device; runs the CUDA path")


@pytest.fixture(scope="session")
def built_library():
    """Build libmlaqp.so if it is missing or stale, then load it."""
    from mla_decode_query_gb300 import build, load_library
    build.build_library()
    return load_library()


@pytest.fixture(scope="session")
def cuda_device(built_library):
    """The GPU tests must run on the CUDA path: fail (never skip) without it."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but CUDA is not available")
    torch.cuda.init()
    return torch.device("cuda:0")
