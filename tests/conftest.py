import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")


import pytest  # noqa: E402


@pytest.fixture(scope="session")
def built_lib():
    """Build libinfllmv2.so (nvcc, sm_103a) once per session and load it."""
    from block_sparse_long_infllm_gb300 import build, infllmv2
    build.build()
    return infllmv2.load()


@pytest.fixture(scope="session")
def cuda_lib(built_lib):
    """The library on a CUDA device (for tests marked gpu)."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("test marked gpu needs a CUDA device")
    return built_lib
