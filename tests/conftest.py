import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


@pytest.fixture(scope="session")
def cuda_lib_path():
    """Path of the in-tree libattn.so, building it (nvcc cross-compiles) when absent or stale."""
    from attention_forward_attn_gb300 import build as pkg_build
    return pkg_build.build_library()
