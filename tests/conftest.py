import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libds4a.so")


def gpu_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def ds4a_lib():
    """The C-ABI library, built in-tree on first use."""
    from compressed_sparse_mqa_gb300 import build as _b
    _b.build()
    from compressed_sparse_mqa_gb300 import ds4a
    return ds4a
