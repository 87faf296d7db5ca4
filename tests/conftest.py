import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: long-running")


@pytest.fixture(scope="session")
def gpu_lib():
    """The product library, built for this machine, with a CUDA device present."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import sparse_top_kv_fathom_gb300 as F
    F.load()
    return F
