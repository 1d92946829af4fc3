import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workloads (minutes)")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built C-ABI library on a machine with a GPU (built on demand)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import mla_decode_attention_paged_gb300 as mla
    mla.load_library(build_if_missing=True)
    return mla
