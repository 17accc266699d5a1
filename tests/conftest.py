import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size parity case")


@pytest.fixture(scope="session")
def cuda_lib():
    """The loaded C-ABI library for GPU tests (fails loudly if the build is missing)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import pagedattention_kv_cache_paged_gb300 as pa
    pa.load_library()
    return pa
