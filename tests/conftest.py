import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built libmla.so")
    config.addinivalue_line("markers", "slow: large CPU oracle work")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="session")
def mla():
    """The ctypes binding of libmla.so, built first if needed (build is CPU-only cross compilation)."""
    from mla_latent_cache_gb300 import build as _build
    if not os.path.exists(_build.LIB):
        _build.build()
    from mla_latent_cache_gb300 import binding
    return binding


@pytest.fixture(scope="session")
def cuda(mla):
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test selected but no CUDA device is visible")
    return torch.device("cuda:0")
