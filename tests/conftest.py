import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle.lib()
    return oracle


def cuda_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def pkv():
    """The CUDA library through its Python binding; it is built on first use
    and never replaced by anything else: without a GPU the tests that ask for
    it are not collected as GPU tests in the first place."""
    if not cuda_available():
        pytest.fail("gpu test run without a CUDA device")
    import paged_kv_decode_pages_gb300 as pkv_mod
    pkv_mod.load()
    return pkv_mod
