import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload, minutes of host time")


@pytest.fixture(scope="session")
def lib():
    """The built C-ABI library (builds it in-tree if it is missing)."""
    from mla_latent_kv_73_b300 import _lib
    return _lib.load(build_if_missing=True)
