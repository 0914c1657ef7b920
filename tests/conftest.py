import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs an sm_103 (GB300) GPU and the CUDA library")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle
    oracle._load()
    return oracle


@pytest.fixture(scope="session")
def fp8g():
    """The CUDA library's Python binding, built for sm_103a and loaded.

    A GPU test that cannot load it fails: there is no fallback path.
    """
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a host without a CUDA device")
    from fp8_block_scaled_nt_gb300 import _build
    _build.build()
    import fp8_block_scaled_nt_gb300 as lib
    lib.load()
    return lib
