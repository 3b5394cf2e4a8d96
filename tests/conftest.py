import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle

    oracle._load()
    return oracle


@pytest.fixture(scope="session")
def gg():
    """The CUDA library binding, built in-tree if needed (fails loudly without it)."""
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import fp8_block_scaled_gb300 as lib

    lib.load()
    return lib
