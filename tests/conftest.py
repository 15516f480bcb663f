import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the CUDA library")


@pytest.fixture(scope="session")
def oracle_mod():
    import oracle

    oracle.build()
    return oracle


@pytest.fixture(scope="session")
def dflash_lib():
    """The CUDA library, built in-tree if it is missing or stale."""
    from speculative_decoding_draft_paged_gb300 import build as _build

    _build.build()
    import speculative_decoding_draft_paged_gb300 as dflash

    return dflash


@pytest.fixture(scope="session")
def cuda_device(dflash_lib):
    import torch

    if not torch.cuda.is_available():
        pytest.fail("the gpu tests need a CUDA device")
    return torch.device("cuda", 0)
