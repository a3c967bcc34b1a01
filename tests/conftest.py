import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def lib():
    """The CUDA library binding; only for tests marked gpu."""
    import torch

    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import weight_only_int4_quant_gb300 as tlq

    tlq.load()
    return tlq
