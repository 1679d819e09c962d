import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: full-size parity cases")


@pytest.fixture(scope="session")
def oracle_lib():
    import oracle
    oracle._load()
    return oracle


@pytest.fixture(scope="session")
def iso():
    """The CUDA library through its C-ABI (GPU tests only)."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without a CUDA device")
    from parallelism_invariant_logprob_gb300 import binding
    return binding.load()
