import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload, minutes of host time")


@pytest.fixture(scope="session")
def gpu_lib():
    """The built C-ABI library with a CUDA device (fails loudly when either is missing)."""
    import torch

    if not torch.cuda.is_available():
        pytest.fail("GPU test collected on a machine without CUDA")
    import tree_speculative_decoding_array_gb300 as tsv

    tsv.load()
    return tsv
