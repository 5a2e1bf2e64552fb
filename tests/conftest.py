import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workload parity (GPU)")


def pytest_collection_modifyitems(config, items):
    # A test marked gpu on a machine without a GPU is a configuration error of
    # the run, not a skip: the driver selects them with -m gpu only on a GPU machine.
    pass


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library's Python binding (builds the .so first if missing)."""
    import torch
    if not torch.cuda.is_available():
        pytest.fail("gpu test selected but no CUDA device is visible")
    from deepseek_v4_sparse_indexer_gb300 import _binding
    _binding.load()
    return _binding
