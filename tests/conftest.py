import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libtt")


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")


@pytest.fixture(scope="session")
def tt():
    """The CUDA library, built in-tree if stale (GPU tests only)."""
    import torch
    from prefix_tree_gb300 import build
    import prefix_tree_gb300
    if not torch.cuda.is_available():
        pytest.fail("GPU test run without a CUDA device")
    build.build()
    prefix_tree_gb300.lib()
    return prefix_tree_gb300
