import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(autouse=True)
def _gpu_guard(request):
    """A gpu-marked test fails (never skips) when no GPU is visible, so a run
    that expects a GPU cannot pass by silently not running the CUDA path."""
    if request.node.get_closest_marker("gpu") is not None:
        import torch
        assert torch.cuda.is_available(), "gpu test run without a visible CUDA device"
    yield
