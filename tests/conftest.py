import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) GPU and the CUDA library")


@pytest.fixture(scope="session")
def cuda_device():
    """The CUDA device for GPU tests; skips only when no GPU is visible at all.

    With a GPU present the CUDA library must load: a missing or broken build is
    a test failure, never a silent fallback."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device visible")
    import mixed_precision_tensor_gb300 as tcg
    tcg.load_library()          # raises if the in-tree libtcg.so is missing
    return torch.device("cuda:0")
