import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a B300 GPU and the built CUDA library")


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library through its Python binding; GPU tests only."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import moe_ragged_bf16_grouped_b300 as gdg
    return gdg
