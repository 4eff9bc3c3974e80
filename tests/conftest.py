import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _load_by_path(name, rel):
    import importlib.util
    spec = importlib.util.spec_from_file_location(name, os.path.join(ROOT, rel))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a B300 GPU and the built CUDA library")
    # Build the CUDA library (nvcc cross-compiles without a GPU) and the oracle if they are
    # missing or stale.  The build script is loaded by path: importing it through the package
    # would run the package's __init__, which refuses to load before libgdg.so exists.
    _load_by_path("_gdg_lib_build", "moe_ragged_bf16_grouped_b300/build.py").build()
    _load_by_path("_gdg_oracle_build", "oracle/build.py").build()


@pytest.fixture(scope="session")
def cuda_lib():
    """The CUDA library through its Python binding; GPU tests only."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no GPU")
    import moe_ragged_bf16_grouped_b300 as gdg
    return gdg
