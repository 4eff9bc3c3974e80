"""The build entry's smoke check (one tiny fwd, dgrad, wgrad and fused accumulate on cuda:0
against the oracle) runs as part of the GPU suite too."""
import importlib.util
import os

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def test_graft_entry_smoke(cuda_lib):
    spec = importlib.util.spec_from_file_location("graft_entry",
                                                  os.path.join(ROOT, "__graft_entry__.py"))
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    mod.smoke()
