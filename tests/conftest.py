import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def _ensure_library_built():
    """Build libattn.so in-tree if it is missing (nvcc cross-compiles without a GPU)."""
    lib = os.path.join(ROOT, "causal_attention_gb300", "lib", "libattn.so")
    if not os.path.exists(lib):
        import importlib.util
        path = os.path.join(ROOT, "causal_attention_gb300", "build.py")
        spec = importlib.util.spec_from_file_location("_attn_build", path)
        mod = importlib.util.module_from_spec(spec)
        spec.loader.exec_module(mod)  # build.py does not import the package itself
        mod.build()


def pytest_configure(config):
    _ensure_library_built()
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


@pytest.fixture(scope="session")
def cuda_lib():
    """The built C-ABI library on a machine with a GPU (fails loudly if it is missing)."""
    import torch
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    import causal_attention_gb300 as ca
    return ca
