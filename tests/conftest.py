import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


import pytest  # noqa: E402


@pytest.fixture(scope="session")
def built_lib():
    """Build libmoelora.so in-tree (nvcc cross-compiles without a GPU) and load it."""
    from routed_moe_expert_gb300 import _build, binding
    _build.build()
    return binding.lib()
