import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session", autouse=True)
def _bounds_build_is_loaded_when_asked():
    """With DIFFATTN_DEBUG=1 every test runs against the bounds-check build: make sure it is the one loaded."""
    if os.environ.get("DIFFATTN_DEBUG", "") == "1":
        from differential_attention_03_gb300 import binding
        assert binding.BOUNDS and binding.LIB_PATH.endswith("libdiffattn_bounds.so")
    yield
