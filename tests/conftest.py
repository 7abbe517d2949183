import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libfd.so")


def pytest_collection_modifyitems(config, items):
    """GPU tests fail loudly (not skip) when no GPU is present but they were
    selected explicitly with -m gpu; otherwise they are skipped on CPU hosts."""
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:
        has_gpu = False
    if has_gpu:
        return
    explicit = "gpu" in (config.getoption("-m") or "") and "not gpu" not in (config.getoption("-m") or "")
    if explicit:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


@pytest.fixture(scope="session")
def fdlib():
    """Build (if needed) and load libfd.so; fail loudly when it cannot load."""
    from split_kv_decode_paged_gb300 import build as fd_build
    from split_kv_decode_paged_gb300 import _lib
    fd_build.build()
    return _lib.load()
