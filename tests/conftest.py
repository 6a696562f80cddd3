import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103) and the built libbsa.so")
    config.addinivalue_line("markers", "slow: full-size workload (minutes)")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


@pytest.fixture(scope="session")
def bsa_lib():
    """Build libbsa.so in-tree if needed (nvcc cross-compiles without a GPU) and load it."""
    from block_sparse_attention_plan_gb300 import build as B
    B.build()
    import block_sparse_attention_plan_gb300 as bsa
    return bsa.library()


@pytest.fixture(scope="session")
def bsa(bsa_lib):
    import block_sparse_attention_plan_gb300 as m
    return m
