import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def _has_gpu():
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


def pytest_collection_modifyitems(config, items):
    if _has_gpu():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session")
def oracle():
    import oracle as o
    o.build()
    return o


@pytest.fixture(autouse=True)
def _device_status_clean(request):
    """Every GPU test also fails if one of its kernels flagged an error (a
    bounded wait that gave up, a skipped bad index) that the test itself did
    not consume, so a stalled kernel can never pass on stale output."""
    yield
    if "gpu" in request.keywords and _has_gpu():
        import mxfp4_quantized_gemm_token_gb300 as mxq
        mxq.sync_status()
