import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the sm_103a kernels)")


def _has_gpu() -> bool:
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


@pytest.fixture(autouse=True)
def _no_refused_access(request):
    """Under the bounds-checking build (SOFTMAX_ROWS_LIB pointing at
    libsoftmax_rows_check.so) every GPU test must end with no access refused."""
    yield
    if "gpu" not in request.keywords or not _has_gpu():
        return
    import memory_bound_row_rows_gb300 as sr
    lib = sr._lib
    if lib is None or lib.softmax_rows_build_flags() != sr.SR_BUILD_BOUNDS_CHECK:
        return
    st = lib.softmax_rows_last_device_error(None)
    addr = lib.softmax_rows_bounds_address()
    assert st != sr.SR_EBOUNDS, "an access was refused (first address 0x%x)" % addr
