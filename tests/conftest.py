import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


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


@pytest.fixture(scope="module")
def device_status_guard():
    """Builds and loads the library, clears its device status word before the
    module's tests and checks afterwards that no kernel raised it (a bounded
    wait that gave up)."""
    import sliding_window_attention_band_gb300 as swab
    from sliding_window_attention_band_gb300 import build as swab_build

    swab_build.build()
    swab.load()
    swab.device_status(reset=True)
    yield
    assert swab.device_status(reset=True) == 0, "a kernel raised the device status word"
