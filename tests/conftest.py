import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


def pytest_collection_modifyitems(config, items):
    try:
        import torch

        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture
def pin():
    """pin(call, form): pin a call's kernel form (moe_tail_set_kernel_form) for
    one test; the library's choice is restored afterwards."""
    import moe_decode_tail_gb300 as mt

    calls = []

    def _pin(call, form):
        mt.moe_tail_set_kernel_form(call, form)
        calls.append(call)

    yield _pin
    for c in calls:
        mt.moe_tail_set_kernel_form(c, 0)
