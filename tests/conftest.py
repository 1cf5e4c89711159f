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

        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture(scope="session", autouse=True)
def _short_device_wait_limit():
    """RA_TEST_WAIT_LIMIT_NS shortens the kernels' bounded waits for a test session."""
    val = os.environ.get("RA_TEST_WAIT_LIMIT_NS")
    if val:
        try:
            import ring_attn_gb300

            ring_attn_gb300.ring_attn_set_knob(ring_attn_gb300.RA_KNOB_WAIT_LIMIT_NS, int(val))
        except Exception:  # library not built yet: the GPU tests build it
            pass
    yield
