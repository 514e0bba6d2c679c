import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device (GB300, sm_103a) and the built library")


def pytest_runtest_setup(item):
    """With TG_REQUIRE_GPU set (not "0"), a GPU test fails instead of
    skipping when no CUDA device is visible."""
    if item.get_closest_marker("gpu") is None:
        return
    if os.environ.get("TG_REQUIRE_GPU", "0") in ("", "0"):
        return
    try:
        import torch

        ok = torch.cuda.is_available()
    except Exception:  # noqa: BLE001 - any import problem means no device
        ok = False
    if not ok:
        pytest.fail("TG_REQUIRE_GPU is set but no CUDA device is visible", pytrace=False)
