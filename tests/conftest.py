import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "exhaustive: sweeps all 2^32 float32 patterns (opt-in, TPS_EXHAUSTIVE=1)")


def pytest_collection_modifyitems(config, items):
    if os.environ.get("TPS_EXHAUSTIVE") == "1":
        return
    skip = pytest.mark.skip(reason="exhaustive sweep: set TPS_EXHAUSTIVE=1")
    for item in items:
        if "exhaustive" in item.keywords:
            item.add_marker(skip)
