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


def pytest_sessionfinish(session, exitstatus):
    """With CA_PARITY_REPORT=<path>, write the largest parity error per test
    and quantity (tests/parity.py) as JSON."""
    path = os.environ.get("CA_PARITY_REPORT")
    if not path:
        return
    import json
    try:
        import parity
    except ImportError:
        return
    with open(path, "w") as f:
        json.dump(parity.REPORT, f, indent=1, sort_keys=True)
