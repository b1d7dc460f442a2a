import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libkda")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_collection_modifyitems(config, items):
    # GPU tests cannot run without a device; skip them instead of failing at import time.
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


@pytest.fixture(autouse=True)
def _parity_record_name(request):
    from tests import _helpers
    _helpers.CURRENT_TEST[0] = request.node.nodeid
    yield


def pytest_sessionfinish(session, exitstatus):
    # KDA_PARITY_REPORT=<path>: every oracle comparison of the session with its measured errors
    path = os.environ.get("KDA_PARITY_REPORT")
    if not path:
        return
    import json
    from tests import _helpers
    os.makedirs(os.path.dirname(os.path.abspath(path)), exist_ok=True)
    with open(path, "w") as f:
        json.dump(_helpers.RECORDS, f, indent=0)
