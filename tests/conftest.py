import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: long-running CPU test")


def pytest_collection_modifyitems(config, items):
    # GPU tests cannot run here without a device; fail loudly on a GPU machine
    # instead of skipping, so a missing library never passes silently.
    import torch
    if torch.cuda.is_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_sessionfinish(session, exitstatus):
    """Write the achieved parity errors of the session (tests/helpers.py
    RECORDED) to $FLASHBOB_PARITY_LOG as JSON lines, when that is set."""
    path = os.environ.get("FLASHBOB_PARITY_LOG")
    if not path:
        return
    try:
        from tests.helpers import RECORDED
    except Exception:
        return
    import json
    with open(path, "w") as fh:
        for check, key, err in RECORDED:
            fh.write(json.dumps({"check": check, "output": key, "rel_err": err}) + "\n")
