import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: takes more than a few seconds")


def pytest_collection_modifyitems(config, items):
    try:
        import torch
        have_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        have_gpu = False
    if have_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def pytest_sessionfinish(session, exitstatus):
    """With GQA_ERR_LOG set, the parity cases' observed errors (relative to
    max|V|, per arithmetic path) are written there as JSON lines."""
    path = os.environ.get("GQA_ERR_LOG")
    if not path:
        return
    mod = sys.modules.get("gpu_cases")
    if mod is None:
        return
    import json
    with open(path, "w") as f:
        for test, p, rel in mod.OBSERVED:
            f.write(json.dumps({"test": test, "path": p, "rel": rel}) + "\n")
