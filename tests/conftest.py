import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
for _p in (ROOT, os.path.join(ROOT, "tests")):
    if _p not in sys.path:
        sys.path.insert(0, _p)


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
    skip = pytest.mark.skip(reason="no CUDA GPU in this environment")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


def pytest_sessionfinish(session, exitstatus):
    """With PA_PARITY_REPORT set to a path, write the realised error of every GPU-vs-oracle
    comparison of the run there (JSON), so the margin left under each bar can be read."""
    path = os.environ.get("PA_PARITY_REPORT")
    if not path:
        return
    helpers = sys.modules.get("gpu_helpers")
    if helpers is None:
        return
    import json
    with open(path, "w") as f:
        json.dump({"bars": {"max_abs": helpers.MAX_ABS, "rel_rms": helpers.REL_RMS, "lse_abs": helpers.LSE_ABS},
                   "comparisons": helpers.REPORT}, f, indent=1)
