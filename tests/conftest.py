import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workloads")


def pytest_collection_modifyitems(config, items):
    # The allocation-free backward's tests run after every other test (whatever
    # order the files were collected in), so a run that stops at the first
    # failure has exercised the rest of the library first.
    last = [it for it in items if it.nodeid.split("::")[0].endswith("test_zz_no_alloc.py")]
    if last:
        items[:] = [it for it in items if it not in last] + last
    # GPU tests only run where a GPU is visible; mark them skipped elsewhere so
    # that `-m gpu` on a CPU host reports skips instead of errors.
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
