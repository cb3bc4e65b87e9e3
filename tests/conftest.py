import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: larger oracle cases")


def pytest_collection_modifyitems(config, items):
    # GPU tests are skipped (not failed) on a machine without a GPU; the
    # product path itself never falls back to the CPU.
    try:
        import torch
        has_gpu = torch.cuda.is_available()
    except Exception:  # pragma: no cover
        has_gpu = False
    if has_gpu:
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for it in items:
        if "gpu" in it.keywords:
            it.add_marker(skip)


def pytest_sessionfinish(session, exitstatus):
    # stop the oracle worker pool of the full-size parity tests, if one was started
    pool = sys.modules.get("tests.oracle_pool")
    if pool is not None:
        pool.close()
