import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "late: kernels new to the suite; run after the rest, so that "
                            "under -x a failure there cannot hide the other results")


# The allocation-free entry point's tests run after everything else, the
# ``late`` ones included.
LAST_FILE = "test_zz_no_alloc.py"


def pytest_collection_modifyitems(config, items):
    def rank(it):
        if it.fspath.basename == LAST_FILE:
            return 2
        return 1 if it.get_closest_marker("late") is not None else 0
    items[:] = sorted(items, key=rank)  # stable: collection order within a rank


def cuda_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")
