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


def pytest_collection_modifyitems(config, items):
    items[:] = ([it for it in items if it.get_closest_marker("late") is None]
                + [it for it in items if it.get_closest_marker("late") is not None])


def cuda_available() -> bool:
    try:
        import torch
        return torch.cuda.is_available()
    except Exception:
        return False


@pytest.fixture(scope="session")
def golden_dir():
    return os.path.join(ROOT, "tests", "golden")
