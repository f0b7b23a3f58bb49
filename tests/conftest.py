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
    # Keep the allocation-free entry point's test file last so that a run that
    # stops at the first failure has already run everything else.
    items.sort(key=lambda it: os.path.basename(str(it.fspath)).startswith("test_zz"))
