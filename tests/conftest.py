import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs an sm_103a GPU (GB300); runs the CUDA path")


def pytest_collection_modifyitems(config, items):
    # keep the no-GPU tests green on a box without CUDA: a gpu test that is
    # selected there fails loudly instead of silently skipping.
    pass
