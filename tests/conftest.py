import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_collection_modifyitems(config, items):
    # A GPU test without a GPU is a failure of the environment, not a pass:
    # keep it selected so `-m gpu` on a CPU machine fails loudly instead of
    # skipping, but let `-m "not gpu"` deselect it as usual.
    pass
