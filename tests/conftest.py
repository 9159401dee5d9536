import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size oracle comparisons (minutes of CPU)")


def pytest_collection_modifyitems(config, items):
    import torch

    if torch.cuda.is_available():
        return
    skip = pytest.mark.skip(reason="no CUDA device")
    for item in items:
        if "gpu" in item.keywords:
            item.add_marker(skip)


@pytest.fixture
def knob():
    """Sets library plan knobs (fsops_debug_set_knob) for one test and puts
    every knob it touched back to its default afterwards."""
    import mxfp8_swiglu_mlp_gb300 as fs

    touched = []

    def set_knob(name, value):
        fs.fsops_debug_set_knob(name, int(value))
        touched.append(name)

    yield set_knob
    for name in touched:
        fs.fsops_debug_set_knob(name, -1)
