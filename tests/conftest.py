"""pytest configuration: the ``gpu`` marker and shared helpers."""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU and the built CUDA library")


def pytest_collection_modifyitems(config, items):
    # The no-GPU suite must never touch CUDA; the GPU suite must never run silently on CPU.
    import torch
    if not torch.cuda.is_available():
        skip = pytest.mark.skip(reason="no CUDA device in this process")
        for item in items:
            if "gpu" in item.keywords:
                item.add_marker(skip)
