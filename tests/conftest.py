import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: large inputs; minutes of CPU or GPU time")


def golden_rows(name):
    """Data rows (whitespace-separated fields) of a fixture under tests/golden."""
    path = os.path.join(ROOT, "tests", "golden", name)
    with open(path) as f:
        return [line.split() for line in f if line.strip() and not line.startswith("#")]
