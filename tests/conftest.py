import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def golden_numbers():
    path = os.path.join(ROOT, "tests", "golden", "page_numbers.txt")
    out = {}
    with open(path) as f:
        for line in f:
            line = line.split("#")[0].strip()
            if line:
                k, v = line.split()
                out[k] = float(v)
    return out
