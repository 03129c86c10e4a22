import functools
import json
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libtq.so")


def golden(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


@functools.lru_cache(maxsize=None)
def codebook(d, mse_bits):
    """Oracle Lloyd-Max codebook, computed once per test session."""
    from oracle import lloyd_max_sphere
    return lloyd_max_sphere(d, mse_bits)
