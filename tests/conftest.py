"""Shared test set-up: repository root on sys.path, the gpu marker, tolerance helpers."""
import os
import sys

import numpy as np
import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU of compute capability 10.3 (GB300)")


def rel_err(got, ref) -> float:
    """max |got - ref| / max(1, |ref|): the error measure the tolerances are stated in."""
    got = np.asarray(got, dtype=np.float64)
    ref = np.asarray(ref, dtype=np.float64)
    if got.size == 0:
        return 0.0
    return float(np.max(np.abs(got - ref) / np.maximum(1.0, np.abs(ref))))


@pytest.fixture
def rel():
    return rel_err
