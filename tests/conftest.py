"""Shared test configuration.

Tests marked ``gpu`` need a CUDA device and the compiled CUDA library; the
rest run on the CPU.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the compiled CUDA library")
    config.addinivalue_line("markers", "slow: large sizes; still part of the normal runs")


@pytest.fixture(scope="session")
def oracle():
    from oracle import Oracle
    return Oracle()


def read_golden(name):
    """Return the non-comment lines of a golden fixture as lists of tokens."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append(line.split())
    return rows
