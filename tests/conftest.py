import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA library)")
    config.addinivalue_line("markers", "slow: long-running parity case")


def read_golden(name):
    """Rows of a tests/golden fixture, comments stripped, whitespace split."""
    rows = []
    with open(os.path.join(ROOT, "tests", "golden", name), encoding="utf-8") as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


@pytest.fixture(scope="session")
def golden():
    return read_golden
