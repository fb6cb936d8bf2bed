import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line(
        "markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")


GOLDEN = os.path.join(ROOT, "tests", "golden")


def read_golden(name):
    """Rows of whitespace-separated fields from a golden file, comments stripped."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                rows.append(line.split())
    return rows


@pytest.fixture(scope="session")
def e2m1_grid():
    return [float(r[0]) for r in read_golden("e2m1_grid.txt")]
