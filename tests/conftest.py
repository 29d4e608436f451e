import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103) GPU and the CUDA library")


def read_golden(name):
    """Rows of a golden fixture: whitespace-separated hex fields before the '|' note."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            fields = line.split("|", 1)[0].split()
            rows.append(tuple(int(v, 16) for v in fields))
    return rows


@pytest.fixture(scope="session")
def orc():
    import oracle

    oracle.build()
    return oracle
