import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built libwq.so")


GOLDEN = os.path.join(ROOT, "tests", "golden")


def read_golden(name):
    """Parse `label ; field ; field` lines of a golden fixture (comments start with #)."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append([p.strip() for p in line.split(";")])
    return rows


@pytest.fixture(scope="session")
def golden():
    return read_golden
