import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built CUDA library")


def read_golden(name):
    """Parse a golden fixture: '#' lines are the citation; 'key: values' lines
    and bare rows are returned in order."""
    entries = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if ":" in line:
                k, v = line.split(":", 1)
                entries.append((k.strip(), v.split()))
            else:
                entries.append(("row", line.split()))
    return entries


@pytest.fixture(scope="session")
def oracle():
    import oracle as o
    o.lib()
    return o
