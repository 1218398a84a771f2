import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built CUDA library")
    config.addinivalue_line("markers", "slow: takes more than a few seconds on the CPU")


def read_golden(name: str) -> dict:
    """Parse a golden fixture: '# comment' lines skipped, 'key v1 v2 ...'
    lines become key -> list of floats; rows with a numeric first column are
    collected under 'rows'."""
    out = {"rows": []}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            parts = line.split()
            try:
                float(parts[0])
                out["rows"].append([float(x) for x in parts])
            except ValueError:
                out[parts[0]] = [float(x) for x in parts[1:]]
    return out


@pytest.fixture
def golden():
    return read_golden
