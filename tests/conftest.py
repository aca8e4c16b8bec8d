import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def read_golden(name):
    """Parse a golden fixture: `key v1 v2 ...` lines, '#' comments ignored.

    Values stay strings; callers convert.  Repeated keys keep every line.
    """
    rows = {}
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            parts = line.split()
            rows.setdefault(parts[0], []).append(parts[1:])
    return rows


def read_golden_table(name):
    """Parse a whitespace table fixture into a list of int rows ('#' comments ignored)."""
    out = []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if line:
                out.append([int(x) for x in line.split()])
    return out


@pytest.fixture(scope="session")
def orc():
    import oracle
    return oracle.default()
