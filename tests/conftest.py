import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def read_table(name):
    """Rows of a '|'-separated golden fixture; '#' lines are comments and
    'key: value' lines are returned as metadata."""
    meta, rows = {}, []
    with open(os.path.join(GOLDEN, name), encoding="utf-8") as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            if "|" not in line and ":" in line:
                k, v = line.split(":", 1)
                meta[k.strip()] = v.strip()
                continue
            rows.append([c.strip() for c in line.split("|")])
    return meta, rows
