import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (B300, sm_103a) and the built library")


def load_golden(name):
    """Parse a tests/golden fixture: `key = value` lines, '#' comments; numbers become floats
    (or lists of floats when several are given)."""
    out = {}
    with open(os.path.join(ROOT, "tests", "golden", name), encoding="utf-8") as fh:
        for line in fh:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            key, val = (s.strip() for s in line.split("=", 1))
            nums = [float(v) for v in val.split()]
            out[key] = nums[0] if len(nums) == 1 else nums
    return out


@pytest.fixture
def golden():
    return load_golden
