import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a GB300 (sm_103a) GPU")
    config.addinivalue_line("markers", "slow: long-running CPU test")


GOLDEN = os.path.join(ROOT, "tests", "golden")


def read_golden(name):
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            rows.append(line.split())
    return rows


def golden_setup():
    """The [FSA] test set-up fixture as a dict: splits and head_dims as int
    lists, seed as an int."""
    out = {}
    for row in read_golden("fsa_pr148_test_setup.txt"):
        vals = [int(x) for x in row[1:]]
        out[row[0]] = vals if len(vals) > 1 else vals[0]
    return out
