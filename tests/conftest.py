import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")
    config.addinivalue_line("markers", "slow: full-size workloads")


def read_golden(name):
    """Parse a whitespace-separated fixture: returns (rows, keyed) where rows are
    the lines whose first token is numeric and keyed maps a leading word to the
    rest of its line."""
    rows, keyed = [], {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.split("#", 1)[0].strip()
            if not line:
                continue
            tok = line.split()
            try:
                float(tok[0])
                rows.append(tok)
            except ValueError:
                keyed[tok[0]] = tok[1:]
    return rows, keyed
