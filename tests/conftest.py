import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")


def read_golden(name):
    """Parse a golden fixture: '#' lines are comments, others 'key v1 v2 ...'."""
    out = {}
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if not line or line.startswith("#"):
                continue
            key, *vals = line.split()
            out.setdefault(key, []).append(vals)
    return out


def pytest_terminal_summary(terminalreporter):
    """Print the error norms of the full-size parity comparisons (also under -q)."""
    try:
        from gpu_util import REPORT
    except Exception:
        return
    if not REPORT:
        return
    tr = terminalreporter
    tr.write_sep("-", "parity against the fp64 oracle over the compared outputs")
    for name in sorted(REPORT):
        tr.write_line(f"{name}: {REPORT[name]}")
