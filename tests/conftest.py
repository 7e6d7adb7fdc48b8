import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def read_golden(name):
    """Rows of integers from a golden fixture (comment lines skipped)."""
    rows = []
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                rows.append([int(x) for x in line.split()])
    return rows


_CPU_ROUNDS = {}


def cpu_round(name, seed=0):
    """A workload generated on the CPU without recurrent state, shared by the
    CPU tests that only read it (generating the large ones takes seconds)."""
    key = (name, seed)
    if key not in _CPU_ROUNDS:
        import workloads
        _CPU_ROUNDS[key] = workloads.make_round(name, seed=seed, device="cpu", with_state=False)
    return _CPU_ROUNDS[key]
