import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a)")


def golden_lines(name):
    """Data lines of a golden fixture (comments and blank lines dropped)."""
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line


def pytest_terminal_summary(terminalreporter):
    """Top-k positions excluded from exact index parity (oracle near-ties),
    per test, when GPU top-k tests ran."""
    mod = sys.modules.get("_gpu")
    rows = getattr(mod, "EXCLUSIONS", None) if mod else None
    if not rows:
        return
    tr = terminalreporter
    tr.section("top-k positions excluded as oracle near-ties (excluded / checked)")
    for nodeid, excluded, positions in rows:
        tr.write_line(f"{excluded:5d} / {positions:5d}  {nodeid}")
    tr.write_line(f"{sum(r[1] for r in rows):5d} / {sum(r[2] for r in rows):5d}  total")
