import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

GOLDEN = os.path.join(ROOT, "tests", "golden")


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs through the C-ABI library)")
    config.addinivalue_line("markers", "slow: takes more than a few seconds")


def golden_lines(name):
    """Non-comment, non-empty lines of a golden fixture, split on whitespace."""
    with open(os.path.join(GOLDEN, name)) as f:
        for line in f:
            line = line.strip()
            if line and not line.startswith("#"):
                yield line.split()


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Print the session's GPU-vs-oracle parity totals (decisions and excused
    decisions per workload and acceptance rule), when any comparison ran."""
    parity = sys.modules.get("parity")
    if parity is None or not getattr(parity, "TALLY", None):
        return
    for line in parity.tally_lines():
        terminalreporter.write_line(line)
