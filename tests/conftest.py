import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")
    config.addinivalue_line("markers", "slow: full-size workload, minutes of host time")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    """Repeats the index-row parity counts of the GPU tests (one line per check) at the end of the run."""
    kp = sys.modules.get("tests.kpool_parity")
    lines = getattr(kp, "PARITY_LOG", None) if kp else None
    if lines:
        terminalreporter.write_sep("-", "index-row parity (rows, bit-exact, boundary rows/pools, hard)")
        for line in lines:
            terminalreporter.write_line(line)
