import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_terminal_summary(terminalreporter):
    """Print the parity margins of the full-size workloads (if any ran)."""
    try:
        import parity
    except Exception:
        return
    if parity.MARGINS:
        terminalreporter.write_sep("-", "parity margins of the full-size workloads")
        for line in parity.MARGINS:
            terminalreporter.write_line(line)
