import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_terminal_summary(terminalreporter, exitstatus, config):
    import flipstats
    if not flipstats.RECORDS:
        return
    terminalreporter.write_sep("-", "tolerated differences per workload (GPU vs oracle)")
    for name, rows, flips, what in flipstats.RECORDS:
        terminalreporter.write_line(f"{name}: {rows} rows checked, {flips} {what}")
