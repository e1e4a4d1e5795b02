import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a) and the built CUDA library")


def pytest_terminal_summary(terminalreporter):
    # The all-rows parity checks of the full-size workloads record their
    # statistics (max error, row-sum error) here; print them even under -q.
    mod = sys.modules.get("_parity")
    lines = getattr(mod, "REPORT", None) if mod else None
    if lines:
        terminalreporter.write_sep("-", "all-rows parity of the full-size workloads")
        for line in lines:
            terminalreporter.write_line(line)
