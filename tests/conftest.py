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
    entries = getattr(mod, "REPORT", None) if mod else None
    if not entries:
        return
    other = [line for group, line in entries if group != "workloads"]
    workloads = [line for group, line in entries if group == "workloads"]
    if other:
        terminalreporter.write_sep("-", "all-rows parity of the other large cases")
        for line in other:
            terminalreporter.write_line(line)
    if workloads:
        terminalreporter.write_sep("-", "all-rows parity of the benchmark workloads at full size")
        for line in workloads:
            terminalreporter.write_line(line)
