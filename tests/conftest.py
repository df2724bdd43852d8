import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_terminal_summary(terminalreporter):
    # the GPU parity tests' near-tie and mismatch counts per workload (printed
    # even under -q); nothing when no parity test ran
    mod = sys.modules.get("compare")
    if mod is None:
        return
    for line in mod.near_tie_summary():
        terminalreporter.write_line(line)
