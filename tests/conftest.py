import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)
HERE = os.path.dirname(os.path.abspath(__file__))
if HERE not in sys.path:
    sys.path.insert(0, HERE)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_terminal_summary(terminalreporter):
    """Prints the non-gating error figures the GPU tests noted (max-abs error
    over the RMS of the reference output), if any ran."""
    helpers = sys.modules.get("gpu_helpers")
    lines = getattr(helpers, "QUALITY", None)
    if lines:
        terminalreporter.section("max-abs error over the RMS of the reference output (not a gate)")
        for line in lines:
            terminalreporter.write_line(line)
