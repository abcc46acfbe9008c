"""Shared pytest setup: the ``gpu`` marker and the repo root on sys.path."""

import os
import sys

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (GB300, sm_103a)")


def pytest_terminal_summary(terminalreporter):
    """With JF_PARITY_REPORT=1: every attention comparison's errors."""
    import os
    if os.environ.get("JF_PARITY_REPORT") != "1":
        return
    try:
        from helpers import REPORT
    except ImportError:
        return
    terminalreporter.write_line("attention parity: test, max-abs, mean-abs, elements above 1e-2")
    for what, mx, mean, over in REPORT:
        terminalreporter.write_line(f"  {what:48s} {mx:.3e} {mean:.3e} {over}")
