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
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (runs the CUDA library)")


def pytest_terminal_summary(terminalreporter):
    """The worst error / tolerance ratio each attention test reached."""
    try:
        import attention_check
    except ImportError:
        return
    if attention_check.WORST:
        terminalreporter.write_sep("-", "attention: worst |o - O| / tolerance per test")
        for k, v in sorted(attention_check.WORST.items()):
            terminalreporter.write_line("%.4f  %s" % (v, k))
