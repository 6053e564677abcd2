import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU (sm_103a) and the built library")


def pytest_terminal_summary(terminalreporter):
    """Prints the whole-tensor parity figures the GPU tests recorded."""
    here = os.path.dirname(os.path.abspath(__file__))
    if here not in sys.path:
        sys.path.insert(0, here)
    try:
        from helpers import PARITY_STATS
    except ImportError:
        return
    if not PARITY_STATS:
        return
    terminalreporter.write_sep("-", "parity against the fp64 oracle, every output element")
    for what, mo, me, ml in PARITY_STATS:
        terminalreporter.write_line(f"{what}: max|dO|={mo:.3e} mean|dO|={me:.3e} max|dLSE|={ml:.3e}")
