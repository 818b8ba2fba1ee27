"""Shared test configuration.

Markers:
  gpu   -- needs a CUDA GPU (GB300, sm_103a); calls the librz C ABI.
Everything else runs on the CPU: the oracle against its pins, host-side logic,
the C-ABI symbol table, and the multi-process (gloo) replica harness.
"""
import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA GPU and the built librz")


# Worst element-wise relative errors of the composite parity checks (layer, stack,
# FFN), reported next to their max/L2 bars at the end of the run.
ELEMENTWISE_REPORT = []


def pytest_terminal_summary(terminalreporter):
    if not ELEMENTWISE_REPORT:
        return
    terminalreporter.section("element-wise relative error of composite outputs")
    terminalreporter.write_line("worst |gpu-ref|/|ref| over elements with |ref| > 1e-2 max|ref|; "
                                "max|gpu-ref|/max|ref| (bar 1e-3)")
    for what, ew, mx in ELEMENTWISE_REPORT:
        terminalreporter.write_line(f"  {what:60s} elementwise {ew:.3e}   max-rel {mx:.3e}")


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.lib()
    return oracle
