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


@pytest.fixture(scope="session")
def orc():
    import oracle
    oracle.lib()
    return oracle
