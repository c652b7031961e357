"""Shared pytest setup.

Tests marked ``gpu`` need a CUDA device and the compiled library; everything
else runs on the CPU (the oracle, its pins, host-side argument validation,
symbol exports and the multi-rank host logic over gloo).
"""

import os
import sys

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
TESTS = os.path.dirname(os.path.abspath(__file__))
for p in (ROOT, TESTS):
    if p not in sys.path:
        sys.path.insert(0, p)


def pytest_configure(config):
    config.addinivalue_line("markers", "gpu: needs a CUDA device and the compiled sm_103a library")
    config.addinivalue_line("markers", "slow: full-size workloads (seconds to a minute each)")
