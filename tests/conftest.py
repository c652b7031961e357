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


@pytest.fixture(scope="session", autouse=True)
def _launch_overrides():
    """DSA_TEST_LAUNCH="knob=value,..." (set by test_launch_shapes_gpu.py for
    its child runs) pins launch shapes through the library's explicit
    override call before any test runs; the library itself never reads the
    environment."""
    spec = os.environ.get("DSA_TEST_LAUNCH", "").strip()
    if not spec:
        yield
        return
    import __graft_entry__

    __graft_entry__.build()
    import deepseek_sparse_attention_row_gb300 as dsa

    for item in spec.split(","):
        knob, value = item.split("=")
        dsa.set_launch_override(knob.strip(), int(value))
    yield
    for knob in dsa.LAUNCH_KNOBS:
        dsa.set_launch_override(knob, 0)
