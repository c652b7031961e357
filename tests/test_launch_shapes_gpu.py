"""Launch shapes that the default choice reaches only for some sizes, forced
through the library's explicit override call (dsa_select_set_launch_override,
applied by conftest.py from DSA_TEST_LAUNCH in a child run), must give the
oracle's results bit for bit like the default ones:

- every row split into 3 or 8 chunk-major parts (long rows normally split
  only when there are few rows), whose keys meet in the workspace;
- short rows handled one per warp in row order instead of last to first;
- short rows handled one per CTA instead of one per warp.

The overrides are process-wide, so each setting re-runs the relevant parity
sweeps in a child process.
"""

import os
import re
import subprocess
import sys

import pytest

pytestmark = pytest.mark.gpu

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
FILES = ["tests/test_parity_gpu.py", "tests/test_bf16_gpu.py"]
# setting -> (overrides, pytest -k selection, least number of tests it must run)
CASES = {
    "split3": ("split=3", "unsharded_sweep or sharded_sweep or starts_sweep", 150),
    "split8": ("split=8", "unsharded_sweep or sharded_sweep or starts_sweep or workspace_reuse",
               150),
    "warp_rows_in_order": ("warp_order=1", "warp", 8),
    "no_warp_kernel": ("warp_rows=1", "warp", 8),
}


@pytest.mark.parametrize("name", sorted(CASES))
def test_forced_launch_shape(name):
    spec, select, least = CASES[name]
    env = dict(os.environ, DSA_TEST_LAUNCH=spec)
    res = subprocess.run([sys.executable, "-m", "pytest", *FILES, "-m", "gpu", "-q", "-x",
                          "-p", "no:cacheprovider", "-k", select],
                         cwd=ROOT, env=env, capture_output=True, text=True, timeout=900)
    assert res.returncode == 0, res.stdout[-4000:] + res.stderr[-2000:]
    passed = re.search(r"(\d+) passed", res.stdout)
    ok = passed and int(passed.group(1)) >= least and " failed" not in res.stdout
    assert ok, res.stdout[-2000:]
