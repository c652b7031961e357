"""Launch shapes that the default choice reaches only for some sizes, forced
through the library's explicit override call (dsa_select_set_launch_override,
applied by conftest.py from DSA_TEST_LAUNCH in a child run), must give the
oracle's results bit for bit like the default ones:

- the row-per-CTA kernel with every row split into 3 or 8 chunk-major parts
  (long rows normally split only when there are few rows), every row ranked
  by the whole CTA or by one warp, the row-per-warp kernel in row order,
  and short rows one per CTA instead of one per warp;
- the pipelined kernels with every warp of a CTA on one row or one row per
  warp, rows cut into 3 or 8 parts that meet in the workspace, the smallest
  rings (2 stages of 4 KiB), rows dealt to CTAs in a fixed order, and rows
  handed out longest first on every call.

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
SWEEPS = "unsharded_sweep or sharded_sweep or starts_sweep"
CASES = {
    # The row-per-CTA and row-per-warp kernels, which take the calls that the
    # pipelined kernels do not (host-mapped logits, odd block sizes, more
    # than 16 shards, more than 4096 blocks or top-256).
    "legacy": ("pipeline=1", SWEEPS + " or warp or workspace_reuse or graph", 190),
    "legacy_split3": ("pipeline=1,split=3", SWEEPS, 150),
    "legacy_split8": ("pipeline=1,split=8", SWEEPS + " or workspace_reuse", 150),
    "legacy_warp_rows_in_order": ("pipeline=1,warp_order=1", "warp", 8),
    "legacy_no_warp_kernel": ("pipeline=1,warp_rows=1", "warp", 8),
    "legacy_rank_cta": ("pipeline=1,rank_cta=1", SWEEPS + " or workspace_reuse", 150),
    "legacy_rank_warp": ("pipeline=1,rank_cta=2", SWEEPS + " or workspace_reuse", 150),
    # The pipelined kernels in shapes the automatic choice reaches only for
    # some sizes.
    "pipe_coop": ("pipeline=2", SWEEPS + " or warp or graph", 190),
    "pipe_solo": ("pipeline=3", "unsharded_sweep or warp", 80),
    "pipe_split3": ("pipeline=2,pipe_split=3", SWEEPS + " or workspace_reuse", 150),
    "pipe_split8": ("pipeline=2,pipe_split=8", SWEEPS, 150),
    "pipe_small_stages": ("pipeline=2,pipe_stage_kb=4,pipe_stages=2", SWEEPS + " or warp", 150),
    "pipe_fixed_order": ("pipeline=2,pipe_sched=1,pipe_split=2", SWEEPS, 150),
    "pipe_8_warps": ("pipeline=2,pipe_warps=8,pipe_ctas=1", SWEEPS + " or graph", 150),
    "pipe_4_warps": ("pipeline=2,pipe_warps=4", SWEEPS + " or full_size_unsharded", 150),
    "pipe_rank_warp": ("pipeline=2,rank_cta=2", SWEEPS + " or full_size_unsharded", 150),
    "pipe_stage_owner": ("pipeline=2,pipe_stage_owner=1", SWEEPS, 150),
    "pipe_longest_first": ("pipeline=2,pipe_order=2", SWEEPS + " or graph", 150),
    "pipe_claim_ahead": ("pipeline=2,pipe_order=3", SWEEPS + " or full_size_unsharded", 150),
    "pipe_solo_small_stages": ("pipeline=3,pipe_stage_kb=4,pipe_ctas=1", "unsharded_sweep or warp",
                               80),
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
