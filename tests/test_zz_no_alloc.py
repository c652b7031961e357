"""The allocation-free entry point, dsa_select_candidate_blocks_sharded_static.

Some callers cannot allocate device memory when they call: serving engines
whose memory planner hands nearly all of HBM to the KV cache at start-up (a
cudaMalloc in the middle of a decode step can fail or stall on the
allocator), and plugin hosts whose operators may not allocate on their own.
This entry point takes no workspace: when a call's workspace fits, it uses a
fixed 8 MiB array that the library holds in device memory; otherwise it runs
without one. These tests call it through the C ABI and compare its ids and
scores with the oracle's, element by element, on two calls in a row:

- 256 rows of up to 256 KiB, whose workspace fits: long rows are cut into
  parts that meet in the array;
- the full [8, 4096, 8192] DCP workload, whose 16.8 MB workspace does not
  fit: the call runs without the array, with the same results.

A row count beyond the library's limit is refused before anything runs (real
device buffers, so that a regression could not reach a wild address).

The file is collected last, so that a run stopping at the first failure has
run every other test before it; it also passes on its own in a fresh process.
"""

import ctypes

import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu

DSA_OK, DSA_EUNSUPPORTED = 0, -3


@pytest.fixture(scope="module")
def env():
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import deepseek_sparse_attention_row_gb300 as dsa

    assert torch.cuda.is_available(), "this test needs a CUDA device"
    lib = dsa.library()
    fn = lib.dsa_select_candidate_blocks_sharded_static
    i64, i32, p = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
    fn.argtypes = [p, i32, i64, i64, i64, i64, p, i32, i32, i32, i32, p, i64, p, i64, p]
    fn.restype = ctypes.c_int
    oracle.build()
    return torch, dsa, fn


def call_static(env, local, gke, wl, out, scores):
    torch, _, fn = env
    D, rows, lw = local.shape
    stream = torch.cuda.current_stream().cuda_stream or None
    return fn(local.data_ptr(), D, rows, lw, local.stride(1), local.stride(0), gke.data_ptr(),
              wl.global_block_size, wl.max_global_blocks, wl.row_repeat, wl.topk_blocks,
              out.data_ptr(), out.stride(0), scores.data_ptr() if scores is not None else None,
              scores.stride(0) if scores is not None else 0, stream)


def check_twice(env, wl, with_scores):
    torch, dsa, _ = env
    want_ids, want_scores = oracle.run_workload(wl, want_scores=with_scores)
    local = torch.from_numpy(wl.logits).cuda()
    gke = torch.from_numpy(wl.global_row_ke).cuda()
    nbg = max(wl.max_global_blocks, 1)
    for _ in range(2):
        out = torch.full((wl.rows, wl.topk_blocks), -7, dtype=torch.int32, device="cuda")
        scores = (torch.full((wl.rows, nbg), -5.0, dtype=torch.float32, device="cuda")
                  if with_scores else None)
        assert call_static(env, local, gke, wl, out, scores) == DSA_OK
        torch.cuda.synchronize()
        np.testing.assert_array_equal(out.cpu().numpy(), want_ids)
        if with_scores:
            np.testing.assert_array_equal(scores.cpu().numpy().view(np.uint32),
                                          want_scores.view(np.uint32))


def test_static_split_rows_match_oracle_twice(env):
    _, dsa, _ = env
    wl, _ = workloads.small_sharded(2024, shards=8, rows=256, global_width=65536,
                                    global_block_size=64, max_global_blocks=1024,
                                    topk_blocks=32, row_repeat=2)
    # The workspace of this call fits in the 8 MiB array.
    assert dsa.workspace_bytes(wl.rows, wl.max_global_blocks) <= 8 << 20
    check_twice(env, wl, with_scores=True)


@pytest.mark.slow
def test_static_full_dcp_workload_matches_oracle_twice(env):
    _, dsa, _ = env
    wl = workloads.make("dcp")
    # 4096 rows x 1024 blocks need more than the array holds: no workspace.
    assert dsa.workspace_bytes(wl.rows, wl.max_global_blocks) > 8 << 20
    check_twice(env, wl, with_scores=False)


def test_static_refuses_rows_beyond_the_limit(env):
    torch, _, fn = env
    # 2^28 + 1 rows exceed the selecting calls' row limit (2^31 / 8): the
    # call returns DSA_EUNSUPPORTED before any launch. Every pointer is a
    # real device buffer (one row group, no local columns, one id per row).
    rows = (1 << 28) + 1
    gke = torch.ones(2, dtype=torch.int32, device="cuda")
    out = torch.empty(rows, dtype=torch.int32, device="cuda")
    local = torch.empty(16, dtype=torch.float32, device="cuda")
    st = fn(local.data_ptr(), 8, rows, 0, 0, 0, gke.data_ptr(), 64, 8, 1 << 28, 1,
            out.data_ptr(), 1, None, 0, None)
    assert st == DSA_EUNSUPPORTED
    del out
    torch.cuda.empty_cache()
