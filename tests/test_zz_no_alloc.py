"""The allocation-free entry point, dsa_select_candidate_blocks_sharded_static.

It exists for callers that must not allocate device memory when they call
(for instance serving engines whose memory planner holds nearly all of HBM,
or plugin hosts whose operators may not allocate on their own); its workspace
is a fixed 8 MiB array inside the library. These tests call it through the C
ABI and check that two calls in a row give exactly what the existing entry
point (with a caller-supplied workspace) gives, ids and scores bit for bit,
and that a request needing more than 8 MiB of workspace is refused.

The file is collected last so that a run stopping at the first failure has
run every other test before it; it also passes on its own in a fresh process.
"""

import ctypes

import numpy as np
import pytest

import workloads

pytestmark = pytest.mark.gpu

DSA_EUNSUPPORTED = -3


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
    return torch, dsa, fn


def call_static(env, local, gke, wl, out, scores):
    torch, dsa, fn = env
    D, rows, lw = local.shape
    stream = torch.cuda.current_stream().cuda_stream or None
    return fn(local.data_ptr(), D, rows, lw, local.stride(1), local.stride(0), gke.data_ptr(),
              wl.global_block_size, wl.max_global_blocks, wl.row_repeat, wl.topk_blocks,
              out.data_ptr(), out.stride(0), scores.data_ptr(), scores.stride(0), stream)


def test_static_matches_workspace_entry_point_twice(env):
    torch, dsa, _ = env
    # 256 rows of up to 256 KiB: the launcher cuts each row into parts of
    # 64 KiB, one CTA each (up to 4 per row), and the parts meet in the fixed
    # array.
    wl, _ = workloads.small_sharded(2024, shards=8, rows=256, global_width=65536,
                                    global_block_size=64, max_global_blocks=1024,
                                    topk_blocks=32, row_repeat=2)
    local = torch.from_numpy(wl.logits).cuda()
    gke = torch.from_numpy(wl.global_row_ke).cuda()
    nbg = wl.max_global_blocks
    ref_out = torch.empty((wl.rows, wl.topk_blocks), dtype=torch.int32, device="cuda")
    ref_scores = torch.empty((wl.rows, nbg), dtype=torch.float32, device="cuda")
    ws = torch.zeros(dsa.workspace_bytes(wl.rows, nbg), dtype=torch.uint8, device="cuda")
    dsa.dsa_select_candidate_blocks_sharded(local, gke, wl.global_block_size, nbg,
                                            wl.topk_blocks, ref_out, wl.row_repeat,
                                            scores_out=ref_scores, workspace=ws)
    torch.cuda.synchronize()
    want_ids = ref_out.cpu().numpy()
    want_scores = ref_scores.cpu().numpy().view(np.uint32)
    for _ in range(2):
        out = torch.full((wl.rows, wl.topk_blocks), -7, dtype=torch.int32, device="cuda")
        scores = torch.full((wl.rows, nbg), -5.0, dtype=torch.float32, device="cuda")
        assert call_static(env, local, gke, wl, out, scores) == 0
        torch.cuda.synchronize()
        np.testing.assert_array_equal(out.cpu().numpy(), want_ids)
        np.testing.assert_array_equal(scores.cpu().numpy().view(np.uint32), want_scores)


def test_static_refuses_requests_beyond_its_array(env):
    torch, dsa, fn = env
    # 4096 rows x 1024 blocks need about 16.8 MB of workspace (> 8 MiB); the
    # call is refused before it touches the device, so the pointers are
    # never read.
    fake = ctypes.c_void_p(0x1000)
    st = fn(fake, 8, 4096, 8192, 8192, 4096 * 8192, fake, 64, 1024, 1, 32, fake, 32, None, 0,
            None)
    assert st == DSA_EUNSUPPORTED
