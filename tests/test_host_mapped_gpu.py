"""Pinned host tensors read and written in place by the kernels.

A pinned (page-locked) host tensor is mapped into the device's address space
(``dsa_mapped_host_pointer``); the binding hands that address to the C entry
points, so the kernels read the in-window logits and the bounds across the
host link and write ids, scores and masked logits straight back into host
memory. Results must equal the oracle's bit for bit, exactly as for device
tensors; pageable and device pointers are refused before anything launches.
"""

import ctypes

import numpy as np
import pytest

import oracle
import workloads
from helpers import assert_bits_equal

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def env():
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import deepseek_sparse_attention_row_gb300 as dsa

    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    return torch, dsa


def pinned(torch, a):
    return torch.from_numpy(np.ascontiguousarray(a)).pin_memory()


def test_select_host_call_reads_pinned_inputs(env):
    torch, dsa = env
    wl = workloads.small_unsharded(21, rows=48, width=9000, block_size=64, topk_blocks=16,
                                   nan_count=5)
    want_ids, _ = oracle.run_workload(wl)
    logits, ks, ke = pinned(torch, wl.logits), pinned(torch, wl.row_ks), pinned(torch, wl.row_ke)
    out = torch.full((wl.rows, wl.topk_blocks), -7, dtype=torch.int32, pin_memory=True)
    got = dsa.select_candidate_blocks_host(logits, ks, ke, wl.topk_blocks, wl.block_size,
                                           wl.row_repeat, wl.pin_newest, out=out)
    assert got is out
    np.testing.assert_array_equal(out.numpy(), want_ids)


@pytest.mark.parametrize("split", [False, True])
def test_select_pinned_strided_view_with_scores(env, split):
    """Rows padded to an odd stride, the view starting three rows into its
    allocation (an interior host address), scores written to host memory;
    with a workspace long rows are split over CTAs that meet in it."""
    torch, dsa = env
    width, ld = 20000, 20037
    wl = workloads.small_unsharded(22, rows=40, width=width, block_size=64, topk_blocks=32,
                                   row_repeat=4, ld=ld)
    want_ids, want_scores = oracle.run_workload(wl)
    big = torch.empty((wl.rows + 3, ld), dtype=torch.float32, pin_memory=True)
    big[3:] = torch.from_numpy(wl.logits)
    view = big[3:, :width]
    ks, ke = pinned(torch, wl.row_ks), pinned(torch, wl.row_ke)
    out = torch.full((wl.rows, 40), -7, dtype=torch.int32, pin_memory=True)
    scores = torch.full((wl.rows, want_scores.shape[1] + 3), 7.0, pin_memory=True)
    ws = (torch.zeros(dsa.workspace_bytes(wl.rows, want_scores.shape[1]), dtype=torch.uint8,
                      device="cuda") if split else False)
    dsa.dsa_select_candidate_blocks(view, ks, ke, wl.topk_blocks, wl.block_size, out,
                                    wl.row_repeat, wl.pin_newest,
                                    scores_out=scores[:, :want_scores.shape[1]], workspace=ws)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.numpy()[:, :wl.topk_blocks], want_ids)
    assert (out.numpy()[:, wl.topk_blocks:] == -7).all()
    assert_bits_equal(scores.numpy()[:, :want_scores.shape[1]], want_scores)
    assert (scores.numpy()[:, want_scores.shape[1]:] == 7.0).all()


def test_select_pinned_bf16(env):
    torch, dsa = env
    wl = workloads.small_unsharded(23, rows=64, width=12288, block_size=128, topk_blocks=16,
                                   bf16_grid=True)
    want_ids, _ = oracle.run_workload(wl)  # bf16-grid values: the fp32 ids
    logits = torch.from_numpy(wl.logits).to(torch.bfloat16).pin_memory()
    got = dsa.select_candidate_blocks_host(logits, pinned(torch, wl.row_ks),
                                           pinned(torch, wl.row_ke), wl.topk_blocks,
                                           wl.block_size, wl.row_repeat, wl.pin_newest)
    np.testing.assert_array_equal(got.numpy(), want_ids)


def test_sharded_host_call_reads_pinned_inputs(env):
    torch, dsa = env
    swl, _ = workloads.small_sharded(24, shards=8, rows=32, global_width=8192,
                                     global_block_size=64, max_global_blocks=128,
                                     topk_blocks=16)
    want_ids, _ = oracle.run_workload(swl)
    got = dsa.select_candidate_blocks_sharded_host(pinned(torch, swl.logits),
                                                   pinned(torch, swl.global_row_ke), 64, 128, 16)
    np.testing.assert_array_equal(got.numpy(), want_ids)


def test_sharded_starts_host_call_reads_pinned_inputs(env):
    torch, dsa = env
    swl, _ = workloads.small_sharded(25, shards=8, rows=32, global_width=8192,
                                     global_block_size=64, max_global_blocks=128,
                                     topk_blocks=16)
    rng = np.random.default_rng(25)
    swl.global_row_ks = rng.integers(0, np.maximum(swl.global_row_ke, 0),
                                     endpoint=True).astype(np.int32)
    want_ids, _ = oracle.run_workload(swl)
    got = dsa.select_candidate_blocks_sharded_host(pinned(torch, swl.logits),
                                                   pinned(torch, swl.global_row_ke), 64, 128, 16,
                                                   global_row_ks=pinned(torch, swl.global_row_ks))
    np.testing.assert_array_equal(got.numpy(), want_ids)


def test_mask_pinned_logits_in_place(env):
    torch, dsa = env
    wl = workloads.small_unsharded(26, rows=24, width=10000, block_size=64, topk_blocks=8)
    ids, _ = oracle.run_workload(wl)
    want = oracle.mask(wl.logits, wl.row_ks, wl.row_ke, ids, wl.block_size, wl.row_repeat)
    logits = pinned(torch, wl.logits)
    dsa.dsa_mask_candidate_logits(logits, pinned(torch, wl.row_ks), pinned(torch, wl.row_ke),
                                  pinned(torch, ids), wl.block_size, wl.row_repeat)
    torch.cuda.synchronize()
    assert_bits_equal(logits.numpy(), want)


def test_merge_pinned_equals_device(env):
    """The LSE merge reading pinned host inputs and writing host outputs
    gives the bits the same kernel gives on device copies of the inputs."""
    torch, dsa = env
    lwl = workloads.make_lse_named("lse_tiny")
    h_outs, h_lses = pinned(torch, lwl.outs), pinned(torch, lwl.lses)
    merged_h, lse_h = dsa.dsa_merge_attn_out(h_outs, h_lses)
    merged_d, lse_d = dsa.dsa_merge_attn_out(h_outs.cuda(), h_lses.cuda())
    torch.cuda.synchronize()
    assert not merged_h.is_cuda and merged_h.is_pinned()
    assert_bits_equal(merged_h.numpy(), merged_d.cpu().numpy())
    assert_bits_equal(lse_h.numpy(), lse_d.cpu().numpy())


def test_unmapped_pointers_are_refused(env):
    torch, dsa = env
    lib = dsa.library()
    dev = ctypes.c_void_p(12345)
    pageable = np.ones(1024, dtype=np.float32)
    assert lib.dsa_mapped_host_pointer(pageable.ctypes.data, ctypes.byref(dev)) == -1
    on_device = torch.ones(1024, device="cuda")
    assert lib.dsa_mapped_host_pointer(on_device.data_ptr(), ctypes.byref(dev)) == -1
    assert dev.value == 12345  # left unchanged
    h = torch.ones(1024).pin_memory()
    assert lib.dsa_mapped_host_pointer(h.data_ptr() + 64, ctypes.byref(dev)) == 0
    assert dev.value is not None
    # The binding refuses pageable host tensors before any launch.
    wl = workloads.small_unsharded(27, rows=4, width=256, block_size=64, topk_blocks=4)
    out = torch.empty((4, 4), dtype=torch.int32, device="cuda")
    with pytest.raises(ValueError, match="pinned host tensor"):
        dsa.dsa_select_candidate_blocks(torch.from_numpy(wl.logits), None,
                                        torch.from_numpy(wl.row_ke).cuda(), 4, 64, out)
    torch.cuda.synchronize()
