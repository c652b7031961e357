"""Multi-rank host logic of the benchmark on CPU (gloo, world size 2).

Rows are independent, so N GPUs run N replicas of the workload with no
data-path collective; the only cross-rank steps are the barriers around the
timed region and the max over ranks of the timed duration. These run here
over gloo exactly as they run over NCCL on GPUs.
"""

import os
import socket

import pytest


def _free_port():
    with socket.socket() as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, results):
    import torch.distributed as dist

    import bench

    os.environ.update(RANK=str(rank), WORLD_SIZE=str(world), LOCAL_RANK=str(rank),
                      MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    dist.init_process_group("gloo", rank=rank, world_size=world)
    try:
        assert bench.dist_env() == (rank, world, rank)
        bench.dist_barrier(world)
        # rank 1 is the slow one: the max must pick its time on every rank
        mine = 10.0 + 5.0 * rank
        worst = bench.dist_max(mine, world)
        rate = bench.whole_job_rate(1000.0, world, worst)
        results[rank] = (worst, rate)
        bench.dist_barrier(world)
    finally:
        dist.destroy_process_group()


def test_two_ranks_max_time_and_weak_aggregate():
    import torch.multiprocessing as mp

    ctx = mp.get_context("spawn")
    with ctx.Manager() as mgr:
        results = mgr.dict()
        port = _free_port()
        procs = [ctx.Process(target=_worker, args=(r, 2, port, results)) for r in range(2)]
        for p in procs:
            p.start()
        for p in procs:
            p.join(timeout=120)
            assert p.exitcode == 0
        res = dict(results)
    assert res[0] == res[1] == (15.0, 1000.0 * 2 / 15.0)


def test_single_rank_needs_no_process_group():
    import bench

    assert bench.dist_max(3.5, 1) == 3.5
    bench.dist_barrier(1)
    assert bench.whole_job_rate(10.0, 1, 2.0) == 5.0


def test_row_slice_keeps_groups():
    import numpy as np

    import bench
    import workloads

    wl = workloads.small_unsharded(3, rows=24, width=512, block_size=64, topk_blocks=4,
                                   row_repeat=8)
    s = bench._row_slice(wl, 8, 20)
    assert s.rows == 12 and s.row_ke.tolist() == wl.row_ke[1:3].tolist()
    swl, _ = workloads.small_sharded(4, shards=8, rows=10, global_width=512,
                                     global_block_size=64, max_global_blocks=8, topk_blocks=4)
    s = bench._row_slice(swl, 2, 5)
    assert s.logits.shape == (8, 3, 64)
    np.testing.assert_array_equal(s.global_row_ke, swl.global_row_ke[2:5])


def test_algorithmic_bytes_count_only_windows():
    import numpy as np

    import bench
    import workloads

    x = np.zeros((3, 100), np.float32)
    wl = workloads.Workload("t", x, np.array([10, 0, 50], np.int32),
                            np.array([30, 200, 40], np.int32), 8, 4, 1, True, 0)
    # windows: [10,30) -> 20, [0,100) -> 100, [50,40) clamps to empty
    assert bench.window_elements(wl) == 120
    assert bench.algorithmic_bytes(wl) == 4 * 120 + 4 * 6 + 4 * 3 * 4
    swl, _ = workloads.small_sharded(1, shards=4, rows=2, global_width=64,
                                     global_block_size=8, max_global_blocks=8, topk_blocks=2)
    swl.global_row_ke[:] = [10, 100]
    # shard ends for gke 10 over 4 shards: 3, 3, 2, 2; gke 100 clamps to 16 each
    assert bench.window_elements(swl) == 10 + 64


def test_window_elements_with_starts_by_brute_force():
    """The bytes a DCP call with starts reads (and the in-place end-to-end call
    moves across the host link): every global token t in a row's window
    [gs, ge) whose local column t // D lies inside the shard width."""
    import numpy as np

    import bench
    import workloads

    for seed in range(6):
        rng = np.random.default_rng(70 + seed)
        D = int(rng.choice([1, 3, 8]))
        lw = int(rng.choice([5, 64, 100]))
        swl, _ = workloads.small_sharded(70 + seed, shards=D, rows=7, global_width=D * lw,
                                         global_block_size=D * 4, max_global_blocks=32,
                                         topk_blocks=4, row_repeat=2, wild_bounds=True)
        groups = swl.global_row_ke.size
        swl.global_row_ks = rng.integers(-5, D * lw + 9, size=groups).astype(np.int32)
        want = 0
        for r in range(swl.rows):
            ge = int(swl.global_row_ke[r // 2])
            gs = min(max(int(swl.global_row_ks[r // 2]), 0), max(ge, 0))
            want += sum(1 for t in range(gs, max(ge, 0)) if t // D < lw)
        assert bench.window_elements(swl) == want, seed


def test_kernel_hash_ignores_comments_only():
    """The traffic figures are keyed by a hash of the kernel code with its
    comments and blank lines removed: comment edits keep it, code edits
    change it."""
    import bench

    src = "int f(int x) {  // doubles\n  /* the\n  answer */\n  return 2 * x;\n}\n"
    same = "// header\nint f(int x) {\n\n    return 2 * x;   /* twice */\n}\n"
    other = "int f(int x) {\n  return 3 * x;\n}\n"
    assert bench.code_only(src) == bench.code_only(same) == "int f(int x) {\nreturn 2 * x;\n}"
    assert bench.code_only(other) != bench.code_only(src)
    assert "ld.global.nc" in bench.code_only('asm("ld.global.nc.b32 %0, [%1];");')
