"""GPU parity: the sm_103a library against the CPU oracle, bit for bit.

Every case compares the ordered id array exactly and the block-score array
bit for bit (integer and index outputs, and fp32 values that are copies of
input elements, so the tolerance is zero). Outputs are written into views
of larger buffers whose guard columns must come back untouched, and rows of
logits can be padded (ld > width) with values that must never win.

Every case runs twice: with a workspace, where rows are split over the 1 to 8
CTAs the launcher picks for the width, and without one (one CTA per row).
Sizes span several 32-block split units, both CTA sizes, both top-k paths
(bound-and-rank, and the exact radix path with its bitonic sort for large
K), every streaming path (vector widths 4 / 2 / 1 and the generic path for
non-power-of-two blocks), ragged window ends and unaligned window starts.
"""

import numpy as np
import pytest

import oracle
import workloads
from helpers import assert_bits_equal, deal_shards

pytestmark = pytest.mark.gpu

GUARD = 3
SENTINEL_ID = -7
SENTINEL_SCORE = np.float32(-12345.5)


@pytest.fixture(scope="module")
def env():
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import deepseek_sparse_attention_row_gb300 as dsa

    assert torch.cuda.is_available(), "GPU parity tests need a CUDA device"
    return torch, dsa


def _dev(torch, a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()


def _padded_logits(torch, logits, width, offset):
    """Device copy of logits [rows, ld] placed `offset` elements into a larger
    buffer, so the row starts get a chosen misalignment."""
    rows, ld = logits.shape
    buf = torch.full((rows * ld + offset + 8,), 1e30, dtype=torch.float32, device="cuda")
    flat = buf[offset:offset + rows * ld]
    flat.copy_(torch.from_numpy(np.ascontiguousarray(logits).reshape(-1)))
    return flat.view(rows, ld)[:, :width]


def run_unsharded(env, wl, *, want_scores=True, offset=0, workspace=None):
    torch, dsa = env
    rows, width, topk = wl.rows, wl.width, wl.topk_blocks
    nb = -(-width // wl.block_size) if width else 0
    logits = _padded_logits(torch, wl.logits, width, offset)
    out_buf = torch.full((rows, topk + GUARD), SENTINEL_ID, dtype=torch.int32, device="cuda")
    sc_buf = torch.full((rows, nb + GUARD), float(SENTINEL_SCORE), dtype=torch.float32,
                        device="cuda")
    dsa.dsa_select_candidate_blocks(logits, _dev(torch, wl.row_ks), _dev(torch, wl.row_ke), topk,
                                    wl.block_size, out_buf[:, :topk], wl.row_repeat,
                                    wl.pin_newest,
                                    scores_out=sc_buf[:, :nb] if want_scores else None,
                                    workspace=workspace)
    torch.cuda.synchronize()
    out_all, sc_all = out_buf.cpu().numpy(), sc_buf.cpu().numpy()
    assert (out_all[:, topk:] == SENTINEL_ID).all(), "guard ids overwritten"
    assert (sc_all[:, nb:] == SENTINEL_SCORE).all(), "guard scores overwritten"
    if not want_scores:
        assert (sc_all == SENTINEL_SCORE).all()
    return out_all[:, :topk], sc_all[:, :nb]


def check_unsharded(env, wl, *, offset=0, with_scores=True):
    ref_ids, ref_scores = oracle.run_workload(wl)
    for ws in (None, False):
        got_ids, got_scores = run_unsharded(env, wl, want_scores=with_scores, offset=offset,
                                            workspace=ws)
        np.testing.assert_array_equal(got_ids, ref_ids)
        if with_scores and ref_scores is not None and wl.width:
            assert_bits_equal(got_scores, ref_scores)


def run_sharded(env, wl, *, offset=0, want_scores=True, workspace=None):
    torch, dsa = env
    D, rows, lw = wl.logits.shape
    topk = wl.topk_blocks
    nbg = max(wl.max_global_blocks, 1)
    buf = torch.full((D * rows * lw + offset + 8,), 1e30, dtype=torch.float32, device="cuda")
    local = buf[offset:offset + D * rows * lw].view(D, rows, lw)
    local.copy_(torch.from_numpy(wl.logits))
    out_buf = torch.full((rows, topk + GUARD), SENTINEL_ID, dtype=torch.int32, device="cuda")
    sc_buf = torch.full((rows, nbg + GUARD), float(SENTINEL_SCORE), dtype=torch.float32,
                        device="cuda")
    dsa.dsa_select_candidate_blocks_sharded(local, _dev(torch, wl.global_row_ke),
                                            wl.global_block_size, wl.max_global_blocks, topk,
                                            out_buf[:, :topk], wl.row_repeat,
                                            scores_out=sc_buf[:, :nbg] if want_scores else None,
                                            workspace=workspace)
    torch.cuda.synchronize()
    out_all, sc_all = out_buf.cpu().numpy(), sc_buf.cpu().numpy()
    assert (out_all[:, topk:] == SENTINEL_ID).all(), "guard ids overwritten"
    assert (sc_all[:, nbg:] == SENTINEL_SCORE).all(), "guard scores overwritten"
    return out_all[:, :topk], sc_all[:, :nbg]


def check_sharded(env, wl, *, offset=0, with_scores=True):
    ref_ids, ref_scores = oracle.run_workload(wl)
    for ws in (None, False):
        got_ids, got_scores = run_sharded(env, wl, offset=offset, want_scores=with_scores,
                                          workspace=ws)
        np.testing.assert_array_equal(got_ids, ref_ids)
        if with_scores:
            assert_bits_equal(got_scores, ref_scores)


# ---------------------------------------------------------------------------
# Randomised sweeps at oracle-friendly sizes
# ---------------------------------------------------------------------------

BLOCK_SIZES = [1, 2, 3, 4, 5, 8, 12, 16, 24, 32, 48, 64, 100, 128, 256, 512]


@pytest.mark.parametrize("seed", range(48))
def test_unsharded_sweep(env, seed):
    rng = np.random.default_rng(seed)
    bs = int(BLOCK_SIZES[seed % len(BLOCK_SIZES)])
    width = int(rng.choice([1, 7, 31, 64, 333, 1000, 4096, 5003, 13000, 30001, 70000]))
    width = min(width, bs * 4000)  # keep nb within the shared-memory limit
    rows = int(rng.integers(1, 40))
    rr = int(rng.choice([1, 1, 2, 3, 8]))
    nb = -(-width // bs)
    topk = int(rng.choice([1, 5, 16, 32, 33, 100, nb, nb + 5]))
    wl = workloads.small_unsharded(
        seed, rows=rows, width=width, block_size=bs, topk_blocks=topk, row_repeat=rr,
        starts=bool(rng.integers(0, 2)), pin_newest=bool(rng.integers(0, 2)),
        nan_count=int(rng.choice([0, 0, 3, 50])), bf16_grid=bool(rng.integers(0, 2)),
        wild_bounds=bool(rng.integers(0, 2)),
        ld=width + int(rng.choice([0, 0, 1, 3, 4])))
    check_unsharded(env, wl, offset=int(rng.choice([0, 0, 1, 2, 3])))


@pytest.mark.parametrize("seed", range(36))
def test_sharded_sweep(env, seed):
    rng = np.random.default_rng(500 + seed)
    shards = int(rng.choice([1, 2, 3, 4, 8, 8, 16]))
    lbs = int(rng.choice([1, 2, 3, 4, 8, 8, 16, 32]))
    gbs = lbs * shards
    lw = int(rng.choice([1, 5, 64, 100, 1024, 2047, 8192]))
    nlb = -(-lw // lbs)
    max_gb = int(rng.choice([0, 1, max(nlb // 2, 1), nlb, nlb + 7]))
    max_gb = min(max_gb, 16384)
    rows = int(rng.integers(1, 40))
    rr = int(rng.choice([1, 1, 2, 5]))
    nbg = max(max_gb, 1)
    topk = int(rng.choice([1, 8, 32, 40, nbg, nbg + 3]))
    wl, _ = workloads.small_sharded(500 + seed, shards=shards, rows=rows,
                                    global_width=lw * shards, global_block_size=gbs,
                                    max_global_blocks=max_gb, topk_blocks=topk, row_repeat=rr,
                                    wild_bounds=bool(rng.integers(0, 2)))
    check_sharded(env, wl, offset=int(rng.choice([0, 0, 1, 2])))


def _run_sharded_starts(env, local, gks, gke, gbs, max_gb, topk, rr, workspace):
    torch, dsa = env
    D, rows, lw = local.shape
    nbg = max(max_gb, 1)
    out = torch.full((rows, topk + GUARD), SENTINEL_ID, dtype=torch.int32, device="cuda")
    sc = torch.full((rows, nbg + GUARD), float(SENTINEL_SCORE), dtype=torch.float32,
                    device="cuda")
    dsa.dsa_select_candidate_blocks_sharded(local, _dev(torch, gke), gbs, max_gb, topk,
                                            out[:, :topk], rr, scores_out=sc[:, :nbg],
                                            workspace=workspace, global_row_ks=_dev(torch, gks))
    torch.cuda.synchronize()
    o, c = out.cpu().numpy(), sc.cpu().numpy()
    assert (o[:, topk:] == SENTINEL_ID).all() and (c[:, nbg:] == SENTINEL_SCORE).all()
    return o[:, :topk], c[:, :nbg]


@pytest.mark.parametrize("seed", range(24))
def test_sharded_starts_sweep(env, seed):
    """The DCP form with global window starts: each shard streams its own
    window (its start sets its alignment) and the keys merge."""
    torch, dsa = env
    rng = np.random.default_rng(27000 + seed)
    shards = int(rng.choice([1, 2, 3, 4, 8, 8, 16]))
    lbs = int(rng.choice([1, 2, 3, 4, 8, 8, 16, 32]))
    gbs = lbs * shards
    lw = int(rng.choice([1, 5, 64, 100, 1024, 2047, 8192]))
    nlb = -(-lw // lbs)
    max_gb = int(min(rng.choice([0, 1, max(nlb // 2, 1), nlb, nlb + 7]), 16384))
    rows, rr = int(rng.integers(1, 40)), int(rng.choice([1, 1, 2, 5]))
    nbg = max(max_gb, 1)
    topk = int(rng.choice([1, 8, 32, 40, nbg, nbg + 3]))
    wl, _ = workloads.small_sharded(27000 + seed, shards=shards, rows=rows,
                                    global_width=lw * shards, global_block_size=gbs,
                                    max_global_blocks=max_gb, topk_blocks=topk, row_repeat=rr,
                                    wild_bounds=bool(rng.integers(0, 2)))
    groups = -(-rows // rr)
    gks = rng.integers(-4, shards * lw + 6, size=groups).astype(np.int32)
    gks[::3] = np.minimum(gks[::3], wl.global_row_ke[::3] - 1)  # mostly non-empty windows
    want_ids, want_sc = oracle.select_sharded_starts(wl.logits, gks, wl.global_row_ke, gbs,
                                                     max_gb, topk, rr)
    offset = int(rng.choice([0, 1, 2, 3]))
    buf = torch.full((shards * rows * lw + offset + 8,), 1e30, dtype=torch.float32,
                     device="cuda")
    local = buf[offset:offset + shards * rows * lw].view(shards, rows, lw)
    local.copy_(torch.from_numpy(wl.logits))
    for ws in (None, False):
        ids, sc = _run_sharded_starts(env, local, gks, wl.global_row_ke, gbs, max_gb, topk, rr,
                                      ws)
        np.testing.assert_array_equal(ids, want_ids)
        assert_bits_equal(sc, want_sc)
    cand = rng.integers(-1, nlb + 2, size=(rows, 6)).astype(np.int32)
    want_mask = oracle.mask_sharded_starts(wl.logits, gks, wl.global_row_ke, gbs, cand, rr)
    dsa.dsa_mask_candidate_logits_sharded(local, _dev(torch, wl.global_row_ke), gbs,
                                          _dev(torch, cand), rr, global_row_ks=_dev(torch, gks))
    torch.cuda.synchronize()
    assert_bits_equal(local.cpu().numpy(), want_mask)


@pytest.mark.slow
def test_sharded_starts_full_size(env):
    """The DCP workload with request starts drawn uniform in [0, gke]."""
    torch, dsa = env
    wl = workloads.make("dcp")
    rng = np.random.default_rng(4004)
    gks = (rng.random(wl.global_row_ke.size) * (wl.global_row_ke + 1)).astype(np.int32)
    want_ids, want_sc = oracle.select_sharded_starts(wl.logits, gks, wl.global_row_ke,
                                                     wl.global_block_size, wl.max_global_blocks,
                                                     wl.topk_blocks)
    local = torch.from_numpy(wl.logits).cuda()
    for ws in (None, False):
        ids, sc = _run_sharded_starts(env, local, gks, wl.global_row_ke, wl.global_block_size,
                                      wl.max_global_blocks, wl.topk_blocks, 1, ws)
        np.testing.assert_array_equal(ids, want_ids)
        assert_bits_equal(sc, want_sc)


@pytest.mark.parametrize("seed", range(12))
def test_block_scores_sweep(env, seed):
    torch, dsa = env
    rng = np.random.default_rng(900 + seed)
    bs = int(rng.choice(BLOCK_SIZES))
    width = int(rng.choice([1, 100, 4096, 20000, 131072]))
    rows = int(rng.integers(1, 24))
    wl = workloads.small_unsharded(900 + seed, rows=rows, width=width, block_size=bs,
                                   topk_blocks=1, row_repeat=int(rng.choice([1, 4])),
                                   pin_newest=bool(rng.integers(0, 2)), nan_count=4,
                                   wild_bounds=bool(rng.integers(0, 2)))
    want = oracle.block_scores(wl.logits, wl.row_ks, wl.row_ke, bs, wl.row_repeat, wl.pin_newest)
    nb = want.shape[1]
    buf = torch.full((rows, nb + GUARD), float(SENTINEL_SCORE), dtype=torch.float32,
                     device="cuda")
    dsa.dsa_block_scores(_dev(torch, wl.logits), _dev(torch, wl.row_ks), _dev(torch, wl.row_ke),
                         bs, wl.row_repeat, wl.pin_newest, scores_out=buf[:, :nb])
    got = buf.cpu().numpy()
    assert (got[:, nb:] == SENTINEL_SCORE).all()
    assert_bits_equal(got[:, :nb], want)


WARP_CASES = [  # (block_size, width, topk, row_repeat, starts, bf16 grid, nan_count, wild)
    (64, 16384, 32, 1, True, False, 40, False),
    (64, 16000, 16, 4, False, True, 0, True),
    (128, 16383, 32, 1, True, False, 0, False),
    (8, 16384, 32, 1, True, False, 5, False),     # 2048 blocks: keys beyond registers
    (3, 4000, 20, 2, True, False, 9, True),       # generic streaming path
    (1, 1500, 32, 1, False, True, 0, False),
    (100, 9000, 7, 8, True, False, 3, False),
]


@pytest.mark.parametrize("case", WARP_CASES, ids=[f"bs{c[0]}-w{c[1]}-k{c[2]}" for c in WARP_CASES])
def test_warp_per_row_sweep(env, case):
    """Many short rows take the one-row-per-warp kernel."""
    bs, width, topk, rr, starts, bf16, nans, wild = case
    wl = workloads.small_unsharded(3000 + bs, rows=1300 + 97 * rr, width=width, block_size=bs,
                                   topk_blocks=topk, row_repeat=rr, starts=starts,
                                   bf16_grid=bf16, nan_count=nans, wild_bounds=wild)
    check_unsharded(env, wl, offset=1 if bs % 4 else 0)


def test_warp_per_row_ties_fallback(env):
    """Rows whose blocks all tie leave more candidates than a warp ranks by
    counting; the warp falls back to repeated maxima."""
    rows, width = 1400, 8192
    x = np.zeros((rows, width), dtype=np.float32)
    x[::2] = 1.5  # even rows: every block ties
    x[1::2] = workloads.round_to_bf16_grid(
        np.random.default_rng(5).standard_normal((rows // 2, width), dtype=np.float32)).round(0)
    wl = workloads.Workload("ties", x, None, np.full(rows, width, np.int32), 32, 32, 1, True, 0)
    check_unsharded(env, wl)


# ---------------------------------------------------------------------------
# Masking to the selected candidate blocks
# ---------------------------------------------------------------------------

def _random_candidates(rng, rows, topk, nb):
    """Ids in [-1, nb + 2): empty slots, duplicates and ids past the row's
    blocks all occur."""
    return rng.integers(-1, nb + 2, size=(rows, topk)).astype(np.int32)


@pytest.mark.parametrize("seed", range(16))
def test_mask_sweep(env, seed):
    torch, dsa = env
    rng = np.random.default_rng(8000 + seed)
    bs = int(BLOCK_SIZES[seed % len(BLOCK_SIZES)])
    width = int(rng.choice([1, 5, 100, 4096, 8191, 8192, 8193, 30001]))
    rows = int(rng.integers(1, 30))
    rr = int(rng.choice([1, 2, 3]))
    topk = int(rng.choice([0, 1, 7, 32, 100]))
    wl = workloads.small_unsharded(8000 + seed, rows=rows, width=width, block_size=bs,
                                   topk_blocks=max(topk, 1), row_repeat=rr,
                                   starts=bool(rng.integers(0, 2)), nan_count=7,
                                   wild_bounds=bool(rng.integers(0, 2)),
                                   ld=width + int(rng.choice([0, 1, 3])))
    nb = -(-width // bs)
    cand = _random_candidates(rng, rows, topk, nb)
    want = oracle.mask(wl.logits, wl.row_ks, wl.row_ke, cand, bs, rr, width=width)
    logits = _padded_logits(torch, wl.logits, width, int(rng.choice([0, 1, 2, 3])))
    dsa.dsa_mask_candidate_logits(logits, _dev(torch, wl.row_ks), _dev(torch, wl.row_ke),
                                  _dev(torch, cand) if topk else None, bs, rr)
    torch.cuda.synchronize()
    got = logits.cpu().numpy()
    assert_bits_equal(got, want[:, :width])


@pytest.mark.parametrize("bs", [2, 1000, 4096, 8193, 20000])
def test_mask_long_kept_runs(env, bs):
    """Kept runs longer than a chunk, runs that start or end inside a 16-byte
    slot, and adjacent candidate blocks whose runs meet inside a slot."""
    torch, dsa = env
    rng = np.random.default_rng(8800 + bs)
    width, rows = 40001, 6
    wl = workloads.small_unsharded(8800 + bs, rows=rows, width=width, block_size=bs,
                                   topk_blocks=8, starts=True, ld=width + 1)
    nb = -(-width // bs)
    cand = np.stack([rng.permutation(nb)[:8] if nb >= 8 else
                     np.concatenate([np.arange(nb), -np.ones(8 - nb, int)])
                     for _ in range(rows)]).astype(np.int32)
    cand[0, :2] = [0, 1]           # adjacent blocks
    want = oracle.mask(wl.logits, wl.row_ks, wl.row_ke, cand, bs, 1, width=width)
    logits = _padded_logits(torch, wl.logits, width, 1)
    dsa.dsa_mask_candidate_logits(logits, _dev(torch, wl.row_ks), _dev(torch, wl.row_ke),
                                  _dev(torch, cand), bs, 1)
    torch.cuda.synchronize()
    assert_bits_equal(logits.cpu().numpy(), want[:, :width])


@pytest.mark.parametrize("seed", range(8))
def test_mask_sharded_sweep(env, seed):
    torch, dsa = env
    rng = np.random.default_rng(8500 + seed)
    shards = int(rng.choice([1, 2, 3, 8]))
    lbs = int(rng.choice([1, 3, 8, 16]))
    lw = int(rng.choice([1, 100, 2047, 8192, 9000]))
    rows, topk = int(rng.integers(1, 20)), int(rng.choice([0, 5, 32]))
    wl, _ = workloads.small_sharded(8500 + seed, shards=shards, rows=rows,
                                    global_width=lw * shards, global_block_size=lbs * shards,
                                    max_global_blocks=-(-lw // lbs), topk_blocks=max(topk, 1),
                                    wild_bounds=True)
    cand = _random_candidates(rng, rows, topk, -(-lw // lbs))
    want = oracle.mask_sharded(wl.logits, wl.global_row_ke, lbs * shards, cand)
    local = torch.from_numpy(wl.logits).cuda()
    dsa.dsa_mask_candidate_logits_sharded(local, _dev(torch, wl.global_row_ke), lbs * shards,
                                          _dev(torch, cand) if topk else None)
    torch.cuda.synchronize()
    assert_bits_equal(local.cpu().numpy(), want)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["decode", "prefill", "dcp"])
def test_select_then_mask_full_size(env, name):
    """The pipeline as used: select on the GPU, then mask on the GPU with the
    selected ids, against the oracle doing both."""
    torch, dsa = env
    wl = workloads.make(name)
    ids, _ = oracle.run_workload(wl, want_scores=False)
    if hasattr(wl, "global_row_ke"):
        want = oracle.mask_sharded(wl.logits, wl.global_row_ke, wl.global_block_size, ids)
        local = torch.from_numpy(wl.logits).cuda()
        gke = _dev(torch, wl.global_row_ke)
        out = torch.empty((wl.rows, wl.topk_blocks), dtype=torch.int32, device="cuda")
        dsa.dsa_select_candidate_blocks_sharded(local, gke, wl.global_block_size,
                                                wl.max_global_blocks, wl.topk_blocks, out)
        dsa.dsa_mask_candidate_logits_sharded(local, gke, wl.global_block_size, out)
    else:
        want = oracle.mask(wl.logits, wl.row_ks, wl.row_ke, ids, wl.block_size, wl.row_repeat)
        local = torch.from_numpy(wl.logits).cuda()
        ks, ke = _dev(torch, wl.row_ks), _dev(torch, wl.row_ke)
        out = torch.empty((wl.rows, wl.topk_blocks), dtype=torch.int32, device="cuda")
        dsa.dsa_select_candidate_blocks(local, ks, ke, wl.topk_blocks, wl.block_size, out,
                                        wl.row_repeat, wl.pin_newest)
        dsa.dsa_mask_candidate_logits(local, ks, ke, out, wl.block_size, wl.row_repeat)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.cpu().numpy(), ids)
    assert_bits_equal(local.cpu().numpy(), want)


def test_sharded_equals_unsharded_on_device(env):
    torch, dsa = env
    wl, g = workloads.small_sharded(4242, shards=8, rows=64, global_width=65536,
                                    global_block_size=64, max_global_blocks=1024, topk_blocks=32)
    ids_s, sc_s = run_sharded(env, wl)
    ids_u, sc_u = run_unsharded(env, workloads.Workload(
        "g", g, None, wl.global_row_ke, 64, 32, 1, True, 0))
    np.testing.assert_array_equal(ids_s, ids_u)
    assert_bits_equal(sc_s, sc_u)


# ---------------------------------------------------------------------------
# Edge cases
# ---------------------------------------------------------------------------

def test_empty_rows_is_noop(env):
    torch, dsa = env
    out = torch.full((0, 4), 5, dtype=torch.int32, device="cuda")
    dsa.dsa_select_candidate_blocks(torch.zeros((0, 16), device="cuda"), None,
                                    torch.zeros(0, dtype=torch.int32, device="cuda"), 4, 4, out)
    torch.cuda.synchronize()


def test_zero_width_gives_minus_one(env):
    torch, dsa = env
    out = torch.full((5, 4), 5, dtype=torch.int32, device="cuda")
    dsa.dsa_select_candidate_blocks(torch.zeros((5, 0), device="cuda"), None,
                                    torch.zeros(5, dtype=torch.int32, device="cuda"), 4, 4, out)
    assert (out.cpu() == -1).all()


def test_topk_zero_with_scores(env):
    wl = workloads.small_unsharded(7, rows=9, width=1000, block_size=16, topk_blocks=0)
    want = oracle.block_scores(wl.logits, wl.row_ks, wl.row_ke, 16, 1, True)
    _, got = run_unsharded(env, wl)
    assert_bits_equal(got, want)


def test_largest_supported_rows(env):
    """nb at the shared-memory limit, K above 32 (shared-memory sort)."""
    torch, dsa = env
    nmax = dsa.max_select_blocks()
    wl = workloads.small_unsharded(8, rows=6, width=nmax, block_size=1, topk_blocks=nmax,
                                   starts=False, nan_count=3, bf16_grid=True)
    check_unsharded(env, wl)
    wl = workloads.small_unsharded(9, rows=5, width=nmax * 4, block_size=4, topk_blocks=600)
    check_unsharded(env, wl)


def test_beyond_limits_raise(env):
    torch, dsa = env
    nmax = dsa.max_select_blocks()
    out = torch.empty((2, 4), dtype=torch.int32, device="cuda")
    with pytest.raises(dsa.DsaError) as e:
        dsa.dsa_select_candidate_blocks(torch.zeros((2, nmax + 1), device="cuda"), None,
                                        torch.ones(2, dtype=torch.int32, device="cuda"), 4, 1, out)
    assert e.value.status == -3
    with pytest.raises(dsa.DsaError) as e:
        dsa.dsa_select_candidate_blocks_sharded(torch.zeros((8, 2, 64), device="cuda"),
                                                torch.ones(2, dtype=torch.int32, device="cuda"),
                                                60, 8, 4, out)
    assert e.value.status == -1


def test_all_nan_and_all_inf_rows(env):
    x = np.full((4, 256), np.nan, dtype=np.float32)
    x[1] = np.inf
    x[2] = -np.inf
    x[3, ::2] = -0.0
    x[3, 1::2] = 0.0
    wl = workloads.Workload("edge", x, None, np.full(4, 256, np.int32), 16, 20, 1, False, 0)
    check_unsharded(env, wl)
    wl.pin_newest = True
    check_unsharded(env, wl)


def test_workspace_reuse_across_shapes(env):
    """A caller-owned, zero-filled workspace serves calls of different shapes
    in turn: key data one call leaves where a later call keeps its arrival
    counters is never taken for a count."""
    torch, dsa = env
    ws = torch.zeros(dsa.workspace_bytes(600, 2048), dtype=torch.uint8, device="cuda")
    cases = [workloads.small_unsharded(40, rows=300, width=131072, block_size=64,
                                       topk_blocks=32, starts=False),
             workloads.small_unsharded(41, rows=17, width=70000, block_size=128, topk_blocks=7),
             workloads.small_unsharded(42, rows=200, width=40000, block_size=32,
                                       topk_blocks=40, bf16_grid=True)]
    for wl in cases:
        ref_ids, _ = oracle.run_workload(wl)
        for _ in range(2):
            got, _ = run_unsharded(env, wl, want_scores=False, workspace=ws)
            np.testing.assert_array_equal(got, ref_ids)
    # the calls above left block keys all over the workspace; a larger call
    # now finds them where its counters are
    wl = workloads.small_unsharded(43, rows=600, width=131072, block_size=128,
                                   topk_blocks=16, starts=False)
    ref_ids, _ = oracle.run_workload(wl)
    for _ in range(2):
        got, _ = run_unsharded(env, wl, want_scores=False, workspace=ws)
        np.testing.assert_array_equal(got, ref_ids)


@pytest.mark.parametrize("sharded", [False, True])
def test_graph_replay_matches_oracle(env, sharded):
    """The bench replays selection from CUDA graphs: replays must give the
    oracle's ids, including the workspace split path."""
    torch, dsa = env
    import bench

    if sharded:
        wl, _ = workloads.small_sharded(60, shards=8, rows=96, global_width=65536,
                                        global_block_size=64, max_global_blocks=1024,
                                        topk_blocks=32)
    else:
        wl = workloads.small_unsharded(61, rows=96, width=65536, block_size=64, topk_blocks=32,
                                       row_repeat=8, starts=False, bf16_grid=True)
    ref_ids, _ = oracle.run_workload(wl)
    step, out = bench.make_runner(wl, dsa, torch, torch.device("cuda"))
    step()
    torch.cuda.synchronize()
    g = bench.graph_of(step, 3, torch)
    out.fill_(-9)
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.cpu().numpy(), ref_ids)


def test_non_default_stream(env):
    torch, dsa = env
    wl = workloads.small_unsharded(10, rows=33, width=9000, block_size=64, topk_blocks=32)
    want_ids, _ = oracle.run_workload(wl)
    s = torch.cuda.Stream()
    out = torch.empty((33, 32), dtype=torch.int32, device="cuda")
    with torch.cuda.stream(s):
        logits = _dev(torch, wl.logits)
        ks, ke = _dev(torch, wl.row_ks), _dev(torch, wl.row_ke)
        dsa.dsa_select_candidate_blocks(logits, ks, ke, 32, 64, out)
    s.synchronize()
    np.testing.assert_array_equal(out.cpu().numpy(), want_ids)


def test_repeated_calls_identical(env):
    wl = workloads.small_unsharded(11, rows=64, width=65536, block_size=64, topk_blocks=32,
                                   bf16_grid=True, starts=False)
    a = run_unsharded(env, wl)
    b = run_unsharded(env, wl)
    np.testing.assert_array_equal(a[0], b[0])
    assert_bits_equal(a[1], b[1])


def test_host_buffer_entry_points(env):
    torch, dsa = env
    wl = workloads.small_unsharded(12, rows=16, width=5000, block_size=64, topk_blocks=16)
    want_ids, _ = oracle.run_workload(wl)
    got = dsa.select_candidate_blocks_host(torch.from_numpy(wl.logits),
                                           torch.from_numpy(wl.row_ks),
                                           torch.from_numpy(wl.row_ke), 16, 64)
    np.testing.assert_array_equal(got.numpy(), want_ids)
    swl, _ = workloads.small_sharded(13, shards=8, rows=16, global_width=4096,
                                     global_block_size=64, max_global_blocks=64, topk_blocks=8)
    want_ids, _ = oracle.run_workload(swl)
    got = dsa.select_candidate_blocks_sharded_host(torch.from_numpy(swl.logits),
                                                   torch.from_numpy(swl.global_row_ke), 64, 64, 8)
    np.testing.assert_array_equal(got.numpy(), want_ids)


# ---------------------------------------------------------------------------
# The workloads at full size (bench launch configuration), every output
# ---------------------------------------------------------------------------

@pytest.mark.slow
@pytest.mark.parametrize("name", ["tiny", "decode", "prefill", "long", "long_pin"])
def test_full_size_unsharded(env, name):
    wl = workloads.make(name)
    check_unsharded(env, wl)
    # the bench calls without scores_out
    want_ids, _ = oracle.run_workload(wl, want_scores=False)
    got_ids, _ = run_unsharded(env, wl, want_scores=False)
    np.testing.assert_array_equal(got_ids, want_ids)


@pytest.mark.slow
def test_full_size_dcp(env):
    wl = workloads.make("dcp")
    check_sharded(env, wl)
    want_ids, _ = oracle.run_workload(wl, want_scores=False)
    got_ids, _ = run_sharded(env, wl, want_scores=False)
    np.testing.assert_array_equal(got_ids, want_ids)


def test_no_pipelined_wait_gave_up(env):
    # Every bounded wait of the pipelined kernels in the calls above (this
    # file and the ones collected before it) completed: none recorded a
    # give-up in the library's device-wide flag.
    _, dsa = env
    assert dsa.pipeline_error() == 0
