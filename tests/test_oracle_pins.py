"""Pins the CPU oracle to things other than itself.

* brute force on tiny inputs: a pure-Python restatement that slices each
  block, takes Python's ``max`` under an explicit rank key and ranks with
  ``sorted`` (no shared code with the C oracle);
* special cases that reduce to library routines: block size 1 (scores are
  the windowed logits), full-width blocks (``numpy.max``), reshaped block
  maxima, ``numpy.argsort`` / ``numpy.lexsort`` ranking;
* invariants at the workloads' shapes: every score is an in-window element
  of its block (or -inf exactly when the block is empty), the pinned block
  is selected, empty windows select nothing, NaN blocks are selected, ids are
  distinct and ranked;
* the interleave identity of the DCP form: the sharded result on
  ``[D, rows, w/D]`` equals the unsharded result on the global rows with the
  global block size (candidate_blocks.py diff, ``_select_candidate_blocks_impl``
  docstring: local block b is this rank's share of global block b, so the
  global score is the max over ranks).
"""

import math

import numpy as np
import pytest

import oracle
import workloads
from helpers import CANONICAL_NAN_BITS, assert_bits_equal, bits, deal_shards

NEG_INF = float("-inf")


# ---------------------------------------------------------------------------
# Brute force (pure Python, tiny inputs only)
# ---------------------------------------------------------------------------

def _rank(x: float):
    """Position of x in the order -inf < ... < -0 < +0 < ... < +inf < NaN."""
    if math.isnan(x):
        return (2, 0.0, 0)
    return (1, x, 0 if math.copysign(1.0, x) < 0 else 1)


def _brute_row(values, s, e, bs, nb, pin):
    scores = []
    for b in range(nb):
        cols = [c for c in range(s, e) if (c - s) // bs == b]
        scores.append(max((float(values[c]) for c in cols), key=_rank) if cols else NEG_INF)
    if pin and e > s:
        scores[(e - s - 1) // bs] = math.inf
    return scores


def _brute_select(scores, topk):
    order = sorted(range(len(scores)), key=lambda b: (_rank(scores[b]), -b), reverse=True)
    k = min(topk, len(scores))
    out = []
    for j in range(topk):
        ok = j < k and _rank(scores[order[j]]) > _rank(NEG_INF)
        out.append(order[j] if ok else -1)
    return out


def _to_f32(scores):
    a = np.array(scores, dtype=np.float32)
    nan = np.isnan(a)
    if nan.any():
        a.view(np.uint32)[nan] = CANONICAL_NAN_BITS
    return a


def brute_unsharded(logits, ks, ke, width, bs, rr, pin, topk):
    rows = logits.shape[0]
    nb = -(-width // bs)
    all_scores, all_ids = [], []
    for r in range(rows):
        g = r // rr
        k_s = 0 if ks is None else int(ks[g])
        e = min(int(ke[g]), width)
        s = min(max(k_s, 0), e)
        sc = _brute_row(logits[r], s, e, bs, nb, pin)
        all_scores.append(_to_f32(sc))
        all_ids.append(_brute_select(sc, topk))
    return (np.array(all_ids, dtype=np.int32).reshape(rows, topk),
            np.array(all_scores, dtype=np.float32).reshape(rows, nb))


def brute_sharded(local, gke_g, gbs, max_gb, rr, topk):
    shards, rows, lw = local.shape
    lbs = gbs // shards
    nbg = max(max_gb, 1)
    nlb = -(-lw // lbs)
    all_scores, all_ids = [], []
    for r in range(rows):
        gke = int(gke_g[r // rr])
        merged = [NEG_INF] * nbg
        for d in range(shards):
            lke = -(-(gke - d) // shards) if gke > d else 0
            sc = _brute_row(local[d, r], 0, min(lke, lw), lbs, nlb, False)
            for b in range(min(nlb, nbg)):
                merged[b] = max(merged[b], sc[b], key=_rank)
        pin = min(max((gke - 1) // gbs, 0), nbg - 1)
        merged[pin] = math.inf
        if gke <= 0:
            merged = [NEG_INF] * nbg
        all_scores.append(_to_f32(merged))
        all_ids.append(_brute_select(merged, topk))
    return (np.array(all_ids, dtype=np.int32).reshape(rows, topk),
            np.array(all_scores, dtype=np.float32).reshape(rows, nbg))


def _tiny_logits(rng, rows, width):
    """Small values with many ties, signed zeros, infinities and NaNs."""
    pool = np.array([-2.0, -1.0, -0.0, 0.0, 0.5, 1.0, 2.0, np.inf, -np.inf], dtype=np.float32)
    x = rng.choice(pool, size=(rows, width)).astype(np.float32)
    x += rng.integers(0, 3, size=(rows, width)).astype(np.float32) * np.float32(0.25) * (
        np.isfinite(x) & (x != 0))
    nan_mask = rng.random((rows, width)) < 0.04
    x[nan_mask] = workloads.random_nan_bits(rng, int(nan_mask.sum()))
    return x


@pytest.mark.parametrize("seed", range(60))
def test_unsharded_matches_brute_force(seed):
    rng = np.random.default_rng(1000 + seed)
    rows = int(rng.integers(0, 7))
    width = int(rng.integers(0, 41))
    bs = int(rng.choice([1, 2, 3, 4, 5, 7, 8, 16, 64]))
    rr = int(rng.integers(1, 4))
    pin = bool(rng.integers(0, 2))
    topk = int(rng.integers(0, 12))
    groups = -(-rows // rr)
    logits = _tiny_logits(rng, rows, width)
    ke = rng.integers(-3, width + 5, size=groups).astype(np.int32)
    ks = rng.integers(-3, width + 3, size=groups).astype(np.int32) if rng.integers(0, 2) else None
    got_ids, got_scores = oracle.select(logits, ks, ke, topk, bs, rr, pin, width=width)
    if rows == 0:
        return
    want_ids, want_scores = brute_unsharded(logits, ks, ke, width, bs, rr, pin, topk)
    np.testing.assert_array_equal(got_ids, want_ids)
    if width:
        assert_bits_equal(got_scores, want_scores)
        s2 = oracle.block_scores(logits, ks, ke, bs, rr, pin, width=width)
        assert_bits_equal(s2, want_scores)


@pytest.mark.parametrize("seed", range(40))
def test_sharded_matches_brute_force(seed):
    rng = np.random.default_rng(5000 + seed)
    shards = int(rng.choice([1, 2, 3, 4, 8]))
    lbs = int(rng.choice([1, 2, 3, 4]))
    gbs = lbs * shards
    lw = int(rng.integers(0, 9))
    rows = int(rng.integers(1, 6))
    rr = int(rng.integers(1, 3))
    max_gb = int(rng.integers(0, 6))
    topk = int(rng.integers(0, 8))
    local = _tiny_logits(rng, shards * rows, lw).reshape(shards, rows, lw)
    groups = -(-rows // rr)
    gke = rng.integers(-2, shards * lw + 6, size=groups).astype(np.int32)
    got_ids, got_scores = oracle.select_sharded(local, gke, gbs, max_gb, topk, rr)
    want_ids, want_scores = brute_sharded(local, gke, gbs, max_gb, rr, topk)
    np.testing.assert_array_equal(got_ids, want_ids)
    assert_bits_equal(got_scores, want_scores)


# ---------------------------------------------------------------------------
# Special cases that reduce to library routines
# ---------------------------------------------------------------------------

def test_block_size_one_gives_windowed_logits():
    rng = np.random.default_rng(7)
    rows, width = 9, 300
    x = rng.standard_normal((rows, width), dtype=np.float32)
    ke = rng.integers(0, width + 1, size=rows).astype(np.int32)
    ks = np.minimum(rng.integers(0, width + 1, size=rows), ke).astype(np.int32)
    s = oracle.block_scores(x, ks, ke, 1, 1, False)
    for r in range(rows):
        want = np.full(width, -np.inf, dtype=np.float32)
        n = ke[r] - ks[r]
        want[:n] = x[r, ks[r]:ke[r]]
        assert_bits_equal(s[r], want)


def test_full_width_block_is_numpy_max():
    rng = np.random.default_rng(8)
    rows, width = 16, 777
    x = rng.standard_normal((rows, width), dtype=np.float32)
    x[3, 100] = np.nan
    ke = rng.integers(1, width + 1, size=rows).astype(np.int32)
    ke[3] = width
    s = oracle.block_scores(x, None, ke, width, 1, False)
    for r in range(rows):
        m = np.max(x[r, :ke[r]])
        if np.isnan(m):
            assert bits(s[r, :1])[0] == CANONICAL_NAN_BITS
        else:
            assert s[r, 0] == m


def test_reshaped_block_max():
    rng = np.random.default_rng(9)
    rows, nb, bs = 12, 33, 16
    x = rng.standard_normal((rows, nb * bs), dtype=np.float32)
    ke = np.full(rows, nb * bs, dtype=np.int32)
    s = oracle.block_scores(x, None, ke, bs, 1, False)
    np.testing.assert_array_equal(s, x.reshape(rows, nb, bs).max(axis=-1))


def test_topk_is_stable_argsort_for_distinct_scores():
    rng = np.random.default_rng(10)
    rows, width, bs, topk = 20, 4096, 64, 16
    x = rng.standard_normal((rows, width), dtype=np.float32)
    ke = np.full(rows, width, dtype=np.int32)
    ids, s = oracle.select(x, None, ke, topk, bs, 1, False)
    for r in range(rows):
        assert len(np.unique(s[r])) == s.shape[1]
        np.testing.assert_array_equal(ids[r], np.argsort(-s[r], kind="stable")[:topk])


def test_ties_rank_lower_id_first_like_lexsort():
    rng = np.random.default_rng(11)
    rows, width, bs, topk = 24, 2048, 8, 40
    x = workloads.round_to_bf16_grid(rng.standard_normal((rows, width), dtype=np.float32))
    x = np.round(x * 2) / 2  # few distinct values: many tied blocks
    x = x.astype(np.float32)
    ke = np.full(rows, width, dtype=np.int32)
    ids, s = oracle.select(x, None, ke, topk, bs, 1, False)
    for r in range(rows):
        order = np.lexsort((np.arange(s.shape[1]), -s[r]))
        np.testing.assert_array_equal(ids[r], order[:topk])


# ---------------------------------------------------------------------------
# Invariants on the workload shapes (scaled down so the suite stays quick)
# ---------------------------------------------------------------------------

def _check_invariants(wl, ids, scores):
    rows, width, bs = wl.rows, wl.width, wl.block_size
    nb = scores.shape[1]
    for r in range(rows):
        g = r // wl.row_repeat
        ks = 0 if wl.row_ks is None else int(wl.row_ks[g])
        e = min(int(wl.row_ke[g]), width)
        s = min(max(ks, 0), e)
        row = wl.logits[r]
        pin_b = (e - s - 1) // bs if (wl.pin_newest and e > s) else -1
        nan_blocks = 0
        for b in range(nb):
            lo, hi = s + b * bs, min(s + (b + 1) * bs, e)
            v = scores[r, b]
            if b == pin_b:
                assert v == np.inf
                continue
            if lo >= hi:
                assert v == -np.inf, (r, b)
                continue
            seg = row[lo:hi]
            if np.isnan(seg).any():
                assert bits(scores[r, b:b + 1])[0] == CANONICAL_NAN_BITS
                nan_blocks += 1
            else:
                assert v in seg and v == seg.max()
        sel = ids[r][ids[r] >= 0]
        assert len(set(sel.tolist())) == len(sel)
        if e <= s:
            assert (ids[r] == -1).all()
        if pin_b >= 0 and nan_blocks < wl.topk_blocks:
            assert pin_b in sel
        key = [(2 if np.isnan(scores[r, b]) else 1, scores[r, b] if not np.isnan(scores[r, b]) else 0, -b)
               for b in sel]
        assert key == sorted(key, reverse=True)


@pytest.mark.parametrize("name", ["tiny", "decode_small", "prefill_small", "long_small"])
def test_invariants_on_workload_shapes(name):
    if name == "tiny":
        wl = workloads.make_tiny()
    elif name == "decode_small":
        wl = workloads.small_unsharded(21, rows=64, width=4096, block_size=64, topk_blocks=32,
                                       row_repeat=8, starts=False, bf16_grid=True)
    elif name == "prefill_small":
        wl = workloads.make_prefill(22, requests=4, tokens=64, max_prefix=192, width=512,
                                    nan_fraction=2e-3)
    else:
        wl = workloads.small_unsharded(23, rows=32, width=8192, block_size=128, topk_blocks=16,
                                       pin_newest=False, nan_count=5)
    ids, scores = oracle.run_workload(wl)
    _check_invariants(wl, ids, scores)
    # a NaN block is always selected when fewer than k blocks are NaN
    for r in range(wl.rows):
        nan_b = np.flatnonzero(np.isnan(scores[r]))
        if 0 < len(nan_b) <= wl.topk_blocks:
            assert set(nan_b.tolist()) <= set(ids[r].tolist())


def test_topk_above_block_count_pads():
    wl = workloads.small_unsharded(31, rows=5, width=100, block_size=32, topk_blocks=9)
    ids, scores = oracle.run_workload(wl)
    assert (ids[:, 4:] == -1).all()  # only 4 blocks exist


def test_empty_shapes():
    ids, s = oracle.select(np.zeros((0, 10), np.float32), None, np.zeros(0, np.int32), 4, 2)
    assert ids.shape == (0, 4)
    ids, s = oracle.select(np.zeros((3, 0), np.float32), None, np.zeros(3, np.int32), 4, 2)
    assert (ids == -1).all()
    ids, s = oracle.select(np.ones((3, 8), np.float32), None, np.full(3, 8, np.int32), 0, 2)
    assert ids.shape == (3, 0)


# ---------------------------------------------------------------------------
# The interleave identity of the DCP form
# ---------------------------------------------------------------------------

@pytest.mark.parametrize("shards,lbs,rows,lw,rr", [(8, 8, 40, 256, 1), (2, 32, 17, 300, 3),
                                                 (4, 1, 9, 64, 2), (1, 64, 10, 1000, 1),
                                                 (3, 5, 12, 61, 1)])
def test_sharded_equals_unsharded_on_global_rows(shards, lbs, rows, lw, rr):
    gbs = lbs * shards
    gw = lw * shards
    wl, g = workloads.small_sharded(77 + shards, shards=shards, rows=rows, global_width=gw,
                                    global_block_size=gbs, max_global_blocks=-(-gw // gbs),
                                    topk_blocks=13, row_repeat=rr)
    wl.global_row_ke[0] = 0
    wl.global_row_ke[-1] = gw
    np.testing.assert_array_equal(wl.logits, deal_shards(g, shards))
    ids_s, sc_s = oracle.run_workload(wl)
    ids_u, sc_u = oracle.select(g, None, wl.global_row_ke, 13, gbs, rr, True)
    np.testing.assert_array_equal(ids_s, ids_u)
    assert_bits_equal(sc_s, sc_u)


def test_single_shard_equals_unsharded():
    rng = np.random.default_rng(12)
    x = rng.standard_normal((7, 333), dtype=np.float32)
    ke = rng.integers(1, 334, size=7).astype(np.int32)
    ids_s, sc_s = oracle.select_sharded(x[None], ke, 16, 21, 8)
    ids_u, sc_u = oracle.select(x, None, ke, 8, 16, 1, True)
    np.testing.assert_array_equal(ids_s, ids_u)
    assert_bits_equal(sc_s, sc_u)


# ---------------------------------------------------------------------------
# Generator checks (inputs, not the method)
# ---------------------------------------------------------------------------

def test_bf16_grid_matches_torch():
    torch = pytest.importorskip("torch")
    rng = np.random.default_rng(13)
    x = rng.standard_normal(100000, dtype=np.float32)
    want = torch.from_numpy(x).bfloat16().float().numpy()
    np.testing.assert_array_equal(workloads.round_to_bf16_grid(x), want)


def test_prefill_layout():
    wl = workloads.make_prefill(2, requests=4, tokens=8, max_prefix=24, width=64,
                                nan_fraction=0.01)
    pre, off = wl.notes["prefixes"], wl.notes["offsets"]
    assert sum(p + 8 for p in pre) <= 64
    for q in range(4):
        for i in range(8):
            r = q * 8 + i
            assert wl.row_ks[r] == off[q] and wl.row_ke[r] == off[q] + pre[q] + i + 1
    assert np.isnan(wl.logits).sum() == wl.notes["nan_count"] == round(0.01 * 32 * 64)
