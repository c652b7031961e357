"""Pins the oracle's DCP form with global window starts (reading R12 in
``oracle/dsa_oracle.c``).

* a hand-computed case (``tests/golden/dcp_starts.json``);
* a pure-Python brute force that walks the global tokens of each row's
  window and finds each token on its shard by the interleave-1 placement
  (token t on shard t % D, local column t // D), counting blocks from the
  global start, instead of computing per-shard windows;
* the interleave identity: on a gathered global matrix, the sharded result
  with starts equals the unsharded result with row starts and the global
  block size (selection with the pin, and masking).
"""

import math

import numpy as np
import pytest

import oracle
import test_oracle_pins as pins
from helpers import assert_bits_equal, deal_shards, load_golden, parse_matrix

FIXTURE = "dcp_starts.json"


def _cases():
    fx = load_golden(FIXTURE)
    assert fx.get("cite") and fx.get("why")
    return [pytest.param(c, id=f"{c['op']}-{i}") for i, c in enumerate(fx["cases"])]


@pytest.mark.parametrize("case", _cases())
def test_golden_starts_case(case):
    local = deal_shards(parse_matrix(case["global_logits"]), case["shards"])
    ids, scores = oracle.select_sharded_starts(
        local, np.array(case["global_row_ks"], np.int32), np.array(case["global_row_ke"], np.int32),
        case["global_block_size"], case["max_global_blocks"], case["topk_blocks"],
        case["row_repeat"])
    np.testing.assert_array_equal(ids, np.array(case["expect_ids"], np.int32))
    assert_bits_equal(scores, parse_matrix(case["expect_scores"]))


def brute_sharded_starts(local, gks, gke, gbs, max_gb, rr, topk):
    D, rows, lw = local.shape
    nbg = max(max_gb, 1)
    all_ids, all_scores = [], []
    for r in range(rows):
        ge = int(gke[r // rr])
        gs = min(max(int(gks[r // rr]), 0), max(ge, 0))
        sc = [-math.inf] * nbg
        for t in range(gs, min(ge, D * lw)):
            b = (t - gs) // gbs
            if b < nbg:
                sc[b] = max(sc[b], float(local[t % D, r, t // D]), key=pins._rank)
        if ge > gs:
            sc[min((ge - gs - 1) // gbs, nbg - 1)] = math.inf
        else:
            sc = [-math.inf] * nbg
        all_scores.append(pins._to_f32(sc))
        all_ids.append(pins._brute_select(sc, topk))
    return (np.array(all_ids, np.int32).reshape(rows, topk),
            np.array(all_scores, np.float32).reshape(rows, nbg))


@pytest.mark.parametrize("seed", range(40))
def test_sharded_starts_matches_brute_force(seed):
    rng = np.random.default_rng(9100 + seed)
    shards, lbs = int(rng.choice([1, 2, 3, 4, 8])), int(rng.choice([1, 2, 3, 4]))
    gbs = lbs * shards
    lw, rows, rr = int(rng.integers(0, 9)), int(rng.integers(1, 6)), int(rng.integers(1, 3))
    max_gb, topk = int(rng.integers(0, 7)), int(rng.integers(0, 8))
    local = pins._tiny_logits(rng, shards * rows, lw).reshape(shards, rows, lw)
    groups = -(-rows // rr)
    gke = rng.integers(-2, shards * lw + 6, size=groups).astype(np.int32)
    gks = rng.integers(-3, shards * lw + 4, size=groups).astype(np.int32)
    got_ids, got_scores = oracle.select_sharded_starts(local, gks, gke, gbs, max_gb, topk, rr)
    want_ids, want_scores = brute_sharded_starts(local, gks, gke, gbs, max_gb, rr, topk)
    np.testing.assert_array_equal(got_ids, want_ids)
    assert_bits_equal(got_scores, want_scores)


@pytest.mark.parametrize("shards,lbs,rows,lw,rr", [(2, 4, 7, 40, 1), (8, 8, 5, 96, 2),
                                                   (3, 2, 6, 33, 3), (1, 16, 4, 100, 1)])
def test_sharded_starts_equals_unsharded_on_global_rows(shards, lbs, rows, lw, rr):
    rng = np.random.default_rng(shards * 100 + lbs)
    gbs, width = lbs * shards, lw * shards
    g = rng.standard_normal((rows, width)).astype(np.float32)
    g[rng.random((rows, width)) < 0.02] = np.nan
    groups = -(-rows // rr)
    gke = rng.integers(0, width, size=groups, endpoint=True).astype(np.int32)
    gks = np.minimum(rng.integers(-4, width, size=groups), gke).astype(np.int32)
    nb = -(-width // gbs)
    topk = 9
    ids, scores = oracle.select_sharded_starts(deal_shards(g, shards), gks, gke, gbs, nb, topk, rr)
    want_ids, want_scores = oracle.select(g, gks, gke, topk, gbs, rr, True)
    np.testing.assert_array_equal(ids, want_ids)
    assert_bits_equal(scores, want_scores)
    cand = rng.integers(-1, nb + 1, size=(rows, 5)).astype(np.int32)
    got = oracle.mask_sharded_starts(deal_shards(g, shards), gks, gke, gbs, cand, rr)
    want = deal_shards(oracle.mask(g, gks, gke, cand, gbs, rr), shards)
    assert_bits_equal(got, want)


def test_null_starts_equal_the_pages_form():
    rng = np.random.default_rng(77)
    local = rng.standard_normal((4, 6, 50)).astype(np.float32)
    gke = rng.integers(-3, 205, size=6).astype(np.int32)
    zeros = np.zeros(6, np.int32)
    a = oracle.select_sharded_starts(local, zeros, gke, 16, 13, 8)
    b = oracle.select_sharded(local, gke, 16, 13, 8)
    np.testing.assert_array_equal(a[0], b[0])
    assert_bits_equal(a[1], b[1])
