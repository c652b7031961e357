"""Pins the masking oracle (the step after selection; see
oracle/dsa_oracle.c, reading R8) to things other than itself: hand-computed
cases, a pure-Python brute force, the selection it follows, and the
interleave identity of the DCP form."""

import numpy as np
import pytest

import oracle
import workloads
from helpers import assert_bits_equal, deal_shards, load_golden, parse_matrix


def test_golden_mask():
    fx = load_golden("mask_to_candidates.json")
    assert fx["cite"] and fx["why"]
    for case in fx["cases"]:
        cand = np.array(case["candidates"], dtype=np.int32)
        if case["op"] == "mask":
            x = parse_matrix(case["logits"])
            got = oracle.mask(x, np.array(case["row_ks"], np.int32),
                              np.array(case["row_ke"], np.int32), cand, case["block_size"],
                              case["row_repeat"], width=case["width"])
            assert_bits_equal(got, parse_matrix(case["expect"]))
        else:
            g = parse_matrix(case["global_logits"])
            got = oracle.mask_sharded(deal_shards(g, case["shards"]),
                                      np.array(case["global_row_ke"], np.int32),
                                      case["global_block_size"], cand, case["row_repeat"])
            assert_bits_equal(got, deal_shards(parse_matrix(case["expect_global"]),
                                               case["shards"]))


def brute_mask(x, ks, ke, cand, bs, rr, width):
    out = x.copy()
    for r in range(x.shape[0]):
        g = r // rr
        e = min(int(ke[g]), width)
        s = min(max(0 if ks is None else int(ks[g]), 0), e)
        keep = {int(c) for c in cand[r] if c >= 0}
        for c in range(width):
            if not (s <= c < e and (c - s) // bs in keep):
                out[r, c] = -np.inf
    return out


@pytest.mark.parametrize("seed", range(30))
def test_mask_matches_brute_force(seed):
    rng = np.random.default_rng(7000 + seed)
    rows, width = int(rng.integers(1, 6)), int(rng.integers(0, 50))
    bs, rr, topk = int(rng.choice([1, 2, 3, 4, 7, 16])), int(rng.integers(1, 3)), int(rng.integers(0, 6))
    groups = -(-rows // rr)
    x = rng.standard_normal((rows, width)).astype(np.float32)
    x[rng.random((rows, width)) < 0.05] = np.nan
    ke = rng.integers(-2, width + 4, size=groups).astype(np.int32)
    ks = rng.integers(-2, width + 2, size=groups).astype(np.int32) if rng.integers(0, 2) else None
    nb = max(-(-width // bs), 1)
    cand = rng.integers(-1, nb + 1, size=(rows, topk)).astype(np.int32)
    got = oracle.mask(x, ks, ke, cand, bs, rr, width=width)
    assert_bits_equal(got, brute_mask(x, ks, ke, cand, bs, rr, width))


def test_mask_after_select_keeps_exactly_the_selected_blocks():
    wl = workloads.small_unsharded(71, rows=40, width=3000, block_size=64, topk_blocks=8,
                                   nan_count=4)
    ids, _ = oracle.run_workload(wl)
    masked = oracle.mask(wl.logits, wl.row_ks, wl.row_ke, ids, 64, 1)
    before = oracle.block_scores(wl.logits, wl.row_ks, wl.row_ke, 64, 1, False)
    after = oracle.block_scores(masked, wl.row_ks, wl.row_ke, 64, 1, False)
    for r in range(wl.rows):
        sel = set(ids[r][ids[r] >= 0].tolist())
        for b in range(before.shape[1]):
            if b in sel:
                assert_bits_equal(after[r, b:b + 1], before[r, b:b + 1])
            else:
                assert after[r, b] == -np.inf


@pytest.mark.parametrize("shards,lbs", [(8, 8), (3, 5), (2, 1)])
def test_mask_sharded_equals_unsharded_on_global_rows(shards, lbs):
    gbs, lw, rows = shards * lbs, 40 * lbs + 3, 11
    wl, g = workloads.small_sharded(90 + shards, shards=shards, rows=rows, global_width=lw * shards,
                                    global_block_size=gbs, max_global_blocks=-(-lw // lbs),
                                    topk_blocks=6)
    ids, _ = oracle.run_workload(wl)
    got = oracle.mask_sharded(wl.logits, wl.global_row_ke, gbs, ids)
    want = oracle.mask(g, None, wl.global_row_ke, ids, gbs)
    assert_bits_equal(got, deal_shards(want, shards))
