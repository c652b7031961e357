"""The oracle's pins must catch plausible mistakes.

Each case below plants one mistake in a temporary copy of ``oracle/dsa_oracle.c``
(the committed source is never touched), builds it with gcc, and runs the
golden fixtures, the brute-force comparisons and the interleave identity
against the planted copy. At least one of them has to fail; a mistake that
passes every pin would mean the pins do not constrain that part of the
oracle. Only in-bounds mistakes are planted, so a planted copy cannot crash
the test process.
"""

import os

import numpy as np
import pytest

import oracle
import test_oracle_golden as golden
import test_oracle_pins as pins

MUTATIONS = [
    ("absolute block origin", "int64_t lo = s + b * bs;", "int64_t lo = b * bs;"),
    ("pin uses the absolute end", "score[(e - s - 1) / bs] = INFINITY;",
     "score[(e - 1) / bs] = INFINITY;"),
    ("NaN ranks lowest", "return a_nan - b_nan;", "return b_nan - a_nan;"),
    ("-0 ranks above +0", "return b_neg - a_neg;", "return a_neg - b_neg;"),
    ("ties rank the higher id first", "return (a->id > b->id) - (a->id < b->id);",
     "return (a->id < b->id) - (a->id > b->id);"),
    ("-inf blocks are emitted", "int keep = j < k && total_cmp(tmp[j].v, -INFINITY) > 0;",
     "int keep = j < k;"),
    ("starts ignored", "int64_t ks = row_ks ? (int64_t)row_ks[g] : 0;", "int64_t ks = 0;"),
    ("block max drops NaN and ignores the zero sign", "if (total_cmp(x, m) > 0)\n                m = x;",
     "if (x > m)\n                m = x;"),
    ("shard end rounds down",
     "(gke - d + shards - 1) / shards : 0;\n            int64_t e = imin64(lke, local_width);\n            int64_t s = imin64(lks, e);\n            if (nlb == 0)",
     "(gke - d) / shards : 0;\n            int64_t e = imin64(lke, local_width);\n            int64_t s = imin64(lks, e);\n            if (nlb == 0)"),
    ("global pin off by one", "pin = floor_div(gke - gs - 1, global_block_size);",
     "pin = floor_div(gke - gs, global_block_size);"),
    ("rows without context keep the pin", "if (gke <= gs)\n            for (b = 0; b < nbg; ++b)",
     "if (gke < gs)\n            for (b = 0; b < nbg; ++b)"),
    ("shard start rounds down",
     "int64_t lks = gs > d ? (gs - d + shards - 1) / shards : 0;\n            int64_t lke = gke > d ? (gke - d + shards - 1) / shards : 0;\n            int64_t e = imin64(lke, local_width);\n            int64_t s = imin64(lks, e);\n            if (nlb == 0)",
     "int64_t lks = gs > d ? (gs - d) / shards : 0;\n            int64_t lke = gke > d ? (gke - d + shards - 1) / shards : 0;\n            int64_t e = imin64(lke, local_width);\n            int64_t s = imin64(lks, e);\n            if (nlb == 0)"),
    ("DCP pin ignores the start", "pin = floor_div(gke - gs - 1, global_block_size);",
     "pin = floor_div(gke - 1, global_block_size);"),
    ("DCP blocks counted from local column 0", "row_block_scores(row, s, e, lbs, nlb, 0, local_score);",
     "row_block_scores(row, 0, e, lbs, nlb, 0, local_score);"),
    ("DCP start not clamped at 0", "int64_t gs = imin64(imax64(gks, 0), imax64(gke, 0));\n        int64_t pin;",
     "int64_t gs = imin64(gks, imax64(gke, 0));\n        int64_t pin;"),
    ("DCP mask keeps columns before the shard start",
     "int keep = c >= s && c < e &&\n                           is_candidate(cand + r * ld_cand, topk, (c - s) / lbs);",
     "int keep = c < e &&\n                           is_candidate(cand + r * ld_cand, topk, (c - s) / lbs);"),
    ("shard merge takes the min", "if (total_cmp(local_score[b], global_score[b]) > 0)",
     "if (total_cmp(local_score[b], global_score[b]) < 0)"),
    ("canonical NaN not written", "uint32_t bits = 0x7FC00000u;", "uint32_t bits = 0x7FC00001u;"),
    ("mask uses absolute blocks", "is_candidate(cand + r * ld_cand, topk, (c - s) / block_size)",
     "is_candidate(cand + r * ld_cand, topk, c / block_size)"),
    ("mask keeps columns before the window",
     "int keep = c >= s && c < e &&\n                       is_candidate(cand + r * ld_cand, topk, (c - s) / block_size);",
     "int keep = c < e &&\n                       is_candidate(cand + r * ld_cand, topk, (c - s) / block_size);"),
    ("mask treats -1 as block 0", "if (cand[j] >= 0 && (int64_t)cand[j] == b)",
     "if ((int64_t)(cand[j] < 0 ? 0 : cand[j]) == b)"),
]


def _battery() -> list:
    """Run the pins against the currently bound oracle; return what failed."""
    failed = []
    for p in golden._cases():
        case = p.values[0]
        try:
            golden.test_golden_case(case)
        except AssertionError:
            failed.append("golden:" + p.id)
    for seed in range(25):
        try:
            pins.test_unsharded_matches_brute_force(seed)
        except AssertionError:
            failed.append(f"brute-unsharded:{seed}")
        try:
            pins.test_sharded_matches_brute_force(seed)
        except AssertionError:
            failed.append(f"brute-sharded:{seed}")
    try:
        pins.test_sharded_equals_unsharded_on_global_rows(4, 1, 9, 64, 2)
    except AssertionError:
        failed.append("interleave-identity")
    import test_oracle_mask as mask_pins
    for name, fn in (("mask-golden", mask_pins.test_golden_mask),
                     ("mask-after-select", mask_pins.test_mask_after_select_keeps_exactly_the_selected_blocks)):
        try:
            fn()
        except AssertionError:
            failed.append(name)
    for seed in range(15):
        try:
            mask_pins.test_mask_matches_brute_force(seed)
        except AssertionError:
            failed.append(f"mask-brute:{seed}")
    import test_oracle_starts as starts
    checks = [(f"starts-golden:{p.id}", lambda c=p.values[0]: starts.test_golden_starts_case(c))
              for p in starts._cases()]
    checks += [(f"starts-brute:{s}", lambda s=s: starts.test_sharded_starts_matches_brute_force(s))
               for s in range(40)]
    checks += [("starts-identity", lambda: starts.test_sharded_starts_equals_unsharded_on_global_rows(
        2, 4, 7, 40, 1))]
    for name, fn in checks:
        try:
            fn()
        except AssertionError:
            failed.append(name)
    return failed


def test_unplanted_oracle_passes_battery():
    assert _battery() == []


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_mistake_is_caught(name, old, new, tmp_path):
    with open(oracle._SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
    so = oracle.build_variant(str(tmp_path), {"dsa_oracle.c": src.replace(old, new)})
    saved = oracle._lib
    oracle._lib = oracle.bind(so)
    try:
        failed = _battery()
    finally:
        oracle._lib = saved
    assert failed, f"planted mistake '{name}' passed every pin"
