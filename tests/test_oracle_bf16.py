"""Pins the oracle's bf16 entry points (``oracle/dsa_oracle_bf16.c``).

* hand-computed cases on explicit bf16 bit patterns
  (``tests/golden/bf16_logits.json``): NaN payloads and signs, signed zeros,
  infinities, request-local blocks, the pin, the DCP merge and masking;
* the pure-Python brute force of ``test_oracle_pins`` / ``test_oracle_mask``
  on the decoded values, with the scores' bf16 bits compared;
* planted mistakes in a copy of ``dsa_oracle_bf16.c`` must fail one of them.
"""

import numpy as np
import pytest

import oracle
import test_oracle_mask as mask_pins
import test_oracle_pins as pins
from helpers import deal_shards, load_golden

FIXTURE = "bf16_logits.json"


def _hex(rows) -> np.ndarray:
    return np.array([[int(t, 16) for t in r] for r in rows], dtype=np.uint16).reshape(
        len(rows), -1 if rows and rows[0] else 0)


def _decode(u16: np.ndarray) -> np.ndarray:
    return (u16.astype(np.uint32) << 16).view(np.float32)


def _bf16_bits_of(f32: np.ndarray) -> np.ndarray:
    """Upper halves of fp32 values that lie on the bf16 grid (scores of the
    brute force: block maxima of bf16 values, +-inf, canonical NaN)."""
    b = np.ascontiguousarray(f32, dtype=np.float32).view(np.uint32)
    assert not (b & 0xFFFF).any()
    return (b >> 16).astype(np.uint16)


def _cases():
    fx = load_golden(FIXTURE)
    assert fx.get("cite") and fx.get("why")
    return [pytest.param(c, id=f"{c['op']}-{i}") for i, c in enumerate(fx["cases"])]


@pytest.mark.parametrize("case", _cases())
def test_golden_bf16_case(case):
    op = case["op"]
    if op == "select_bf16":
        x = _hex(case["logits"])
        ks = None if case["row_ks"] is None else np.array(case["row_ks"], np.int32)
        ke = np.array(case["row_ke"], np.int32)
        ids, scores = oracle.select_bf16(x, ks, ke, case["topk_blocks"], case["block_size"],
                                         case["row_repeat"], case["pin_newest"],
                                         width=case["width"])
        np.testing.assert_array_equal(ids, np.array(case["expect_ids"], np.int32))
        np.testing.assert_array_equal(scores, _hex(case["expect_scores"]))
        s2 = oracle.block_scores_bf16(x, ks, ke, case["block_size"], case["row_repeat"],
                                      case["pin_newest"], width=case["width"])
        np.testing.assert_array_equal(s2, _hex(case["expect_scores"]))
    elif op == "sharded_bf16":
        local = deal_shards(_hex(case["global_logits"]), case["shards"])
        ids, scores = oracle.select_sharded_bf16(local, np.array(case["global_row_ke"], np.int32),
                                                 case["global_block_size"],
                                                 case["max_global_blocks"], case["topk_blocks"],
                                                 case["row_repeat"])
        np.testing.assert_array_equal(ids, np.array(case["expect_ids"], np.int32))
        np.testing.assert_array_equal(scores, _hex(case["expect_scores"]))
    else:
        x = _hex(case["logits"])
        got = oracle.mask_bf16(x, np.array(case["row_ks"], np.int32),
                               np.array(case["row_ke"], np.int32),
                               np.array(case["candidates"], np.int32), case["block_size"],
                               case["row_repeat"], width=case["width"])
        np.testing.assert_array_equal(got, _hex(case["expect"]))


def _tiny_bf16(rng, rows, width):
    """The brute-force pool (ties, signed zeros, infinities) with NaNs whose
    payload and sign live in the upper 16 bits, as bf16 bit patterns."""
    x = pins._tiny_logits(rng, rows, width)
    bits = x.view(np.uint32).copy()
    nan = np.isnan(x)
    payload = rng.integers(1, 64, size=int(nan.sum())).astype(np.uint32) << np.uint32(16)
    bits[nan] = (bits[nan] & np.uint32(0x80000000)) | np.uint32(0x7FC00000) | payload
    return (bits >> 16).astype(np.uint16)


@pytest.mark.parametrize("seed", range(30))
def test_select_bf16_matches_brute_force(seed):
    rng = np.random.default_rng(3100 + seed)
    rows, width = int(rng.integers(1, 6)), int(rng.integers(0, 33))
    bs = int(rng.choice([1, 2, 3, 4, 8]))
    rr, pin, topk = int(rng.integers(1, 3)), bool(rng.integers(0, 2)), int(rng.integers(0, 9))
    groups = -(-rows // rr)
    x = _tiny_bf16(rng, rows, width)
    ke = rng.integers(-2, width + 4, size=groups).astype(np.int32)
    ks = rng.integers(-2, width + 2, size=groups).astype(np.int32) if rng.integers(0, 2) else None
    ids, scores = oracle.select_bf16(x, ks, ke, topk, bs, rr, pin, width=width)
    want_ids, want_scores = pins.brute_unsharded(_decode(x), ks, ke, width, bs, rr, pin, topk)
    np.testing.assert_array_equal(ids, want_ids)
    if width:
        np.testing.assert_array_equal(scores, _bf16_bits_of(want_scores))


@pytest.mark.parametrize("seed", range(20))
def test_sharded_bf16_matches_brute_force(seed):
    rng = np.random.default_rng(3300 + seed)
    shards, lbs = int(rng.choice([1, 2, 3, 8])), int(rng.choice([1, 2, 3]))
    lw, rows, rr = int(rng.integers(0, 8)), int(rng.integers(1, 5)), int(rng.integers(1, 3))
    max_gb, topk = int(rng.integers(0, 6)), int(rng.integers(0, 7))
    local = _tiny_bf16(rng, shards * rows, lw).reshape(shards, rows, lw)
    gke = rng.integers(-2, shards * lw + 5, size=-(-rows // rr)).astype(np.int32)
    ids, scores = oracle.select_sharded_bf16(local, gke, lbs * shards, max_gb, topk, rr)
    want_ids, want_scores = pins.brute_sharded(_decode(local), gke, lbs * shards, max_gb, rr,
                                               topk)
    np.testing.assert_array_equal(ids, want_ids)
    np.testing.assert_array_equal(scores, _bf16_bits_of(want_scores))


@pytest.mark.parametrize("seed", range(15))
def test_mask_bf16_matches_brute_force(seed):
    rng = np.random.default_rng(3500 + seed)
    rows, width = int(rng.integers(1, 5)), int(rng.integers(0, 40))
    bs, rr, topk = int(rng.choice([1, 2, 3, 5])), int(rng.integers(1, 3)), int(rng.integers(0, 5))
    groups = -(-rows // rr)
    x = _tiny_bf16(rng, rows, width)
    ke = rng.integers(-2, width + 3, size=groups).astype(np.int32)
    ks = rng.integers(-2, width + 2, size=groups).astype(np.int32) if rng.integers(0, 2) else None
    cand = rng.integers(-1, max(-(-width // bs), 1) + 1, size=(rows, topk)).astype(np.int32)
    got = oracle.mask_bf16(x, ks, ke, cand, bs, rr, width=width)
    want = mask_pins.brute_mask(_decode(x), ks, ke, cand, bs, rr, width)
    np.testing.assert_array_equal(got, (want.view(np.uint32) >> 16).astype(np.uint16))


def test_mask_sharded_bf16_keeps_selected_global_blocks():
    rng = np.random.default_rng(3700)
    shards, lbs, rows, lw = 4, 2, 3, 6
    g = _tiny_bf16(rng, rows, shards * lw)
    gke = np.array([24, 9, 0], np.int32)
    cand = np.array([[0, 2], [1, -1], [0, 1]], np.int32)
    got = oracle.mask_sharded_bf16(deal_shards(g, shards), gke, lbs * shards, cand)
    want = mask_pins.brute_mask(_decode(g), None, gke, cand, lbs * shards, 1, shards * lw)
    np.testing.assert_array_equal(got, deal_shards((want.view(np.uint32) >> 16).astype(np.uint16),
                                                   shards))


# --------------------------------------------------------------------------
# Planted mistakes
# --------------------------------------------------------------------------

MUTATIONS = [
    ("widening shifts by 15", "uint32_t bits = (uint32_t)h << 16;",
     "uint32_t bits = (uint32_t)h << 15;"),
    ("narrowing keeps the wrong half", "return (uint16_t)(bits >> 16);",
     "return (uint16_t)(bits >> 15);"),
    ("last score not written",
     "    if (rc == 0 && scores)\n        narrow(s, rows, nb, scores, ld_scores);",
     "    if (rc == 0 && scores)\n        narrow(s, rows, nb - 1, scores, ld_scores);"),
    ("every shard reads shard 0",
     "float *part = widen(logits + d * shard_stride, rows, local_width, ld_logits);\n        if (!part) {\n            free(x);\n            free(s);",
     "float *part = widen(logits, rows, local_width, ld_logits);\n        if (!part) {\n            free(x);\n            free(s);"),
    ("masked values not written back",
     "    if (rc == 0)\n        narrow(x, rows, width, logits, ld_logits);", ""),
]


def _battery():
    failed = []
    checks = [(f"golden:{p.id}", lambda c=p.values[0]: test_golden_bf16_case(c))
              for p in _cases()]
    checks += [(f"brute:{s}", lambda s=s: test_select_bf16_matches_brute_force(s))
               for s in range(30)]
    checks += [(f"brute-sharded:{s}", lambda s=s: test_sharded_bf16_matches_brute_force(s))
               for s in range(20)]
    checks += [(f"mask:{s}", lambda s=s: test_mask_bf16_matches_brute_force(s))
               for s in range(15)]
    checks += [("mask-sharded", test_mask_sharded_bf16_keeps_selected_global_blocks)]
    for name, fn in checks:
        try:
            fn()
        except AssertionError:
            failed.append(name)
    return failed


def test_unplanted_bf16_oracle_passes_battery():
    assert _battery() == []


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_bf16_mistake_is_caught(name, old, new, tmp_path):
    with open(oracle._BF16_SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
    so = oracle.build_variant(str(tmp_path), {"dsa_oracle_bf16.c": src.replace(old, new)})
    saved = oracle._lib
    oracle._lib = oracle.bind(so)
    try:
        failed = _battery()
    finally:
        oracle._lib = saved
    assert failed, f"planted mistake '{name}' passed every pin"
