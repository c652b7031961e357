"""Pins the CPU oracle to hand-computed cases (``tests/golden/*.json``).

Each fixture names the passage it follows and how its expected values were
worked out by hand; none of them came from either implementation.
"""

import numpy as np
import pytest

import oracle
from helpers import assert_bits_equal, deal_shards, golden_files, load_golden, parse_matrix


def _cases():
    for name in golden_files():
        fx = load_golden(name)
        assert fx.get("cite") and fx.get("why"), name
        for i, case in enumerate(fx["cases"]):
            if case["op"] in ("select", "block_scores", "sharded"):  # masking: test_oracle_mask
                yield pytest.param(case, id=f"{name[:-5]}-{i}")


def run_oracle_case(case):
    op = case["op"]
    if op == "sharded":
        g = parse_matrix(case["global_logits"])
        local = deal_shards(g, case["shards"])
        gke = np.array(case["global_row_ke"], dtype=np.int32)
        return oracle.select_sharded(local, gke, case["global_block_size"],
                                     case["max_global_blocks"], case["topk_blocks"],
                                     case["row_repeat"])
    logits = parse_matrix(case["logits"])
    ks = None if case["row_ks"] is None else np.array(case["row_ks"], dtype=np.int32)
    ke = np.array(case["row_ke"], dtype=np.int32)
    if op == "block_scores":
        s = oracle.block_scores(logits, ks, ke, case["block_size"], case["row_repeat"],
                                case["pin_newest"], width=case["width"])
        return None, s
    return oracle.select(logits, ks, ke, case["topk_blocks"], case["block_size"],
                         case["row_repeat"], case["pin_newest"], width=case["width"])


@pytest.mark.parametrize("case", list(_cases()))
def test_golden_case(case):
    ids, scores = run_oracle_case(case)
    want_scores = parse_matrix(case["expect_scores"])
    assert_bits_equal(scores, want_scores)
    if case["expect_ids"] is not None:
        np.testing.assert_array_equal(ids, np.array(case["expect_ids"], dtype=np.int32))
