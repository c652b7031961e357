"""Pins the CPU oracle of the DCP partial-attention LSE correction.

What fixes it, apart from its own formula:
- hand-computed cases (``tests/golden/dcp_lse_correction.json``, powers of
  two so that the expected values are exact);
- a closed form: when each shard's partial output and LSE come from a
  softmax over its own keys, the merged output is the softmax attention over
  all keys at once, and the combined LSE is the log-sum-exp of all scores
  (computed here in one pass with numpy, never through the oracle);
- ``numpy.logaddexp2.reduce`` for the combined LSE of arbitrary values;
- invariants: the shares of the shards add up to one; equal LSEs on a
  power-of-two count of shards give a share of exactly 1/N; the output is
  head-major.
Planted mistakes in a temporary copy of ``oracle/dcp_lse_oracle.c`` must
fail at least one of these.
"""

import math

import numpy as np
import pytest

import oracle
import workloads
from helpers import load_golden

FIXTURE = "dcp_lse_correction.json"


def _arr(nested) -> np.ndarray:
    return np.array(nested, dtype=object).astype(str).astype(np.float64)


def _golden_cases():
    fx = load_golden(FIXTURE)
    assert fx.get("cite") and fx.get("why")
    return [pytest.param(c, id=f"{c['op']}-{i}") for i, c in enumerate(fx["cases"])]


def _close(got, want, rel=1e-12):
    got, want = np.asarray(got, np.float64), np.asarray(want, np.float64)
    assert got.shape == want.shape, (got.shape, want.shape)
    same_special = (np.isnan(got) == np.isnan(want)).all() and (
        np.isinf(got) == np.isinf(want)).all()
    assert same_special, (got, want)
    fin = np.isfinite(want)
    assert (got[~fin & ~np.isnan(want)] == want[~fin & ~np.isnan(want)]).all(), (got, want)
    err = np.abs(got[fin] - want[fin])
    assert (err <= rel * np.maximum(1.0, np.abs(want[fin]))).all(), (got, want)


@pytest.mark.parametrize("case", _golden_cases())
def test_golden_lse_case(case):
    lses = _arr(case["lses"]).astype(np.float32)
    if case["op"] == "correct":
        out = _arr(case["out"]).astype(np.float32)
        got_out, got_lse = oracle.correct_attn_out(out, lses, case["rank"])
    else:
        outs = _arr(case["outs"]).astype(np.float32)
        got_out, got_lse = oracle.merge_attn_out(outs, lses)
    _close(got_lse, _arr(case["expect_lse"]))
    _close(got_out, _arr(case["expect_out"]))


def _split_attention(seed: int, shards: int, batch: int, heads: int, head_dim: int):
    """A softmax attention problem split over shards by keys: per (b, h)
    random base-2 scores and values, dealt to shards at random (a shard may
    get no key). Returns the partials (fp32, as the method receives them)
    and the one-pass result over all keys (float64)."""
    rng = np.random.default_rng(seed)
    outs = np.zeros((shards, batch, heads, head_dim))
    lses = np.full((shards, batch, heads), -np.inf)
    full = np.zeros((batch, heads, head_dim))
    full_lse = np.zeros((batch, heads))
    for b in range(batch):
        for h in range(heads):
            nk = int(rng.integers(1, 40))
            t = rng.normal(0.0, 3.0, size=nk) + rng.uniform(-30, 30)
            v = rng.normal(size=(nk, head_dim))
            owner = rng.integers(0, shards, size=nk)
            # one pass over all keys
            w = np.exp2(t - t.max())
            full[b, h] = (w[:, None] * v).sum(0) / w.sum()
            full_lse[b, h] = math.log2(w.sum()) + t.max()
            for n in range(shards):
                sel = owner == n
                if sel.any():
                    tn, vn = t[sel], v[sel]
                    wn = np.exp2(tn - tn.max())
                    outs[n, b, h] = (wn[:, None] * vn).sum(0) / wn.sum()
                    lses[n, b, h] = math.log2(wn.sum()) + tn.max()
    return outs.astype(np.float32), lses.astype(np.float32), full, full_lse


@pytest.mark.parametrize("seed", range(6))
def test_merge_equals_one_pass_attention(seed):
    shards = [1, 2, 3, 4, 8, 5][seed]
    outs, lses, full, full_lse = _split_attention(seed, shards, 3, 4, 8)
    merged, lse = oracle.merge_attn_out(outs, lses)
    # inputs were rounded to fp32: LSEs to 2^-24 relative (|lse| < 64 here),
    # outputs likewise; the shares then move by at most ~1e-5 relative.
    np.testing.assert_allclose(lse, full_lse, rtol=0, atol=2e-5)
    np.testing.assert_allclose(merged, full.transpose(1, 0, 2), rtol=0, atol=5e-5)
    # the per-shard corrections add up to the merge
    acc = sum(oracle.correct_attn_out(outs[n], lses, n)[0] for n in range(shards))
    np.testing.assert_allclose(acc, merged, rtol=1e-12, atol=1e-12)


@pytest.mark.parametrize("seed", range(4))
def test_combined_lse_matches_logaddexp2(seed):
    rng = np.random.default_rng(100 + seed)
    N, B, H = 5, 7, 6
    lses = rng.normal(0, 40, size=(N, B, H)).astype(np.float32)
    specials = rng.integers(0, 8, size=(N, B, H))
    lses[specials == 0] = -np.inf
    lses[specials == 1] = np.inf
    lses[specials == 2] = np.nan
    lses[:, 0, 0] = -np.inf          # a row with no finite value at all
    lses[:, 0, 1] = [np.nan, np.inf, -np.inf, np.nan, np.inf]
    clean = np.where(np.isnan(lses) | (lses == np.inf), -np.inf, lses).astype(np.float64)
    want = np.logaddexp2.reduce(clean, axis=0)
    _, got = oracle.correct_attn_out(np.zeros((B, H, 1), np.float32), lses, 0)
    _close(got, want, rel=1e-13)


@pytest.mark.parametrize("seed", range(3))
def test_shares_add_up_to_one(seed):
    wl = workloads.make_lse(seed, shards=4, batch=9, heads=5, head_dim=1, specials=True)
    N, B, H = wl.lses.shape
    ones = np.ones((B, H, 1), np.float32)
    total = sum(oracle.correct_attn_out(ones, wl.lses, n)[0][:, :, 0] for n in range(N))
    clean = np.where(np.isnan(wl.lses) | (wl.lses == np.inf), -np.inf, wl.lses)
    any_finite = np.isfinite(clean).any(axis=0).T          # [H, B]
    np.testing.assert_allclose(total[any_finite], 1.0, rtol=0, atol=1e-12)
    assert (total[~any_finite] == 0).all()
    # and each local NaN or +inf gets share 0
    for n in range(N):
        share = oracle.correct_attn_out(ones, wl.lses, n)[0][:, :, 0]
        bad = (np.isnan(wl.lses[n]) | (wl.lses[n] == np.inf)).T
        assert (share[bad] == 0).all()


def test_equal_lses_give_one_over_n_head_major():
    rng = np.random.default_rng(9)
    B, H, D = 3, 5, 4
    out = rng.normal(size=(B, H, D)).astype(np.float32)
    for N in (1, 2, 4, 8):
        lses = np.full((N, B, H), 7.25, np.float32)
        for rank in range(N):
            new, lse = oracle.correct_attn_out(out, lses, rank)
            assert new.shape == (H, B, D)
            np.testing.assert_array_equal(new, out.transpose(1, 0, 2).astype(np.float64) / N)
            np.testing.assert_array_equal(lse, np.full((B, H), 7.25 + math.log2(N)))


# --------------------------------------------------------------------------
# Planted mistakes
# --------------------------------------------------------------------------

MUTATIONS = [
    ("natural exponent", "acc += exp2(sanitize", "acc += exp(sanitize"),
    ("max not subtracted", "- m);\n    return log2(acc) + m;", ");\n    return log2(acc);"),
    ("+inf kept", "if (isnan(x) || x == INFINITY)", "if (isnan(x))"),
    ("NaN kept", "if (isnan(x) || x == INFINITY)", "if (x == INFINITY)"),
    ("empty rows keep a -inf max", "if (m == -INFINITY)\n        m = 0.0;", ""),
    ("NaN difference kept", "if (isnan(d) || d == INFINITY)", "if (d == INFINITY)"),
    ("+inf difference kept", "if (isnan(d) || d == INFINITY)", "if (isnan(d))"),
    ("output not transposed", "double *dst = new_out + (h * batch + b) * head_dim;",
     "double *dst = new_out + (b * heads + h) * head_dim;"),
    ("local LSE of the wrong shard", "share((double)col[rank * step], F)",
     "share((double)col[0], F)"),
    ("LSE stride of one token", "int64_t step = batch * heads;\n            double F = combined_lse(col, step, shards);\n            double f",
     "int64_t step = heads;\n            double F = combined_lse(col, step, shards);\n            double f"),
    ("merge overwrites", "dst[c] += f * (double)src[c];", "dst[c] = f * (double)src[c];"),
    ("merge uses shard 0's LSE", "share((double)col[n * step], F)", "share((double)col[0], F)"),
    ("merge reads shard 0's output",
     "const float *src = outs + ((n * batch + b) * heads + h) * head_dim;",
     "const float *src = outs + (b * heads + h) * head_dim;"),
]


def _battery() -> list:
    failed = []
    checks = [(f"golden:{p.id}", lambda c=p.values[0]: test_golden_lse_case(c))
              for p in _golden_cases()]
    checks += [(f"one-pass:{s}", lambda s=s: test_merge_equals_one_pass_attention(s))
               for s in range(6)]
    checks += [(f"logaddexp2:{s}", lambda s=s: test_combined_lse_matches_logaddexp2(s))
               for s in range(4)]
    checks += [(f"shares:{s}", lambda s=s: test_shares_add_up_to_one(s)) for s in range(3)]
    checks += [("one-over-n", test_equal_lses_give_one_over_n_head_major)]
    for name, fn in checks:
        try:
            fn()
        except AssertionError:
            failed.append(name)
    return failed


def test_unplanted_lse_oracle_passes_battery():
    assert _battery() == []


@pytest.mark.parametrize("name,old,new", MUTATIONS, ids=[m[0] for m in MUTATIONS])
def test_planted_lse_mistake_is_caught(name, old, new, tmp_path):
    with open(oracle._LSE_SRC) as f:
        src = f.read()
    assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
    so = oracle.build_variant(str(tmp_path), {"dcp_lse_oracle.c": src.replace(old, new)})
    saved = oracle._lib
    oracle._lib = oracle.bind(so)
    try:
        failed = _battery()
    finally:
        oracle._lib = saved
    assert failed, f"planted mistake '{name}' passed every pin"
