"""GPU parity for bf16 logits: the ``*_bf16`` entry points against the
oracle's bf16 entry points, ids exactly and score / logit bits exactly.

Inputs are drawn as fp32 and put on the bf16 grid (finite values rounded to
nearest even, NaNs truncated so that their payload and sign survive), then
moved to the device bit for bit as uint16 patterns viewed as bfloat16 (a
float -> bfloat16 conversion would canonicalise NaN payloads). Every case
runs with a workspace (rows split over CTAs) and without one. Outputs land
in views of larger buffers whose guard columns must come back untouched.
"""

import numpy as np
import pytest

import oracle
import workloads
from helpers import deal_shards

pytestmark = pytest.mark.gpu

GUARD = 3
SENTINEL_ID = -7
SENTINEL_BITS = 0x1234  # a bf16 pattern no score takes here


@pytest.fixture(scope="module")
def env():
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import deepseek_sparse_attention_row_gb300 as dsa

    assert torch.cuda.is_available(), "GPU parity tests need a CUDA device"
    return torch, dsa


def to_bf16_bits(x: np.ndarray) -> np.ndarray:
    """uint16 bf16 patterns of fp32 values: finite values rounded to nearest
    even, infinities kept, NaNs truncated (payload and sign kept)."""
    x = np.ascontiguousarray(x, dtype=np.float32)
    nan = np.isnan(x)
    fin = np.where(nan, np.float32(0), x)
    r = workloads.round_to_bf16_grid(fin).view(np.uint32)
    r = np.where(nan, x.view(np.uint32) & np.uint32(0xFFFF0000), r)
    return (r >> 16).astype(np.uint16)


def widen(bits: np.ndarray) -> np.ndarray:
    return (bits.astype(np.uint32) << 16).view(np.float32)


def dev_bf16(torch, bits: np.ndarray, offset: int = 0, fill: int = 0x7F7F):
    """Device bfloat16 copy of uint16 patterns, `offset` elements into a
    larger buffer filled with `fill` (a large finite bf16)."""
    flat = np.ascontiguousarray(bits).reshape(-1)
    buf = torch.full((flat.size + offset + 16,), fill, dtype=torch.int16, device="cuda")
    buf[offset:offset + flat.size].copy_(torch.from_numpy(flat.view(np.int16)))
    return buf[offset:offset + flat.size].view(torch.bfloat16).view(bits.shape)


def host_bits(t) -> np.ndarray:
    return t.contiguous().view(__import__("torch").int16).cpu().numpy().view(np.uint16)


def _dev(torch, a):
    return None if a is None else torch.from_numpy(np.ascontiguousarray(a)).cuda()


def check_unsharded(env, bits, ks, ke, width, bs, topk, rr, pin, offset=0):
    torch, dsa = env
    rows = bits.shape[0]
    nb = -(-width // bs)
    want_ids, want_sc = oracle.select_bf16(bits, ks, ke, topk, bs, rr, pin, width=width)
    logits = dev_bf16(torch, bits, offset)[:, :width]
    for ws in (None, False):
        out = torch.full((rows, topk + GUARD), SENTINEL_ID, dtype=torch.int32, device="cuda")
        sc = torch.full((rows, nb + GUARD), SENTINEL_BITS, dtype=torch.int16,
                        device="cuda").view(torch.bfloat16)
        dsa.dsa_select_candidate_blocks(logits, _dev(torch, ks), _dev(torch, ke), topk, bs,
                                        out[:, :topk], rr, pin, scores_out=sc[:, :nb],
                                        workspace=ws)
        torch.cuda.synchronize()
        o, s = out.cpu().numpy(), host_bits(sc)
        assert (o[:, topk:] == SENTINEL_ID).all() and (s[:, nb:] == SENTINEL_BITS).all()
        np.testing.assert_array_equal(o[:, :topk], want_ids)
        if want_sc is not None:
            np.testing.assert_array_equal(s[:, :nb], want_sc)


BLOCK_SIZES = [1, 2, 3, 4, 8, 12, 16, 32, 64, 100, 128, 256]


@pytest.mark.parametrize("seed", range(32))
def test_bf16_unsharded_sweep(env, seed):
    rng = np.random.default_rng(20000 + seed)
    bs = int(BLOCK_SIZES[seed % len(BLOCK_SIZES)])
    width = int(min(rng.choice([1, 9, 64, 333, 4096, 5003, 30001, 70000]), bs * 4000))
    rows, rr = int(rng.integers(1, 30)), int(rng.choice([1, 2, 3, 8]))
    nb = -(-width // bs)
    topk = int(rng.choice([1, 5, 16, 32, 33, 100, nb, nb + 5]))
    pad = int(rng.choice([0, 0, 1, 3, 8]))
    wl = workloads.small_unsharded(20000 + seed, rows=rows, width=width, block_size=bs,
                                   topk_blocks=topk, row_repeat=rr,
                                   starts=bool(rng.integers(0, 2)),
                                   nan_count=int(rng.choice([0, 3, 40])),
                                   wild_bounds=bool(rng.integers(0, 2)), ld=width + pad)
    bits = to_bf16_bits(wl.logits)
    check_unsharded(env, bits, wl.row_ks, wl.row_ke, width, bs, topk, rr,
                    bool(rng.integers(0, 2)), offset=int(rng.choice([0, 0, 1, 3, 5])))


@pytest.mark.parametrize("seed", range(20))
def test_bf16_sharded_sweep(env, seed):
    torch, dsa = env
    rng = np.random.default_rng(21000 + seed)
    shards = int(rng.choice([1, 2, 3, 8, 8, 16]))
    lbs = int(rng.choice([1, 2, 3, 4, 8, 8, 16, 32]))
    lw = int(rng.choice([1, 5, 64, 100, 1024, 2047, 8192]))
    nlb = -(-lw // lbs)
    max_gb = int(min(rng.choice([0, 1, max(nlb // 2, 1), nlb, nlb + 7]), 16384))
    rows, rr = int(rng.integers(1, 30)), int(rng.choice([1, 2, 5]))
    nbg = max(max_gb, 1)
    topk = int(rng.choice([1, 8, 32, 40, nbg, nbg + 3]))
    wl, _ = workloads.small_sharded(21000 + seed, shards=shards, rows=rows,
                                    global_width=lw * shards, global_block_size=lbs * shards,
                                    max_global_blocks=max_gb, topk_blocks=topk, row_repeat=rr,
                                    wild_bounds=bool(rng.integers(0, 2)))
    bits = to_bf16_bits(wl.logits)
    nan_pos = rng.random(bits.shape) < 0.001
    bits[nan_pos] = 0x7FC3
    want_ids, want_sc = oracle.select_sharded_bf16(bits, wl.global_row_ke, lbs * shards, max_gb,
                                                   topk, rr)
    local = dev_bf16(torch, bits, int(rng.choice([0, 0, 1, 4])))
    for ws in (None, False):
        out = torch.full((rows, topk + GUARD), SENTINEL_ID, dtype=torch.int32, device="cuda")
        sc = torch.full((rows, nbg + GUARD), SENTINEL_BITS, dtype=torch.int16,
                        device="cuda").view(torch.bfloat16)
        dsa.dsa_select_candidate_blocks_sharded(local, _dev(torch, wl.global_row_ke),
                                                lbs * shards, max_gb, topk, out[:, :topk], rr,
                                                scores_out=sc[:, :nbg], workspace=ws)
        torch.cuda.synchronize()
        o, s = out.cpu().numpy(), host_bits(sc)
        assert (o[:, topk:] == SENTINEL_ID).all() and (s[:, nbg:] == SENTINEL_BITS).all()
        np.testing.assert_array_equal(o[:, :topk], want_ids)
        np.testing.assert_array_equal(s[:, :nbg], want_sc)


@pytest.mark.parametrize("seed", range(10))
def test_bf16_sharded_starts_sweep(env, seed):
    """bf16 DCP form with global starts against the fp32 oracle on the
    widened values (ids equal; bf16 scores are the fp32 scores' upper
    halves)."""
    torch, dsa = env
    rng = np.random.default_rng(28000 + seed)
    shards, lbs = int(rng.choice([2, 3, 8])), int(rng.choice([1, 2, 8, 16]))
    lw, rows = int(rng.choice([5, 100, 2047, 8192])), int(rng.integers(1, 30))
    nlb = -(-lw // lbs)
    max_gb, topk = nlb, int(rng.choice([1, 8, 32]))
    wl, _ = workloads.small_sharded(28000 + seed, shards=shards, rows=rows,
                                    global_width=lw * shards, global_block_size=lbs * shards,
                                    max_global_blocks=max_gb, topk_blocks=topk)
    bits = to_bf16_bits(wl.logits)
    gks = rng.integers(-3, shards * lw + 3, size=rows).astype(np.int32)
    gks[::2] = np.minimum(gks[::2], wl.global_row_ke[::2] - 1)
    want_ids, want_sc = oracle.select_sharded_starts(widen(bits), gks, wl.global_row_ke,
                                                     lbs * shards, max_gb, topk)
    local = dev_bf16(torch, bits, int(rng.choice([0, 1, 5])))
    for ws in (None, False):
        out = torch.full((rows, topk), SENTINEL_ID, dtype=torch.int32, device="cuda")
        sc = torch.empty((rows, max_gb), dtype=torch.bfloat16, device="cuda")
        dsa.dsa_select_candidate_blocks_sharded(local, _dev(torch, wl.global_row_ke),
                                                lbs * shards, max_gb, topk, out, scores_out=sc,
                                                workspace=ws, global_row_ks=_dev(torch, gks))
        torch.cuda.synchronize()
        np.testing.assert_array_equal(out.cpu().numpy(), want_ids)
        np.testing.assert_array_equal(host_bits(sc),
                                      (want_sc.view(np.uint32) >> 16).astype(np.uint16))
    cand = rng.integers(-1, nlb + 1, size=(rows, 4)).astype(np.int32)
    want_mask = oracle.mask_sharded_starts(widen(bits), gks, wl.global_row_ke, lbs * shards,
                                           cand)
    dsa.dsa_mask_candidate_logits_sharded(local, _dev(torch, wl.global_row_ke), lbs * shards,
                                          _dev(torch, cand), global_row_ks=_dev(torch, gks))
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host_bits(local),
                                  (want_mask.view(np.uint32) >> 16).astype(np.uint16))


@pytest.mark.parametrize("seed", range(8))
def test_bf16_block_scores_sweep(env, seed):
    torch, dsa = env
    rng = np.random.default_rng(22000 + seed)
    bs = int(rng.choice(BLOCK_SIZES))
    width = int(rng.choice([1, 100, 4096, 20000, 131072]))
    rows = int(rng.integers(1, 20))
    wl = workloads.small_unsharded(22000 + seed, rows=rows, width=width, block_size=bs,
                                   topk_blocks=1, row_repeat=int(rng.choice([1, 4])),
                                   nan_count=4, wild_bounds=bool(rng.integers(0, 2)))
    bits = to_bf16_bits(wl.logits)
    pin = bool(rng.integers(0, 2))
    want = oracle.block_scores_bf16(bits, wl.row_ks, wl.row_ke, bs, wl.row_repeat, pin)
    nb = want.shape[1]
    sc = torch.full((rows, nb + GUARD), SENTINEL_BITS, dtype=torch.int16,
                    device="cuda").view(torch.bfloat16)
    dsa.dsa_block_scores(dev_bf16(torch, bits), _dev(torch, wl.row_ks), _dev(torch, wl.row_ke),
                         bs, wl.row_repeat, pin, scores_out=sc[:, :nb])
    torch.cuda.synchronize()
    s = host_bits(sc)
    assert (s[:, nb:] == SENTINEL_BITS).all()
    np.testing.assert_array_equal(s[:, :nb], want)


@pytest.mark.parametrize("bs,width,topk", [(64, 32768, 32), (8, 16384, 32), (3, 4000, 20)])
def test_bf16_warp_per_row(env, bs, width, topk):
    """Many short rows (up to 64 KiB of bf16) take the one-row-per-warp kernel."""
    wl = workloads.small_unsharded(23000 + bs, rows=1400, width=width, block_size=bs,
                                   topk_blocks=topk, starts=True, nan_count=30)
    check_unsharded(env, to_bf16_bits(wl.logits), wl.row_ks, wl.row_ke, width, bs, topk, 1,
                    True, offset=1)


def test_bf16_ids_equal_fp32_ids_on_widened_logits(env):
    """Selection ranks exact values: the bf16 call and the fp32 call on the
    widened logits give the same ids (both on the GPU)."""
    torch, dsa = env
    wl = workloads.small_unsharded(24000, rows=300, width=50000, block_size=64, topk_blocks=32,
                                   starts=True, nan_count=20)
    bits = to_bf16_bits(wl.logits)
    ks, ke = _dev(torch, wl.row_ks), _dev(torch, wl.row_ke)
    o16 = torch.empty((300, 32), dtype=torch.int32, device="cuda")
    o32 = torch.empty((300, 32), dtype=torch.int32, device="cuda")
    dsa.dsa_select_candidate_blocks(dev_bf16(torch, bits), ks, ke, 32, 64, o16)
    dsa.dsa_select_candidate_blocks(_dev(torch, widen(bits)), ks, ke, 32, 64, o32)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(o16.cpu().numpy(), o32.cpu().numpy())


@pytest.mark.parametrize("seed", range(14))
def test_bf16_mask_sweep(env, seed):
    torch, dsa = env
    rng = np.random.default_rng(25000 + seed)
    bs = int(rng.choice([1, 3, 8, 64, 100, 4096]))
    width = int(rng.choice([1, 9, 100, 8192, 16383, 16384, 16385, 40001]))
    rows, rr, topk = int(rng.integers(1, 20)), int(rng.choice([1, 2])), int(rng.choice([0, 3, 32]))
    wl = workloads.small_unsharded(25000 + seed, rows=rows, width=width, block_size=bs,
                                   topk_blocks=max(topk, 1), row_repeat=rr,
                                   starts=bool(rng.integers(0, 2)), nan_count=5,
                                   wild_bounds=bool(rng.integers(0, 2)))
    bits = to_bf16_bits(wl.logits)
    nb = -(-width // bs)
    cand = rng.integers(-1, nb + 2, size=(rows, topk)).astype(np.int32)
    want = oracle.mask_bf16(bits, wl.row_ks, wl.row_ke, cand, bs, rr, width=width)
    logits = dev_bf16(torch, bits, int(rng.choice([0, 1, 3, 7])))
    dsa.dsa_mask_candidate_logits(logits, _dev(torch, wl.row_ks), _dev(torch, wl.row_ke),
                                  _dev(torch, cand) if topk else None, bs, rr)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host_bits(logits), want)


@pytest.mark.parametrize("seed", range(4))
def test_bf16_mask_sharded_sweep(env, seed):
    torch, dsa = env
    rng = np.random.default_rng(26000 + seed)
    shards, lbs = int(rng.choice([2, 3, 8])), int(rng.choice([1, 3, 8]))
    lw, rows = int(rng.choice([100, 2047, 9000])), int(rng.integers(1, 12))
    topk = int(rng.choice([0, 5, 32]))
    wl, _ = workloads.small_sharded(26000 + seed, shards=shards, rows=rows,
                                    global_width=lw * shards, global_block_size=lbs * shards,
                                    max_global_blocks=-(-lw // lbs), topk_blocks=max(topk, 1),
                                    wild_bounds=True)
    bits = to_bf16_bits(wl.logits)
    cand = rng.integers(-1, -(-lw // lbs) + 2, size=(rows, topk)).astype(np.int32)
    want = oracle.mask_sharded_bf16(bits, wl.global_row_ke, lbs * shards, cand)
    local = dev_bf16(torch, bits)
    dsa.dsa_mask_candidate_logits_sharded(local, _dev(torch, wl.global_row_ke), lbs * shards,
                                          _dev(torch, cand) if topk else None)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(host_bits(local), want)


@pytest.mark.slow
@pytest.mark.parametrize("name", ["decode_bf16", "dcp_bf16"])
def test_bf16_full_size(env, name):
    """The bench's bf16 workloads: select, then mask with the selected ids."""
    torch, dsa = env
    wl = workloads.make(name)
    bits = to_bf16_bits(wl.logits)
    if hasattr(wl, "global_row_ke"):
        want_ids, _ = oracle.select_sharded_bf16(bits, wl.global_row_ke, wl.global_block_size,
                                                 wl.max_global_blocks, wl.topk_blocks,
                                                 wl.row_repeat, want_scores=False)
        local = dev_bf16(torch, bits)
        gke = _dev(torch, wl.global_row_ke)
        out = torch.empty((wl.rows, wl.topk_blocks), dtype=torch.int32, device="cuda")
        dsa.dsa_select_candidate_blocks_sharded(local, gke, wl.global_block_size,
                                                wl.max_global_blocks, wl.topk_blocks, out)
        dsa.dsa_mask_candidate_logits_sharded(local, gke, wl.global_block_size, out)
        want_mask = oracle.mask_sharded_bf16(bits, wl.global_row_ke, wl.global_block_size,
                                             want_ids)
    else:
        want_ids, _ = oracle.select_bf16(bits, wl.row_ks, wl.row_ke, wl.topk_blocks,
                                         wl.block_size, wl.row_repeat, wl.pin_newest,
                                         want_scores=False)
        local = dev_bf16(torch, bits)
        ks, ke = _dev(torch, wl.row_ks), _dev(torch, wl.row_ke)
        out = torch.empty((wl.rows, wl.topk_blocks), dtype=torch.int32, device="cuda")
        dsa.dsa_select_candidate_blocks(local, ks, ke, wl.topk_blocks, wl.block_size, out,
                                        wl.row_repeat, wl.pin_newest)
        dsa.dsa_mask_candidate_logits(local, ks, ke, out, wl.block_size, wl.row_repeat)
        want_mask = oracle.mask_bf16(bits, wl.row_ks, wl.row_ke, want_ids, wl.block_size,
                                     wl.row_repeat)
    torch.cuda.synchronize()
    np.testing.assert_array_equal(out.cpu().numpy(), want_ids)
    np.testing.assert_array_equal(host_bits(local), want_mask)
