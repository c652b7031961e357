"""Seeded synthetic inputs for DSA candidate-block selection.

This module only draws inputs. It holds none of the selection arithmetic
(no windowing, block maxima, pins, shard ends or top-k): both the CPU oracle
and the CUDA path receive exactly the arrays built here.

Every workload follows the shapes, value distributions and structure of the
indexer-logit rows that candidate selection consumes on the page
"launcher/dcp2/diffs/02-model_executor_kernels_attention_dsa_candidate_blocks.py.diff"
(``select_candidate_blocks`` / ``_select_candidate_blocks_impl``): fp32 logits
in packed column space, int32 per-group ``row_ks`` / ``row_ke`` bounds shared by
``row_repeat`` rows, and for the DCP form an interleave-1 shard layout
(global token t lives on shard t % D at local column t // D, as in the
SGLang ``dcp/kernels.py`` page, ``create_triton_kv_indices_for_dcp_triton``).

The DCP partial-attention LSE correction (SGLang ``dcp/kernels.py`` page,
``correct_attn_out``) gets its own inputs at the end: partial outputs and
base-2 LSEs of N context shards (``make_lse``).

Generators use ``numpy.random.Generator(PCG64(seed))``. Nothing here needs a
GPU; arrays are C-contiguous numpy arrays.
"""

from __future__ import annotations

import dataclasses
from typing import Optional

import numpy as np

__all__ = [
    "Workload",
    "ShardedWorkload",
    "CONFIG_NAMES",
    "make",
    "make_tiny",
    "make_decode",
    "make_prefill",
    "make_long",
    "make_dcp",
    "round_to_bf16_grid",
    "deal_to_shards",
    "gather_from_shards",
    "random_nan_bits",
    "small_unsharded",
    "small_sharded",
    "LseWorkload",
    "LSE_NAMES",
    "make_lse",
    "make_lse_named",
]


@dataclasses.dataclass
class Workload:
    """One unsharded selection problem.

    ``logits`` is ``[rows, width]`` fp32. ``row_ks`` (or None) and ``row_ke`` are
    int32 of length ``ceil(rows / row_repeat)``.
    """

    name: str
    logits: np.ndarray
    row_ks: Optional[np.ndarray]
    row_ke: np.ndarray
    block_size: int
    topk_blocks: int
    row_repeat: int
    pin_newest: bool
    seed: int
    notes: dict = dataclasses.field(default_factory=dict)
    logical_width: Optional[int] = None
    dtype: str = "f32"  # "bf16": the values lie on the bf16 grid, stored as bf16

    @property
    def rows(self) -> int:
        return int(self.logits.shape[0])

    @property
    def width(self) -> int:
        """Logical row length; rows may be padded up to ``logits.shape[1]``."""
        if self.logical_width is not None:
            return int(self.logical_width)
        return int(self.logits.shape[1])


@dataclasses.dataclass
class ShardedWorkload:
    """One selection problem held as D interleave-1 shards on one device.

    ``logits`` is ``[D, rows, local_width]`` fp32; ``global_row_ke`` is int32 of
    length ``ceil(rows / row_repeat)``.
    """

    name: str
    logits: np.ndarray
    global_row_ke: np.ndarray
    global_block_size: int
    max_global_blocks: int
    topk_blocks: int
    row_repeat: int
    seed: int
    notes: dict = dataclasses.field(default_factory=dict)
    dtype: str = "f32"  # "bf16": the values lie on the bf16 grid, stored as bf16
    global_row_ks: Optional[np.ndarray] = None  # global window starts (None: all 0)

    @property
    def shards(self) -> int:
        return int(self.logits.shape[0])

    @property
    def rows(self) -> int:
        return int(self.logits.shape[1])

    @property
    def local_width(self) -> int:
        return int(self.logits.shape[2])


def _rng(seed: int) -> np.random.Generator:
    return np.random.Generator(np.random.PCG64(seed))


def round_to_bf16_grid(x: np.ndarray, *, inplace: bool = False) -> np.ndarray:
    """Round fp32 values to the nearest bf16-representable value (ties to even).

    Works on the bit pattern: add 0x7FFF plus the lowest kept bit, then clear
    the low 16 bits. Inputs must be finite (normal draws are). Processes the
    array in chunks so that large inputs need no large temporaries.
    """
    x = np.ascontiguousarray(x, dtype=np.float32)
    if not inplace:
        x = x.copy()
    u = x.reshape(-1).view(np.uint32)
    step = 1 << 20
    lsb = np.empty(min(step, u.size), dtype=np.uint32)
    for i in range(0, u.size, step):
        c = u[i:i + step]
        t = lsb[:c.size]
        np.right_shift(c, np.uint32(16), out=t)
        np.bitwise_and(t, np.uint32(1), out=t)
        t += np.uint32(0x7FFF)
        c += t
        c &= np.uint32(0xFFFF0000)
    return x


def _normal(rng: np.random.Generator, shape) -> np.ndarray:
    """fp32 N(0, 1) draws written straight into one new array."""
    out = np.empty(shape, dtype=np.float32)
    rng.standard_normal(out=out, dtype=np.float32)
    return out


def deal_to_shards(g: np.ndarray, shards: int) -> np.ndarray:
    """Interleave-1 layout: global token t of each row goes to shard t % D at
    local column t // D. ``g`` is [rows, D * local_width]."""
    rows, gw = g.shape
    return np.ascontiguousarray(g.reshape(rows, gw // shards, shards).transpose(2, 0, 1))


def gather_from_shards(local: np.ndarray) -> np.ndarray:
    """Inverse of ``deal_to_shards``: [D, rows, lw] back to [rows, D * lw]."""
    shards, rows, lw = local.shape
    return np.ascontiguousarray(local.transpose(1, 2, 0)).reshape(rows, lw * shards)


def random_nan_bits(rng: np.random.Generator, n: int) -> np.ndarray:
    """``n`` quiet NaNs with random sign and random payload, as fp32."""
    sign = rng.integers(0, 2, size=n, dtype=np.uint32) << np.uint32(31)
    payload = rng.integers(0, 1 << 22, size=n, dtype=np.uint32)
    bits = sign | np.uint32(0x7FC00000) | payload
    return bits.view(np.float32)


# --------------------------------------------------------------------------
# The five workloads
# --------------------------------------------------------------------------

CONFIG_NAMES = ("tiny", "decode", "prefill", "long", "long_pin", "dcp")
BF16_NAMES = ("decode_bf16", "dcp_bf16")
EXTRA_NAMES = BF16_NAMES + ("dcp_starts",)


def make_tiny(seed: int = 0) -> Workload:
    """[64, 4096] N(0,1); no starts; ends uniform in [0, 4096] with one 0 and
    one 4096 forced; block 64, top-16, pinned."""
    rng = _rng(seed)
    rows, width = 64, 4096
    logits = _normal(rng, (rows, width))
    ke = rng.integers(0, width, size=rows, endpoint=True).astype(np.int32)
    ke[0] = 0
    ke[1] = width
    return Workload("tiny", logits, None, ke, 64, 16, 1, True, seed)


def make_decode(seed: int = 1) -> Workload:
    """64 sequences x 8 heads = 512 rows of [65536] N(0,1) on the bf16 grid
    (forces ties); per-sequence ends uniform in [1, 65536]; no starts;
    block 64, top-32, pinned, row_repeat 8."""
    rng = _rng(seed)
    seqs, heads, width = 64, 8, 65536
    rows = seqs * heads
    logits = round_to_bf16_grid(_normal(rng, (rows, width)), inplace=True)
    ke = rng.integers(1, width, size=seqs, endpoint=True).astype(np.int32)
    return Workload("decode", logits, None, ke, 64, 32, heads, True, seed)


def make_prefill(seed: int = 2, *, requests: int = 4, tokens: int = 2048,
                 max_prefix: int = 6144, width: int = 16384,
                 nan_fraction: float = 1e-6, sigma: float = 2.0) -> Workload:
    """A packed multi-request prefill chunk.

    ``requests`` requests of ``tokens`` query tokens each; request q has a
    cached prefix p_q uniform in [0, max_prefix] and occupies packed columns
    [off_q, off_q + p_q + tokens), requests back to back. Row (q, i) has
    ks = off_q and ke = off_q + p_q + i + 1 (causal). Logits ~ N(0, sigma)
    (sigma is the standard deviation) with round(nan_fraction * rows * width)
    NaNs of random sign and payload at distinct uniform positions.

    The four prefixes can need more than ``width`` columns; all four are
    redrawn until they fit.
    """
    rng = _rng(seed)
    rows = requests * tokens
    draws = 0
    while True:
        draws += 1
        prefix = rng.integers(0, max_prefix, size=requests, endpoint=True)
        if int(np.sum(prefix + tokens)) <= width:
            break
    offsets = np.concatenate([[0], np.cumsum(prefix + tokens)[:-1]])
    ks = np.repeat(offsets, tokens).astype(np.int32)
    tok = np.tile(np.arange(tokens), requests)
    ke = (np.repeat(offsets + prefix, tokens) + tok + 1).astype(np.int32)
    logits = _normal(rng, (rows, width))
    logits *= np.float32(sigma)
    n_nan = int(round(nan_fraction * rows * width))
    pos = rng.choice(rows * width, size=n_nan, replace=False)
    logits.reshape(-1)[pos] = random_nan_bits(rng, n_nan)
    notes = {"prefixes": [int(p) for p in prefix], "offsets": [int(o) for o in offsets],
             "prefix_draws": draws, "nan_count": n_nan}
    return Workload("prefill", logits, ks, ke, 64, 32, 1, True, seed, notes)


def make_long(seed: int = 3, *, pin_newest: bool = False, rows: int = 1024,
              width: int = 131072, spikes: int = 64) -> Workload:
    """[1024, 131072] N(0,1) plus, per row, ``spikes`` distinct in-window
    columns raised by U(3, 6); ends uniform in [65536, 131072], starts uniform
    in [0, 4096]; block 128, top-16."""
    rng = _rng(seed)
    logits = _normal(rng, (rows, width))
    ke = rng.integers(width // 2, width, size=rows, endpoint=True).astype(np.int32)
    ks = rng.integers(0, 4096, size=rows, endpoint=True).astype(np.int32)
    for r in range(rows):
        span = int(ke[r]) - int(ks[r])
        cols = int(ks[r]) + rng.choice(span, size=min(spikes, span), replace=False)
        logits[r, cols] += rng.uniform(3.0, 6.0, size=cols.size).astype(np.float32)
    name = "long_pin" if pin_newest else "long"
    return Workload(name, logits, ks, ke, 128, 16, 1, pin_newest, seed)


def make_dcp(seed: int = 4, *, shards: int = 8, rows: int = 4096,
             global_width: int = 65536, global_block_size: int = 64,
             max_global_blocks: int = 1024, topk_blocks: int = 32) -> ShardedWorkload:
    """Simulated DCP layout: a global [rows, global_width] N(0,1) matrix G
    dealt over ``shards`` interleave-1 shards, L[d, r, c] = G[r, shards*c + d];
    global ends uniform in [1, global_width].

    Dealing an i.i.d. N(0,1) matrix gives an i.i.d. N(0,1) array, so L is
    drawn directly in the shard layout and G is defined as its inverse deal
    (``gather_from_shards``); this avoids a 1 GiB strided copy."""
    rng = _rng(seed)
    lw = global_width // shards
    local = _normal(rng, (shards, rows, lw))
    gke = rng.integers(1, global_width, size=rows, endpoint=True).astype(np.int32)
    return ShardedWorkload("dcp", local, gke, global_block_size, max_global_blocks,
                           topk_blocks, 1, seed)


def make(name: str):
    """Build one named workload at full size."""
    if name == "tiny":
        return make_tiny()
    if name == "decode":
        return make_decode()
    if name == "prefill":
        return make_prefill()
    if name == "long":
        return make_long(pin_newest=False)
    if name == "long_pin":
        return make_long(pin_newest=True)
    if name == "dcp":
        return make_dcp()
    if name == "dcp_starts":
        # The DCP workload with a request start per row, uniform in [0, gke]
        # (window lengths uniform in [0, gke], so about half the bytes).
        wl = make_dcp()
        rng = _rng(40)
        g = wl.global_row_ke.astype(np.int64)
        wl.global_row_ks = rng.integers(0, g + 1).astype(np.int32)
        wl.name = "dcp_starts"
        return wl
    if name == "decode_bf16":
        wl = make_decode()  # already on the bf16 grid
        wl.name, wl.dtype = "decode_bf16", "bf16"
        return wl
    if name == "dcp_bf16":
        wl = make_dcp()
        round_to_bf16_grid(wl.logits, inplace=True)
        wl.name, wl.dtype = "dcp_bf16", "bf16"
        return wl
    raise KeyError(name)


# --------------------------------------------------------------------------
# Small randomized problems for parity sweeps and edge cases
# --------------------------------------------------------------------------

def small_unsharded(seed: int, *, rows: int, width: int, block_size: int,
                    topk_blocks: int, row_repeat: int = 1, starts: bool = True,
                    pin_newest: bool = True, nan_count: int = 0,
                    bf16_grid: bool = False, wild_bounds: bool = False,
                    ld: Optional[int] = None) -> Workload:
    """A random unsharded problem. ``wild_bounds`` draws bounds outside
    [0, width] and starts above ends too. ``ld`` > width pads each row (the
    pad holds large values that must never be read)."""
    rng = _rng(seed)
    groups = -(-rows // row_repeat) if rows else 0
    ld = width if ld is None else ld
    buf = _normal(rng, (rows, ld))
    if bf16_grid:
        buf = round_to_bf16_grid(buf, inplace=True)
    if ld > width:
        buf[:, width:] = np.float32(1e30)
    if nan_count and rows and width:
        pos = rng.choice(rows * width, size=min(nan_count, rows * width), replace=False)
        buf[pos // width, pos % width] = random_nan_bits(rng, pos.size)
    if wild_bounds:
        ke = rng.integers(-3, width + 8, size=groups, endpoint=True).astype(np.int32)
        ks = rng.integers(-5, width + 4, size=groups, endpoint=True).astype(np.int32)
    else:
        ke = rng.integers(0, width, size=groups, endpoint=True).astype(np.int32)
        ks = np.minimum(rng.integers(0, max(width, 1), size=groups, endpoint=True),
                        ke).astype(np.int32)
    return Workload("small", buf, ks if starts else None, ke, block_size,
                    topk_blocks, row_repeat, pin_newest, seed, {"ld": ld}, width)


def small_sharded(seed: int, *, shards: int, rows: int, global_width: int,
                  global_block_size: int, max_global_blocks: int,
                  topk_blocks: int, row_repeat: int = 1,
                  wild_bounds: bool = False) -> tuple[ShardedWorkload, np.ndarray]:
    """A random sharded problem plus its global matrix G (so that tests can
    compare against the unsharded form). ``global_width`` must be a multiple
    of ``shards``."""
    rng = _rng(seed)
    assert global_width % shards == 0
    g = _normal(rng, (rows, global_width))
    local = deal_to_shards(g, shards)
    groups = -(-rows // row_repeat) if rows else 0
    lo, hi = (-4, global_width + 40) if wild_bounds else (0, global_width)
    gke = rng.integers(lo, hi, size=groups, endpoint=True).astype(np.int32)
    wl = ShardedWorkload("small_sharded", local, gke, global_block_size,
                         max_global_blocks, topk_blocks, row_repeat, seed)
    return wl, g


# --------------------------------------------------------------------------
# DCP partial-attention LSE correction inputs
# --------------------------------------------------------------------------

@dataclasses.dataclass
class LseWorkload:
    """Partial attention results of ``shards`` context shards.

    ``outs`` is ``[N, B, H, Dh]`` fp32 (values on the bf16 grid when
    ``dtype == "bf16"``), ``lses`` ``[N, B, H]`` fp32 base-2 log-sum-exps.
    A shard that holds no key for a (token, head) has LSE -inf and a zero
    partial output.
    """

    name: str
    outs: np.ndarray
    lses: np.ndarray
    dtype: str
    seed: int
    notes: dict = dataclasses.field(default_factory=dict)

    @property
    def shards(self) -> int:
        return int(self.outs.shape[0])

    @property
    def batch(self) -> int:
        return int(self.outs.shape[1])

    @property
    def heads(self) -> int:
        return int(self.outs.shape[2])

    @property
    def head_dim(self) -> int:
        return int(self.outs.shape[3])


LSE_NAMES = ("lse_decode", "lse_decode_bf16", "lse_tiny")


def make_lse(seed: int = 5, *, shards: int = 8, batch: int = 512, heads: int = 128,
             head_dim: int = 512, dtype: str = "f32", empty_rate: float = 1 / 32,
             specials: bool = False) -> LseWorkload:
    """Random partial results of an MLA decode step split over ``shards``.

    Per (token, head) a centre mu ~ U(4, 20); each shard's LSE is
    mu + N(0, 1). With probability ``empty_rate`` a (shard, token) pair holds
    no keys (every head's LSE -inf, output 0), as for short contexts.
    Partial outputs are N(0, 1). ``specials`` also plants NaN and +inf LSEs
    (1 in 64 entries each, random payload NaNs) and makes token 0 empty on
    every shard.
    """
    assert dtype in ("f32", "bf16")
    rng = _rng(seed)
    outs = _normal(rng, (shards, batch, heads, head_dim))
    if dtype == "bf16":
        outs = round_to_bf16_grid(outs, inplace=True)
    mu = rng.uniform(4.0, 20.0, size=(batch, heads)).astype(np.float32)
    lses = mu[None] + _normal(rng, (shards, batch, heads))
    empty = rng.random((shards, batch)) < empty_rate
    if specials and batch:
        empty[:, 0] = True
    lses[empty] = -np.inf
    outs[empty] = 0.0
    if specials and lses.size:
        flat = lses.reshape(-1)
        k = max(1, flat.size // 64)
        pos = rng.choice(flat.size, size=2 * k, replace=False)
        flat[pos[:k]] = random_nan_bits(rng, k)
        flat[pos[k:]] = np.inf
    return LseWorkload("lse", outs, lses.astype(np.float32), dtype, seed,
                       {"empty_rate": empty_rate, "specials": specials})


def make_lse_named(name: str) -> LseWorkload:
    """The named LSE-correction workloads (full size, plus a small one)."""
    if name == "lse_decode":
        return make_lse(5)
    if name == "lse_decode_bf16":
        return make_lse(6, dtype="bf16")
    if name == "lse_tiny":
        return make_lse(7, shards=4, batch=16, heads=8, head_dim=64, specials=True)
    raise KeyError(name)
