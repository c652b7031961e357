"""Helpers shared by the tests: fixture parsing and bit-level comparison."""

from __future__ import annotations

import json
import math
import os
import struct

import numpy as np

GOLDEN = os.path.join(os.path.dirname(os.path.abspath(__file__)), "golden")
CANONICAL_NAN_BITS = 0x7FC00000


def parse_float(tok: str) -> np.float32:
    """'1.5', 'inf', '-inf', '-0.0', 'nan' (canonical) or 'nan:0xBITS'."""
    if tok.startswith("nan:"):
        return np.array([int(tok[4:], 16)], dtype=np.uint32).view(np.float32)[0]
    if tok == "nan":
        return np.array([CANONICAL_NAN_BITS], dtype=np.uint32).view(np.float32)[0]
    return np.float32(float(tok))


def parse_matrix(rows) -> np.ndarray:
    return np.array([[parse_float(t) for t in r] for r in rows], dtype=np.float32).reshape(
        len(rows), -1 if rows and rows[0] else 0)


def load_golden(name: str) -> dict:
    with open(os.path.join(GOLDEN, name)) as f:
        return json.load(f)


def golden_files():
    return sorted(f for f in os.listdir(GOLDEN) if f.endswith(".json"))


def deal_shards(g: np.ndarray, shards: int) -> np.ndarray:
    """Input layout only: global token t of each row goes to shard t % D at
    local column t // D."""
    rows, gw = g.shape
    return np.ascontiguousarray(g.reshape(rows, gw // shards, shards).transpose(2, 0, 1))


def bits(a: np.ndarray) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float32).view(np.uint32)


def assert_bits_equal(got: np.ndarray, want: np.ndarray, what: str = "scores"):
    gb, wb = bits(got), bits(want)
    if gb.shape != wb.shape or not np.array_equal(gb, wb):
        bad = np.argwhere(gb != wb) if gb.shape == wb.shape else None
        raise AssertionError(f"{what} differ: shapes {gb.shape} vs {wb.shape}; "
                             f"first mismatches {bad[:8].tolist() if bad is not None else ''}")


def f32_bits(x: float) -> int:
    return struct.unpack("<I", struct.pack("<f", x))[0]
