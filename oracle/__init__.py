"""CPU oracle for DSA candidate-block selection (ctypes over plain C).

TEST INFRASTRUCTURE. Only ``tests/``, ``__graft_entry__.smoke()`` and the
benchmark's CPU-baseline / reference leg may import this package. The
product path (``deepseek_sparse_attention_row_gb300``) never imports it and
shares no code with it.

``dsa_oracle.c`` states the definition each function follows and the
readings taken where the pages are silent. Every function here is pinned by
``tests/test_oracle_pins.py`` and ``tests/test_oracle_golden.py``.

``dcp_lse_oracle.c`` does the same for the DCP partial-attention LSE
correction (``correct_attn_out``, ``merge_attn_out``); its pins are in
``tests/test_oracle_lse.py``.

``dsa_oracle_bf16.c`` gives the selection, block-score and masking entry
points for bf16 logits (``*_bf16``: uint16 bit patterns in and out); its pins
are in ``tests/test_oracle_bf16.py``.

``build()`` compiles the C files with gcc into one library in
``oracle/_build``.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from typing import Optional

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "dsa_oracle.c")
_HDR = os.path.join(_HERE, "dsa_oracle.h")
_LSE_SRC = os.path.join(_HERE, "dcp_lse_oracle.c")
_LSE_HDR = os.path.join(_HERE, "dcp_lse_oracle.h")
_BF16_SRC = os.path.join(_HERE, "dsa_oracle_bf16.c")
SOURCES = (_SRC, _LSE_SRC, _BF16_SRC)
HEADERS = (_HDR, _LSE_HDR)
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "libdsa_oracle.so")

_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle (portable C, no target-specific flags)."""
    os.makedirs(_BUILD, exist_ok=True)
    fresh = (os.path.exists(_LIB_PATH)
             and os.path.getmtime(_LIB_PATH) >= max(os.path.getmtime(f)
                                                    for f in SOURCES + HEADERS))
    if fresh and not force:
        return _LIB_PATH
    tmp = _LIB_PATH + f".tmp{os.getpid()}"
    compile_sources(SOURCES, tmp, warnings=True)
    os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def build_variant(directory: str, replacements: dict) -> str:
    """Build a copy of the oracle library in ``directory`` with the given
    ``{file name: new text}`` replacing those sources (used by the tests to
    plant mistakes); returns the library's path."""
    srcs = []
    for f in SOURCES + HEADERS:
        name = os.path.basename(f)
        with open(f) as fh:
            text = fh.read()
        dst = os.path.join(directory, name)
        with open(dst, "w") as fh:
            fh.write(replacements.get(name, text))
        if name.endswith(".c"):
            srcs.append(dst)
    path = os.path.join(directory, "libvariant.so")
    compile_sources(srcs, path)
    return path


def compile_sources(sources, path: str, warnings: bool = False) -> None:
    """gcc the given C sources (with the headers beside them) into a shared
    library at ``path``."""
    cmd = ["gcc", "-std=c99", "-O2", "-fPIC", "-shared"]
    if warnings:
        cmd += ["-Wall", "-Wextra"]
    subprocess.run(cmd + ["-o", path, *sources, "-lm"], check=True)


def bind(path: str):
    """Load an oracle library built from the C sources and declare its entry
    points."""
    lib = ctypes.CDLL(path)
    i64, i32, p = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
    lib.dsa_oracle_block_scores.argtypes = [p, i64, i64, i64, p, p, i32, i32, i32, p, i64]
    lib.dsa_oracle_select.argtypes = [p, i64, i64, i64, p, p, i32, i32, i32, i32, p, i64, p, i64]
    lib.dsa_oracle_select_sharded.argtypes = [p, i32, i64, i64, i64, i64, p, i32, i32, i32, i32,
                                              p, i64, p, i64]
    lib.dsa_oracle_mask.argtypes = [p, i64, i64, i64, p, p, p, i64, i64, i32, i32]
    lib.dsa_oracle_mask_sharded.argtypes = [p, i32, i64, i64, i64, i64, p, i32, i32, p, i64, i64]
    lib.dsa_oracle_select_sharded_starts.argtypes = [p, i32, i64, i64, i64, i64, p, p, i32, i32,
                                                     i32, i32, p, i64, p, i64]
    lib.dsa_oracle_mask_sharded_starts.argtypes = [p, i32, i64, i64, i64, i64, p, p, i32, i32,
                                                   p, i64, i64]
    lib.dsa_oracle_block_scores_bf16.argtypes = lib.dsa_oracle_block_scores.argtypes
    lib.dsa_oracle_select_bf16.argtypes = lib.dsa_oracle_select.argtypes
    lib.dsa_oracle_select_sharded_bf16.argtypes = lib.dsa_oracle_select_sharded.argtypes
    lib.dsa_oracle_mask_bf16.argtypes = lib.dsa_oracle_mask.argtypes
    lib.dsa_oracle_mask_sharded_bf16.argtypes = lib.dsa_oracle_mask_sharded.argtypes
    lib.dcp_oracle_correct_attn_out.argtypes = [p, p, i32, i64, i64, i64, i32, p, p]
    lib.dcp_oracle_merge_attn_out.argtypes = [p, p, i32, i64, i64, i64, p, p]
    for f in (lib.dsa_oracle_block_scores, lib.dsa_oracle_select,
              lib.dsa_oracle_select_sharded, lib.dsa_oracle_mask, lib.dsa_oracle_mask_sharded,
              lib.dcp_oracle_correct_attn_out, lib.dcp_oracle_merge_attn_out,
              lib.dsa_oracle_block_scores_bf16, lib.dsa_oracle_select_bf16,
              lib.dsa_oracle_select_sharded_bf16, lib.dsa_oracle_mask_bf16,
              lib.dsa_oracle_mask_sharded_bf16, lib.dsa_oracle_select_sharded_starts,
              lib.dsa_oracle_mask_sharded_starts):
        f.restype = ctypes.c_int
    return lib


def _load():
    global _lib
    if _lib is None:
        _lib = bind(build())
    return _lib


def _ptr(a: Optional[np.ndarray]):
    return None if a is None else a.ctypes.data


def _f32(a):
    a = np.asarray(a, dtype=np.float32)
    assert a.flags.c_contiguous
    return a


def _u16(a):
    """bf16 logits as their uint16 bit patterns (a numpy uint16 array, or a
    float32 array whose values are exactly bf16-representable)."""
    a = np.asarray(a)
    if a.dtype == np.float32:
        bits = a.view(np.uint32)
        assert not (bits & 0xFFFF).any(), "float32 values are not on the bf16 grid"
        a = (bits >> 16).astype(np.uint16)
    assert a.dtype == np.uint16
    return np.ascontiguousarray(a)


def _i32(a):
    if a is None:
        return None
    return np.ascontiguousarray(a, dtype=np.int32)


def nblocks(width: int, block_size: int) -> int:
    return -(-width // block_size)


def block_scores(logits: np.ndarray, row_ks, row_ke, block_size: int,
                 row_repeat: int = 1, pin_newest: bool = True,
                 width: Optional[int] = None) -> np.ndarray:
    """Block scores ``[rows, ceil(width / block_size)]`` (fp32).

    ``logits`` is ``[rows, ld]``; ``width`` (default ``ld``) is the logical
    row length."""
    logits = _f32(logits)
    rows, ld = logits.shape
    width = ld if width is None else width
    ks, ke = _i32(row_ks), _i32(row_ke)
    nb = nblocks(width, block_size)
    scores = np.zeros((rows, nb), dtype=np.float32)
    rc = _load().dsa_oracle_block_scores(_ptr(logits), rows, width, ld, _ptr(ks), _ptr(ke),
                                         block_size, row_repeat, int(pin_newest),
                                         _ptr(scores), nb)
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (status {rc})")
    return scores


def select(logits: np.ndarray, row_ks, row_ke, topk_blocks: int, block_size: int,
           row_repeat: int = 1, pin_newest: bool = True,
           width: Optional[int] = None, want_scores: bool = True):
    """Ordered candidate ids ``[rows, topk_blocks]`` (int32, -1 padded) and,
    when ``want_scores``, the block scores they were ranked by."""
    logits = _f32(logits)
    rows, ld = logits.shape
    width = ld if width is None else width
    ks, ke = _i32(row_ks), _i32(row_ke)
    nb = nblocks(width, block_size)
    out = np.full((rows, topk_blocks), -7, dtype=np.int32)
    scores = np.zeros((rows, nb), dtype=np.float32) if want_scores and nb else None
    rc = _load().dsa_oracle_select(_ptr(logits), rows, width, ld, _ptr(ks), _ptr(ke),
                                   topk_blocks, block_size, row_repeat, int(pin_newest),
                                   _ptr(out), topk_blocks, _ptr(scores), max(nb, 1))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (status {rc})")
    return out, scores


def select_sharded(logits: np.ndarray, global_row_ke, global_block_size: int,
                   max_global_blocks: int, topk_blocks: int, row_repeat: int = 1,
                   want_scores: bool = True):
    """Ordered candidate ids for a ``[shards, rows, local_width]`` DCP layout,
    and the merged global block scores ``[rows, max(max_global_blocks, 1)]``."""
    logits = _f32(logits)
    shards, rows, lw = logits.shape
    gke = _i32(global_row_ke)
    nbg = max(int(max_global_blocks), 1)
    out = np.full((rows, topk_blocks), -7, dtype=np.int32)
    scores = np.zeros((rows, nbg), dtype=np.float32) if want_scores else None
    rc = _load().dsa_oracle_select_sharded(_ptr(logits), shards, rows, lw, lw, rows * lw,
                                           _ptr(gke), global_block_size, max_global_blocks,
                                           row_repeat, topk_blocks, _ptr(out), topk_blocks,
                                           _ptr(scores), nbg)
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (status {rc})")
    return out, scores


def select_sharded_starts(logits: np.ndarray, global_row_ks, global_row_ke,
                          global_block_size: int, max_global_blocks: int, topk_blocks: int,
                          row_repeat: int = 1, want_scores: bool = True):
    """``select_sharded`` with global window starts (reading R12): ids and the
    merged global block scores."""
    logits = _f32(logits)
    shards, rows, lw = logits.shape
    nbg = max(int(max_global_blocks), 1)
    out = np.full((rows, topk_blocks), -7, dtype=np.int32)
    scores = np.zeros((rows, nbg), dtype=np.float32) if want_scores else None
    rc = _load().dsa_oracle_select_sharded_starts(
        _ptr(logits), shards, rows, lw, lw, rows * lw, _ptr(_i32(global_row_ks)),
        _ptr(_i32(global_row_ke)), global_block_size, max_global_blocks, row_repeat,
        topk_blocks, _ptr(out), topk_blocks, _ptr(scores), nbg)
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (status {rc})")
    return out, scores


def mask_sharded_starts(logits: np.ndarray, global_row_ks, global_row_ke,
                        global_block_size: int, candidates: np.ndarray,
                        row_repeat: int = 1) -> np.ndarray:
    """Masked copy of a ``[shards, rows, local_width]`` layout with global
    window starts (reading R12)."""
    out = np.array(_f32(logits), copy=True)
    shards, rows, lw = out.shape
    cand = np.ascontiguousarray(candidates, dtype=np.int32)
    topk = cand.shape[1] if cand.ndim == 2 else 0
    rc = _load().dsa_oracle_mask_sharded_starts(
        _ptr(out), shards, rows, lw, lw, rows * lw, _ptr(_i32(global_row_ks)),
        _ptr(_i32(global_row_ke)), global_block_size, row_repeat, _ptr(cand), topk,
        max(topk, 1))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (status {rc})")
    return out


def run_workload(wl, want_scores: bool = True):
    """Run the oracle on a ``workloads.Workload`` or ``ShardedWorkload``."""
    if getattr(wl, "global_row_ks", None) is not None:
        return select_sharded_starts(wl.logits, wl.global_row_ks, wl.global_row_ke,
                                     wl.global_block_size, wl.max_global_blocks, wl.topk_blocks,
                                     wl.row_repeat, want_scores=want_scores)
    if hasattr(wl, "global_row_ke"):
        return select_sharded(wl.logits, wl.global_row_ke, wl.global_block_size,
                              wl.max_global_blocks, wl.topk_blocks, wl.row_repeat,
                              want_scores=want_scores)
    return select(wl.logits, wl.row_ks, wl.row_ke, wl.topk_blocks, wl.block_size,
                  wl.row_repeat, wl.pin_newest, width=wl.width,
                  want_scores=want_scores)


def mask(logits: np.ndarray, row_ks, row_ke, candidates: np.ndarray, block_size: int,
         row_repeat: int = 1, width: Optional[int] = None) -> np.ndarray:
    """Masked copy of ``logits`` [rows, ld]: -inf outside each row's window
    and outside its candidate blocks (``candidates`` [rows, topk], -1 = empty)."""
    out = np.array(_f32(logits), copy=True)
    rows, ld = out.shape
    width = ld if width is None else width
    cand = np.ascontiguousarray(candidates, dtype=np.int32)
    ks, ke = _i32(row_ks), _i32(row_ke)
    topk = cand.shape[1] if cand.ndim == 2 else 0
    rc = _load().dsa_oracle_mask(_ptr(out), rows, width, ld, _ptr(ks), _ptr(ke), _ptr(cand),
                                 topk, max(topk, 1), block_size, row_repeat)
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (status {rc})")
    return out


def mask_sharded(logits: np.ndarray, global_row_ke, global_block_size: int,
                 candidates: np.ndarray, row_repeat: int = 1) -> np.ndarray:
    """Masked copy of a ``[shards, rows, local_width]`` DCP layout."""
    out = np.array(_f32(logits), copy=True)
    shards, rows, lw = out.shape
    cand = np.ascontiguousarray(candidates, dtype=np.int32)
    topk = cand.shape[1] if cand.ndim == 2 else 0
    rc = _load().dsa_oracle_mask_sharded(_ptr(out), shards, rows, lw, lw, rows * lw,
                                         _ptr(_i32(global_row_ke)), global_block_size,
                                         row_repeat, _ptr(cand), topk, max(topk, 1))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (status {rc})")
    return out


def correct_attn_out(out: np.ndarray, lses: np.ndarray, rank: int):
    """DCP LSE correction of one shard's partial attention output.

    ``out`` [B, H, Dh] and ``lses`` [N, B, H] (base-2 LSEs of all N shards)
    are read as fp32 (bf16 inputs widen exactly). Returns ``new_out``
    [H, B, Dh] and the combined LSE [B, H], both float64."""
    out = np.ascontiguousarray(out, dtype=np.float32)
    lses = np.ascontiguousarray(lses, dtype=np.float32)
    B, H, Dh = out.shape
    N = lses.shape[0]
    assert lses.shape == (N, B, H)
    new_out = np.zeros((H, B, Dh), dtype=np.float64)
    lse = np.zeros((B, H), dtype=np.float64)
    rc = _load().dcp_oracle_correct_attn_out(_ptr(out), _ptr(lses), N, B, H, Dh, rank,
                                             _ptr(new_out), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (status {rc})")
    return new_out, lse


def merge_attn_out(outs: np.ndarray, lses: np.ndarray):
    """Sum over shards of the corrected partial outputs.

    ``outs`` [N, B, H, Dh], ``lses`` [N, B, H]. Returns the merged output
    [H, B, Dh] and the combined LSE [B, H], both float64."""
    outs = np.ascontiguousarray(outs, dtype=np.float32)
    lses = np.ascontiguousarray(lses, dtype=np.float32)
    N, B, H, Dh = outs.shape
    assert lses.shape == (N, B, H)
    merged = np.zeros((H, B, Dh), dtype=np.float64)
    lse = np.zeros((B, H), dtype=np.float64)
    rc = _load().dcp_oracle_merge_attn_out(_ptr(outs), _ptr(lses), N, B, H, Dh,
                                           _ptr(merged), _ptr(lse))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (status {rc})")
    return merged, lse


# --------------------------------------------------------------------------
# bf16 logits (dsa_oracle_bf16.c): inputs and scores are uint16 bit patterns
# --------------------------------------------------------------------------

def block_scores_bf16(logits, row_ks, row_ke, block_size: int, row_repeat: int = 1,
                      pin_newest: bool = True, width: Optional[int] = None) -> np.ndarray:
    """bf16 block scores (uint16 bits) of bf16 logits ``[rows, ld]``."""
    x = _u16(logits)
    rows, ld = x.shape
    width = ld if width is None else width
    nb = nblocks(width, block_size)
    scores = np.zeros((rows, nb), dtype=np.uint16)
    rc = _load().dsa_oracle_block_scores_bf16(_ptr(x), rows, width, ld, _ptr(_i32(row_ks)),
                                              _ptr(_i32(row_ke)), block_size, row_repeat,
                                              int(pin_newest), _ptr(scores), nb)
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (status {rc})")
    return scores


def select_bf16(logits, row_ks, row_ke, topk_blocks: int, block_size: int, row_repeat: int = 1,
                pin_newest: bool = True, width: Optional[int] = None, want_scores: bool = True):
    """``select`` on bf16 logits: ids and bf16 scores (uint16 bits)."""
    x = _u16(logits)
    rows, ld = x.shape
    width = ld if width is None else width
    nb = nblocks(width, block_size)
    out = np.full((rows, topk_blocks), -7, dtype=np.int32)
    scores = np.zeros((rows, nb), dtype=np.uint16) if want_scores and nb else None
    rc = _load().dsa_oracle_select_bf16(_ptr(x), rows, width, ld, _ptr(_i32(row_ks)),
                                        _ptr(_i32(row_ke)), topk_blocks, block_size, row_repeat,
                                        int(pin_newest), _ptr(out), topk_blocks, _ptr(scores),
                                        max(nb, 1))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (status {rc})")
    return out, scores


def select_sharded_bf16(logits, global_row_ke, global_block_size: int, max_global_blocks: int,
                        topk_blocks: int, row_repeat: int = 1, want_scores: bool = True):
    """``select_sharded`` on bf16 logits ``[shards, rows, local_width]``."""
    x = _u16(logits)
    shards, rows, lw = x.shape
    nbg = max(int(max_global_blocks), 1)
    out = np.full((rows, topk_blocks), -7, dtype=np.int32)
    scores = np.zeros((rows, nbg), dtype=np.uint16) if want_scores else None
    rc = _load().dsa_oracle_select_sharded_bf16(_ptr(x), shards, rows, lw, lw, rows * lw,
                                                _ptr(_i32(global_row_ke)), global_block_size,
                                                max_global_blocks, row_repeat, topk_blocks,
                                                _ptr(out), topk_blocks, _ptr(scores), nbg)
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (status {rc})")
    return out, scores


def mask_bf16(logits, row_ks, row_ke, candidates, block_size: int, row_repeat: int = 1,
              width: Optional[int] = None) -> np.ndarray:
    """Masked copy (uint16 bits) of bf16 logits ``[rows, ld]``."""
    out = np.array(_u16(logits), copy=True)
    rows, ld = out.shape
    width = ld if width is None else width
    cand = np.ascontiguousarray(candidates, dtype=np.int32)
    topk = cand.shape[1] if cand.ndim == 2 else 0
    rc = _load().dsa_oracle_mask_bf16(_ptr(out), rows, width, ld, _ptr(_i32(row_ks)),
                                      _ptr(_i32(row_ke)), _ptr(cand), topk, max(topk, 1),
                                      block_size, row_repeat)
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (status {rc})")
    return out


def mask_sharded_bf16(logits, global_row_ke, global_block_size: int, candidates,
                      row_repeat: int = 1) -> np.ndarray:
    """Masked copy (uint16 bits) of bf16 logits ``[shards, rows, local_width]``."""
    out = np.array(_u16(logits), copy=True)
    shards, rows, lw = out.shape
    cand = np.ascontiguousarray(candidates, dtype=np.int32)
    topk = cand.shape[1] if cand.ndim == 2 else 0
    rc = _load().dsa_oracle_mask_sharded_bf16(_ptr(out), shards, rows, lw, lw, rows * lw,
                                              _ptr(_i32(global_row_ke)), global_block_size,
                                              row_repeat, _ptr(cand), topk, max(topk, 1))
    if rc != 0:
        raise ValueError(f"oracle rejected the arguments (status {rc})")
    return out


def run_workload_bf16(wl, want_scores: bool = True):
    """Run the bf16 oracle on a workload whose logits are on the bf16 grid."""
    if hasattr(wl, "global_row_ke"):
        return select_sharded_bf16(wl.logits, wl.global_row_ke, wl.global_block_size,
                                   wl.max_global_blocks, wl.topk_blocks, wl.row_repeat,
                                   want_scores=want_scores)
    return select_bf16(wl.logits, wl.row_ks, wl.row_ke, wl.topk_blocks, wl.block_size,
                       wl.row_repeat, wl.pin_newest, width=wl.width, want_scores=want_scores)
