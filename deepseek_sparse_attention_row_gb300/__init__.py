"""GB300 (sm_103a) DSA candidate-block selection.

A thin binding over ``libdsa_cb.so`` (C ABI declared in ``include/dsa_cb.h``
and ``include/dsa_dcp_attn.h``):
argument marshalling only. Every step of the computation runs in the
library's CUDA kernels; there is no CPU or PyTorch fallback, and every call
raises if the library is missing or a call fails.

Functions carry the C ABI's names:

* ``dsa_block_scores`` -- per-block windowed maxima (candidate_blocks.py diff,
  ``_block_scores``).
* ``dsa_select_candidate_blocks`` -- ranked top-k block ids, -1 padded
  (``select_candidate_blocks`` without a DCP group).
* ``dsa_select_candidate_blocks_sharded`` -- the DCP form with the ranks'
  local logits held as a leading ``[D, rows, local_width]`` axis.
* ``dsa_mask_candidate_logits[_sharded]`` -- the masking pass after
  selection: -inf outside each row's window and candidate blocks.
* ``dsa_correct_attn_out`` / ``dsa_merge_attn_out`` -- the DCP partial-
  attention LSE correction (sglang ``dcp/kernels.py``, ``correct_attn_out``;
  C ABI in ``include/dsa_dcp_attn.h``) and the sum over shards after it.

Tensors are PyTorch CUDA tensors (PyTorch supplies device memory and the
current stream) or pinned host tensors, which the kernels read and write in
place through ``dsa_mapped_host_pointer`` (across NVLink-C2C on Grace
systems). Logits may be float32 or bfloat16 (the ``*_bf16`` C entry points);
scores follow the logits' dtype. ``select_candidate_blocks[_sharded]_host``
take host tensors and wait for the ids: pinned inputs are read in place
(only the in-window logits cross the link), other host tensors are copied to
the device first.
"""

from __future__ import annotations

import ctypes
import os
from typing import Optional

__all__ = [
    "DsaError",
    "library",
    "library_path",
    "dsa_block_scores",
    "dsa_select_candidate_blocks",
    "dsa_select_candidate_blocks_sharded",
    "dsa_mask_candidate_logits",
    "dsa_mask_candidate_logits_sharded",
    "dsa_correct_attn_out",
    "dsa_merge_attn_out",
    "select_candidate_blocks_host",
    "select_candidate_blocks_sharded_host",
    "max_select_blocks",
    "mapped_host_pointer",
    "set_launch_override",
    "pipeline_error",
    "EXPORTED_SYMBOLS",
]

_PKG = os.path.dirname(os.path.abspath(__file__))
library_path = os.path.join(_PKG, "_build", "libdsa_cb.so")

EXPORTED_SYMBOLS = (
    "dsa_status_string",
    "dsa_select_max_blocks",
    "dsa_select_max_shards",
    "dsa_select_workspace_bytes",
    "dsa_block_scores",
    "dsa_select_candidate_blocks",
    "dsa_select_candidate_blocks_sharded",
    "dsa_mask_candidate_logits",
    "dsa_mask_candidate_logits_sharded",
    "dsa_select_candidate_blocks_sharded_static",
    "dsa_mapped_host_pointer",
    "dsa_attn_max_shards",
    "dsa_correct_attn_out",
    "dsa_merge_attn_out",
    "dsa_block_scores_bf16",
    "dsa_select_candidate_blocks_bf16",
    "dsa_select_candidate_blocks_sharded_bf16",
    "dsa_mask_candidate_logits_bf16",
    "dsa_mask_candidate_logits_sharded_bf16",
    "dsa_select_candidate_blocks_sharded_starts",
    "dsa_select_candidate_blocks_sharded_starts_bf16",
    "dsa_mask_candidate_logits_sharded_starts",
    "dsa_mask_candidate_logits_sharded_starts_bf16",
    "dsa_select_set_launch_override",
    "dsa_pipeline_error",
)

# Knobs of dsa_select_set_launch_override (include/dsa_cb.h).
LAUNCH_KNOBS = {"split": 1, "threads": 2, "warp_rows": 3, "warp_order": 4, "pipeline": 5,
                "pipe_split": 6, "pipe_stages": 7, "pipe_stage_kb": 8, "pipe_sched": 9,
                "pipe_warps": 10, "pipe_ctas": 11, "pipe_stage_owner": 12, "pipe_order": 13,
                "rank_cta": 14}

_lib = None


class DsaError(RuntimeError):
    """A library call returned a status other than DSA_OK."""

    def __init__(self, fn: str, status: int, text: str):
        super().__init__(f"{fn} failed: {text} (status {status})")
        self.status = status


def library():
    """Load libdsa_cb.so (build it with ``__graft_entry__.build()``)."""
    global _lib
    if _lib is not None:
        return _lib
    if not os.path.exists(library_path):
        raise RuntimeError(f"libdsa_cb.so is not built ({library_path}); "
                           "run __graft_entry__.build() first")
    lib = ctypes.CDLL(library_path)
    i64, i32, p = ctypes.c_int64, ctypes.c_int32, ctypes.c_void_p
    lib.dsa_status_string.argtypes = [ctypes.c_int]
    lib.dsa_status_string.restype = ctypes.c_char_p
    lib.dsa_select_max_blocks.argtypes = []
    lib.dsa_select_max_blocks.restype = i32
    lib.dsa_select_max_shards.argtypes = []
    lib.dsa_select_max_shards.restype = i32
    lib.dsa_select_workspace_bytes.argtypes = [i64, i64]
    lib.dsa_select_workspace_bytes.restype = ctypes.c_size_t
    lib.dsa_pipeline_error.argtypes = [ctypes.c_int]
    lib.dsa_pipeline_error.restype = ctypes.c_int
    lib.dsa_select_set_launch_override.argtypes = [i32, i32]
    lib.dsa_select_set_launch_override.restype = ctypes.c_int
    lib.dsa_block_scores.argtypes = [p, i64, i64, i64, p, p, i32, i32, i32, p, i64, p]
    sz = ctypes.c_size_t
    lib.dsa_select_candidate_blocks.argtypes = [p, i64, i64, i64, p, p, i32, i32, i32, i32,
                                                p, i64, p, i64, p, sz, p]
    lib.dsa_select_candidate_blocks_sharded.argtypes = [p, i32, i64, i64, i64, i64, p, i32, i32,
                                                        i32, i32, p, i64, p, i64, p, sz, p]
    lib.dsa_mask_candidate_logits.argtypes = [p, i64, i64, i64, p, p, p, i32, i64, i32, i32, p]
    lib.dsa_mask_candidate_logits_sharded.argtypes = [p, i32, i64, i64, i64, i64, p, i32, i32, p,
                                                      i32, i64, p]
    lib.dsa_mapped_host_pointer.argtypes = [p, ctypes.POINTER(ctypes.c_void_p)]
    lib.dsa_mapped_host_pointer.restype = ctypes.c_int
    lib.dsa_attn_max_shards.argtypes = []
    lib.dsa_attn_max_shards.restype = i32
    lib.dsa_correct_attn_out.argtypes = [p, i32, i64, i64, i64, i64, i64, i64, p, i32, i64, i64,
                                         i64, i32, p, i64, i64, i64, p, i64, i64, p]
    lib.dsa_merge_attn_out.argtypes = [p, i32, i32, i64, i64, i64, i64, i64, i64, i64, p, i64,
                                       i64, i64, p, i64, i64, i64, p, i64, i64, p]
    lib.dsa_select_candidate_blocks_sharded_starts.argtypes = [
        p, i32, i64, i64, i64, i64, p, p, i32, i32, i32, i32, p, i64, p, i64, p, sz, p]
    lib.dsa_mask_candidate_logits_sharded_starts.argtypes = [p, i32, i64, i64, i64, i64, p, p,
                                                             i32, i32, p, i32, i64, p]
    for name in ("dsa_block_scores", "dsa_select_candidate_blocks",
                 "dsa_select_candidate_blocks_sharded", "dsa_mask_candidate_logits",
                 "dsa_mask_candidate_logits_sharded", "dsa_select_candidate_blocks_sharded_starts",
                 "dsa_mask_candidate_logits_sharded_starts"):
        getattr(lib, name + "_bf16").argtypes = getattr(lib, name).argtypes
    for f in (lib.dsa_block_scores, lib.dsa_select_candidate_blocks,
              lib.dsa_select_candidate_blocks_sharded, lib.dsa_mask_candidate_logits,
              lib.dsa_mask_candidate_logits_sharded, lib.dsa_correct_attn_out,
              lib.dsa_merge_attn_out, lib.dsa_block_scores_bf16,
              lib.dsa_select_candidate_blocks_bf16, lib.dsa_select_candidate_blocks_sharded_bf16,
              lib.dsa_mask_candidate_logits_bf16, lib.dsa_mask_candidate_logits_sharded_bf16,
              lib.dsa_select_candidate_blocks_sharded_starts,
              lib.dsa_select_candidate_blocks_sharded_starts_bf16,
              lib.dsa_mask_candidate_logits_sharded_starts,
              lib.dsa_mask_candidate_logits_sharded_starts_bf16):
        f.restype = ctypes.c_int
    _lib = lib
    return lib


def set_launch_override(knob: str, value: int) -> None:
    """Pin one launch-shape choice of the selecting calls for this process
    (value 0 hands it back to the launcher); for tests and tuning sweeps."""
    _check("dsa_select_set_launch_override",
           library().dsa_select_set_launch_override(LAUNCH_KNOBS[knob], int(value)))


def pipeline_error(clear: bool = False) -> int:
    """The pipelined kernels' give-up flag (0: none of their waits ever gave
    up); see dsa_pipeline_error."""
    return int(library().dsa_pipeline_error(1 if clear else 0))


def _check(fn: str, status: int):
    if status != 0:
        raise DsaError(fn, status, library().dsa_status_string(status).decode())


def max_select_blocks() -> int:
    return int(library().dsa_select_max_blocks())


def _torch():
    import torch
    return torch


def workspace_bytes(rows: int, nblocks: int) -> int:
    """Bytes of workspace that let a selecting call split rows over CTAs."""
    return int(library().dsa_select_workspace_bytes(rows, nblocks))


_ws_cache = {}


def _workspace(workspace, rows: int, nblocks: int, device, stream_handle):
    """(pointer, bytes) of the workspace for one call.

    ``workspace`` may be a CUDA tensor (zero-filled before its first use,
    written by nothing but these calls, and not shared by calls that can
    overlap), ``False`` (no workspace: one CTA per row) or ``None``: a
    zero-filled workspace cached per (device, stream) and grown when a call
    needs more."""
    torch = _torch()
    if workspace is False:
        return None, 0
    if workspace is not None:
        if not workspace.is_cuda:
            raise ValueError("workspace must be a CUDA tensor")
        return workspace.data_ptr(), workspace.numel() * workspace.element_size()
    need = workspace_bytes(rows, nblocks)
    key = (device.index if device.index is not None else torch.cuda.current_device(),
           stream_handle)
    buf = _ws_cache.get(key)
    if buf is None or buf.numel() < need:
        buf = torch.zeros(need, dtype=torch.uint8, device=device)
        _ws_cache[key] = buf
    return buf.data_ptr(), buf.numel()


def _stream_handle(stream) -> Optional[int]:
    torch = _torch()
    s = torch.cuda.current_stream() if stream is None else stream
    return s.cuda_stream or None


def mapped_host_pointer(t) -> int:
    """Device address of a pinned (page-locked) host tensor's data, under
    which kernels read and write it in place (``dsa_mapped_host_pointer``)."""
    if t.is_cuda or not t.is_pinned():
        raise ValueError("expected a pinned host tensor")
    dev = ctypes.c_void_p()
    _check("dsa_mapped_host_pointer", library().dsa_mapped_host_pointer(t.data_ptr(),
                                                                         ctypes.byref(dev)))
    return dev.value


def _dev_ptr(t, dtype, name, *, allow_none=False):
    """Device address of a CUDA tensor, or of a pinned host tensor (read and
    written in place across the host link)."""
    if t is None:
        if allow_none:
            return None
        raise ValueError(f"{name} is required")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        if not t.is_pinned():
            raise ValueError(f"{name} must be a CUDA tensor or a pinned host tensor")
        return (mapped_host_pointer(t) if t.numel() else None) or None
    return t.data_ptr() or None


def _empty_beside(shape, dtype, t):
    """An output tensor where input ``t`` lives: on its CUDA device, or in
    pinned host memory for a host input."""
    torch = _torch()
    if t.is_cuda:
        return torch.empty(shape, dtype=dtype, device=t.device)
    return torch.empty(shape, dtype=dtype, pin_memory=True)


def _cuda_device(t):
    """The device a call on tensor ``t`` runs on: its own, or the current
    CUDA device for a pinned host tensor."""
    torch = _torch()
    return t.device if t.is_cuda else torch.device("cuda", torch.cuda.current_device())


def _logits_kind(t, name="logits"):
    """(dtype, C-ABI name suffix) of a logits tensor: fp32 or bf16."""
    torch = _torch()
    if t.dtype == torch.float32:
        return torch.float32, ""
    if t.dtype == torch.bfloat16:
        return torch.bfloat16, "_bf16"
    raise TypeError(f"{name} must be float32 or bfloat16, got {t.dtype}")


def _row_major(t, name):
    if t.stride(-1) != 1:
        raise ValueError(f"{name} must have unit stride in its last dimension")
    return t.stride(-2) if t.dim() >= 2 else t.shape[-1]


def dsa_block_scores(logits, row_ks, row_ke, block_size: int, row_repeat: int = 1,
                     pin_newest: bool = True, scores_out=None, stream=None):
    """Block scores ``[rows, ceil(width / block_size)]`` in the logits' dtype
    (fp32 or bf16; returned)."""
    torch = _torch()
    dt, sfx = _logits_kind(logits)
    rows, width = logits.shape
    nb = -(-width // block_size) if block_size > 0 else 0
    if scores_out is None:
        scores_out = _empty_beside((rows, nb), dt, logits)
    st = getattr(library(), "dsa_block_scores" + sfx)(
        _dev_ptr(logits, dt, "logits"), rows, width, _row_major(logits, "logits"),
        _dev_ptr(row_ks, torch.int32, "row_ks", allow_none=True),
        _dev_ptr(row_ke, torch.int32, "row_ke"), block_size, row_repeat, int(bool(pin_newest)),
        _dev_ptr(scores_out, dt, "scores_out"),
        _row_major(scores_out, "scores_out") if scores_out.numel() else nb,
        _stream_handle(stream))
    _check("dsa_block_scores" + sfx, st)
    return scores_out


def dsa_select_candidate_blocks(logits, row_ks, row_ke, topk_blocks: int, block_size: int,
                                out, row_repeat: int = 1, pin_newest: bool = True,
                                scores_out=None, stream=None, workspace=None):
    """Write ranked candidate block ids (-1 padded) into ``out`` [rows, >=topk]
    int32; optionally the block scores into ``scores_out`` (the logits'
    dtype). Logits are fp32 or bf16. ``workspace``: see ``_workspace``."""
    torch = _torch()
    dt, sfx = _logits_kind(logits)
    rows, width = logits.shape
    nb = -(-width // block_size) if block_size > 0 else 0
    handle = _stream_handle(stream)
    ws_ptr, ws_bytes = _workspace(workspace, rows, nb, _cuda_device(logits), handle)
    st = getattr(library(), "dsa_select_candidate_blocks" + sfx)(
        _dev_ptr(logits, dt, "logits"), rows, width, _row_major(logits, "logits"),
        _dev_ptr(row_ks, torch.int32, "row_ks", allow_none=True),
        _dev_ptr(row_ke, torch.int32, "row_ke"), topk_blocks, block_size, row_repeat,
        int(bool(pin_newest)), _dev_ptr(out, torch.int32, "out"),
        _row_major(out, "out") if out.dim() == 2 else topk_blocks,
        _dev_ptr(scores_out, dt, "scores_out", allow_none=True),
        _row_major(scores_out, "scores_out") if scores_out is not None else 0,
        ws_ptr, ws_bytes, handle)
    _check("dsa_select_candidate_blocks" + sfx, st)
    return out


def dsa_select_candidate_blocks_sharded(logits, global_row_ke, global_block_size: int,
                                        max_global_blocks: int, topk_blocks: int, out,
                                        row_repeat: int = 1, scores_out=None, stream=None,
                                        workspace=None, global_row_ks=None):
    """DCP form: ``logits`` is ``[D, rows, local_width]`` (unit stride in the last
    dimension); writes ranked global block ids into ``out``. ``global_row_ks``
    (optional) gives global window starts (the ``_starts`` C entry point).
    ``workspace``: see ``_workspace``."""
    torch = _torch()
    dt, sfx = _logits_kind(logits)
    shards, rows, lw = logits.shape
    handle = _stream_handle(stream)
    ws_ptr, ws_bytes = _workspace(workspace, rows, max(int(max_global_blocks), 1),
                                  _cuda_device(logits), handle)
    if logits.stride(2) != 1:
        raise ValueError("logits must have unit stride in its last dimension")
    name = "dsa_select_candidate_blocks_sharded" + ("_starts" if global_row_ks is not None
                                                    else "") + sfx
    starts = (_dev_ptr(global_row_ks, torch.int32, "global_row_ks"),) \
        if global_row_ks is not None else ()
    st = getattr(library(), name)(
        _dev_ptr(logits, dt, "logits"), shards, rows, lw, logits.stride(1),
        logits.stride(0), *starts, _dev_ptr(global_row_ke, torch.int32, "global_row_ke"),
        global_block_size, max_global_blocks, row_repeat, topk_blocks,
        _dev_ptr(out, torch.int32, "out"), _row_major(out, "out") if out.dim() == 2 else topk_blocks,
        _dev_ptr(scores_out, dt, "scores_out", allow_none=True),
        _row_major(scores_out, "scores_out") if scores_out is not None else 0,
        ws_ptr, ws_bytes, handle)
    _check(name, st)
    return out


def dsa_mask_candidate_logits(logits, row_ks, row_ke, candidates, block_size: int,
                              row_repeat: int = 1, stream=None):
    """In place: -inf for every logit outside its row's window or outside the
    row's candidate blocks (``candidates`` [rows, topk] int32, -1 = empty)."""
    torch = _torch()
    dt, sfx = _logits_kind(logits)
    rows, width = logits.shape
    topk = candidates.shape[1] if candidates is not None else 0
    st = getattr(library(), "dsa_mask_candidate_logits" + sfx)(
        _dev_ptr(logits, dt, "logits"), rows, width, _row_major(logits, "logits"),
        _dev_ptr(row_ks, torch.int32, "row_ks", allow_none=True),
        _dev_ptr(row_ke, torch.int32, "row_ke"),
        _dev_ptr(candidates, torch.int32, "candidates", allow_none=True), topk,
        _row_major(candidates, "candidates") if candidates is not None else 0, block_size,
        row_repeat, _stream_handle(stream))
    _check("dsa_mask_candidate_logits" + sfx, st)
    return logits


def dsa_mask_candidate_logits_sharded(logits, global_row_ke, global_block_size: int, candidates,
                                      row_repeat: int = 1, stream=None, global_row_ks=None):
    """DCP form of ``dsa_mask_candidate_logits`` on ``[D, rows, local_width]``;
    ``global_row_ks`` (optional) gives global window starts."""
    torch = _torch()
    dt, sfx = _logits_kind(logits)
    shards, rows, lw = logits.shape
    if logits.stride(2) != 1:
        raise ValueError("logits must have unit stride in its last dimension")
    topk = candidates.shape[1] if candidates is not None else 0
    name = "dsa_mask_candidate_logits_sharded" + ("_starts" if global_row_ks is not None
                                                  else "") + sfx
    starts = (_dev_ptr(global_row_ks, torch.int32, "global_row_ks"),) \
        if global_row_ks is not None else ()
    st = getattr(library(), name)(
        _dev_ptr(logits, dt, "logits"), shards, rows, lw, logits.stride(1),
        logits.stride(0), *starts, _dev_ptr(global_row_ke, torch.int32, "global_row_ke"),
        global_block_size, row_repeat,
        _dev_ptr(candidates, torch.int32, "candidates", allow_none=True), topk,
        _row_major(candidates, "candidates") if candidates is not None else 0,
        _stream_handle(stream))
    _check(name, st)
    return logits


DTYPE_F32, DTYPE_BF16 = 0, 1


def _attn_dtype(t, name):
    torch = _torch()
    if t.dtype == torch.float32:
        return DTYPE_F32
    if t.dtype == torch.bfloat16:
        return DTYPE_BF16
    raise TypeError(f"{name} must be float32 or bfloat16, got {t.dtype}")


def _attn_ptr(t, name, dtype_code):
    torch = _torch()
    want = torch.float32 if dtype_code == DTYPE_F32 else torch.bfloat16
    return _dev_ptr(t, want, name)


def dsa_correct_attn_out(out, lses, rank: int, new_out=None, lse_out=None, stream=None):
    """DCP LSE correction of shard ``rank``'s partial attention output.

    ``out`` [B, H, Dh] (or [B, 1, H, Dh]) fp32 or bf16; ``lses`` [N, B, H]
    fp32 base-2 LSEs of all shards (a trailing or second size-1 dimension is
    squeezed, as on the page). Writes ``new_out`` [H, B, Dh] (allocated when
    None, same dtype as ``out``) and the combined LSE ``lse_out`` [B, H]
    fp32 (allocated when None); returns both."""
    torch = _torch()
    if out.dim() == 4 and out.shape[1] == 1:
        out = out.squeeze(1)
    if lses.dim() == 4 and lses.shape[-1] == 1:
        lses = lses.squeeze(-1)
    if lses.dim() == 4 and lses.shape[1] == 1:
        lses = lses.squeeze(1)
    if out.dim() != 3 or lses.dim() != 3:
        raise ValueError("expected out [B, H, Dh] and lses [N, B, H]")
    B, H, D = out.shape
    N = lses.shape[0]
    if tuple(lses.shape[1:]) != (B, H):
        raise ValueError(f"lses {tuple(lses.shape)} does not match out {tuple(out.shape)}")
    code = _attn_dtype(out, "out")
    if new_out is None:
        new_out = _empty_beside((H, B, D), out.dtype, out)
    if lse_out is None:
        lse_out = _empty_beside((B, H), torch.float32, out)
    if tuple(new_out.shape) != (H, B, D) or tuple(lse_out.shape) != (B, H):
        raise ValueError("new_out must be [H, B, Dh] and lse_out [B, H]")
    st = library().dsa_correct_attn_out(
        _attn_ptr(out, "out", code), code, B, H, D, *out.stride(),
        _dev_ptr(lses, torch.float32, "lses"), N, *lses.stride(), rank,
        _attn_ptr(new_out, "new_out", code), *new_out.stride(),
        _dev_ptr(lse_out, torch.float32, "lse_out"), *lse_out.stride(), _stream_handle(stream))
    _check("dsa_correct_attn_out", st)
    return new_out, lse_out


def dsa_merge_attn_out(outs, lses, merged=None, lse_out=None, stream=None):
    """Sum over shards of the corrected partial outputs.

    ``outs`` [N, B, H, Dh] fp32 or bf16, ``lses`` [N, B, H] fp32. Writes
    ``merged`` [H, B, Dh] (same dtype as ``outs``) and ``lse_out`` [B, H]
    fp32, allocating them when None; returns both."""
    torch = _torch()
    if outs.dim() != 4 or lses.dim() != 3:
        raise ValueError("expected outs [N, B, H, Dh] and lses [N, B, H]")
    N, B, H, D = outs.shape
    if tuple(lses.shape) != (N, B, H):
        raise ValueError(f"lses {tuple(lses.shape)} does not match outs {tuple(outs.shape)}")
    code = _attn_dtype(outs, "outs")
    if merged is None:
        merged = _empty_beside((H, B, D), outs.dtype, outs)
    if lse_out is None:
        lse_out = _empty_beside((B, H), torch.float32, outs)
    if tuple(merged.shape) != (H, B, D) or tuple(lse_out.shape) != (B, H):
        raise ValueError("merged must be [H, B, Dh] and lse_out [B, H]")
    st = library().dsa_merge_attn_out(
        _attn_ptr(outs, "outs", code), code, N, B, H, D, *outs.stride(),
        _dev_ptr(lses, torch.float32, "lses"), *lses.stride(),
        _attn_ptr(merged, "merged", code), *merged.stride(),
        _dev_ptr(lse_out, torch.float32, "lse_out"), *lse_out.stride(), _stream_handle(stream))
    _check("dsa_merge_attn_out", st)
    return merged, lse_out


def _to_device(host, dev_buf, stream):
    torch = _torch()
    if host is None:
        return None
    if dev_buf is None:
        dev_buf = torch.empty(host.shape, dtype=host.dtype, device="cuda")
    with torch.cuda.stream(stream):
        dev_buf.copy_(host, non_blocking=True)
    return dev_buf


def _all_pinned(*ts) -> bool:
    return all(t is None or (not t.is_cuda and t.is_pinned()) for t in ts)


def select_candidate_blocks_host(logits, row_ks, row_ke, topk_blocks: int, block_size: int,
                                 row_repeat: int = 1, pin_newest: bool = True, *,
                                 out=None, device_buffers: Optional[dict] = None, stream=None,
                                 in_place: bool = True):
    """Host-memory form of ``dsa_select_candidate_blocks``; waits for the
    result and returns the ids in host tensor ``out`` (pinned; allocated when
    None).

    Pinned inputs are read in place (unless ``in_place`` is False): the
    kernel reads only the in-window logits across the host link and writes
    the ids straight into ``out``. Other host tensors are first copied to the
    device whole; ``device_buffers``
    may then hold preallocated device tensors under 'logits', 'row_ks',
    'row_ke', 'out' so that repeated calls allocate nothing. A device
    tensor under 'workspace' is passed on as the call's workspace."""
    torch = _torch()
    stream = torch.cuda.current_stream() if stream is None else stream
    db = device_buffers if device_buffers is not None else {}
    rows = logits.shape[0]
    if out is None:
        out = torch.empty((rows, topk_blocks), dtype=torch.int32, pin_memory=True)
    if in_place and _all_pinned(logits, row_ks, row_ke, out):
        dsa_select_candidate_blocks(logits, row_ks, row_ke, topk_blocks, block_size, out,
                                    row_repeat, pin_newest, stream=stream,
                                    workspace=db.get("workspace"))
        stream.synchronize()
        return out
    d_logits = _to_device(logits, db.get("logits"), stream)
    d_ks = _to_device(row_ks, db.get("row_ks"), stream)
    d_ke = _to_device(row_ke, db.get("row_ke"), stream)
    d_out = db.get("out")
    if d_out is None:
        d_out = torch.empty((rows, topk_blocks), dtype=torch.int32, device="cuda")
    dsa_select_candidate_blocks(d_logits, d_ks, d_ke, topk_blocks, block_size, d_out,
                                row_repeat, pin_newest, stream=stream,
                                workspace=db.get("workspace"))
    with torch.cuda.stream(stream):
        out.copy_(d_out, non_blocking=True)
    stream.synchronize()
    return out


def select_candidate_blocks_sharded_host(logits, global_row_ke, global_block_size: int,
                                         max_global_blocks: int, topk_blocks: int,
                                         row_repeat: int = 1, *, out=None,
                                         device_buffers: Optional[dict] = None, stream=None,
                                         global_row_ks=None, in_place: bool = True):
    """Host-memory form of ``dsa_select_candidate_blocks_sharded`` (see
    ``select_candidate_blocks_host``: pinned inputs are read in place;
    ``device_buffers`` may also hold 'global_row_ke' and 'global_row_ks')."""
    torch = _torch()
    stream = torch.cuda.current_stream() if stream is None else stream
    db = device_buffers if device_buffers is not None else {}
    rows = logits.shape[1]
    if out is None:
        out = torch.empty((rows, topk_blocks), dtype=torch.int32, pin_memory=True)
    if in_place and _all_pinned(logits, global_row_ke, global_row_ks, out):
        dsa_select_candidate_blocks_sharded(logits, global_row_ke, global_block_size,
                                            max_global_blocks, topk_blocks, out, row_repeat,
                                            stream=stream, workspace=db.get("workspace"),
                                            global_row_ks=global_row_ks)
        stream.synchronize()
        return out
    d_logits = _to_device(logits, db.get("logits"), stream)
    d_gke = _to_device(global_row_ke, db.get("global_row_ke"), stream)
    d_gks = _to_device(global_row_ks, db.get("global_row_ks"), stream)
    d_out = db.get("out")
    if d_out is None:
        d_out = torch.empty((rows, topk_blocks), dtype=torch.int32, device="cuda")
    dsa_select_candidate_blocks_sharded(d_logits, d_gke, global_block_size, max_global_blocks,
                                        topk_blocks, d_out, row_repeat, stream=stream,
                                        global_row_ks=d_gks, workspace=db.get("workspace"))
    with torch.cuda.stream(stream):
        out.copy_(d_out, non_blocking=True)
    stream.synchronize()
    return out
