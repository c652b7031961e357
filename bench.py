#!/usr/bin/env python3
"""Throughput of DSA candidate-block selection on GB300.

One step = one call of the selection over one batch of synthetic rows with
the inputs resident in HBM. The default workload is the simulated DCP layout
(8 interleave-1 shards of a [4096, 65536] fp32 indexer-logit matrix, global
block 64, 1024 global blocks, top-32): the largest configuration, and the
one whose call covers every step of the path (window, block max, shard
merge, pin, top-k, -1 store).

Metric: algorithmic logits GB/s = (in-window logit bytes + bound bytes read +
id bytes written) / time, with rows/s beside it. Window bytes only: the
columns outside each row's window are never read and are not counted.

    python bench.py [--gpus N] [--steps K] [--warmup W] [--workload NAME]
                    [--impl reference] [--op select|mask]

--op mask times the masking pass that follows selection instead: one step
sets every logit outside the selected candidate blocks (or outside the
window) to -inf, in place; its bytes are the -inf stores plus the bounds and
ids read.

Prints one JSON line on rank 0. For N > 1 launch one process per GPU with
torch.distributed.run; every rank runs the same workload on its own GPU
(weak scaling, no data-path collective) and the slowest rank's time counts.
"""

from __future__ import annotations

import argparse
import csv
import hashlib
import io
import json
import os
import re
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
if ROOT not in sys.path:
    sys.path.insert(0, ROOT)

METRIC = "candidate-select logits GB/s (% of GB300 HBM peak) and rows/s"
MASK_METRIC = "candidate-mask -inf write GB/s (% of GB300 HBM peak) and rows/s"
LSE_METRICS = {
    "correct": "DCP LSE-correction GB/s (% of GB300 HBM peak) and (token, head) rows/s",
    "merge": "DCP LSE-merge GB/s (% of GB300 HBM peak) and (token, head) rows/s",
}
LSE_OPS = tuple(LSE_METRICS)
LSE_NAMES = ("lse_decode", "lse_decode_bf16", "lse_tiny")
UNIT = "GB/s"
L2_BYTES = 129 * 1000 * 1000
FALLBACK_HBM_GBS = 6800.0
_CSRC = "deepseek_sparse_attention_row_gb300/csrc/"
# The sources each timed kernel is built from; a committed traffic figure
# counts only while their hash still matches.
KERNEL_SOURCES = {
    "select": tuple(_CSRC + f for f in ("dsa_cb.cu", "stream.cuh", "topk.cuh", "topk_warp.cuh",
                                        "keys.cuh", "select_pipe.cu", "select_pipe.h",
                                        "pipe.cuh")),
    "mask": tuple(_CSRC + f for f in ("mask.cu", "keys.cuh")),
    "correct": (_CSRC + "dcp_lse.cu",),
    "merge": (_CSRC + "dcp_lse.cu",),
}


# ---------------------------------------------------------------------------
# Workload bookkeeping (host only)
# ---------------------------------------------------------------------------

def window_elements(wl) -> int:
    """Number of in-window logits the selection must read."""
    import numpy as np

    if hasattr(wl, "global_row_ke"):
        rows = wl.rows
        g = np.repeat(wl.global_row_ke.astype(np.int64), wl.row_repeat)[:rows]
        ks = getattr(wl, "global_row_ks", None)
        gs = (np.zeros(rows, np.int64) if ks is None else
              np.minimum(np.maximum(np.repeat(ks.astype(np.int64), wl.row_repeat)[:rows], 0),
                         np.maximum(g, 0)))
        # shard d reads columns [ceil((gs - d) / D), ceil((gke - d) / D)), clamped to lw
        total = 0
        D = wl.shards
        for d in range(D):
            lke = np.minimum(np.where(g > d, (g - d + D - 1) // D, 0), wl.local_width)
            lks = np.minimum(np.where(gs > d, (gs - d + D - 1) // D, 0), lke)
            total += int((lke - lks).sum())
        return total
    rows, width = wl.rows, wl.width
    ke = np.repeat(wl.row_ke.astype(np.int64), wl.row_repeat)[:rows]
    ks = (np.zeros(rows, np.int64) if wl.row_ks is None
          else np.repeat(wl.row_ks.astype(np.int64), wl.row_repeat)[:rows])
    e = np.minimum(ke, width)
    s = np.minimum(np.maximum(ks, 0), e)
    return int((e - s).sum())


def esize(wl) -> int:
    """Bytes per logit: 2 for the bf16 workloads, else 4."""
    return 2 if getattr(wl, "dtype", "f32") == "bf16" else 4


def algorithmic_bytes(wl) -> int:
    """Bytes one call must move: in-window logits (fp32 or bf16), the int32
    bounds it reads, the int32 ids it writes."""
    bounds = (wl.global_row_ke.size + (0 if getattr(wl, "global_row_ks", None) is None
                                       else wl.global_row_ks.size)
              if hasattr(wl, "global_row_ke") else
              wl.row_ke.size + (0 if wl.row_ks is None else wl.row_ks.size))
    return esize(wl) * window_elements(wl) + 4 * bounds + 4 * wl.rows * wl.topk_blocks


def workload_config(wl, name: str) -> dict:
    if hasattr(wl, "global_row_ke"):
        cfg = {"workload": f"dcp-sim D={wl.shards} [{wl.shards},{wl.rows},{wl.local_width}] "
                           f"{'bf16' if esize(wl) == 2 else 'fp32'}",
               "shards": wl.shards, "rows": wl.rows, "local_width": wl.local_width,
               "global_width": wl.shards * wl.local_width,
               "global_block_size": wl.global_block_size,
               "max_global_blocks": wl.max_global_blocks}
    else:
        cfg = {"workload": f"{name} [{wl.rows},{wl.width}] {'bf16' if esize(wl) == 2 else 'fp32'}",
               "rows": wl.rows,
               "width": wl.width, "block_size": wl.block_size,
               "pin_newest": bool(wl.pin_newest), "starts": wl.row_ks is not None}
    cfg.update({"topk_blocks": wl.topk_blocks, "row_repeat": wl.row_repeat, "seed": wl.seed,
                "window_bytes": esize(wl) * window_elements(wl)})
    if wl.notes:
        cfg["notes"] = wl.notes
    return cfg


def selection_kernel(wl, sms: int = 152) -> str:
    """The selecting kernel the library's default launch choice takes for a
    workload (the rule of select_impl / pipe_takes, restated for the report):
    the DCP forms stay on select_kernel; unsharded rows go to the pipelined
    kernels, one row per warp for many short rows with top-k <= 32."""
    if hasattr(wl, "global_row_ke"):
        return "select_kernel (row per CTA, one launch per step)"
    nb = -(-wl.width // wl.block_size)
    solo = (wl.topk_blocks <= 32 and nb <= 2048 and wl.width * esize(wl) <= 64 * 1024
            and wl.rows >= 8 * sms)
    return ("pipe_solo_kernel (bulk-copy staged, one row per warp, one launch per step)" if solo
            else "pipe_coop_kernel (bulk-copy staged, warps of a CTA on one row, one launch "
                 "per step)")


def measured_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(path) as f:
            v = float(json.load(f)["hbm_gbs"])
        return v, "measured"
    except (OSError, KeyError, ValueError):
        return FALLBACK_HBM_GBS, "fallback"


def code_only(text: str) -> str:
    """C / CUDA source without its comments and blank lines, each line
    stripped: what decides the compiled kernel (no string literal in the
    kernel sources holds a comment marker)."""
    text = re.sub(r"/\*.*?\*/", " ", text, flags=re.S)
    text = re.sub(r"//[^\n]*", "", text)
    return "\n".join(line.strip() for line in text.splitlines() if line.strip())


def kernel_source_hash(op: str = "select") -> str:
    """Hash of the code (comments and blank lines removed) of the sources the
    op's kernel is built from: a committed traffic figure stays valid across
    comment edits and lapses with any change to the code."""
    h = hashlib.sha256()
    for rel in KERNEL_SOURCES[op]:
        with open(os.path.join(ROOT, rel), encoding="utf-8") as f:
            h.update(code_only(f.read()).encode())
    return h.hexdigest()[:16]


def profiled_traffic(op: str, workload: str):
    """Per-launch DRAM bytes of the op's kernel on this workload from the
    committed ncu summary, if it was taken on the current kernel sources;
    else None."""
    path = os.path.join(ROOT, "profiles", "traffic.json")
    try:
        with open(path) as f:
            rec = json.load(f).get(f"{op}/{workload}")
    except (OSError, ValueError):
        return None
    if not rec or rec.get("kernel_sources") != kernel_source_hash(op):
        return None
    return rec.get("dram_bytes_per_launch")


# ---------------------------------------------------------------------------
# Multi-rank plumbing (also exercised on CPU with gloo by the tests)
# ---------------------------------------------------------------------------

def dist_env():
    return (int(os.environ.get("RANK", "0")), int(os.environ.get("WORLD_SIZE", "1")),
            int(os.environ.get("LOCAL_RANK", "0")))


def dist_barrier(world: int):
    if world > 1:
        import torch.distributed as dist

        dist.barrier()


def dist_max(value: float, world: int, device=None) -> float:
    if world == 1:
        return value
    import torch
    import torch.distributed as dist

    t = torch.tensor([value], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


def whole_job_rate(units_per_rank: float, world: int, max_seconds: float) -> float:
    """Every rank processes the same units; the slowest rank's time counts."""
    return units_per_rank * world / max_seconds


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------

CLOCK_QUERY = ("index,uuid,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
               "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
               "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")
REASONS = ("hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap")


class ClockSampler:
    """nvidia-smi sampling of SM clocks and throttle reasons (read only)."""

    def __init__(self, uuid: str, period_ms: int = 100):
        self.cmd = ["nvidia-smi", f"--query-gpu={CLOCK_QUERY}", "--format=csv,noheader,nounits",
                    f"-lms={period_ms}"]
        self.uuid = uuid.lower().replace("gpu-", "")
        self.proc = None
        self.text = ""

    def __enter__(self):
        try:
            self.proc = subprocess.Popen(self.cmd, stdout=subprocess.PIPE,
                                         stderr=subprocess.DEVNULL, text=True)
            time.sleep(0.3)
        except OSError:
            self.proc = None
        return self

    def __exit__(self, *exc):
        self.text = ""
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.text, _ = self.proc.communicate(timeout=5)
            except subprocess.TimeoutExpired:
                self.proc.kill()
                self.text, _ = self.proc.communicate()
        return False

    def summary(self):
        rows = [[c.strip() for c in r] for r in csv.reader(io.StringIO(self.text)) if len(r) >= 10]
        mine = [r for r in rows if self.uuid and self.uuid in r[1].lower()]
        if not mine and len({r[0] for r in rows}) == 1:
            mine = rows
        sm, mx, reasons = [], [], set()
        for r in mine:
            try:
                sm.append(float(r[2]))
                mx.append(float(r[3]))
            except ValueError:
                continue
            for name, val in zip(REASONS, r[6:10]):
                if val.strip().lower() == "active":
                    reasons.add(name)
        if not sm:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": [], "samples": 0}
        return {"sm_mhz": statistics.median(sm), "sm_max_mhz": max(mx),
                "reasons": sorted(reasons), "samples": len(sm)}


# ---------------------------------------------------------------------------
# Our arm
# ---------------------------------------------------------------------------

def device_logits(wl, torch, device):
    """The workload's logits on the device, as fp32 or (for the bf16
    workloads, whose values lie on the bf16 grid) bf16."""
    t = torch.from_numpy(wl.logits).to(device)
    return t.to(torch.bfloat16) if esize(wl) == 2 else t


def make_runner(wl, dsa, torch, device, copies: int = 1):
    """Device-resident inputs, an explicit workspace (so that graph capture
    allocates nothing) and one-call step functions. With copies = 2 the
    logits are held twice and the two steps read different copies, so that a
    step never finds the previous step's lines in L2."""
    out = torch.empty((wl.rows, wl.topk_blocks), dtype=torch.int32, device=device)
    if hasattr(wl, "global_row_ke"):
        gke = torch.from_numpy(wl.global_row_ke).to(device)
        ws = torch.zeros(dsa.workspace_bytes(wl.rows, max(wl.max_global_blocks, 1)),
                         dtype=torch.uint8, device=device)
        gks = (None if getattr(wl, "global_row_ks", None) is None
               else torch.from_numpy(wl.global_row_ks).to(device))

        def make_step(logits):
            def step():
                dsa.dsa_select_candidate_blocks_sharded(logits, gke, wl.global_block_size,
                                                        wl.max_global_blocks, wl.topk_blocks,
                                                        out, wl.row_repeat, workspace=ws,
                                                        global_row_ks=gks)
            return step
    else:
        ks = None if wl.row_ks is None else torch.from_numpy(wl.row_ks).to(device)
        ke = torch.from_numpy(wl.row_ke).to(device)
        ws = torch.zeros(dsa.workspace_bytes(wl.rows, -(-wl.width // wl.block_size)),
                         dtype=torch.uint8, device=device)

        def make_step(logits):
            def step():
                dsa.dsa_select_candidate_blocks(logits, ks, ke, wl.topk_blocks, wl.block_size,
                                                out, wl.row_repeat, wl.pin_newest, workspace=ws)
            return step
    first = device_logits(wl, torch, device)
    steps = [make_step(first)] + [make_step(first.clone()) for _ in range(copies - 1)]
    if copies == 1:
        return steps[0], out
    return steps, out


def mask_written_elements(wl, ids) -> int:
    """Logits the masking pass sets to -inf: every column of every (shard)
    row minus the columns of selected blocks inside the window."""
    import numpy as np

    if hasattr(wl, "global_row_ke"):
        D, rows, lw = wl.logits.shape
        lbs = wl.global_block_size // D
        g = np.repeat(wl.global_row_ke.astype(np.int64), wl.row_repeat)[:rows]
        ks = getattr(wl, "global_row_ks", None)
        gs = (np.zeros(rows, np.int64) if ks is None else
              np.minimum(np.maximum(np.repeat(ks.astype(np.int64), wl.row_repeat)[:rows], 0),
                         np.maximum(g, 0)))
        kept = 0
        for d in range(D):
            e = np.minimum(np.where(g > d, (g - d + D - 1) // D, 0), lw)
            st = np.minimum(np.where(gs > d, (gs - d + D - 1) // D, 0), e)
            for j in range(ids.shape[1]):
                b = ids[:, j].astype(np.int64)
                lo = st + b * lbs
                kept += int(np.where(b >= 0, np.clip(np.minimum(lo + lbs, e) - lo, 0, None),
                                     0).sum())
        return D * rows * lw - kept
    rows, width, bs = wl.rows, wl.logits.shape[1], wl.block_size
    ke = np.repeat(wl.row_ke.astype(np.int64), wl.row_repeat)[:rows]
    ks = (np.zeros(rows, np.int64) if wl.row_ks is None
          else np.repeat(wl.row_ks.astype(np.int64), wl.row_repeat)[:rows])
    e = np.minimum(ke, width)
    s = np.minimum(np.maximum(ks, 0), e)
    kept = 0
    for j in range(ids.shape[1]):
        b = ids[:, j].astype(np.int64)
        lo = s + b * bs
        kept += int(np.where(b >= 0, np.clip(np.minimum(lo + bs, e) - lo, 0, None), 0).sum())
    return rows * width - kept


def make_mask_runner(wl, dsa, torch, device):
    """Device-resident logits and the ids the selection picks for them, and a
    one-call masking step (idempotent: it only writes -inf)."""
    step_sel, ids_dev = make_runner(wl, dsa, torch, device)
    step_sel()
    torch.cuda.synchronize()
    if hasattr(wl, "global_row_ke"):
        logits = device_logits(wl, torch, device)
        gke = torch.from_numpy(wl.global_row_ke).to(device)

        gks = (None if getattr(wl, "global_row_ks", None) is None
               else torch.from_numpy(wl.global_row_ks).to(device))

        def step():
            dsa.dsa_mask_candidate_logits_sharded(logits, gke, wl.global_block_size, ids_dev,
                                                  wl.row_repeat, global_row_ks=gks)
    else:
        logits = device_logits(wl, torch, device)
        ks = None if wl.row_ks is None else torch.from_numpy(wl.row_ks).to(device)
        ke = torch.from_numpy(wl.row_ke).to(device)

        def step():
            dsa.dsa_mask_candidate_logits(logits, ks, ke, ids_dev, wl.block_size, wl.row_repeat)
    ids = ids_dev.cpu().numpy()
    bounds = wl.global_row_ke.size if hasattr(wl, "global_row_ke") else (
        wl.row_ke.size + (0 if wl.row_ks is None else wl.row_ks.size))
    nbytes = esize(wl) * mask_written_elements(wl, ids) + 4 * bounds + 4 * ids.size
    return step, nbytes, ids


def lse_algorithmic_bytes(wl, op: str) -> int:
    """Bytes one LSE call must move: the partial output(s) read, the LSEs
    read, the corrected / merged output and the combined LSE written."""
    esize = 2 if wl.dtype == "bf16" else 4
    N, B, H, D = wl.outs.shape
    plane = B * H * D * esize
    reads = (N if op == "merge" else 1) * plane + 4 * N * B * H
    return reads + plane + 4 * B * H


def lse_workload_config(wl, name: str) -> dict:
    N, B, H, D = wl.outs.shape
    return {"workload": f"{name} N={N} [B={B}, H={H}, Dh={D}] {wl.dtype}", "shards": N,
            "batch": B, "heads": H, "head_dim": D, "dtype": wl.dtype, "seed": wl.seed,
            "notes": wl.notes}


def make_lse_runner(wl, op: str, dsa, torch, device):
    """Device-resident partial outputs and LSEs, preallocated results, and a
    one-call step."""
    tdt = torch.bfloat16 if wl.dtype == "bf16" else torch.float32
    N, B, H, D = wl.outs.shape
    lses = torch.from_numpy(wl.lses).to(device)
    lse_out = torch.empty((B, H), dtype=torch.float32, device=device)
    res = torch.empty((H, B, D), dtype=tdt, device=device)
    if op == "merge":
        outs = torch.from_numpy(wl.outs).to(device).to(tdt)

        def step():
            dsa.dsa_merge_attn_out(outs, lses, res, lse_out)
    else:
        out = torch.from_numpy(wl.outs[N // 2]).to(device).to(tdt)

        def step():
            dsa.dsa_correct_attn_out(out, lses, N // 2, res, lse_out)
    return step


def oracle_lse_baseline(wl, op: str, budget_s: float = 10.0):
    """The LSE oracle as it stands, single-threaded, over the whole workload."""
    import oracle

    oracle.build()
    N = wl.shards
    reps, t0 = 0, time.perf_counter()
    while True:
        if op == "merge":
            oracle.merge_attn_out(wl.outs, wl.lses)
        else:
            oracle.correct_attn_out(wl.outs[N // 2], wl.lses, N // 2)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 50:
            break
    return el / reps, reps


def graph_of(step, n: int, torch):
    """A CUDA graph of n consecutive steps (launch cost paid once per replay,
    not per step); ``step`` is one callable or a list taken in turn. Every
    step must have run once before, outside capture."""
    steps = step if isinstance(step, (list, tuple)) else [step]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(n):
            steps[i % len(steps)]()
    return g


def steps_per_graph(k: int) -> int:
    """Largest divisor of k up to 64: k steps are k / g replays of g steps."""
    return max(d for d in range(1, min(k, 64) + 1) if k % d == 0)


def e2e_measure(wl, dsa, torch, device, steps: int, flush=None):
    """Same metric through the host-buffer API, one call per step from pinned
    host inputs to the ids in pinned host memory, each step timed on its own
    (the call waits for its result). ``in_place`` (the headline): the kernel
    reads the in-window logits and the bounds across the host link and
    writes the ids straight into host memory. ``staged``: the whole logits
    tensor and the bounds are copied to the device first and the ids copied
    back. ``flush`` (a callable) runs untimed between steps when the bytes a
    step reads fit in L2."""
    sharded = hasattr(wl, "global_row_ke")
    h_logits = torch.from_numpy(wl.logits)
    if esize(wl) == 2:
        h_logits = h_logits.to(torch.bfloat16)  # values on the bf16 grid: exact
    h_logits = h_logits.pin_memory()
    h_out = torch.empty((wl.rows, wl.topk_blocks), dtype=torch.int32).pin_memory()
    bufs = {"logits": torch.empty(h_logits.shape, dtype=h_logits.dtype, device=device),
            "out": torch.empty((wl.rows, wl.topk_blocks), dtype=torch.int32, device=device)}
    if sharded:
        nb = max(wl.max_global_blocks, 1)
        h_b = [torch.from_numpy(wl.global_row_ke).pin_memory()]
        bufs["global_row_ke"] = torch.empty(h_b[0].shape, dtype=torch.int32, device=device)
        h_ks = None
        if getattr(wl, "global_row_ks", None) is not None:
            h_ks = torch.from_numpy(wl.global_row_ks).pin_memory()
            h_b.append(h_ks)
            bufs["global_row_ks"] = torch.empty(h_ks.shape, dtype=torch.int32, device=device)

        def call(in_place):
            dsa.select_candidate_blocks_sharded_host(h_logits, h_b[0], wl.global_block_size,
                                                     wl.max_global_blocks, wl.topk_blocks,
                                                     wl.row_repeat, out=h_out,
                                                     device_buffers=bufs, global_row_ks=h_ks,
                                                     in_place=in_place)
    else:
        nb = -(-wl.width // wl.block_size)
        h_b = [None if wl.row_ks is None else torch.from_numpy(wl.row_ks).pin_memory(),
               torch.from_numpy(wl.row_ke).pin_memory()]
        if h_b[0] is not None:
            bufs["row_ks"] = torch.empty(h_b[0].shape, dtype=torch.int32, device=device)
        bufs["row_ke"] = torch.empty(h_b[1].shape, dtype=torch.int32, device=device)

        def call(in_place):
            dsa.select_candidate_blocks_host(h_logits, h_b[0], h_b[1], wl.topk_blocks,
                                             wl.block_size, wl.row_repeat, wl.pin_newest,
                                             out=h_out, device_buffers=bufs, in_place=in_place)
    bufs["workspace"] = torch.zeros(dsa.workspace_bytes(wl.rows, nb), dtype=torch.uint8,
                                    device=device)
    bound_bytes = sum(b.numel() * 4 for b in h_b if b is not None)
    d2h = h_out.numel() * 4
    res = {}
    for in_place in (True, False):
        call(in_place)
        torch.cuda.synchronize()
        total = 0.0
        for _ in range(steps):
            if flush is not None:
                flush()
                torch.cuda.synchronize()
            t0 = time.perf_counter()
            call(in_place)
            total += time.perf_counter() - t0
        # in place: the bytes the kernel reads across the link; staged: the
        # tensors copied in
        h2d = (esize(wl) * window_elements(wl) if in_place else h_logits.numel() * esize(wl)) \
            + bound_bytes
        res["in_place" if in_place else "staged"] = (total / steps, h2d, d2h)
    return res


def oracle_cpu_baseline(wl, budget_s: float = 10.0):
    """The oracle as it stands, single-threaded on a host core, repeated over
    the whole workload until about budget_s seconds have passed."""
    import oracle

    oracle.build()
    run = oracle.run_workload_bf16 if esize(wl) == 2 else oracle.run_workload
    reps, t0 = 0, time.perf_counter()
    while True:
        run(wl, want_scores=False)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 50:
            break
    return el / reps, reps


def host_threads() -> int:
    """Host cores this process may run on."""
    try:
        return len(os.sched_getaffinity(0))
    except (AttributeError, OSError):
        return os.cpu_count() or 1


def oracle_cpu_baseline_threads(wl, budget_s: float = 10.0, threads: int = 0):
    """The same oracle function over ``threads`` contiguous row ranges on as
    many host threads (the C calls release the GIL), repeated over the whole
    workload until about budget_s seconds have passed; seconds per pass."""
    from concurrent.futures import ThreadPoolExecutor

    import oracle

    oracle.build()
    run = oracle.run_workload_bf16 if esize(wl) == 2 else oracle.run_workload
    threads = max(1, threads or host_threads())
    groups = -(-wl.rows // wl.row_repeat)
    cuts = [min(wl.rows, (groups * i // threads) * wl.row_repeat) for i in range(threads + 1)]
    parts = [_row_slice(wl, a, b) for a, b in zip(cuts, cuts[1:]) if b > a]
    reps, t0 = 0, time.perf_counter()
    with ThreadPoolExecutor(max_workers=len(parts)) as pool:
        while True:
            list(pool.map(lambda w: run(w, want_scores=False), parts))
            reps += 1
            el = time.perf_counter() - t0
            if el >= budget_s or reps >= 50:
                break
    return el / reps, reps


def oracle_mask(oracle, wl, ids):
    """One masking pass of the oracle (the entry point for the workload's
    layout and dtype) on a copy of the workload's logits."""
    bf16 = esize(wl) == 2
    if getattr(wl, "global_row_ks", None) is not None:
        return oracle.mask_sharded_starts(wl.logits, wl.global_row_ks, wl.global_row_ke,
                                          wl.global_block_size, ids, wl.row_repeat)
    if hasattr(wl, "global_row_ke"):
        return (oracle.mask_sharded_bf16 if bf16 else oracle.mask_sharded)(
            wl.logits, wl.global_row_ke, wl.global_block_size, ids, wl.row_repeat)
    return (oracle.mask_bf16 if bf16 else oracle.mask)(
        wl.logits, wl.row_ks, wl.row_ke, ids, wl.block_size, wl.row_repeat,
        width=wl.logits.shape[1])


def oracle_mask_baseline(wl, ids, budget_s: float = 10.0):
    """The masking oracle as it stands, single-threaded, repeated over the
    whole workload until about budget_s seconds have passed."""
    import oracle

    oracle.build()
    reps, t0 = 0, time.perf_counter()
    while True:
        oracle_mask(oracle, wl, ids)
        reps += 1
        el = time.perf_counter() - t0
        if el >= budget_s or reps >= 50:
            break
    return el / reps, reps


class StepTimer:
    """Times K steps on the device with CUDA events on the launching stream.

    Steps whose inputs fit in L2 twice over (``flush``) are timed one by one
    with L2 flushed before each (a 256 MB write, and for read-dominated steps
    a 256 MB read of another buffer after it); the others are replayed from
    a CUDA graph of up to 64 steps so that host launch cost never starves
    the GPU between short steps. ``step`` is one callable or a list taken in
    turn (e.g. two copies of the inputs, so that no step finds the previous
    step's lines in L2)."""

    def __init__(self, torch, device, read_after_flush: bool):
        self.torch = torch
        self.read_after_flush = read_after_flush
        self.scratch = torch.empty(256 * 1000 * 1000 // 4, dtype=torch.float32, device=device)
        self.scratch2 = (torch.ones(256 * 1000 * 1000 // 4, dtype=torch.float32, device=device)
                         if read_after_flush else None)
        self.flush = False
        self.clean = False

    def flush_l2(self):
        self.scratch.fill_(1.0)
        if self.clean:
            self.scratch2.amax()

    def prepare(self, step, steps: int, warmup: int, flush: bool):
        torch = self.torch
        self.flush = flush
        self.clean = flush and self.read_after_flush
        seq = list(step) if isinstance(step, (list, tuple)) else [step]
        for i in range(max(warmup, len(seq))):
            seq[i % len(seq)]()
        torch.cuda.synchronize()
        self.one = graph_of(seq[0], 1, torch)
        self.per = steps_per_graph(steps)
        self.many = graph_of(seq, self.per, torch)
        for _ in range(2):
            self.one.replay()
            self.many.replay()
        torch.cuda.synchronize()

    def run(self, steps: int, stream) -> float:
        """Device milliseconds of ``steps`` steps (prepare() first)."""
        torch = self.torch
        if self.flush:
            evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True))
                   for _ in range(steps)]
            for a, b in evs:
                self.flush_l2()
                a.record(stream)
                self.one.replay()
                b.record(stream)
            torch.cuda.synchronize()
            return sum(a.elapsed_time(b) for a, b in evs)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(stream)
        for _ in range(steps // self.per):
            self.many.replay()
        b.record(stream)
        torch.cuda.synchronize()
        return a.elapsed_time(b)

    def l2_note(self) -> str:
        if self.clean:
            return "flushed before every step (256 MB write, then 256 MB read of another buffer)"
        if self.flush:
            return "flushed before every step (256 MB write)"
        return ("inputs larger than L2 (bytes per step > 2 x 129 MB); two copies of the logits "
                "read in turn" if self.read_after_flush else
                "inputs larger than L2 (bytes per step > 2 x 129 MB)")


# The configurations besides the headline one, each timed briefly in the same
# run (selection only, one GPU) so that the bench line carries all of them.
OTHER_WORKLOADS = ("tiny", "decode", "prefill", "long", "long_pin", "decode_bf16", "dcp_bf16",
                   "dcp_starts")


def time_other_workloads(names, dsa, torch, device, timer, steps: int, warmup: int,
                         peak: float):
    """ms per step, GB/s, roofline fraction and rows/s of each workload's
    selection, by the headline's method (flushed per step when its window
    bytes fit in L2 twice over, else graph-replayed over two logits copies)."""
    import workloads

    res = {}
    stream = torch.cuda.current_stream()
    for name in names:
        wl = workloads.make(name)
        nbytes = algorithmic_bytes(wl)
        flush = esize(wl) * window_elements(wl) < 2 * L2_BYTES
        step, _ = make_runner(wl, dsa, torch, device, copies=1 if flush else 2)
        n = steps if not flush else max(steps // 4, 20)
        timer.prepare(step, n, warmup, flush)
        ms = timer.run(n, stream) / n
        res[name] = {"ms_per_step": round(ms, 5), "value": round(nbytes / ms / 1e6, 3),
                     "unit": UNIT, "frac": round(nbytes / ms / 1e6 / peak, 4),
                     "rows_per_s": round(wl.rows / ms * 1e3, 1),
                     "algorithmic_bytes_per_step": nbytes, "steps": n,
                     "workload": workload_config(wl, name)["workload"], "l2": timer.l2_note(),
                     "kernel": selection_kernel(wl, torch.cuda.get_device_properties(device)
                                                .multi_processor_count),
                     "traffic": profiled_traffic("select", name)}
        del step
        timer.one = timer.many = None
        torch.cuda.empty_cache()
        if flush:
            res[name]["streamed"] = time_streamed(wl, dsa, torch, device, timer, steps, warmup,
                                                  peak, nbytes)
        del wl
        timer.one = timer.many = None
        torch.cuda.empty_cache()
    return res


def time_streamed(wl, dsa, torch, device, timer, steps: int, warmup: int, peak: float,
                  nbytes: int):
    """A step of a workload whose window fits in L2, in steady state: steps
    replayed back to back from a CUDA graph over C copies of the logits taken
    in turn, C chosen so that the C - 1 other steps between two reads of a
    copy stream at least twice the L2 capacity (no L2 flush; each step's
    window is out of L2 when it is read again). Null when that needs more
    than 16 copies or 8 GB."""
    window = esize(wl) * window_elements(wl)
    copies = 2 + -(-2 * L2_BYTES // max(window, 1))
    tensor = esize(wl) * wl.logits.size
    if copies > 16 or copies * tensor > 8e9:
        return None
    step, _ = make_runner(wl, dsa, torch, device, copies=copies)
    stream = torch.cuda.current_stream()
    # One graph replay is a whole number of rounds over the copies, so the
    # order never restarts early.
    per = copies * (64 // copies)
    total = per * max(1, steps // per)
    timer.prepare(step, per, warmup, False)
    ms = timer.run(total, stream) / total
    del step
    return {"ms_per_step": round(ms, 5), "value": round(nbytes / ms / 1e6, 3), "unit": UNIT,
            "frac": round(nbytes / ms / 1e6 / peak, 4), "steps": total, "copies": copies,
            "l2": f"no flush; {copies} logits copies read in turn, each re-read after "
                  f"{(copies - 1) * window / 1e6:.0f} MB of other windows (L2 "
                  f"{L2_BYTES / 1e6:.0f} MB)"}


def run_ours(args):
    import numpy as np
    import torch

    import __graft_entry__
    import workloads

    rank, world, local_rank = dist_env()
    if world > 1:
        import torch.distributed as dist

        torch.cuda.set_device(local_rank)
        dist.init_process_group("nccl", device_id=torch.device("cuda", local_rank))
    device = torch.device("cuda", local_rank)
    torch.cuda.set_device(device)
    __graft_entry__.build()
    import deepseek_sparse_attention_row_gb300 as dsa

    for item in filter(None, args.launch.split(",")):
        knob, val = item.split("=")
        dsa.set_launch_override(knob.strip(), int(val))
    if args.op in LSE_OPS:
        wl = workloads.make_lse_named(args.workload)
        step = make_lse_runner(wl, args.op, dsa, torch, device)
        nbytes = lse_algorithmic_bytes(wl, args.op)
        flush = nbytes < 2 * L2_BYTES
    elif args.op == "mask":
        wl = workloads.make(args.workload)
        step, nbytes, mask_ids = make_mask_runner(wl, dsa, torch, device)
        flush = nbytes < 2 * L2_BYTES
    else:
        wl = workloads.make(args.workload)
        nbytes = algorithmic_bytes(wl)
        window_bytes = esize(wl) * window_elements(wl)
        flush = window_bytes < 2 * L2_BYTES
        step, out = make_runner(wl, dsa, torch, device, copies=1 if flush else 2)
    # Read-dominated steps (selection) also read a second 256 MB buffer after
    # the flush write, so that the flush's own dirty lines are written back
    # before the timed step rather than during it; write-heavy steps (masking,
    # LSE) keep the write-only flush, so that their stores cannot sit in a
    # clean L2 when the step ends.
    timer = StepTimer(torch, device, read_after_flush=args.op == "select")
    stream = torch.cuda.current_stream()
    props = torch.cuda.get_device_properties(device)
    uuid = str(getattr(props, "uuid", "") or "")
    timer.prepare(step, args.steps, args.warmup, flush)

    with ClockSampler(uuid) as sampler:
        dist_barrier(world)
        torch.cuda.synchronize()
        t_wall = time.perf_counter()
        gpu_ms = timer.run(args.steps, stream)
        dist_barrier(world)
        wall_s = time.perf_counter() - t_wall
    clocks = sampler.summary()

    max_ms = dist_max(gpu_ms, world, device)
    ms_per_step = max_ms / args.steps
    value = whole_job_rate(nbytes * args.steps, world, max_ms / 1e3) / 1e9
    nrows = wl.batch * wl.heads if args.op in LSE_OPS else wl.rows
    rows_per_s = whole_job_rate(nrows * args.steps, world, max_ms / 1e3)
    launch_s = (gpu_ms / args.steps) / 1e3
    achieved = nbytes / launch_s / 1e9
    peak, peak_src = measured_peak()

    e2e = None
    cpu = None
    if rank == 0 and not args.no_e2e and args.op == "select":
        res = e2e_measure(wl, dsa, torch, device, args.e2e_steps,
                          flush=timer.flush_l2 if flush else None)
        sec, h2d, d2h = res["in_place"]
        ssec, sh2d, sd2h = res["staged"]
        e2e = {"value": round(nbytes / sec / 1e9 * world, 3), "unit": UNIT,
               "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
               "ms_per_step": round(sec * 1e3, 4), "steps": args.e2e_steps,
               "path": "pinned host inputs read in place by the kernel (in-window logits and "
                       "bounds across the host link), ids written to pinned host memory",
               "staged": {"value": round(nbytes / ssec / 1e9 * world, 3), "unit": UNIT,
                          "h2d_bytes_per_step": sh2d, "d2h_bytes_per_step": sd2h,
                          "ms_per_step": round(ssec * 1e3, 4),
                          "path": "whole logits tensor and bounds copied to the device, "
                                  "ids copied back"}}
    if rank == 0 and world == 1 and not args.no_cpu_baseline and args.op in LSE_OPS:
        sec, reps = oracle_lse_baseline(wl, args.op, args.cpu_budget)
        cpu = {"value": round(nbytes / sec / 1e9, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"the whole {args.workload} workload, {reps} pass(es), single-threaded "
                         f"C oracle ({args.op}), {sec:.3f} s per pass"}
    elif rank == 0 and world == 1 and not args.no_cpu_baseline and args.op == "mask":
        sec, reps = oracle_mask_baseline(wl, mask_ids, args.cpu_budget)
        cpu = {"value": round(nbytes / sec / 1e9, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
               "sample": f"the whole {args.workload} workload, {reps} pass(es), single-threaded "
                         f"C oracle masking, {sec:.3f} s per pass"}
    elif rank == 0 and world == 1 and not args.no_cpu_baseline:
        nthr = host_threads()
        msec, mreps = oracle_cpu_baseline_threads(wl, args.cpu_budget, nthr)
        sec, reps = oracle_cpu_baseline(wl, args.cpu_budget)
        cpu = {"value": round(nbytes / msec / 1e9, 4), "unit": UNIT, "cores": nthr,
               "kind": "oracle",
               "sample": f"the whole {args.workload} workload, {mreps} pass(es), the C oracle "
                         f"over {nthr} row ranges on {nthr} threads, {msec:.3f} s per pass",
               "single_core": {"value": round(nbytes / sec / 1e9, 4), "unit": UNIT, "cores": 1,
                               "sample": f"the whole {args.workload} workload, {reps} pass(es), "
                                         f"single-threaded C oracle, {sec:.3f} s per pass"}}
    others = None
    if rank == 0 and world == 1 and args.op == "select" and not args.no_other_workloads:
        others = time_other_workloads([n for n in OTHER_WORKLOADS if n != args.workload], dsa,
                                      torch, device, timer, 500, 5, peak)

    if rank == 0:
        metric = {"select": METRIC, "mask": MASK_METRIC}.get(args.op) or LSE_METRICS[args.op]
        if args.op in LSE_OPS:
            config = lse_workload_config(wl, args.workload)
            full_gbs = None
            kernel = "lse_kernel (one launch per step)"
            dtype = "f32" if wl.dtype == "f32" else "f32 arithmetic, bf16 data"
        else:
            config = workload_config(wl, args.workload)
            full_gbs = round(whole_job_rate(wl.logits.size * esize(wl) * args.steps, world,
                                            max_ms / 1e3) / 1e9, 3)
            kernel = (selection_kernel(wl, torch.cuda.get_device_properties(device)
                                       .multi_processor_count)
                      if args.op == "select" else "mask_kernel (one launch per step)")
            dtype = "f32" if esize(wl) == 4 else "bf16 data, exact compares"
        line = {
            "metric": metric, "value": round(value, 3), "unit": UNIT, "n_gpus": world,
            "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(ms_per_step, 5),
            "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": dtype,
            "data": "synthetic (seeded numpy PCG64; shapes and distributions of the workload)",
            "config": {**config,
                       "parallelism": f"replicas x{world}" if world > 1 else "single GPU",
                       "l2": timer.l2_note()},
            "rows_per_s": round(rows_per_s, 1),
            "algorithmic_bytes_per_step": nbytes,
            "full_tensor_equivalent_gbs": full_gbs,
            "roofline": {"bound": "hbm", "achieved": round(achieved, 3), "peak": peak,
                         "unit": UNIT, "frac": round(achieved / peak, 4),
                         "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                         if peak_src == "measured" else "fallback 6.8 TB/s",
                         "traffic": profiled_traffic(args.op, args.workload),
                         "kernel": kernel},
            "clocks": clocks,
            "gpu_launches": args.steps,
            "wall_s_timed_region": round(wall_s, 3),
            "e2e": e2e,
            "cpu_baseline": cpu,
        }
        if others is not None:
            line["workloads"] = others
        print(json.dumps(line), flush=True)
    if world > 1:
        import torch.distributed as dist

        dist.destroy_process_group()


# ---------------------------------------------------------------------------
# Reference arm: the oracle, timed on the host cores
# ---------------------------------------------------------------------------

def run_reference(args):
    rank, world, _ = dist_env()
    if rank != 0:
        return
    import numpy as np

    import oracle
    import workloads

    oracle.build()
    if args.op in LSE_OPS:
        return run_reference_lse(args, oracle, workloads, world)
    wl = workloads.make(args.workload)

    bf16 = esize(wl) == 2
    run_select = oracle.run_workload_bf16 if bf16 else oracle.run_workload

    def oracle_mask_step(w, ids):
        oracle_mask(oracle, w, ids)

    def prepare(w):
        """(step, algorithmic bytes) of one oracle pass over workload w."""
        if args.op == "select":
            return (lambda: run_select(w, want_scores=False)), algorithmic_bytes(w)
        ids, _ = run_select(w, want_scores=False)
        nb = (w.global_row_ke.size if hasattr(w, "global_row_ke")
              else w.row_ke.size + (0 if w.row_ks is None else w.row_ks.size))
        return ((lambda: oracle_mask_step(w, ids)),
                esize(w) * mask_written_elements(w, ids) + 4 * nb + 4 * ids.size)

    # Calibrate on a slice of rows, then size each step's sample so that the
    # whole run stays within about args.ref_budget seconds. The sample's rows
    # are cut into one contiguous range per host thread and each step runs
    # the oracle on all ranges at once (the C calls release the GIL).
    from concurrent.futures import ThreadPoolExecutor

    rows = wl.rows
    nthr = host_threads()
    rr = wl.row_repeat
    probe = max(rr, (rows // 64) // rr * rr)
    probe_step, _ = prepare(_row_slice(wl, 0, probe))
    t0 = time.perf_counter()
    probe_step()
    per_row = max((time.perf_counter() - t0) / probe, 1e-7)
    total_steps = args.steps + args.warmup
    sample_rows = int(max(1, min(rows, args.ref_budget * nthr / total_steps / per_row)))
    groups = -(-sample_rows // rr)
    cuts = [min(sample_rows, (groups * i // nthr) * rr) for i in range(nthr + 1)]
    parts = [prepare(_row_slice(wl, a, b)) for a, b in zip(cuts, cuts[1:]) if b > a]
    sample_bytes = sum(nb for _, nb in parts)
    with ThreadPoolExecutor(max_workers=len(parts)) as pool:
        def ref_step():
            list(pool.map(lambda part: part[0](), parts))
        for _ in range(args.warmup):
            ref_step()
        t0 = time.perf_counter()
        for _ in range(args.steps):
            ref_step()
        sec = (time.perf_counter() - t0) / args.steps
    value = sample_bytes / sec / 1e9
    desc = (f"first {sample_rows} of {rows} rows of the {args.workload} workload per step, "
            f"cut into {len(parts)} row ranges run on {len(parts)} host threads "
            f"({sample_bytes} algorithmic bytes)")
    line = {
        "impl": "reference", "metric": METRIC if args.op == "select" else MASK_METRIC,
        "value": round(value, 4), "unit": UNIT,
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sec * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f32" if esize(wl) == 4 else "bf16 data, exact compares",
        "data": "synthetic (seeded numpy PCG64; shapes and distributions of the workload)",
        "config": {**workload_config(wl, args.workload),
                   "parallelism": f"host, {len(parts)} threads"},
        "rows_per_s": round(sample_rows / sec, 1),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": len(parts),
                         "kind": "oracle", "sample": desc},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def run_reference_lse(args, oracle, workloads, world):
    """Reference arm for the LSE ops: the oracle on the first tokens of the
    workload, sized so that the whole run takes about args.ref_budget s."""
    import copy

    wl = workloads.make_lse_named(args.workload)
    N, B = wl.shards, wl.batch

    def sliced(b):
        w = copy.copy(wl)
        w.outs = np.ascontiguousarray(wl.outs[:, :b])
        w.lses = np.ascontiguousarray(wl.lses[:, :b])
        return w

    def run(w):
        if args.op == "merge":
            oracle.merge_attn_out(w.outs, w.lses)
        else:
            oracle.correct_attn_out(w.outs[N // 2], w.lses, N // 2)

    import numpy as np

    probe = sliced(max(1, B // 32))
    t0 = time.perf_counter()
    run(probe)
    per_tok = max((time.perf_counter() - t0) / probe.batch, 1e-7)
    total_steps = args.steps + args.warmup
    b = int(max(1, min(B, args.ref_budget / total_steps / per_tok)))
    sample = sliced(b)
    sample_bytes = lse_algorithmic_bytes(sample, args.op)
    for _ in range(args.warmup):
        run(sample)
    t0 = time.perf_counter()
    for _ in range(args.steps):
        run(sample)
    sec = (time.perf_counter() - t0) / args.steps
    value = sample_bytes / sec / 1e9
    desc = (f"first {b} of {B} tokens (all heads) of the {args.workload} workload per step "
            f"({sample_bytes} algorithmic bytes)")
    line = {
        "impl": "reference", "metric": LSE_METRICS[args.op], "value": round(value, 4),
        "unit": UNIT, "n_gpus": world, "steps": args.steps, "warmup": args.warmup,
        "ms_per_step": round(sec * 1e3, 4), "higher_is_better": True, "scaling": "weak",
        "vs_baseline": None, "dtype": "f64",
        "data": "synthetic (seeded numpy PCG64; shapes and distributions of the workload)",
        "config": {**lse_workload_config(wl, args.workload), "parallelism": "host, 1 thread"},
        "rows_per_s": round(b * wl.heads / sec, 1),
        "cpu_baseline": {"value": round(value, 4), "unit": UNIT, "cores": 1, "kind": "oracle",
                         "sample": desc},
        "e2e": {"value": round(value, 4), "unit": UNIT, "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }
    print(json.dumps(line), flush=True)


def _row_slice(wl, r0: int, r1: int):
    """The same workload restricted to rows [r0, r1) (r0 a multiple of
    row_repeat)."""
    import copy

    import numpy as np

    assert r0 % wl.row_repeat == 0
    g0, g1 = r0 // wl.row_repeat, -(-r1 // wl.row_repeat)
    s = copy.copy(wl)
    if hasattr(wl, "global_row_ke"):
        s.logits = np.ascontiguousarray(wl.logits[:, r0:r1])
        s.global_row_ke = wl.global_row_ke[g0:g1].copy()
        if getattr(wl, "global_row_ks", None) is not None:
            s.global_row_ks = wl.global_row_ks[g0:g1].copy()
    else:
        s.logits = wl.logits[r0:r1]
        s.row_ke = wl.row_ke[g0:g1].copy()
        s.row_ks = None if wl.row_ks is None else wl.row_ks[g0:g1].copy()
    return s


def main(argv=None):
    p = argparse.ArgumentParser(description=__doc__.split("\n\n")[0])
    p.add_argument("--gpus", type=int, default=1)
    p.add_argument("--steps", type=int, default=2000)
    p.add_argument("--warmup", type=int, default=20)
    p.add_argument("--impl", choices=("ours", "reference"), default="ours")
    p.add_argument("--op", choices=("select", "mask") + LSE_OPS, default="select",
                   help="select: candidate selection (the bench line); mask: the masking "
                        "pass that follows it; correct / merge: the DCP partial-attention "
                        "LSE correction of one shard / merge of all shards")
    p.add_argument("--workload", default=None,
                   choices=("dcp", "decode", "prefill", "long", "long_pin", "tiny",
                            "dcp_bf16", "decode_bf16", "dcp_starts") + tuple(LSE_NAMES),
                   help="default: dcp for select / mask, lse_decode for correct / merge")
    p.add_argument("--e2e-steps", type=int, default=10)
    p.add_argument("--no-e2e", action="store_true")
    p.add_argument("--no-cpu-baseline", action="store_true")
    p.add_argument("--launch", default="",
                   help="tuning sweeps: knob=value,... pinned through the library's launch "
                        "overrides (see dsa_select_set_launch_override)")
    p.add_argument("--no-other-workloads", action="store_true",
                   help="select only: skip timing the other configurations after the headline")
    p.add_argument("--cpu-budget", type=float, default=10.0)
    p.add_argument("--ref-budget", type=float, default=90.0)
    args = p.parse_args(argv)
    if args.warmup < 3:
        p.error("--warmup must be at least 3")
    if args.workload is None:
        args.workload = "lse_decode" if args.op in LSE_OPS else "dcp"
    if (args.op in LSE_OPS) != (args.workload in LSE_NAMES):
        p.error(f"--op {args.op} does not run on --workload {args.workload}")
    _, world, _ = dist_env()
    if args.gpus > 1 and world == 1 and args.impl == "ours":
        p.error("--gpus N > 1 needs torch.distributed.run with N processes")
    if args.impl == "reference":
        run_reference(args)
    else:
        run_ours(args)


if __name__ == "__main__":
    main()
