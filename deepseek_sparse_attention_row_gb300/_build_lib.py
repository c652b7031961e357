"""Compile libdsa_cb.so (sm_103a) in tree, under ``_build/``.

Each ``csrc/*.cu`` is compiled by nvcc for
``-gencode arch=compute_103a,code=sm_103a`` (in parallel, one object each)
and the objects are linked into one shared library with the CUDA runtime
linked statically, so it loads next to any PyTorch build without a runtime
search.
"""

from __future__ import annotations

import os
import subprocess
import sys

PKG = os.path.dirname(os.path.abspath(__file__))
ROOT = os.path.dirname(PKG)
CSRC = os.path.join(PKG, "csrc")
BUILD = os.path.join(PKG, "_build")
LIB = os.path.join(BUILD, "libdsa_cb.so")
INCLUDE = os.path.join(ROOT, "include")
ARCH = ["-gencode", "arch=compute_103a,code=sm_103a"]


def sources() -> list:
    return (sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC)
                   if f.endswith((".cu", ".cuh", ".h")))
            + sorted(os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h")))


def nvcc() -> str:
    for cand in (os.environ.get("NVCC"), "/usr/local/cuda/bin/nvcc", "nvcc"):
        if cand and (os.path.sep not in cand or os.path.exists(cand)):
            return cand
    return "nvcc"


def units() -> list:
    """The translation units, one object each."""
    return sorted(os.path.join(CSRC, f) for f in os.listdir(CSRC) if f.endswith(".cu"))


def build(force: bool = False, verbose: bool = False) -> str:
    os.makedirs(BUILD, exist_ok=True)
    if (not force and os.path.exists(LIB)
            and os.path.getmtime(LIB) >= max(os.path.getmtime(s) for s in sources())):
        return LIB
    tag = f"tmp{os.getpid()}"
    flags = [*ARCH, "-O3", "-lineinfo", "-std=c++17", "-Xcompiler", "-fPIC"]
    if verbose:
        flags.append("-Xptxas=-v")
    procs, objs = [], []
    for cu in units():
        obj = os.path.join(BUILD, os.path.basename(cu)[:-3] + f".{tag}.o")
        objs.append(obj)
        procs.append((cu, subprocess.Popen([nvcc(), *flags, "-c", "-o", obj, cu],
                                           stdout=subprocess.PIPE, stderr=subprocess.PIPE,
                                           text=True)))
    failed = False
    for cu, p in procs:
        out, err = p.communicate()
        if p.returncode != 0 or verbose:
            sys.stderr.write(f"== {os.path.basename(cu)}\n" + out + err)
        failed |= p.returncode != 0
    try:
        if failed:
            raise RuntimeError("nvcc failed to build libdsa_cb.so")
        tmp = f"{LIB}.{tag}"
        res = subprocess.run([nvcc(), *ARCH, "-shared", "-o", tmp, *objs],
                             capture_output=True, text=True)
        if res.returncode != 0:
            sys.stderr.write(res.stdout + res.stderr)
            raise RuntimeError("nvcc failed to link libdsa_cb.so")
        os.replace(tmp, LIB)
    finally:
        for obj in objs:
            if os.path.exists(obj):
                os.remove(obj)
    return LIB


if __name__ == "__main__":
    print(build(force="--force" in sys.argv, verbose="-v" in sys.argv))
