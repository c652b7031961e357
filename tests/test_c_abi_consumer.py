"""The C ABI from plain C: ``tests/c_abi_consumer.c`` includes only
``include/dsa_cb.h`` and the CUDA runtime API, allocates its own device
memory and stream, and calls the library. Without a GPU the program must
compile (C99, warnings as errors) and link against ``libdsa_cb.so``; on a
GPU its ids must equal the oracle's."""

import os
import subprocess

import numpy as np
import pytest

import oracle
import workloads

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
CUDA = os.environ.get("CUDA_HOME", "/usr/local/cuda")
SOURCE = os.path.join(ROOT, "tests", "c_abi_consumer.c")


def build_consumer(out_dir: str) -> str:
    from deepseek_sparse_attention_row_gb300 import _build_lib

    lib = _build_lib.build()
    lib_dir = os.path.dirname(lib)
    exe = os.path.join(out_dir, "c_abi_consumer")
    cmd = ["gcc", "-std=c99", "-O2", "-Wall", "-Wextra", "-Werror",
           "-I", os.path.join(ROOT, "include"), "-I", os.path.join(CUDA, "include"),
           SOURCE, "-o", exe, "-L", lib_dir, "-ldsa_cb",
           "-L", os.path.join(CUDA, "lib64"), "-lcudart",
           f"-Wl,-rpath,{lib_dir}:{os.path.join(CUDA, 'lib64')}"]
    res = subprocess.run(cmd, capture_output=True, text=True)
    assert res.returncode == 0, res.stdout + res.stderr
    return exe


def test_c_consumer_compiles_and_links(tmp_path):
    exe = build_consumer(str(tmp_path))
    assert os.path.exists(exe)


@pytest.mark.gpu
@pytest.mark.parametrize("seed,rows,width,bs,topk,rr", [
    (31, 40, 5000, 64, 16, 4),      # starts, row groups, a ragged last block
    (32, 24, 70000, 128, 32, 1),    # rows long enough to be split over CTAs
])
def test_c_consumer_matches_oracle(tmp_path, seed, rows, width, bs, topk, rr):
    exe = build_consumer(str(tmp_path))
    wl = workloads.small_unsharded(seed, rows=rows, width=width, block_size=bs,
                                   topk_blocks=topk, row_repeat=rr, nan_count=3)
    want, _ = oracle.run_workload(wl, want_scores=False)
    hdr = np.array([rows, width, bs, topk, rr, int(wl.pin_newest)], dtype=np.int64)
    inp, out = tmp_path / "in.bin", tmp_path / "out.bin"
    with open(inp, "wb") as f:
        f.write(hdr.tobytes())
        f.write(np.ascontiguousarray(wl.logits, dtype=np.float32).tobytes())
        f.write(np.ascontiguousarray(wl.row_ke, dtype=np.int32).tobytes())
        f.write(np.ascontiguousarray(wl.row_ks, dtype=np.int32).tobytes())
    res = subprocess.run([exe, str(inp), str(out)], capture_output=True, text=True, timeout=300)
    assert res.returncode == 0, res.stdout + res.stderr
    got = np.fromfile(out, dtype=np.int32).reshape(rows, topk)
    np.testing.assert_array_equal(got, want)
