"""The C ABI without a GPU: the library builds for sm_103a, loads, exports
every function that the headers in ``include/`` declare, and rejects invalid
arguments on the host before touching the device (no call below reaches a
CUDA API)."""

import ctypes
import os
import re
import subprocess

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
INCLUDE = os.path.join(ROOT, "include")
HEADERS = sorted(os.path.join(INCLUDE, f) for f in os.listdir(INCLUDE) if f.endswith(".h"))

DSA_OK, DSA_EINVAL, DSA_ECUDA, DSA_EUNSUPPORTED = 0, -1, -2, -3


@pytest.fixture(scope="module")
def lib():
    from deepseek_sparse_attention_row_gb300 import _build_lib

    _build_lib.build()
    import deepseek_sparse_attention_row_gb300 as dsa

    return dsa.library()


def declared_functions():
    names = set()
    for h in HEADERS:
        text = re.sub(r"/\*.*?\*/", "", open(h).read(), flags=re.S)
        names.update(re.findall(r"\b(dsa_[a-z0-9_]+)\s*\(", text))
    return sorted(names)


def test_headers_declare_the_operations():
    names = declared_functions()
    for n in ("dsa_block_scores", "dsa_select_candidate_blocks",
              "dsa_select_candidate_blocks_sharded", "dsa_mask_candidate_logits",
              "dsa_mask_candidate_logits_sharded", "dsa_correct_attn_out",
              "dsa_merge_attn_out"):
        assert n in names


def test_every_declared_symbol_is_exported(lib):
    import deepseek_sparse_attention_row_gb300 as dsa

    names = declared_functions()
    assert sorted(dsa.EXPORTED_SYMBOLS) == names
    nm = subprocess.run(["nm", "-D", "--defined-only", dsa.library_path], capture_output=True,
                        text=True, check=True).stdout
    exported = set(re.findall(r"\bT (\w+)", nm))
    for n in names:
        assert n in exported, n
        assert hasattr(lib, n)


def test_status_strings(lib):
    for st in (DSA_OK, DSA_EINVAL, DSA_ECUDA, DSA_EUNSUPPORTED, 12345):
        assert lib.dsa_status_string(st)


def test_workspace_bytes(lib):
    # a 256-byte queue header, one counter per row and rows * nblocks keys,
    # each part 256-byte aligned
    assert lib.dsa_select_workspace_bytes(4096, 1024) == 256 + 16384 + 4096 * 1024 * 4
    assert lib.dsa_select_workspace_bytes(3, 5) == 256 + 256 + 256
    assert lib.dsa_select_workspace_bytes(0, 7) == 0
    assert lib.dsa_select_workspace_bytes(-1, 7) == 0


def test_limits(lib):
    assert lib.dsa_select_max_blocks() >= 1024
    assert lib.dsa_select_max_shards() >= 8


def test_launch_override_validation(lib):
    # Only the explicit call sets a launch shape: out-of-range values and
    # unknown knobs are refused, and 0 hands every knob back to the launcher.
    set_ = lib.dsa_select_set_launch_override
    set_.argtypes = [ctypes.c_int32, ctypes.c_int32]
    set_.restype = ctypes.c_int
    for knob, good, bad in ((1, (0, 1, 3, 8), (-1, 9)), (2, (0, 128, 256), (64, 512, -1)),
                            (3, (0, 1), (2, -1)), (4, (0, 1), (2, -1))):
        for v in good:
            assert set_(knob, v) == DSA_OK
        for v in bad:
            assert set_(knob, v) == DSA_EINVAL
        assert set_(knob, 0) == DSA_OK
    for knob, good, bad in ((5, (0, 1, 2, 3), (4, -1)), (6, (0, 1, 8), (9, -1)),
                            (7, (0, 2, 16), (1, 17)), (8, (0, 4, 64), (3, 65)),
                            (9, (0, 1), (2, -1)), (10, (0, 4, 8), (2, 16)),
                            (11, (0, 1, 4), (5, -1)), (12, (0, 1), (2, -1)),
                            (13, (0, 1, 2, 3), (4, -1)), (14, (0, 1, 2), (3, -1))):
        for v in good:
            assert set_(knob, v) == DSA_OK
        for v in bad:
            assert set_(knob, v) == DSA_EINVAL
        assert set_(knob, 0) == DSA_OK
    for knob in (0, 15, 99, -3):
        assert set_(knob, 0) == DSA_EINVAL


def test_library_reads_no_environment():
    # Launch shapes are plain function arguments or explicit calls: no source
    # of the library asks the process environment for anything.
    csrc = os.path.join(ROOT, "deepseek_sparse_attention_row_gb300", "csrc")
    for f in sorted(os.listdir(csrc)):
        text = open(os.path.join(csrc, f)).read()
        assert "getenv" not in text and "environ" not in text, f


FAKE = ctypes.c_void_p(0x1000)  # never dereferenced: every call below fails validation first


@pytest.mark.parametrize("kw,want", [
    (dict(rows=-1), DSA_EINVAL),
    (dict(width=-1), DSA_EINVAL),
    (dict(block_size=0), DSA_EINVAL),
    (dict(row_repeat=0), DSA_EINVAL),
    (dict(ld=5), DSA_EINVAL),
    (dict(scores=None), DSA_EINVAL),
    (dict(ld_scores=1), DSA_EINVAL),
    (dict(rows=0), DSA_OK),
    (dict(width=0), DSA_OK),
    (dict(width=1 << 31, ld=1 << 31, ld_scores=1 << 31), DSA_EUNSUPPORTED),
])
def test_block_scores_validation(lib, kw, want):
    a = dict(logits=FAKE, rows=4, width=10, ld=10, ks=None, ke=FAKE, block_size=4,
             row_repeat=1, pin=1, scores=FAKE, ld_scores=3)
    a.update(kw)
    st = lib.dsa_block_scores(a["logits"], a["rows"], a["width"], a["ld"], a["ks"], a["ke"],
                              a["block_size"], a["row_repeat"], a["pin"], a["scores"],
                              a["ld_scores"], None)
    assert st == want


@pytest.mark.parametrize("kw,want", [
    (dict(rows=-2), DSA_EINVAL),
    (dict(topk=-1), DSA_EINVAL),
    (dict(block_size=-3), DSA_EINVAL),
    (dict(row_repeat=0), DSA_EINVAL),
    (dict(out=None), DSA_EINVAL),
    (dict(ld_out=3), DSA_EINVAL),
    (dict(logits=None), DSA_EINVAL),
    (dict(ke=None), DSA_EINVAL),
    (dict(ld=99), DSA_EINVAL),
    (dict(scores=FAKE, ld_scores=2), DSA_EINVAL),
    (dict(rows=0), DSA_OK),
    (dict(topk=0, out=None), DSA_OK),
    (dict(block_size=1, width=20000, ld=20000), DSA_EUNSUPPORTED),
])
def test_select_validation(lib, kw, want):
    a = dict(logits=FAKE, rows=4, width=100, ld=100, ks=None, ke=FAKE, topk=4, block_size=8,
             row_repeat=1, pin=1, out=FAKE, ld_out=4, scores=None, ld_scores=0, ws=FAKE,
             ws_bytes=1 << 20)
    a.update(kw)
    st = lib.dsa_select_candidate_blocks(a["logits"], a["rows"], a["width"], a["ld"], a["ks"],
                                         a["ke"], a["topk"], a["block_size"], a["row_repeat"],
                                         a["pin"], a["out"], a["ld_out"], a["scores"],
                                         a["ld_scores"], a["ws"], a["ws_bytes"], None)
    assert st == want


@pytest.mark.parametrize("kw,want", [
    (dict(shards=0), DSA_EINVAL),
    (dict(gbs=60), DSA_EINVAL),          # not a multiple of 8 shards
    (dict(gbs=0), DSA_EINVAL),
    (dict(rows=-1), DSA_EINVAL),
    (dict(lw=-1), DSA_EINVAL),
    (dict(topk=-1), DSA_EINVAL),
    (dict(row_repeat=0), DSA_EINVAL),
    (dict(ld=10), DSA_EINVAL),
    (dict(shard_stride=-1), DSA_EINVAL),
    (dict(gke=None), DSA_EINVAL),
    (dict(out=None), DSA_EINVAL),
    (dict(ld_out=1), DSA_EINVAL),
    (dict(logits=None), DSA_EINVAL),
    (dict(scores=FAKE, ld_scores=7), DSA_EINVAL),
    (dict(rows=0), DSA_OK),
    (dict(topk=0, out=None), DSA_OK),
    (dict(max_gb=20000, scores=None), DSA_EUNSUPPORTED),
    (dict(shards=2048, gbs=2048), DSA_EUNSUPPORTED),
])
def test_sharded_validation(lib, kw, want):
    a = dict(logits=FAKE, shards=8, rows=4, lw=64, ld=64, shard_stride=256, gke=FAKE, gbs=64,
             max_gb=8, row_repeat=1, topk=4, out=FAKE, ld_out=4, scores=None, ld_scores=0,
             ws=None, ws_bytes=0)
    a.update(kw)
    st = lib.dsa_select_candidate_blocks_sharded(
        a["logits"], a["shards"], a["rows"], a["lw"], a["ld"], a["shard_stride"], a["gke"],
        a["gbs"], a["max_gb"], a["row_repeat"], a["topk"], a["out"], a["ld_out"], a["scores"],
        a["ld_scores"], a["ws"], a["ws_bytes"], None)
    assert st == want


@pytest.mark.parametrize("kw,want", [
    (dict(rows=-1), DSA_EINVAL),
    (dict(width=-1), DSA_EINVAL),
    (dict(block_size=0), DSA_EINVAL),
    (dict(row_repeat=0), DSA_EINVAL),
    (dict(topk=-1), DSA_EINVAL),
    (dict(ld=5), DSA_EINVAL),
    (dict(logits=None), DSA_EINVAL),
    (dict(ke=None), DSA_EINVAL),
    (dict(cand=None), DSA_EINVAL),
    (dict(ld_cand=1), DSA_EINVAL),
    (dict(rows=0), DSA_OK),
    (dict(width=0), DSA_OK),
])
def test_mask_validation(lib, kw, want):
    a = dict(logits=FAKE, rows=4, width=100, ld=100, ks=None, ke=FAKE, cand=FAKE, topk=4,
             ld_cand=4, block_size=8, row_repeat=1)
    a.update(kw)
    st = lib.dsa_mask_candidate_logits(a["logits"], a["rows"], a["width"], a["ld"], a["ks"],
                                       a["ke"], a["cand"], a["topk"], a["ld_cand"],
                                       a["block_size"], a["row_repeat"], None)
    assert st == want


@pytest.mark.parametrize("kw,want", [
    (dict(shards=0), DSA_EINVAL),
    (dict(gbs=60), DSA_EINVAL),
    (dict(row_repeat=0), DSA_EINVAL),
    (dict(ld=10), DSA_EINVAL),
    (dict(gke=None), DSA_EINVAL),
    (dict(cand=None), DSA_EINVAL),
    (dict(rows=0), DSA_OK),
    (dict(lw=0, ld=0), DSA_OK),
])
def test_mask_sharded_validation(lib, kw, want):
    a = dict(logits=FAKE, shards=8, rows=4, lw=64, ld=64, shard_stride=256, gke=FAKE, gbs=64,
             row_repeat=1, cand=FAKE, topk=4, ld_cand=4)
    a.update(kw)
    st = lib.dsa_mask_candidate_logits_sharded(a["logits"], a["shards"], a["rows"], a["lw"],
                                               a["ld"], a["shard_stride"], a["gke"], a["gbs"],
                                               a["row_repeat"], a["cand"], a["topk"],
                                               a["ld_cand"], None)
    assert st == want


@pytest.mark.parametrize("kw,want", [
    (dict(dtype=2), DSA_EINVAL),
    (dict(shards=0), DSA_EINVAL),
    (dict(rank=-1), DSA_EINVAL),
    (dict(rank=8), DSA_EINVAL),
    (dict(batch=-1), DSA_EINVAL),
    (dict(head_dim=-1), DSA_EINVAL),
    (dict(lses=None), DSA_EINVAL),
    (dict(out=None), DSA_EINVAL),
    (dict(new_out=None), DSA_EINVAL),
    (dict(shards=33, rank=0), DSA_EUNSUPPORTED),
    (dict(batch=0), DSA_OK),
    (dict(heads=0), DSA_OK),
])
def test_correct_attn_out_validation(lib, kw, want):
    a = dict(out=FAKE, dtype=0, batch=4, heads=8, head_dim=64, lses=FAKE, shards=8, rank=3,
             new_out=FAKE)
    a.update(kw)
    B, H, D = a["batch"], a["heads"], a["head_dim"]
    st = lib.dsa_correct_attn_out(a["out"], a["dtype"], B, H, D, H * D, D, 1, a["lses"],
                                  a["shards"], B * H, H, 1, a["rank"], a["new_out"], B * D, D, 1,
                                  None, H, 1, None)
    assert st == want


@pytest.mark.parametrize("kw,want", [
    (dict(dtype=-1), DSA_EINVAL),
    (dict(shards=0), DSA_EINVAL),
    (dict(heads=-1), DSA_EINVAL),
    (dict(lses=None), DSA_EINVAL),
    (dict(outs=None), DSA_EINVAL),
    (dict(merged=None), DSA_EINVAL),
    (dict(shards=64), DSA_EUNSUPPORTED),
    (dict(batch=0), DSA_OK),
])
def test_merge_attn_out_validation(lib, kw, want):
    a = dict(outs=FAKE, dtype=1, shards=4, batch=4, heads=8, head_dim=64, lses=FAKE,
             merged=FAKE)
    a.update(kw)
    N, B, H, D = a["shards"], a["batch"], a["heads"], a["head_dim"]
    st = lib.dsa_merge_attn_out(a["outs"], a["dtype"], N, B, H, D, B * H * D, H * D, D, 1,
                                a["lses"], B * H, H, 1, a["merged"], B * D, D, 1, None, H, 1,
                                None)
    assert st == want


def test_attn_limits(lib):
    assert lib.dsa_attn_max_shards() == 32


def test_mapped_host_pointer_null_arguments(lib):
    out = ctypes.c_void_p(7)
    assert lib.dsa_mapped_host_pointer(None, ctypes.byref(out)) == DSA_EINVAL
    buf = ctypes.create_string_buffer(64)
    assert lib.dsa_mapped_host_pointer(ctypes.addressof(buf), None) == DSA_EINVAL
    assert out.value == 7
