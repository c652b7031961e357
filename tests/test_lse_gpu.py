"""GPU parity of the DCP partial-attention LSE correction and merge against
the CPU oracle (``oracle/dcp_lse_oracle.c``), through the C ABI.

The kernels compute in fp32 (exp2f, log2f, fp32 products and fused
multiply-adds) and the oracle in double, so results are compared within a
bound derived from fp32 rounding, per (token, head), from the inputs:

* u = 2^-24 (fp32 unit roundoff); M = the largest |finite LSE| of the row;
  N shards.
* The combined LSE F: the shifted exponents x_n - m round by u|x_n - m|
  <= 2uM, exp2f is within 2 ulp (4u relative), the sum of N terms in [0, N]
  adds N u relative, log2f adds 1 ulp of a value below log2 N + 1, and the
  final + m rounds by u|F|. Converting the relative error of the sum to an
  absolute error of its log2 divides by ln 2, so
      eps_F <= u (3M + 1.45 N + 3 log2 N + 8).
* A share f = exp2f(l - F): the difference adds u(|l| + |F|) to eps_F, and
  exp2f turns an absolute exponent error e into a relative error ln2 e, plus
  its own 4u:  rel_f <= ln2 (eps_F + u(|l| + |F|)) + 4u.
* f * o rounds once more (u for fp32 output, 2^-9 for bf16 output).
* The merge sums N such products with N fused multiply-adds: the bound is
  (max_n rel_f_n + N u) * sum_n |f_n o_n| (+ the output rounding).
Every bound is doubled, and an absolute 2^-146 (|o| + 1) covers shares in
fp32's subnormal range, where exp2f's 2 ulp are absolute. NaN and infinite
results must match exactly in position.
"""

import math

import numpy as np
import pytest

import oracle
import workloads

pytestmark = pytest.mark.gpu

U = 2.0 ** -24


@pytest.fixture(scope="module")
def env():
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import deepseek_sparse_attention_row_gb300 as dsa

    assert torch.cuda.is_available(), "these tests need a CUDA device"
    return torch, dsa


def _clean(lses):
    return np.where(np.isnan(lses) | (lses == np.inf), -np.inf, lses).astype(np.float64)


def _eps_F(lses):
    """Bound on the combined LSE's absolute error, per [B, H]."""
    N = lses.shape[0]
    c = _clean(lses)
    fin = np.where(np.isfinite(c), np.abs(c), 0.0)
    M = fin.max(axis=0)
    return U * (3 * M + 1.45 * N + 3 * math.log2(max(N, 1)) + 8)


def _rel_share(lses, F, eps_F, n):
    """Bound on shard n's share's relative error, per [B, H]."""
    l = lses[n].astype(np.float64)
    la = np.where(np.isfinite(l), np.abs(l), 0.0)
    Fa = np.where(np.isfinite(F), np.abs(F), 0.0)
    return math.log(2) * (eps_F + U * (la + Fa)) + 4 * U


def _assert_within(got, want, tol, what):
    got = np.asarray(got, np.float64)
    want = np.asarray(want, np.float64)
    assert got.shape == want.shape, (what, got.shape, want.shape)
    nan_g, nan_w = np.isnan(got), np.isnan(want)
    assert np.array_equal(nan_g, nan_w), f"{what}: NaN positions differ"
    inf_w = np.isinf(want)
    assert np.array_equal(got[inf_w], want[inf_w]), f"{what}: infinities differ"
    assert not np.isinf(got[~inf_w & ~nan_w]).any(), f"{what}: unexpected infinity"
    fin = ~nan_w & ~inf_w
    err = np.abs(np.where(fin, got, 0.0) - np.where(fin, want, 0.0))
    bad = fin & (err > np.broadcast_to(tol, got.shape))
    if bad.any():
        idx = np.argwhere(bad)[:5]
        raise AssertionError(f"{what}: {int(bad.sum())} values outside the bound, e.g. "
                             + ", ".join(f"{tuple(i)} got {got[tuple(i)]!r} want "
                                         f"{want[tuple(i)]!r} tol "
                                         f"{np.broadcast_to(tol, got.shape)[tuple(i)]!r}"
                                         for i in idx))


def _out_rounding(dtype):
    return 2.0 ** -9 if dtype == "bf16" else U


def _tdtype(torch, dtype):
    return torch.bfloat16 if dtype == "bf16" else torch.float32


def check_correct(env, outs, lses, rank, dtype, out_dev=None, lses_dev=None):
    """Run the correction of shard `rank` on the GPU and compare."""
    torch, dsa = env
    o = outs[rank]
    if out_dev is None:
        out_dev = torch.from_numpy(np.ascontiguousarray(o)).cuda().to(_tdtype(torch, dtype))
    if lses_dev is None:
        lses_dev = torch.from_numpy(lses).cuda()
    new, lse = dsa.dsa_correct_attn_out(out_dev, lses_dev, rank)
    torch.cuda.synchronize()
    want, want_lse = oracle.correct_attn_out(o, lses, rank)
    eF = _eps_F(lses)
    _assert_within(lse.cpu().numpy(), want_lse, 2 * eF, "combined LSE")
    rel = 2 * (_rel_share(lses, want_lse, eF, rank) + _out_rounding(dtype))   # [B, H]
    tol = rel.T[:, :, None] * np.abs(want) + 2.0 ** -146 * (np.abs(o).transpose(1, 0, 2) + 1)
    _assert_within(new.float().cpu().numpy(), want, tol, f"corrected output (rank {rank})")


def check_merge(env, outs, lses, dtype, outs_dev=None):
    torch, dsa = env
    N = outs.shape[0]
    if outs_dev is None:
        outs_dev = torch.from_numpy(np.ascontiguousarray(outs)).cuda().to(_tdtype(torch, dtype))
    merged, lse = dsa.dsa_merge_attn_out(outs_dev, torch.from_numpy(lses).cuda())
    torch.cuda.synchronize()
    want, want_lse = oracle.merge_attn_out(outs, lses)
    eF = _eps_F(lses)
    _assert_within(lse.cpu().numpy(), want_lse, 2 * eF, "combined LSE")
    mag = np.zeros_like(want)
    rel = np.zeros(lses.shape[1:])
    for n in range(N):
        mag += oracle.correct_attn_out(np.abs(outs[n]), lses, n)[0]
        rel = np.maximum(rel, _rel_share(lses, want_lse, eF, n))
    tol = 2 * ((rel.T[:, :, None] + N * U) * mag + _out_rounding(dtype) * np.abs(want)) \
        + 2.0 ** -146 * (mag + 1)
    _assert_within(merged.float().cpu().numpy(), want, tol, "merged output")


# ---------------------------------------------------------------------------
# Small and mid-size sweeps
# ---------------------------------------------------------------------------

SHAPES = [  # (N, B, H, Dh)
    (1, 3, 2, 64), (2, 5, 4, 128), (3, 7, 3, 4), (4, 16, 8, 64), (5, 2, 9, 512),
    (8, 33, 16, 512), (8, 64, 128, 576), (16, 9, 7, 3), (32, 4, 5, 256), (8, 1, 1, 1),
]


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
@pytest.mark.parametrize("shape", SHAPES, ids=[str(s) for s in SHAPES])
def test_correct_and_merge_sweep(env, shape, dtype):
    N, B, H, D = shape
    wl = workloads.make_lse(1000 + N * 7 + D, shards=N, batch=B, heads=H, head_dim=D,
                            dtype=dtype, specials=True)
    for rank in sorted({0, N // 2, N - 1}):
        check_correct(env, wl.outs, wl.lses, rank, dtype)
    check_merge(env, wl.outs, wl.lses, dtype)


@pytest.mark.parametrize("dtype", ["f32", "bf16"])
def test_named_tiny(env, dtype):
    wl = workloads.make_lse_named("lse_tiny")
    outs = workloads.round_to_bf16_grid(wl.outs) if dtype == "bf16" else wl.outs
    for rank in range(wl.shards):
        check_correct(env, outs, wl.lses, rank, dtype)
    check_merge(env, outs, wl.lses, dtype)


def test_strided_views(env):
    """Views the page passes: [B, 1, H, D] outputs and [N, B, H, 1] LSEs
    (squeezed), an output transposed in memory, a misaligned base, and a
    non-contiguous LSE buffer; all must give the dense results."""
    torch, dsa = env
    N, B, H, D = 4, 6, 5, 64
    wl = workloads.make_lse(77, shards=N, batch=B, heads=H, head_dim=D, specials=True)
    lses_t = torch.from_numpy(wl.lses).cuda()
    # [B, 1, H, D] output and [N, B, H, 1] LSEs
    o4 = torch.from_numpy(wl.outs[2]).cuda().unsqueeze(1)
    check_correct(env, wl.outs, wl.lses, 2, "f32", out_dev=o4,
                  lses_dev=lses_t.unsqueeze(-1))
    # output stored [H, B, D] in memory, viewed as [B, H, D]
    ot = torch.from_numpy(np.ascontiguousarray(wl.outs[1].transpose(1, 0, 2))).cuda()
    check_correct(env, wl.outs, wl.lses, 1, "f32", out_dev=ot.permute(1, 0, 2))
    # misaligned base (4 bytes past a 16-byte boundary)
    buf = torch.zeros(B * H * D + 1, dtype=torch.float32, device="cuda")
    mis = buf[1:].view(B, H, D)
    mis.copy_(torch.from_numpy(wl.outs[3]))
    check_correct(env, wl.outs, wl.lses, 3, "f32", out_dev=mis)
    # LSEs as a strided slice of a wider buffer
    wide = torch.zeros((N, B, H + 3), dtype=torch.float32, device="cuda")
    wide[:, :, :H] = lses_t
    check_correct(env, wl.outs, wl.lses, 0, "f32", lses_dev=wide[:, :, :H])
    # merge over a non-contiguous shard axis
    big = torch.zeros((N, B, H, D + 4), dtype=torch.float32, device="cuda")
    big[..., :D] = torch.from_numpy(wl.outs).cuda()
    check_merge(env, wl.outs, wl.lses, "f32", outs_dev=big[..., :D])


def test_head_dim_zero_writes_only_the_lse(env):
    torch, dsa = env
    N, B, H = 3, 4, 5
    wl = workloads.make_lse(5, shards=N, batch=B, heads=H, head_dim=1, specials=True)
    out = torch.empty((B, H, 0), dtype=torch.float32, device="cuda")
    new, lse = dsa.dsa_correct_attn_out(out, torch.from_numpy(wl.lses).cuda(), 1)
    torch.cuda.synchronize()
    _, want_lse = oracle.correct_attn_out(wl.outs[1], wl.lses, 1)
    _assert_within(lse.cpu().numpy(), want_lse, 2 * _eps_F(wl.lses), "combined LSE")
    assert new.shape == (H, B, 0)


def test_invalid_arguments_raise(env):
    torch, dsa = env
    out = torch.zeros((2, 3, 8), device="cuda")
    lses = torch.zeros((33, 2, 3), device="cuda")
    with pytest.raises(dsa.DsaError):
        dsa.dsa_correct_attn_out(out, lses, 0)          # 33 shards: unsupported
    with pytest.raises(dsa.DsaError):
        dsa.dsa_correct_attn_out(out, lses[:4], 4)      # rank outside [0, 4)
    with pytest.raises(TypeError):
        dsa.dsa_correct_attn_out(out.half(), lses[:4], 0)


def test_graph_replay(env):
    torch, dsa = env
    wl = workloads.make_lse(11, shards=8, batch=32, heads=16, head_dim=512)
    outs = torch.from_numpy(wl.outs).cuda()
    lses = torch.from_numpy(wl.lses).cuda()
    merged = torch.empty((16, 32, 512), device="cuda")
    lse = torch.empty((32, 16), device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        dsa.dsa_merge_attn_out(outs, lses, merged, lse)
    torch.cuda.current_stream().wait_stream(s)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        dsa.dsa_merge_attn_out(outs, lses, merged, lse)
    merged.zero_()
    g.replay()
    torch.cuda.synchronize()
    want, _ = oracle.merge_attn_out(wl.outs, wl.lses)
    assert np.abs(merged.cpu().numpy() - want).max() < 1e-4


# ---------------------------------------------------------------------------
# Full size (the bench's workloads), sampled where the oracle is slow
# ---------------------------------------------------------------------------

@pytest.mark.slow
@pytest.mark.parametrize("name", ["lse_decode", "lse_decode_bf16"])
def test_full_size(env, name):
    wl = workloads.make_lse_named(name)
    check_correct(env, wl.outs, wl.lses, 3, wl.dtype)
    check_merge(env, wl.outs, wl.lses, wl.dtype)
