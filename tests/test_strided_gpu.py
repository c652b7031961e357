"""The DCP form on shard and row strides other than the packed ones.

The sharded entry points take any row stride (ld >= local_width) and shard
stride, and pick the vector width from the alignment of every shard and row
origin. Each case here passes a view into a padded buffer,
[D, rows + 2, local_width + pad] with the view starting one row in, and
fills the padding with 1e30, which would win any max if it were read. Ids
and scores must equal the oracle's on the packed logits, the padding must
come back untouched, and the masking pass must write the same bits as on
packed logits.
"""

import numpy as np
import pytest

import oracle
import workloads
from helpers import assert_bits_equal

pytestmark = pytest.mark.gpu

PAD_FILL = np.float32(1e30)


@pytest.fixture(scope="module")
def env():
    import torch

    import __graft_entry__

    __graft_entry__.build()
    import deepseek_sparse_attention_row_gb300 as dsa

    if not torch.cuda.is_available():
        pytest.skip("needs a CUDA device")
    return torch, dsa


def padded_view(torch, local, pad, dtype):
    """[D, rows, lw] values inside a [D, rows + 2, lw + pad] buffer."""
    D, rows, lw = local.shape
    buf = torch.full((D, rows + 2, lw + pad), float(PAD_FILL), dtype=dtype, device="cuda")
    view = buf[:, 1:rows + 1, :lw]
    view.copy_(torch.from_numpy(local).to(dtype))
    return buf, view


def padding_intact(torch, buf, rows, lw):
    host = buf.float().cpu().numpy()
    inner = np.zeros(host.shape, dtype=bool)
    inner[:, 1:rows + 1, :lw] = True
    fill = torch.tensor(float(PAD_FILL), dtype=buf.dtype).float().item()  # as stored
    return bool((host[~inner] == np.float32(fill)).all())


CASES = [(pad, starts, bf16) for pad in (0, 1, 2, 4, 8) for starts in (False, True)
         for bf16 in (False, True)]


@pytest.mark.parametrize("pad,starts,bf16", CASES,
                         ids=[f"pad{p}-{'starts' if s else 'nostarts'}-{'bf16' if b else 'f32'}"
                              for p, s, b in CASES])
def test_sharded_select_and_mask_on_padded_view(env, pad, starts, bf16):
    torch, dsa = env
    seed = 900 + 10 * pad + 2 * int(starts) + int(bf16)
    wl, _ = workloads.small_sharded(seed, shards=8, rows=12, global_width=8 * 1000,
                                    global_block_size=64, max_global_blocks=125,
                                    topk_blocks=16, row_repeat=3)
    if bf16:
        wl.logits = workloads.round_to_bf16_grid(wl.logits)
    gks = None
    if starts:
        rng = np.random.default_rng(seed)
        gks = rng.integers(0, np.maximum(wl.global_row_ke, 0), endpoint=True).astype(np.int32)
        wl.global_row_ks = gks
    want_ids, want_scores = oracle.run_workload(wl)
    D, rows, lw = wl.logits.shape
    dtype = torch.bfloat16 if bf16 else torch.float32
    buf, view = padded_view(torch, wl.logits, pad, dtype)
    gke_d = torch.from_numpy(wl.global_row_ke).cuda()
    gks_d = None if gks is None else torch.from_numpy(gks).cuda()
    out = torch.full((rows, 16), -7, dtype=torch.int32, device="cuda")
    scores = torch.empty((rows, 125), dtype=dtype, device="cuda")
    for ws in (None, False):
        out.fill_(-7)
        dsa.dsa_select_candidate_blocks_sharded(view, gke_d, 64, 125, 16, out, 3,
                                                scores_out=scores, workspace=ws,
                                                global_row_ks=gks_d)
        torch.cuda.synchronize()
        np.testing.assert_array_equal(out.cpu().numpy(), want_ids)
        assert_bits_equal(scores.float().cpu().numpy(), want_scores)
    assert padding_intact(torch, buf, rows, lw), "padding was written"

    # The masking pass after it, in place on the strided view.
    ids = want_ids
    if starts:
        want_masked = oracle.mask_sharded_starts(wl.logits, gks, wl.global_row_ke, 64, ids, 3)
    else:
        want_masked = oracle.mask_sharded(wl.logits, wl.global_row_ke, 64, ids, 3)
    dsa.dsa_mask_candidate_logits_sharded(view, gke_d, 64, out, 3, global_row_ks=gks_d)
    torch.cuda.synchronize()
    assert_bits_equal(view.float().cpu().numpy(), want_masked)
    assert padding_intact(torch, buf, rows, lw), "masking wrote into the padding"
