"""Pools of 16 tokens: NeMo AutoModel's Glm5NextTextConfig default
(index_kpool 16), next to the checkpoint's 4.  Same method with kpool = 16: a
pooled key per 16 keys, n_full(t) = floor((t + 1) / 16), a tail of up to 15
tokens, topk_tokens / 16 pools selected.  Compared with the oracle run with
kpool = 16, and the paged layout with the contiguous one, bit for bit.
"""
import numpy as np
import pytest
import torch

import kpool_inputs as KI
import parity_lib as PL
from dsa_indexer_sparse_kpool_b300 import COMPRESS_MEAN

pytestmark = pytest.mark.gpu


def spec(lens, n_q, topk, seed, **kw):
    return KI.Spec("kp16", list(lens), list(n_q), topk_tokens=topk, seed=seed, kpool=16, **kw)


def test_kpool16_multi_tile_ragged():
    wl = KI.make(spec([1000, 1537, 2050], [1, 3, 5], 256, 91))
    assert wl.k_pools == 16
    PL.full_check(wl)
    PL.fused_check(wl)


def test_kpool16_every_tail_length():
    # 16 consecutive positions: tails of 0 .. 15 tokens, and more pools than K
    wl = KI.make(spec([2700], [16], 512, 92))
    PL.full_check(wl)


def test_kpool16_mean_mode_without_tail():
    wl = KI.make(spec([901, 1026], [3, 2], 128, 93))
    cfg = PL.cfg_of(wl, compress_mode=COMPRESS_MEAN, always_select_tail=False)
    PL.full_check(wl, cfg=cfg)


@pytest.mark.parametrize("page_tokens", [64, 1024])
def test_kpool16_paged_equals_contiguous(page_tokens):
    wl = KI.make(spec([1000, 1537, 515], [1, 3, 9], 256, 94))
    a_sess, a_step = PL.make_gpu(wl)
    a_step.run()
    b_sess, b_step = PL.make_gpu(wl, page_tokens=page_tokens, page_seed=5)
    b_step.run()
    torch.cuda.synchronize()
    assert int(a_sess.status.item()) == 0 and int(b_sess.status.item()) == 0
    for s in range(wl.B):
        assert np.array_equal(PL.gpu_pooled_of_seq(a_sess, wl, s), PL.gpu_pooled_of_seq(b_sess, wl, s))
    assert torch.equal(a_step.pool_idx, b_step.pool_idx) and torch.equal(a_step.out, b_step.out)
    assert torch.equal(a_step.lse, b_step.lse)


def test_kpool16_decode_full_size():
    s = KI.named("decode")
    s.kpool = 16
    wl = KI.make(s)
    assert wl.k_pools == 128
    PL.fused_check(wl, queries=[0, 9, 31], check_all_pooled=False)
