"""Paged caches: the latent and pooled caches split into pages named by a
per-sequence block table (the KV-pool pages of the MAX docs,
Glm5NextConfig.infer_optimal_batch_size; the Rust loader's persistent block
table, Mixer::Dsa), with pages handed out in a shuffled order.

The arithmetic does not depend on where a row lives, so a paged step must give
the contiguous step's results bit for bit (pooled keys in pool order,
selection, outputs, lse), and the oracle comparison must hold as well.
"""
import numpy as np
import pytest
import torch

import kpool_inputs as KI
import parity_lib as PL

pytestmark = pytest.mark.gpu

BOUNDS = 5


def _run(wl, page_tokens, page_seed=0):
    sess, step = PL.make_gpu(wl, page_tokens=page_tokens, page_seed=page_seed)
    step.run()
    torch.cuda.synchronize()
    assert int(sess.status.item()) == 0, f"device status {int(sess.status.item())}"
    return sess, step


def _same(wl, a, b):
    (sa, ta), (sb, tb) = a, b
    for s in range(wl.B):
        assert np.array_equal(PL.gpu_pooled_of_seq(sa, wl, s), PL.gpu_pooled_of_seq(sb, wl, s))
    assert torch.equal(ta.n_sel, tb.n_sel) and torch.equal(ta.pool_idx, tb.pool_idx)
    assert torch.equal(ta.out, tb.out) and torch.equal(ta.lse, tb.lse)


@pytest.mark.parametrize("page_tokens", [16, 64, 256, 2048])
def test_paged_equals_contiguous_and_oracle(page_tokens):
    # several 128-pool score tiles per sequence (tiles span 1 .. 32 pages),
    # ragged tails, a 9-query group
    wl = KI.make(KI.Spec("paged", [1000, 1537, 2050, 515], [1, 3, 5, 9], topk_tokens=256, seed=61))
    contiguous = _run(wl, None)
    paged = _run(wl, page_tokens, page_seed=page_tokens)
    _same(wl, contiguous, paged)
    PL.full_check(wl, page_tokens=page_tokens)


def test_paged_decode_full_size():
    wl = KI.make(KI.named("decode"))
    _same(wl, _run(wl, None), _run(wl, 64, page_seed=1))
    PL.fused_check(wl, queries=[0, 17, 31], check_all_pooled=False, page_tokens=64)


def test_paged_ragged_full_size():
    wl = KI.make(KI.named("ragged"))
    _same(wl, _run(wl, None), _run(wl, 128, page_seed=2))
    PL.fused_check(wl, queries=[1, 8, 14], check_all_pooled=False, page_tokens=128)


def test_paged_prefill_full_size():
    wl = KI.make(KI.named("prefill"))
    _same(wl, _run(wl, None), _run(wl, 64, page_seed=3))
    PL.fused_check(wl, queries=[0, 2049, 4095], check_all_pooled=False, page_tokens=64)


def test_bad_page_id_is_skipped_and_reported():
    wl = KI.make(KI.Spec("paged-bad", [1000, 1537], [2, 3], topk_tokens=256, seed=62))
    sess, step = _run(wl, 64)
    n_pages = sess.latent.shape[0] // 64
    sess.block_table[1, 3] = n_pages + 7       # a page id past the caches
    sess.block_table[0, 1] = -3
    step.run()
    torch.cuda.synchronize()
    assert int(sess.status.item()) == BOUNDS
