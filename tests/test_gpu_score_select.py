"""GPU parity of kp_indexer_score_select, the scores and the top-k selection in
one kernel with the scores kept on chip: its pool_idx and n_sel must equal,
bit for bit, those of kp_indexer_score followed by kp_topk_select on the same
inputs (the staged calls, themselves checked against the oracle in the other
parity tests, and checked here against the oracle's fp64 scores on sampled
queries).

Cases span the kernel's layouts: one CTA per group (rows up to 2048 pools),
clusters of 2, 4 and 8 CTAs (rows up to 16,384 pools) with several rounds of
rows per cluster, rows of at most K pools (no selection), queries that see no
pool, the plan built in the kernel (<= 510 queries) and by the plan kernel,
paged caches and pools of 16 tokens.
"""
import dataclasses

import numpy as np
import pytest
import torch

import kpool_inputs as KI
import parity_lib as PL
import dsa_indexer_sparse_kpool_b300 as kp

pytestmark = pytest.mark.gpu

BOUNDS = 5


def _fused(sess, step, queries=None):
    q = queries or step.queries
    nq = q.q_seq.numel()
    K = sess.cfg.k_pools
    idx = torch.full((nq, K), -7, dtype=torch.int32, device=sess.device)
    nsel = torch.full((nq,), -7, dtype=torch.int32, device=sess.device)
    ws = torch.empty(kp.kp_score_workspace_size(nq), dtype=torch.uint8, device=sess.device)
    kp.kp_indexer_score_select(sess.cfg, step.seqs, q, step.q_idx, step.w, sess.pooled, idx, nsel, ws,
                               d_status=sess.status)
    return idx, nsel


def _check_against_staged(wl, cfg=None, page_tokens=None, sample=(0,)):
    cfg = cfg or PL.cfg_of(wl)
    sess, step = PL.make_gpu(wl, cfg, page_tokens=page_tokens)
    scores = step.run_stages()
    torch.cuda.synchronize()
    assert int(sess.status.item()) == 0
    idx, nsel = _fused(sess, step)
    torch.cuda.synchronize()
    assert int(sess.status.item()) == 0
    assert torch.equal(nsel, step.n_sel), "n_sel differs from the staged calls"
    assert torch.equal(idx, step.pool_idx), "selection differs from the staged calls"
    # and against the oracle's fp64 scores on a few queries
    g_idx, g_n = idx.cpu().numpy(), nsel.cpu().numpy()
    for qi in sample:
        qi = qi % wl.NQ
        o_sc = PL.oracle_scores_on(PL.gpu_pooled_of_seq(sess, wl, int(wl.q_seq[qi])), wl, qi)
        PL.check_selection_fp64(g_idx[qi], g_n[qi], o_sc, cfg.k_pools)
    return sess, step, scores


@pytest.mark.parametrize("lens,n_q,topk", [
    ([7, 300, 5000, 8195], [3, 5, 6, 9], 256),       # rows of 0 .. 2048 pools: one CTA, trivial rows
    ([20000, 41000], [3, 10], 2048),                 # 5,000 and 10,250 pools: clusters of 4 and 8
    ([9000], [21], 1024),                            # 2250 pools: 6 groups over 2-CTA clusters, 2 rounds
])
def test_matches_staged_calls(lens, n_q, topk):
    wl = KI.make(KI.Spec("ss", lens, n_q, topk_tokens=topk, seed=91))
    _check_against_staged(wl, sample=(0, -1, 7))


def test_decode_shape():
    wl = KI.make(KI.named("decode"))
    _check_against_staged(wl, sample=(0, 13, 31))


def test_plan_from_the_plan_kernel():
    # 1,100 queries: above the in-kernel plan's 510, so the plan kernel builds it
    wl = KI.make(KI.Spec("ss", [2600, 2100], [600, 500], topk_tokens=256, seed=92))
    _check_against_staged(wl, sample=(0, 599, 600, 1099))


def test_paged_caches():
    wl = KI.make(KI.Spec("ss", [3000, 9001, 257], [4, 6, 2], topk_tokens=512, seed=93))
    _check_against_staged(wl, page_tokens=64, sample=(0, 5, 11))


def test_pools_of_16():
    wl = KI.make(KI.Spec("ss", [5000, 70001], [3, 5], topk_tokens=2048, seed=94, kpool=16))
    _check_against_staged(wl, sample=(0, 4, 7))


def test_row_past_max_pools_is_cut_and_reported():
    # max_pools claims 2000 pools, but the last query sees 3000: the kernel
    # (one CTA of 2048 pools per group) scores and selects only what fits,
    # reports KP_ERR_DEVICE_BOUNDS, and reads nothing past its buffers.  The
    # first sequence's queries stay exact.
    wl = KI.make(KI.Spec("ss", [1500, 12000], [3, 1], topk_tokens=256, seed=95))
    sess, step = PL.make_gpu(wl)
    step.run_stages()
    torch.cuda.synchronize()
    assert int(sess.status.item()) == 0
    short = dataclasses.replace(step.queries, max_pools=2000)
    idx, nsel = _fused(sess, step, short)
    assert kp.kp_read_device_status(sess.status) == BOUNDS
    for q in range(3):
        assert torch.equal(idx[q], step.pool_idx[q]) and int(nsel[q]) == int(step.n_sel[q])
    sel = idx[3].cpu().numpy()
    assert int(nsel[3]) == 64 and (np.diff(sel) > 0).all() and sel[0] >= 0 and sel[-1] < 2048
