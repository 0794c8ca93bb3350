"""Shared selection (MAX docs, Glm5NextConfig.index_share_for_mtp_iteration,
read for the MTP verification query of a step): a query q with share_src[q] >= 0
attends the selection of that source query (a query of the same sequence that
selects for itself) plus its own tail, and is not selected itself.

Checks, on the GPU against the oracle:
  * source queries give the bits of a run without sharing;
  * a shared query's pool_idx row and n_sel are left as they were (top-k and
    the fused select both skip it);
  * a shared query's output and lse equal the oracle's attention over the
    source's selection and the query's own tail positions;
  * a bad source (another sequence, a shared query, out of range) is reported
    as KP_ERR_DEVICE_BOUNDS and the query attends its tail alone.
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
SENTINEL = -7


def _mtp_share(wl):
    """Each sequence's second query (t = L - 1) shares its first's (t = L - 2)."""
    share = []
    for q in range(wl.NQ):
        share.append(q - 1 if q > 0 and wl.q_seq[q] == wl.q_seq[q - 1] else -1)
    return share


def _run(wl, mode, share):
    sess, step = PL.make_gpu(wl, PL.cfg_of(wl, select_mode=mode))
    step.set_share(share)
    step.pool_idx.fill_(SENTINEL)
    step.n_sel.fill_(SENTINEL)
    step.run()
    torch.cuda.synchronize()
    return sess, step


def _check_shared(wl, share, sess, step, ref_step, queries=None):
    g_idx = step.pool_idx.cpu().numpy()
    g_n = step.n_sel.cpu().numpy()
    out = step.out.float().cpu().numpy()
    lse = step.lse.cpu().numpy()
    for q in (range(wl.NQ) if queries is None else queries):
        src = share[q]
        if src < 0:   # selects for itself: the unshared run's bits
            assert np.array_equal(g_idx[q], ref_step.pool_idx[q].cpu().numpy())
            assert int(g_n[q]) == int(ref_step.n_sel[q])
            assert torch.equal(step.out[q], ref_step.out[q]) and torch.equal(step.lse[q], ref_step.lse[q])
        else:         # shared: row untouched, attention on the source's selection + own tail
            assert (g_idx[q] == SENTINEL).all() and int(g_n[q]) == SENTINEL
            ns = int(g_n[src])
            o_out, o_lse = PL.oracle_attend_on_selection(wl, q, g_idx[src][:ns])
            PL.check_attend(out[q], lse[q], o_out, o_lse)


@pytest.mark.parametrize("mode", [kp.SELECT_STAGED, kp.SELECT_FUSED])
def test_mtp_query_attends_the_previous_querys_selection(mode):
    # 3 sequences x (t = L - 2, t = L - 1).  In the 5000-token sequence the
    # last query (t = 4999) completes pool 1249, which its source (t = 4998)
    # cannot select: the shared query attends without it (and has no tail).
    wl = KI.make(KI.Spec("mtp", [5000, 9003, 3001], [2, 2, 2], topk_tokens=512, seed=61))
    share = _mtp_share(wl)
    assert share == [-1, 0, -1, 2, -1, 4]
    _, ref_step = PL.make_gpu(wl, PL.cfg_of(wl, select_mode=mode))
    ref_step.run()
    sess, step = _run(wl, mode, share)
    assert int(sess.status.item()) == 0
    _check_shared(wl, share, sess, step, ref_step)


def test_staged_topk_skips_shared_rows():
    wl = KI.make(KI.Spec("mtp", [3000, 4097], [2, 3], topk_tokens=256, seed=62))
    sess, step = PL.make_gpu(wl)
    scores = step.run_stages()
    torch.cuda.synchronize()
    share = [-1, 0, -1, 2, 2]
    queries = dataclasses.replace(step.queries, share_src=torch.tensor(share, dtype=torch.int32, device="cuda"))
    idx = torch.full_like(step.pool_idx, SENTINEL)
    nsel = torch.full_like(step.n_sel, SENTINEL)
    kp.kp_topk_select(sess.cfg, queries, scores, idx, nsel, d_status=sess.status)
    torch.cuda.synchronize()
    assert int(sess.status.item()) == 0
    for q, src in enumerate(share):
        if src < 0:
            assert torch.equal(idx[q], step.pool_idx[q]) and int(nsel[q]) == int(step.n_sel[q])
        else:
            assert bool((idx[q] == SENTINEL).all()) and int(nsel[q]) == SENTINEL


def test_bad_share_source_attends_the_tail_alone():
    wl = KI.make(KI.Spec("mtp", [3000, 4099], [2, 3], topk_tokens=256, seed=63))
    # q1 -> q2 (another sequence), q3 -> q4 (a shared query), q4 -> 9 (out of range)
    share = [-1, 2, -1, 4, 9]
    sess, step = _run(wl, kp.SELECT_STAGED, share)
    assert kp.kp_read_device_status(sess.status) == BOUNDS
    out, lse = step.out.float().cpu().numpy(), step.lse.cpu().numpy()
    for q in (1, 3, 4):
        o_out, o_lse = PL.oracle_attend_on_selection(wl, q, np.zeros(0, np.int32))
        PL.check_attend(out[q], lse[q], o_out, o_lse)


def test_ragged_mtp_full_size_shared():
    wl = KI.make(KI.named("ragged"))
    share = _mtp_share(wl)
    assert sum(s >= 0 for s in share) == 8
    _, ref_step = PL.make_gpu(wl)
    ref_step.run()
    sess, step = _run(wl, kp.SELECT_AUTO, share)
    assert int(sess.status.item()) == 0
    _check_shared(wl, share, sess, step, ref_step, queries=[0, 1, 6, 7, 14, 15])
