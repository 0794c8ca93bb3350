"""Failure detection on the GPU, in the forms that leave the context usable.

* A wait that runs out: KP_DEBUG_STALL_FIRST_WAIT makes the first pipeline
  wait of the scoring or attention kernel wait on a barrier that nothing
  completes, with a short per-call limit (kp_config.wait_limit_us).  The
  kernel must record KP_ERR_DEVICE_TIMEOUT, let every copy and MMA it issued
  finish, free its tensor memory and return; the next call on the same stream
  must then give the same bits as before.
* Bad data: an out-of-range pool index or a query past its sequence's length
  is skipped (never dereferenced) and reported as KP_ERR_DEVICE_BOUNDS.

No test here faults, traps or hangs the GPU: every wait has a limit and the
bad indices are caught before any memory access.
"""
import dataclasses

import pytest
import torch

import kpool_inputs as KI
import parity_lib as PL
import dsa_indexer_sparse_kpool_b300 as kp

pytestmark = pytest.mark.gpu

TIMEOUT, BOUNDS = 4, 5


def _ready(lens, n_q, seed):
    wl = KI.make(KI.Spec("fail", lens, n_q, topk_tokens=256, seed=seed))
    sess, step = PL.make_gpu(wl)
    step.run()
    torch.cuda.synchronize()
    assert int(sess.status.item()) == 0
    return wl, sess, step


def _attend(sess, step, cfg, out, lse, seqs=None, pool_idx=None):
    NQ = out.shape[0]
    aws = torch.empty(max(256, kp.kp_attend_workspace_size(cfg, NQ)), dtype=torch.uint8, device=sess.device)
    kp.kp_sparse_mla_attend(cfg, seqs or step.seqs, step.queries, step.q_lat, sess.latent,
                            step.pool_idx if pool_idx is None else pool_idx, step.n_sel, out, lse, aws,
                            d_status=sess.status)


@pytest.mark.parametrize("lens,n_q", [
    ([1000, 1537], [2, 3]),      # 5 queries: each split over a 4-CTA cluster
    ([3000], [100]),             # 100 queries: one CTA each
])
def test_attention_wait_runs_out_then_next_call_is_exact(lens, n_q):
    wl, sess, step = _ready(lens, n_q, seed=51)
    stall = dataclasses.replace(sess.cfg, wait_limit_us=2000, debug_flags=kp.DEBUG_STALL_FIRST_WAIT)
    out, lse = torch.empty_like(step.out), torch.empty_like(step.lse)
    _attend(sess, step, stall, out, lse)
    assert kp.kp_read_device_status(sess.status) == TIMEOUT
    sess.status.zero_()
    out2, lse2 = torch.empty_like(step.out), torch.empty_like(step.lse)
    _attend(sess, step, sess.cfg, out2, lse2)
    assert kp.kp_read_device_status(sess.status) == 0
    assert torch.equal(out2, step.out) and torch.equal(lse2, step.lse)


def test_scorer_wait_runs_out_then_next_call_is_exact():
    wl, sess, step = _ready([1000, 1537, 2050], [1, 3, 5], seed=52)
    NQ = wl.NQ
    stride = kp.score_stride(step.queries.max_pools)
    ws = torch.empty(kp.kp_score_workspace_size(NQ), dtype=torch.uint8, device=sess.device)
    ref = torch.empty(NQ, stride, dtype=torch.float32, device=sess.device)
    kp.kp_indexer_score(sess.cfg, step.seqs, step.queries, step.q_idx, step.w, sess.pooled, ref, ws,
                        d_status=sess.status)
    assert kp.kp_read_device_status(sess.status) == 0
    stall = dataclasses.replace(sess.cfg, wait_limit_us=2000, debug_flags=kp.DEBUG_STALL_FIRST_WAIT)
    junk = torch.empty_like(ref)
    kp.kp_indexer_score(stall, step.seqs, step.queries, step.q_idx, step.w, sess.pooled, junk, ws,
                        d_status=sess.status)
    assert kp.kp_read_device_status(sess.status) == TIMEOUT
    sess.status.zero_()
    again = torch.empty_like(ref)
    kp.kp_indexer_score(sess.cfg, step.seqs, step.queries, step.q_idx, step.w, sess.pooled, again, ws,
                        d_status=sess.status)
    assert kp.kp_read_device_status(sess.status) == 0
    for q in range(NQ):
        n = (int(wl.q_pos[q]) + 1) // 4
        assert torch.equal(again[q, :n], ref[q, :n])


def test_out_of_range_pool_index_is_skipped_and_reported():
    wl, sess, step = _ready([1000, 1537], [2, 3], seed=53)
    bad = step.pool_idx.clone()
    nf = (int(wl.q_pos[2]) + 1) // 4
    bad[2, 0] = nf + 5           # past the query's complete pools
    bad[2, 7] = -7
    out, lse = torch.empty_like(step.out), torch.empty_like(step.lse)
    _attend(sess, step, sess.cfg, out, lse, pool_idx=bad)
    assert kp.kp_read_device_status(sess.status) == BOUNDS
    # the other queries are untouched by query 2's bad entries
    for q in (0, 1, 3, 4):
        assert torch.equal(out[q], step.out[q]) and torch.equal(lse[q], step.lse[q])
    sess.status.zero_()
    _attend(sess, step, sess.cfg, out, lse)
    assert kp.kp_read_device_status(sess.status) == 0
    assert torch.equal(out, step.out)


def test_query_past_its_sequence_is_skipped_and_reported():
    wl, sess, step = _ready([1000, 1537], [2, 3], seed=54)
    short = sess.seq_len.clone()
    short[1] = int(wl.q_pos[4])          # the last query of sequence 1 sits at its length
    seqs = dataclasses.replace(sess.seqs(), seq_len=short)
    out, lse = torch.empty_like(step.out), torch.empty_like(step.lse)
    _attend(sess, step, sess.cfg, out, lse, seqs=seqs)
    assert kp.kp_read_device_status(sess.status) == BOUNDS
    assert int(torch.count_nonzero(out[4])) == 0 and bool(torch.isneginf(lse[4]).all())
    for q in range(4):
        assert torch.equal(out[q], step.out[q]) and torch.equal(lse[q], step.lse[q])
