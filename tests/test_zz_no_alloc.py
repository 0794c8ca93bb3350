"""kp_indexer_score_noalloc against kp_indexer_score, through the C ABI.

The no-allocation variant serves callers that cannot allocate device memory
when they score (their framework's allocator forbids raw allocations, or they
are handed only input and output buffers): it keeps its work plan in a device
array inside the library instead of a caller workspace.  It must give the same
scores as the workspace variant, and a second call must not be disturbed by
what the first left in the shared array.  This file is named to be collected
last, so that a run stopping at the first failure has run every other test.
"""
import numpy as np
import pytest
import torch

import kpool_inputs as KI
import parity_lib as PL
import dsa_indexer_sparse_kpool_b300 as kp

pytestmark = pytest.mark.gpu


def _scores_both_ways(wl):
    sess, step = PL.make_gpu(wl)
    step.run()                                  # appends the step's tokens to the pooled cache
    cfg, NQ = sess.cfg, wl.NQ
    stride = kp.score_stride(step.queries.max_pools)
    ref = torch.full((NQ, stride), float("nan"), dtype=torch.float32, device=sess.device)
    got = torch.full((NQ, stride), float("nan"), dtype=torch.float32, device=sess.device)
    ws = torch.empty(kp.kp_score_workspace_size(NQ), dtype=torch.uint8, device=sess.device)
    kp.kp_indexer_score(cfg, step.seqs, step.queries, step.q_idx, step.w, sess.pooled, ref, ws,
                        d_status=sess.status)
    kp.kp_indexer_score_noalloc(cfg, step.seqs, step.queries, step.q_idx, step.w, sess.pooled, got,
                                d_status=sess.status)
    torch.cuda.synchronize()
    assert int(sess.status.item()) == 0
    return wl, ref.cpu().numpy(), got.cpu().numpy()


def _compare(wl, ref, got):
    for q in range(wl.NQ):
        nf = (int(wl.q_pos[q]) + 1) // wl.spec.kpool
        span = (nf + 127) // 128 * 128
        # the masked entries n_full .. next multiple of 128 are -inf in both
        assert np.array_equal(np.isneginf(ref[q, :span]), np.isneginf(got[q, :span]))
        PL.check_scores_row(got[q], ref[q, :nf].astype(np.float64))


def test_noalloc_scores_match_workspace_variant_twice():
    # first call: three sequences, ragged tails, several 128-pool tiles
    first = KI.make(KI.Spec("noalloc-a", [1000, 1537, 2050], [1, 3, 5], topk_tokens=256, seed=21))
    _compare(*_scores_both_ways(first))
    # second call right after: more queries and a different grouping, so any
    # plan entries left over from the first call would be read if they leaked
    second = KI.make(KI.Spec("noalloc-b", [515, 4099, 600], [9, 8, 2], topk_tokens=256, seed=22))
    _compare(*_scores_both_ways(second))



def test_noalloc_at_the_query_limit_and_past_the_shared_plan_stage():
    # 8,192 queries (KP_NOALLOC_MAX_QUERIES: the plan fills the whole device
    # array) and then 5,003: both too many for the scorer to hold the plan's
    # group table in shared memory, so it reads the table from the array
    assert kp.NOALLOC_MAX_QUERIES == 8192
    full = KI.make(KI.Spec("noalloc-c", [2100, 2200, 2300, 2400], [2048] * 4, topk_tokens=256, seed=23))
    assert full.NQ == kp.NOALLOC_MAX_QUERIES
    _compare(*_scores_both_ways(full))
    mid = KI.make(KI.Spec("noalloc-d", [2000, 2500, 1100], [2000, 2000, 1003], topk_tokens=256, seed=24))
    assert 4096 < mid.NQ < kp.NOALLOC_MAX_QUERIES
    _compare(*_scores_both_ways(mid))
