"""Edge cases of the step through the C ABI, against the oracle:

  * the largest top-k budget (KP_MAX_TOPK_POOLS = 1024 pools, 4096 tokens);
  * pools of 16 tokens through the fused score-and-select and with a shared
    selection;
  * the allocation-free scorer on paged caches;
  * a step with new tokens and no queries (compression only).
"""
import numpy as np
import pytest
import torch

import kpool_inputs as KI
import oracle
import parity_lib as PL
import dsa_indexer_sparse_kpool_b300 as kp

pytestmark = pytest.mark.gpu


def test_largest_topk_budget():
    # K = 4096 / 4 = 1024 pools: 64 tiles of attention per query; the second
    # sequence's rows have more pools than K, the first's fewer
    wl = KI.make(KI.Spec("edge", [3001, 20003], [2, 3], topk_tokens=4 * kp.MAX_TOPK_POOLS, seed=71))
    PL.fused_check(wl, queries=[0, 1, 2, 4])


def test_kpool16_fused_select_and_shared_selection():
    wl = KI.make(KI.Spec("edge", [5000, 40001], [2, 2], topk_tokens=2048, seed=72, kpool=16))
    PL.fused_check(wl)   # the forward in both select modes, bit for bit against the staged calls
    sess, step = PL.make_gpu(wl, PL.cfg_of(wl, select_mode=kp.SELECT_FUSED))
    share = [-1, 0, -1, 2]
    step.set_share(share)
    step.run()
    torch.cuda.synchronize()
    assert int(sess.status.item()) == 0
    g_idx, g_n = step.pool_idx.cpu().numpy(), step.n_sel.cpu().numpy()
    out, lse = step.out.float().cpu().numpy(), step.lse.cpu().numpy()
    for q in (1, 3):
        src = share[q]
        o_out, o_lse = PL.oracle_attend_on_selection(wl, q, g_idx[src][:int(g_n[src])])
        PL.check_attend(out[q], lse[q], o_out, o_lse)


@pytest.mark.parametrize("page_tokens", [64, 512])
def test_noalloc_scorer_on_paged_caches(page_tokens):
    wl = KI.make(KI.Spec("edge", [1000, 4099, 2050], [1, 3, 5], topk_tokens=256, seed=73))
    sess, step = PL.make_gpu(wl, page_tokens=page_tokens)
    step.run()
    NQ = wl.NQ
    stride = kp.score_stride(step.queries.max_pools)
    ref = torch.full((NQ, stride), float("nan"), dtype=torch.float32, device=sess.device)
    got = torch.full((NQ, stride), float("nan"), dtype=torch.float32, device=sess.device)
    ws = torch.empty(kp.kp_score_workspace_size(NQ), dtype=torch.uint8, device=sess.device)
    kp.kp_indexer_score(sess.cfg, step.seqs, step.queries, step.q_idx, step.w, sess.pooled, ref, ws,
                        d_status=sess.status)
    kp.kp_indexer_score_noalloc(sess.cfg, step.seqs, step.queries, step.q_idx, step.w, sess.pooled, got,
                                d_status=sess.status)
    torch.cuda.synchronize()
    assert int(sess.status.item()) == 0
    ref, got = ref.cpu().numpy(), got.cpu().numpy()
    for q in range(NQ):
        nf = (int(wl.q_pos[q]) + 1) // 4
        assert np.array_equal(ref[q, :nf], got[q, :nf])
        o_sc = PL.oracle_scores_on(PL.gpu_pooled_of_seq(sess, wl, int(wl.q_seq[q])), wl, q)
        PL.check_scores_row(got[q], o_sc)


def test_step_with_new_tokens_and_no_queries():
    from dsa_indexer_sparse_kpool_b300.session import Step, build_session
    wl = KI.make(KI.Spec("edge", [1030, 515], [6, 3], topk_tokens=256, seed=74))
    cfg = PL.cfg_of(wl)
    sess = build_session(cfg, wl.lens.tolist(), wl.prev_len.tolist(), wl.tok_off.tolist(), wl.pool_off.tolist(),
                         wl.pool_rows, wl.latent, wl.keys, wl.gates, wl.ape)
    counts = [int(x) for x in (wl.lens - wl.prev_len)]
    idx = torch.cat([torch.arange(int(wl.tok_off[b] + wl.prev_len[b]), int(wl.tok_off[b] + wl.lens[b]))
                     for b in range(wl.B)])
    step = Step(sess, wl.prev_len.tolist(), counts, wl.keys[idx], wl.gates[idx], [], [], wl.q_idx[:0], wl.w[:0],
                wl.q_lat[:0])
    assert step.launches_per_step() == 1
    step.run()
    torch.cuda.synchronize()
    assert int(sess.status.item()) == 0
    PL.check_pooled(sess, wl)     # the appended pools (and the older ones) against the oracle


@pytest.mark.parametrize("nq", [16, 26, 40])
def test_cluster_sizes_that_do_not_divide_the_heads(nq):
    # 16, 26 and 40 queries take clusters of 6, 5 and 3 CTAs on a 148-SM B300
    # (the largest split count whose clusters all fit at once), so the CTAs
    # merge 10-11, 12-13 and 21-22 of the 64 heads; every stage of every
    # query against the oracle, through the forward call
    lens = [6000 + 37 * i for i in range(4)]
    per = [nq // 4 + (1 if i < nq % 4 else 0) for i in range(4)]
    wl = KI.make(KI.Spec("edge", lens, per, topk_tokens=2048, seed=90 + nq))
    PL.full_check(wl, stages=False)
