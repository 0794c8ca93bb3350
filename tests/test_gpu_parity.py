"""GPU parity of the four stages and the fused step against the fp64 oracle.

Every test calls the library through its C ABI (ctypes binding) on seeded
synthetic inputs and compares stage by stage (see parity_lib for the rules).
"""
import numpy as np
import pytest
import torch

import kpool_inputs as KI
import oracle
import parity_lib as PL
import dsa_indexer_sparse_kpool_b300 as kp
from dsa_indexer_sparse_kpool_b300 import COMPRESS_MEAN

pytestmark = pytest.mark.gpu


def small_spec(lens, n_q, topk_tokens=256, seed=11, **kw):
    return KI.Spec("small", list(lens), list(n_q), topk_tokens=topk_tokens, seed=seed, **kw)


def test_tiny_all_stages_and_fused():
    wl = KI.make(KI.named("tiny"))
    sess, step, rep = PL.full_check(wl)
    # the whole-step call on fresh state, in either select mode, gives the same
    # bits as the staged calls
    for mode in (kp.SELECT_AUTO, kp.SELECT_FUSED):
        sess2, step2 = PL.make_gpu(wl, PL.cfg_of(wl, select_mode=mode))
        step2.run()
        torch.cuda.synchronize()
        assert torch.equal(step2.pool_idx, step.pool_idx) and torch.equal(step2.n_sel, step.n_sel)
        assert torch.equal(step2.out, step.out)
        assert torch.equal(step2.lse, step.lse)
        assert int(sess2.status.item()) == 0


def test_tiny_end_to_end_against_oracle_pipeline():
    """The whole fused step against the oracle's whole pipeline (its own fp64
    pooled keys, scores and selection): every query is compared; where the
    two selections differ, every differing pool must be a near tie of the
    oracle's K-th score, and the output is then compared with the oracle's
    attention on the GPU's selection."""
    wl = KI.make(KI.named("tiny"))
    sess, step = PL.make_gpu(wl)
    step.run()
    torch.cuda.synchronize()
    assert int(sess.status.item()) == 0
    pooled, _ = oracle.kpool_compress(KI.bits(wl.keys), KI.bits(wl.gates), KI.bits(wl.ape), 4)
    ref = oracle.dsa_queries(wl.q_seq, wl.q_pos, np.zeros(1, np.int64), np.zeros(1, np.int64), 4, wl.k_pools, 1,
                             KI.bits(wl.q_idx), wl.w.numpy(), pooled, KI.bits(wl.q_lat), KI.bits(wl.latent),
                             wl.spec.sm_scale)
    g_idx = step.pool_idx.cpu().numpy()
    assert np.array_equal(step.n_sel.cpu().numpy(), ref["n_sel"])
    compared = 0
    for q in range(wl.NQ):
        g_out, g_lse = step.out[q].float().cpu().numpy(), step.lse[q].cpu().numpy()
        if np.array_equal(g_idx[q], ref["sel"][q]):
            PL.check_attend(g_out, g_lse, ref["out"][q], ref["lse"][q])
        else:
            o_sc = oracle.indexer_score(KI.bits(wl.q_idx[q]), wl.w[q].numpy(), pooled,
                                        (int(wl.q_pos[q]) + 1) // 4)
            PL.check_selection_fp64(g_idx[q], step.n_sel[q].item(), o_sc, wl.k_pools)
            ns = int(step.n_sel[q].item())
            o_out, o_lse = PL.oracle_attend_on_selection(wl, q, g_idx[q][:ns])
            PL.check_attend(g_out, g_lse, o_out, o_lse)
        compared += 1
    assert compared == wl.NQ


@pytest.mark.parametrize("lens,n_q,topk", [
    ([1000, 1537, 2050], [1, 3, 5], 256),      # several score tiles, ragged tails, active selection
    ([515, 600], [9, 2], 128),                  # 9 queries of one sequence: two query groups
    ([130], [4], 2048),                          # budget covers every pool
    ([4099], [8], 64),                           # K = 16
])
def test_multi_tile_ragged(lens, n_q, topk):
    wl = KI.make(small_spec(lens, n_q, topk))
    PL.full_check(wl)


def test_peaked_softmax_and_rope_columns():
    spec = small_spec([777, 1203], [2, 3], 256, q_scale=16.0, q_rope_random=True)
    wl = KI.make(spec)
    PL.full_check(wl)


def test_mean_mode_and_no_tail():
    wl = KI.make(small_spec([901, 1026], [3, 2], 128))
    cfg = PL.cfg_of(wl, compress_mode=COMPRESS_MEAN, always_select_tail=False)
    PL.full_check(wl, cfg=cfg)


def test_very_short_sequences():
    # positions 0..3: n_full 0 or 1, tails of 1..3 tokens
    wl = KI.make(small_spec([4, 3, 1, 6], [4, 3, 1, 2], 64))
    PL.full_check(wl)


# The four full-size workloads run through kp_dsa_forward -- the call the
# bench times, in the launch configuration it times -- and are compared bit
# for bit with the four stage calls on fresh state, and with the oracle on
# sampled queries.
def test_decode_config_fused_sampled():
    wl = KI.make(KI.named("decode"))
    PL.fused_check(wl, queries=[0, 13, 31], check_all_pooled=False)


def test_ragged_config_fused_sampled():
    wl = KI.make(KI.named("ragged"))
    PL.fused_check(wl, queries=[0, 5, 15], check_all_pooled=False)


def test_large_logits_exercise_running_max_rescale():
    # logits spread over tens of log2 units, so later tiles raise the running
    # max and the accumulated O and row sums are rescaled
    spec = small_spec([1000, 1537, 2050], [1, 3, 2], 256, q_scale=64.0)
    spec.sm_scale = 4.0
    wl = KI.make(spec)
    PL.full_check(wl)


def test_prefill_chunk_of_64_queries():
    # 64 consecutive positions of one sequence: per-query causal pool limits,
    # all four tail lengths, several score query groups
    wl = KI.make(small_spec([3000], [64], 512, seed=13))
    PL.full_check(wl)


def test_prefill_config_fused_sampled():
    # 4096 queries: above the scorer's shared-memory plan limit, so the fused
    # step builds the plan in the compression launch's extra grid row and the
    # scorer runs with the plan ready
    wl = KI.make(KI.named("prefill"))
    PL.fused_check(wl, queries=[0, 1, 2, 3, 1023, 2047, 4095], check_all_pooled=False)


def test_long_config_fused_sampled():
    wl = KI.make(KI.named("long"))
    PL.fused_check(wl, queries=[0, 1, 2, 3], check_all_pooled=False)


def test_fused_over_1022_queries_small():
    # 1,100 queries over two sequences: the fused step's plan-in-compression
    # branch on a case the oracle checks in full at every 9th query
    wl = KI.make(small_spec([3000, 2500], [700, 400], 256, seed=41))
    assert wl.NQ > 1022
    qs = sorted(set(range(0, wl.NQ, 9)) | {wl.NQ - 1, 699, 700})
    PL.fused_check(wl, queries=qs)


def test_few_queries_full_budget_widest_split():
    # 3 queries with the full 2048-token budget: each query's 32 tiles go to a
    # cluster of 8 CTAs (4 tiles each), whose merge gives every CTA 8 heads;
    # one query has a 3-token tail.
    wl = KI.make(small_spec([9000, 12003], [1, 2], 2048, seed=33))
    PL.fused_check(wl)


def test_exact_ties_in_scores():
    # sequence 0: every pool identical -> all 5000 scores equal (the radix
    # levels run down to a single key value shared by every pool); sequence 1:
    # pooled keys repeat every 10 pools -> 75-fold ties at the threshold.  Ties
    # go to the lower pool index in both.
    wl = KI.make(small_spec([20000, 3000], [1, 2], 256, seed=17))
    a, e = int(wl.tok_off[0]), int(wl.tok_off[0] + wl.lens[0])
    wl.keys[a:e] = wl.keys[a:a + 4].repeat((e - a) // 4, 1)
    wl.gates[a:e] = wl.gates[a:a + 4].repeat((e - a) // 4, 1)
    a, e = int(wl.tok_off[1]), int(wl.tok_off[1] + wl.lens[1])
    wl.keys[a:e] = wl.keys[a:a + 40].repeat((e - a) // 40, 1)
    wl.gates[a:e] = wl.gates[a:a + 40].repeat((e - a) // 40, 1)
    sess, step, rep = PL.full_check(wl)
    sel0 = step.pool_idx[0].cpu().numpy()
    assert np.array_equal(sel0, np.arange(64)), "equal scores must select the lowest pool indices"
    # the same ties through the step with the scores kept on chip
    PL.fused_check(wl, modes=(kp.SELECT_FUSED,))


@pytest.mark.parametrize("lens,n_q", [
    ([1000, 1537], [2, 3]),          # scorer builds its plan in shared memory
    ([2600, 2100], [600, 500]),      # 1,100 queries: the scorer's own plan kernel
])
def test_forward_without_new_tokens(lens, n_q):
    # every token is already cached: the step only queries, so there is no
    # compression launch
    from dsa_indexer_sparse_kpool_b300.session import Step, build_session
    wl = KI.make(small_spec(lens, n_q, 256, seed=23))
    cfg = PL.cfg_of(wl)
    lens = wl.lens.tolist()
    sess = build_session(cfg, lens, lens, wl.tok_off.tolist(), wl.pool_off.tolist(), wl.pool_rows, wl.latent,
                         wl.keys, wl.gates, wl.ape)
    empty = torch.zeros(0, 128, dtype=torch.bfloat16)
    step = Step(sess, lens, [0] * wl.B, empty, empty, wl.q_seq.tolist(), wl.q_pos.tolist(), wl.q_idx, wl.w,
                wl.q_lat)
    assert step.launches_per_step() == (3 if wl.NQ <= 1022 else 4)
    step.run()
    torch.cuda.synchronize()
    assert int(sess.status.item()) == 0
    PL.check_pooled(sess, wl)
    qs = range(wl.NQ) if wl.NQ < 64 else sorted(set(range(0, wl.NQ, 11)) | {wl.NQ - 1})
    rep = PL._oracle_checks(sess, wl, qs, cfg, None, step.pool_idx.cpu().numpy(), step.n_sel.cpu().numpy(),
                            step.out.float().cpu().numpy(), step.lse.cpu().numpy())
    assert rep["checked"] == len(qs)


def test_mtp_draft_layer_reuses_target_selection():
    """index_share_for_mtp_iteration (MAX docs, Glm5NextConfig): the MTP draft
    layer reuses the target layer's top-k selection.  The draft layer's step is
    then attention only: kp_sparse_mla_attend over the draft layer's own latent
    cache and absorbed queries, with the target's pool_idx / n_sel.  Checked
    against the oracle's attention on the draft data with that selection."""
    lens, n_q = [300, 517, 1030], [2, 2, 1]
    wl = KI.make(small_spec(lens, n_q, topk_tokens=256, seed=11))
    draft = KI.make(small_spec(lens, n_q, topk_tokens=256, seed=12))  # same layout, other values
    assert np.array_equal(wl.tok_off, draft.tok_off) and np.array_equal(wl.q_pos, draft.q_pos)
    cfg = PL.cfg_of(wl)
    sess, step = PL.make_gpu(wl, cfg)
    step.run()
    latent_d = draft.latent.to(sess.device).contiguous()
    q_lat_d = draft.q_lat.to(sess.device).contiguous()
    out_d = torch.empty_like(step.out)
    lse_d = torch.empty_like(step.lse)
    aws = torch.empty(max(256, kp.kp_attend_workspace_size(cfg, wl.NQ)), dtype=torch.uint8, device=sess.device)
    kp.kp_sparse_mla_attend(cfg, step.seqs, step.queries, q_lat_d, latent_d, step.pool_idx, step.n_sel, out_d,
                            lse_d, aws, d_status=sess.status)
    torch.cuda.synchronize()
    assert int(sess.status.item()) == 0
    g_idx, g_ns = step.pool_idx.cpu().numpy(), step.n_sel.cpu().numpy()
    for qi in range(wl.NQ):
        ns = int(g_ns[qi])
        o_out, o_lse = PL.oracle_attend_on_selection(draft, qi, g_idx[qi][:ns], int(cfg.always_select_tail))
        PL.check_attend(out_d[qi].float().cpu().numpy(), lse_d[qi].cpu().numpy(), o_out, o_lse)
    # the target layer's own output is untouched by the draft call
    o_out, o_lse = PL.oracle_attend_on_selection(wl, 0, g_idx[0][:int(g_ns[0])], int(cfg.always_select_tail))
    PL.check_attend(step.out[0].float().cpu().numpy(), step.lse[0].cpu().numpy(), o_out, o_lse)


def test_two_steps_with_the_tail_ring_equal_one_step():
    """Appending a chunk in one step or in two steps (the tail ring of the
    incomplete pool carried between them) gives the same pooled cache and the
    same outputs for the final step's queries, bit for bit."""
    from dsa_indexer_sparse_kpool_b300.session import build_session, build_step
    lens, n_q = [203, 346], [13, 11]          # 13 and 11 new tokens, split 6 + 7 and 5 + 6
    wl = KI.make(small_spec(lens, n_q, topk_tokens=64, seed=31))
    cfg = PL.cfg_of(wl)
    prev = wl.prev_len.tolist()
    mid = [int(wl.prev_len[0]) + 6, int(wl.prev_len[1]) + 5]
    args = (wl.lens.tolist(), wl.tok_off.tolist(), wl.pool_off.tolist(), wl.pool_rows, wl.latent, wl.keys,
            wl.gates, wl.ape)

    def session():
        return build_session(cfg, args[0], prev, args[1], args[2], args[3], args[4], args[5], args[6], args[7])

    # one step: all new tokens, queries = the last two positions of each sequence
    last = [qi for qi in range(wl.NQ) if int(wl.q_pos[qi]) >= int(wl.lens[int(wl.q_seq[qi])]) - 2]
    qs = lambda sel: (wl.q_seq[sel], wl.q_pos[sel], wl.q_idx[sel], wl.w[sel], wl.q_lat[sel])
    sA = session()
    stA = build_step(sA, args[0], prev, args[1], wl.keys, wl.gates, *qs(last))
    stA.run()
    # two steps: first up to `mid` (queries at the first new position of each sequence), then the rest
    sB = session()
    first = [qi for qi in range(wl.NQ) if int(wl.q_pos[qi]) == int(wl.prev_len[int(wl.q_seq[qi])])]
    st1 = build_step(sB, mid, prev, args[1], wl.keys, wl.gates, *qs(first))
    st1.run()
    st2 = build_step(sB, args[0], mid, args[1], wl.keys, wl.gates, *qs(last))
    st2.run()
    torch.cuda.synchronize()
    assert int(sA.status.item()) == 0 and int(sB.status.item()) == 0
    assert torch.equal(sA.pooled, sB.pooled)
    assert torch.equal(stA.pool_idx, st2.pool_idx) and torch.equal(stA.n_sel, st2.n_sel)
    assert torch.equal(stA.out, st2.out) and torch.equal(stA.lse, st2.lse)
    # and the one-step path matches the oracle
    PL.check_pooled(sA, wl)
