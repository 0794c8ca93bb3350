"""Shared pieces of the GPU parity tests: run a workload through the C ABI and
compare every stage with the fp64 oracle on the same seeded inputs.

Comparison rules (from the method's precision and the workloads' tolerances):
  * pooled keys: within 1 bf16 ulp of the oracle's pooled key (fp32 vs fp64
    before the same round-to-nearest-even), or, where the 4-term weighted sum
    cancels, within half an ulp plus the fp32 error bound 2^-20 * sum|k_i|;
  * scores: |gpu - oracle| <= 1e-2 * max(|oracle|, rms(oracle row)) -- the
    floor keeps scores that sit near zero from demanding absolute accuracy;
  * selection: exactly the oracle's selection when the oracle selects from the
    GPU's own fp32 scores; against fp64 oracle scores, every differing pool
    lies within the near-tie band |s - s_K| <= 1e-4 * |s_K|;
  * attention: computed by the oracle on the GPU's selection (so the stage is
    isolated); max |gpu - oracle| <= 2e-2 absolute AND <= 2e-2 * max |oracle|
    (outputs are ~1e-3 in size, so the absolute bound alone would be vacuous);
    lse within 1e-3 absolute.
"""
from __future__ import annotations

import math

import dataclasses

import numpy as np
import torch

import kpool_inputs as KI
import oracle
import dsa_indexer_sparse_kpool_b300 as kp
from dsa_indexer_sparse_kpool_b300 import Config, COMPRESS_LEARNED
from dsa_indexer_sparse_kpool_b300.session import build_session, build_step

SCORE_RTOL = 1e-2
NEAR_TIE = 1e-4
OUT_TOL = 2e-2
LSE_ATOL = 1e-3


def cfg_of(wl, **kw) -> Config:
    c = Config(topk_tokens=wl.spec.topk_tokens, sm_scale=wl.spec.sm_scale, kpool=wl.spec.kpool)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def make_gpu(wl, cfg=None, max_pools=None, page_tokens=None, page_seed=0):
    cfg = cfg or cfg_of(wl)
    sess = build_session(cfg, wl.lens.tolist(), wl.prev_len.tolist(), wl.tok_off.tolist(), wl.pool_off.tolist(),
                         wl.pool_rows, wl.latent, wl.keys, wl.gates, wl.ape, page_tokens=page_tokens,
                         page_seed=page_seed)
    step = build_step(sess, wl.lens.tolist(), wl.prev_len.tolist(), wl.tok_off.tolist(), wl.keys, wl.gates,
                      wl.q_seq, wl.q_pos, wl.q_idx, wl.w, wl.q_lat, max_pools)
    return sess, step


def host(t):
    return t.detach().cpu()


def bf16_bits(t):
    return host(t).contiguous().view(torch.int16).numpy().view(np.uint16)


def gpu_pooled_of_seq(sess, wl, b):
    """The pooled keys of sequence b's complete pools, in pool order, wherever
    the session keeps them (row offsets or pages)."""
    n = int(wl.lens[b]) // wl.spec.kpool
    rows = sess.pool_rows_of(b, torch.arange(n)).to(sess.pooled.device)
    return bf16_bits(sess.pooled.index_select(0, rows))


def oracle_pooled_of_seq(wl, b, mode=0):
    a, e = int(wl.tok_off[b]), int(wl.tok_off[b] + wl.lens[b])
    pooled, exact = oracle.kpool_compress(KI.bits(wl.keys[a:e]), KI.bits(wl.gates[a:e]), KI.bits(wl.ape),
                                          wl.spec.kpool, mode)
    return pooled, exact


def ulp_distance(a_bits, b_bits):
    """Distance in representable bf16 steps (sign-magnitude aware)."""
    def ordered(x):
        x = x.astype(np.int32)
        return np.where(x & 0x8000, 0x8000 - (x & 0x7fff), 0x8000 + (x & 0x7fff))
    return np.abs(ordered(a_bits) - ordered(b_bits))


def bf16_half_ulp(v):
    v = np.abs(v)
    e = np.floor(np.log2(np.maximum(v, 2.0 ** -126)))
    return 2.0 ** (e - 8)


def check_pooled(sess, wl, seqs=None, mode=0):
    """GPU pooled keys vs the oracle: within 1 bf16 ulp of the oracle's rounded
    value, or -- where the weighted sum cancels -- within half an ulp of the
    exact value plus the fp32 error bound of a 4-term weighted sum,
    2^-20 * sum_i |k_i| (alpha_i <= 1)."""
    seqs = range(wl.B) if seqs is None else seqs
    worst = 0
    kp = wl.spec.kpool
    for b in seqs:
        g = gpu_pooled_of_seq(sess, wl, b)
        o, exact = oracle_pooled_of_seq(wl, b, mode)
        assert g.shape == o.shape
        d = ulp_distance(g, o)
        bad = d > 1
        if bad.any():
            a = int(wl.tok_off[b])
            n = g.shape[0]
            k = oracle.bf16_to_double(KI.bits(wl.keys[a:a + n * kp])).reshape(n, kp, -1)
            sum_abs = np.abs(k).sum(axis=1)
            gv = oracle.bf16_to_double(g)
            bound = bf16_half_ulp(gv) + 2.0 ** -20 * sum_abs
            still = bad & (np.abs(gv - exact) > bound)
            assert not still.any(), f"pooled keys off by {int(d[still].max())} ulp beyond the fp32 bound"
        worst = max(worst, int(d.max()) if d.size else 0)
    return worst


def oracle_scores_on(pooled_bits_seq, wl, qi):
    t = int(wl.q_pos[qi])
    nf = (t + 1) // wl.spec.kpool
    return oracle.indexer_score(KI.bits(wl.q_idx[qi]), wl.w[qi].numpy(), pooled_bits_seq, nf)


def check_scores_row(g_row, o_row):
    nf = o_row.shape[0]
    g = g_row[:nf].astype(np.float64)
    floor = math.sqrt(float(np.mean(o_row ** 2))) if nf else 0.0
    bound = SCORE_RTOL * np.maximum(np.abs(o_row), floor)
    err = np.abs(g - o_row)
    assert (err <= bound).all(), f"score error {err.max():.3e} > bound at {int(np.argmax(err - bound))}"
    return float((err / np.maximum(bound / SCORE_RTOL, 1e-30)).max()) if nf else 0.0


def check_selection(g_sel, g_nsel, g_scores_row, o_scores_row, k_pools):
    nf = o_scores_row.shape[0]
    ns = int(g_nsel)
    assert ns == min(k_pools, nf)
    sel = np.asarray(g_sel[:ns])
    assert (np.asarray(g_sel[ns:]) == -1).all()
    # exact against the oracle's selection on the GPU's own fp32 scores
    own = oracle.topk_select(g_scores_row[:nf].astype(np.float64), k_pools)
    assert np.array_equal(sel, own), "selection differs from the oracle's on the same scores"
    # near-tie band against fp64 scores
    ref = oracle.topk_select(o_scores_row, k_pools)
    diff = np.setxor1d(sel, ref)
    if diff.size and ns < nf:
        sK = np.sort(o_scores_row)[::-1][k_pools - 1]
        gap = np.abs(o_scores_row[diff] - sK)
        assert (gap <= NEAR_TIE * abs(sK)).all(), f"selection differs beyond near ties: {gap.max()}"
    return int(diff.size)


def oracle_attend_on_selection(wl, qi, sel, always_select_tail=1):
    t = int(wl.q_pos[qi])
    b = int(wl.q_seq[qi])
    pos = oracle.token_set(t, wl.spec.kpool, np.asarray(sel, np.int32), always_select_tail)
    rows = pos + int(wl.tok_off[b])
    return oracle.attend(KI.bits(wl.q_lat[qi]), KI.bits(wl.latent), rows, wl.spec.sm_scale)


def check_attend(g_out, g_lse, o_out, o_lse):
    g = g_out.astype(np.float64)
    err = np.abs(g - o_out).max()
    mx = np.abs(o_out).max()
    assert err <= OUT_TOL, f"output abs error {err}"
    assert err <= OUT_TOL * mx, f"output error {err:.3e} > {OUT_TOL} x max|o| ({mx:.3e})"
    fin = np.isfinite(o_lse)
    assert np.array_equal(np.isfinite(g_lse), fin)
    if fin.any():
        assert np.abs(g_lse[fin] - o_lse[fin]).max() <= LSE_ATOL
    return err / max(mx, 1e-30)


def check_selection_fp64(g_sel, g_nsel, o_scores_row, k_pools):
    """Selection of a path whose fp32 scores are not exposed (the fused step):
    the count is exact, the list ascending and -1 padded, and every pool that
    differs from the oracle's fp64 selection lies within the near-tie band."""
    nf = o_scores_row.shape[0]
    ns = int(g_nsel)
    assert ns == min(k_pools, nf)
    sel = np.asarray(g_sel[:ns])
    assert (np.asarray(g_sel[ns:]) == -1).all()
    assert (np.diff(sel) > 0).all() and (ns == 0 or (sel[0] >= 0 and sel[-1] < nf))
    ref = oracle.topk_select(o_scores_row, k_pools)
    diff = np.setxor1d(sel, ref)
    if diff.size and ns < nf:
        sK = np.sort(o_scores_row)[::-1][k_pools - 1]
        gap = np.abs(o_scores_row[diff] - sK)
        assert (gap <= NEAR_TIE * abs(sK)).all(), f"selection differs beyond near ties: {gap.max()}"
    return int(diff.size)


def _oracle_checks(sess, wl, queries, cfg, g_scores, g_idx, g_nsel, g_out, g_lse):
    """Per-query comparison with the oracle on the GPU's own inputs to each
    stage: scores (when given) on the GPU's pooled cache, the selection (exact
    on the GPU's scores when given, near-tie band against fp64 scores always),
    attention on the GPU's selection."""
    report = dict(max_sel_diff=0, max_out_rel=0.0, checked=0)
    for qi in queries:
        b = int(wl.q_seq[qi])
        pooled_gpu = gpu_pooled_of_seq(sess, wl, b)
        o_sc = oracle_scores_on(pooled_gpu, wl, qi)
        if g_scores is not None:
            check_scores_row(g_scores[qi], o_sc)
            d = check_selection(g_idx[qi], g_nsel[qi], g_scores[qi], o_sc, cfg.k_pools)
        else:
            d = check_selection_fp64(g_idx[qi], g_nsel[qi], o_sc, cfg.k_pools)
        report["max_sel_diff"] = max(report["max_sel_diff"], d)
        ns = int(g_nsel[qi])
        o_out, o_lse = oracle_attend_on_selection(wl, qi, g_idx[qi][:ns], int(cfg.always_select_tail))
        r = check_attend(g_out[qi], g_lse[qi], o_out, o_lse)
        report["max_out_rel"] = max(report["max_out_rel"], r)
        report["checked"] += 1
    return report


def full_check(wl, queries=None, cfg=None, stages=True, check_all_pooled=True, page_tokens=None):
    """Runs the step on the GPU (the four stage calls, or the fused
    kp_dsa_forward when stages is False) and checks every stage for the given
    queries."""
    cfg = cfg or cfg_of(wl)
    sess, step = make_gpu(wl, cfg, page_tokens=page_tokens)
    if stages:
        scores = step.run_stages()
    else:
        step.run()
        scores = None
    torch.cuda.synchronize()
    assert int(sess.status.item()) == 0, f"device status {int(sess.status.item())}"
    queries = list(range(wl.NQ) if queries is None else queries)
    seqs_needed = sorted({int(wl.q_seq[q]) for q in queries}) if not check_all_pooled else None
    check_pooled(sess, wl, seqs_needed, cfg.compress_mode)
    g_scores = host(scores).numpy() if scores is not None else None
    report = _oracle_checks(sess, wl, queries, cfg, g_scores, host(step.pool_idx).numpy(),
                            host(step.n_sel).numpy(), host(step.out.float()).numpy(), host(step.lse).numpy())
    assert report["checked"] == len(queries)
    return sess, step, report


def fused_check(wl, queries=None, cfg=None, check_all_pooled=True, page_tokens=None,
                modes=(kp.SELECT_AUTO, kp.SELECT_FUSED)):
    """The path the bench times: kp_dsa_forward on fresh state, in each of the
    given select modes, against the four stage calls on other fresh state (bit
    for bit: pooled cache, tail rings, selection, outputs) and against the
    oracle on the sampled queries (scores from the staged run, selection and
    attention from the forward)."""
    cfg = cfg or cfg_of(wl)
    sess_s, step_s = make_gpu(wl, cfg, page_tokens=page_tokens)
    scores = step_s.run_stages()
    torch.cuda.synchronize()
    assert int(sess_s.status.item()) == 0, f"staged: device status {int(sess_s.status.item())}"
    out = None
    for mode in modes:
        cfg_m = dataclasses.replace(cfg, select_mode=mode)
        sess_f, step_f = make_gpu(wl, cfg_m, page_tokens=page_tokens)
        step_f.run()
        torch.cuda.synchronize()
        tag = f"select_mode {mode}"
        assert int(sess_f.status.item()) == 0, f"{tag}: device status {int(sess_f.status.item())}"
        assert torch.equal(sess_f.pooled, sess_s.pooled), f"{tag}: pooled caches differ"
        assert torch.equal(sess_f.tail_keys, sess_s.tail_keys) and torch.equal(sess_f.tail_gates, sess_s.tail_gates)
        assert torch.equal(step_f.n_sel, step_s.n_sel), f"{tag}: n_sel differs"
        assert torch.equal(step_f.pool_idx, step_s.pool_idx), f"{tag}: selection differs"
        assert torch.equal(step_f.out, step_s.out), f"{tag}: outputs differ"
        assert torch.equal(step_f.lse, step_s.lse), f"{tag}: lse differs"
        queries = list(range(wl.NQ) if queries is None else queries)
        seqs_needed = sorted({int(wl.q_seq[q]) for q in queries}) if not check_all_pooled else None
        check_pooled(sess_f, wl, seqs_needed, cfg.compress_mode)
        report = _oracle_checks(sess_f, wl, queries, cfg, host(scores).numpy(), host(step_f.pool_idx).numpy(),
                                host(step_f.n_sel).numpy(), host(step_f.out.float()).numpy(),
                                host(step_f.lse).numpy())
        assert report["checked"] == len(queries)
        out = (sess_f, step_f, report)
    return out
