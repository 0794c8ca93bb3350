"""Pins of the fp64 oracle against closed forms, special cases and invariants.

None of these re-types the oracle's formula: each check comes from a property
the method (or plain mathematics) fixes, chosen so that a plausible slip in the
oracle -- a dropped term, a wrong sign, a transposed index, a wrong pool or
tail boundary -- fails at least one of them.

Sources of the properties (pages about GLM-5.3-Flash):
  * MAX docs, glm5_next.Glm5NextConfig: index_kpool_compress (learned weighted
    average from gate logits + intra-pool position embedding, else a plain
    mean), index_kpool_always_select_tail, mla_use_nope / build_layers (the 64
    rotary latent columns are zero).
  * llama.cpp PR "add GLM-5.3-Flash (GLM5-Next) support": pools of 4
    consecutive tokens, incomplete tail always kept, pooling softmax over the
    4 in-pool positions of a [4, 128, n_pool] tensor.
  * llm-atlas GLM-5.3-Flash card, raw config: index_topk 2048 tokens, 32
    indexer heads x 128, kv_lora_rank 512, 64 attention heads.
"""
import json
import math
import os

import numpy as np
import pytest
import torch

import oracle
import kpool_inputs as KI

HERE = os.path.dirname(os.path.abspath(__file__))
rng = np.random.default_rng(1234)


def to_bf16_bits(x):
    """float64 array -> bf16 bits via torch's float32 -> bf16 (round to nearest even).

    Only used on values exactly representable in float32."""
    t = torch.tensor(np.asarray(x, dtype=np.float32))
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def rand_bf16(shape, std=1.0):
    return to_bf16_bits(rng.standard_normal(shape) * std)


# ------------------------------------------------------------------ bf16 rounding

def test_double_to_bf16_ties_to_even_and_edges():
    cases = {
        1.0 + 2.0 ** -8: 1.0,                      # halfway, even is 1.0
        1.0 + 3 * 2.0 ** -8: 1.0 + 2.0 ** -6,      # halfway, even is the upper
        1.0 + 2.0 ** -8 + 2.0 ** -30: 1.0 + 2.0 ** -7,   # just above halfway (not float-representable)
        -(1.0 + 2.0 ** -8 + 2.0 ** -30): -(1.0 + 2.0 ** -7),
        3.0e38 * 1.2: math.inf,
        0.0: 0.0,
    }
    for x, want in cases.items():
        got = oracle.bf16_to_double(oracle.double_to_bf16(np.array([x])))[0]
        assert got == want, (x, got, want)
    # -0.0 keeps its sign bit
    assert oracle.double_to_bf16(np.array([-0.0]))[0] == 0x8000


def test_double_to_bf16_matches_float32_rne_on_float_values():
    x = rng.standard_normal(20000) * np.exp(rng.uniform(-30, 30, 20000))
    x = x.astype(np.float32).astype(np.float64)          # float32-representable
    assert (oracle.double_to_bf16(x) == to_bf16_bits(x)).all()


# ------------------------------------------------------------------ step 1: compress

def test_compress_hand_worked_fixture():
    fx = json.load(open(os.path.join(HERE, "golden", "compress_hand.json")))
    for case in fx["cases"]:
        keys = to_bf16_bits(np.array(case["keys"]))
        gates = to_bf16_bits(np.array(case["gates"]))
        ape = to_bf16_bits(np.array(case["ape"]))
        pooled, exact = oracle.kpool_compress(keys, gates, ape, kpool=4, mode=case["mode"])
        np.testing.assert_allclose(exact, np.array(case["pooled"]), rtol=0, atol=1e-12,
                                   err_msg=case["what"])


def test_compress_equal_logits_is_plain_mean():
    # equal gate+ape logits within a pool (per dim) -> alpha = 1/4
    n_pool, dim = 6, 128
    keys = rand_bf16((n_pool * 4, dim), 1 / math.sqrt(128))
    ape = np.zeros((4, dim), np.uint16)
    g = np.repeat(rng.standard_normal((n_pool, 1, dim)), 4, axis=1).reshape(n_pool * 4, dim)
    gates = to_bf16_bits(g)
    _, exact = oracle.kpool_compress(keys, gates, ape, 4, mode=0)
    k = oracle.bf16_to_double(keys).reshape(n_pool, 4, dim)
    np.testing.assert_allclose(exact, k.mean(axis=1), rtol=0, atol=1e-15)
    _, exact_mean = oracle.kpool_compress(keys, rand_bf16((n_pool * 4, dim)), rand_bf16((4, dim)), 4, mode=1)
    np.testing.assert_allclose(exact_mean, k.mean(axis=1), rtol=0, atol=1e-15)


def test_compress_identical_keys_return_the_key():
    n_pool, dim = 5, 128
    one = rand_bf16((n_pool, 1, dim))
    keys = np.repeat(one, 4, axis=1).reshape(n_pool * 4, dim)
    pooled, exact = oracle.kpool_compress(keys, rand_bf16((n_pool * 4, dim)), rand_bf16((4, dim), 0.1), 4)
    np.testing.assert_allclose(exact, oracle.bf16_to_double(one[:, 0]), rtol=1e-14, atol=0)
    assert (pooled == one[:, 0]).all()


@pytest.mark.parametrize("via", ["gate", "ape"])
def test_compress_dominant_logit_selects_that_position(via):
    # A logit 80 above the rest makes alpha one-hot (e^-80 ~ 1.8e-35): the pooled
    # key is that position's key, exactly after bf16 rounding.  The dominant
    # position varies with the dimension, so a transposed gate/ape or a shifted
    # pool boundary lands on a different key.
    n_pool, dim = 4, 128
    keys = rand_bf16((n_pool * 4, dim))
    star = (np.arange(dim)[None, :] * 7 + np.arange(n_pool)[:, None] * 3) % 4    # [pool, dim]
    if via == "gate":
        g = rng.uniform(-1, 1, (n_pool, 4, dim))
        for p in range(n_pool):
            for d in range(dim):
                g[p, star[p, d], d] = 80.0
        gates = to_bf16_bits(g.reshape(n_pool * 4, dim))
        ape = rand_bf16((4, dim), 0.1)
    else:
        star[:] = star[0]                       # the ape is shared by all pools
        a = np.zeros((4, dim))
        for d in range(dim):
            a[star[0, d], d] = 80.0
        ape = to_bf16_bits(a)
        gates = to_bf16_bits(rng.uniform(-1, 1, (n_pool * 4, dim)))
    pooled, _ = oracle.kpool_compress(keys, gates, ape, 4)
    k = keys.reshape(n_pool, 4, dim)
    want = np.take_along_axis(k, star[:, None, :], axis=1)[:, 0, :]
    assert (pooled == want).all()


def test_compress_two_position_closed_form():
    # logits (a, b, -80, -80): alpha = (sigmoid(a-b), 1 - sigmoid(a-b), 0, 0)
    dim = 128
    a = rng.uniform(-2, 2, dim)
    b = rng.uniform(-2, 2, dim)
    g = np.stack([a, b, np.full(dim, -80.0), np.full(dim, -80.0)])
    gates = to_bf16_bits(g)
    ga = oracle.bf16_to_double(gates)
    keys = rand_bf16((4, dim))
    k = oracle.bf16_to_double(keys)
    _, exact = oracle.kpool_compress(keys, gates, np.zeros((4, dim), np.uint16), 4)
    sig = 1.0 / (1.0 + np.exp(-(ga[0] - ga[1])))
    np.testing.assert_allclose(exact[0], sig * k[0] + (1 - sig) * k[1], rtol=1e-12, atol=1e-30)


def test_compress_only_complete_pools():
    keys = rand_bf16((4 * 3 + 3, 8))
    pooled, _ = oracle.kpool_compress(keys, rand_bf16((15, 8)), rand_bf16((4, 8)), 4)
    assert pooled.shape == (3, 8)


# ------------------------------------------------------------------ step 2: score

def test_score_one_head_unit_weight_is_relu_dot():
    q = rand_bf16((1, 128))
    pooled = rand_bf16((50, 128))
    s = oracle.indexer_score(q, np.ones(1, np.float32), pooled, 50)
    dots = oracle.bf16_to_double(pooled) @ oracle.bf16_to_double(q)[0]
    np.testing.assert_allclose(s, np.maximum(dots, 0.0), rtol=1e-12, atol=1e-15)
    assert (s[dots < 0] == 0).all() and (dots < 0).any()


def test_score_unit_vector_queries_read_single_dims():
    # head h has q = e_{d_h}: its dot is k_pool[p, d_h]; with w = 2^h the score
    # is sum_h 2^h * relu(k[p, d_h]) -- a wrong head/dim index or w index fails.
    H = 32
    d_of_h = rng.permutation(128)[:H]
    q = np.zeros((H, 128))
    q[np.arange(H), d_of_h] = 1.0
    w = (2.0 ** -np.arange(H)).astype(np.float32)
    pooled = rand_bf16((40, 128))
    s = oracle.indexer_score(to_bf16_bits(q), w, pooled, 40)
    k = oracle.bf16_to_double(pooled)
    want = (np.maximum(k[:, d_of_h], 0) * w.astype(np.float64)[None, :]).sum(axis=1)
    np.testing.assert_allclose(s, want, rtol=1e-13, atol=1e-300)


def test_score_weight_sign_and_zero_and_head_permutation():
    H = 32
    q = rand_bf16((H, 128))
    pooled = rand_bf16((30, 128))
    w = np.abs(rng.standard_normal(H)).astype(np.float32)
    s_pos = oracle.indexer_score(q, w, pooled, 30)
    s_neg = oracle.indexer_score(q, -w, pooled, 30)
    assert (s_pos >= 0).all() and (s_pos > 0).any()
    np.testing.assert_array_equal(s_neg, -s_pos)          # ReLU before the weight
    assert (oracle.indexer_score(q, np.zeros(H, np.float32), pooled, 30) == 0).all()
    perm = rng.permutation(H)
    s_perm = oracle.indexer_score(q[perm], w[perm], pooled, 30)
    np.testing.assert_allclose(s_perm, s_pos, rtol=1e-13, atol=0)


# ------------------------------------------------------------------ step 3: select

def test_topk_takes_all_when_budget_covers():
    s = rng.standard_normal(37)
    assert oracle.topk_select(s, 37).tolist() == list(range(37))
    assert oracle.topk_select(s, 100).tolist() == list(range(37))
    assert oracle.topk_select(np.zeros(0), 5).tolist() == []


def test_topk_properties_random():
    for n, k in [(1000, 16), (8192, 512), (513, 512), (700, 1)]:
        s = rng.standard_normal(n)
        idx = oracle.topk_select(s, k)
        assert len(idx) == k
        assert (np.diff(idx) > 0).all()
        mask = np.zeros(n, bool)
        mask[idx] = True
        assert s[mask].min() > s[~mask].max()


def test_topk_ties_go_to_lower_index():
    s = np.zeros(50)
    assert oracle.topk_select(s, 10).tolist() == list(range(10))
    s = np.array([5.0, 1.0, 3.0, 3.0, 3.0, 0.0, 3.0, 9.0])
    # best 9 (7), 5 (0), then the 3s in index order: 2, 3
    assert oracle.topk_select(s, 4).tolist() == [0, 2, 3, 7]


def test_topk_nan_ranks_below_minus_inf():
    s = np.array([np.nan, -np.inf, 1.0, np.nan, 2.0])
    assert oracle.topk_select(s, 3).tolist() == [1, 2, 4]
    assert oracle.topk_select(s, 4).tolist() == [0, 1, 2, 4]


# ------------------------------------------------------------------ forced tail

@pytest.mark.parametrize("t,tail", [(257, [256, 257]), (255, []), (254, [252, 253, 254]),
                                    (256, [256]), (0, [0]), (3, [])])
def test_tail_positions(t, tail):
    n_full = (t + 1) // 4
    sel = np.arange(min(n_full, 2), dtype=np.int32)
    pos = oracle.token_set(t, 4, sel, 1).tolist()
    want = [4 * p + i for p in sel for i in range(4)] + tail
    assert pos == want
    assert oracle.token_set(t, 4, sel, 0).tolist() == [4 * p + i for p in sel for i in range(4)]


def test_tiny_budget_covering_all_selects_256_tokens_plus_tail():
    # tiny shape with the budget raised to cover all 64 pools: 64 x 4 = 256 pooled
    # tokens (+ tail) per query
    spec = KI.named("tiny")
    spec.topk_tokens = 4 * 64
    wl = KI.make(spec)
    pooled, _ = oracle.kpool_compress(KI.bits(wl.keys), KI.bits(wl.gates), KI.bits(wl.ape), 4)
    res = oracle.dsa_queries(wl.q_seq, wl.q_pos, np.zeros(1, np.int64), np.zeros(1, np.int64), 4,
                             64, 1, KI.bits(wl.q_idx), wl.w.numpy(), pooled, KI.bits(wl.q_lat),
                             KI.bits(wl.latent), spec.sm_scale)
    tails = [(t + 1) % 4 for t in wl.q_pos]
    assert tails == [3, 0, 1, 2]
    n_full = [(t + 1) // 4 for t in wl.q_pos]
    assert n_full == [63, 64, 64, 64]
    assert res["n_sel"].tolist() == n_full
    assert [4 * n + tl for n, tl in zip(n_full, tails)] == [255, 256, 257, 258]


def test_forced_tail_present_even_with_hostile_affinity():
    # the tail tokens get a very negative logit; they still carry (tiny) weight,
    # and an output computed without them differs
    L, t = 23, 22                     # n_full = 5, tail = 20, 21, 22
    lat = np.zeros((L, 576))
    lat[:, :512] = rng.standard_normal((L, 512)) * 0.05
    q = rng.standard_normal((2, 576)) * 0.05
    q[:, 512:] = 0
    lat[20:23, :512] = -q[0, :512] * 3            # hostile to head 0
    pos = oracle.token_set(t, 4, np.array([1, 3], np.int32), 1)
    assert pos.tolist()[-3:] == [20, 21, 22]
    out, lse = oracle.attend(to_bf16_bits(q), to_bf16_bits(lat), pos, 1.0)
    out2, lse2 = oracle.attend(to_bf16_bits(q), to_bf16_bits(lat), pos[:-3], 1.0)
    assert (lse > lse2).all()                   # more tokens, larger log-sum-exp
    assert not np.allclose(out, out2)


# ------------------------------------------------------------------ step 4: attend

def test_attend_single_token_returns_that_row():
    lat = rand_bf16((10, 576), 0.1)
    lat[:, 512:] = 0
    q = rand_bf16((64, 576), 0.1)
    out, lse = oracle.attend(q, lat, np.array([7]), 0.0625)
    c = oracle.bf16_to_double(lat)[7]
    np.testing.assert_array_equal(out, np.repeat(c[None, :512], 64, axis=0))
    np.testing.assert_allclose(lse, 0.0625 * (oracle.bf16_to_double(q) @ c), rtol=1e-13, atol=1e-15)


def test_attend_zero_query_is_uniform_mean():
    lat = rand_bf16((40, 576), 0.1)
    rows = np.array([3, 9, 11, 12, 30, 31])
    out, lse = oracle.attend(np.zeros((4, 576), np.uint16), lat, rows, 0.0625)
    c = oracle.bf16_to_double(lat)[rows, :512].mean(axis=0)
    np.testing.assert_allclose(out, np.repeat(c[None], 4, 0), rtol=1e-13, atol=1e-16)
    np.testing.assert_allclose(lse, np.log(len(rows)), rtol=1e-15)


def test_attend_empty_set():
    out, lse = oracle.attend(rand_bf16((2, 576)), rand_bf16((3, 576)), np.zeros(0, np.int64), 1.0)
    assert (out == 0).all() and np.isneginf(lse).all()


def test_attend_large_logits_stay_finite_and_peak():
    lat = rand_bf16((16, 576), 0.05)
    lat[:, 512:] = 0
    q = lat[5:6].copy().repeat(3, 0)
    out, lse = oracle.attend(q, lat, np.arange(16), 4000.0)
    assert np.isfinite(out).all() and np.isfinite(lse).all()
    np.testing.assert_allclose(out, np.repeat(oracle.bf16_to_double(lat)[5:6, :512], 3, 0), atol=1e-6)


def _dense_reference(q_lat, latent, t, scale):
    """Textbook causal softmax attention over positions 0..t (numpy, float64)."""
    qd = q_lat.astype(np.float64)
    k = latent[: t + 1].astype(np.float64)
    z = scale * qd @ k.T                           # [H, t+1]
    z = z - z.max(axis=1, keepdims=True)
    p = np.exp(z)
    p /= p.sum(axis=1, keepdims=True)
    return p @ k[:, :512]


@pytest.mark.parametrize("rope_random", [False, True])
def test_sparse_equals_dense_when_budget_covers_all(rope_random):
    spec = KI.named("tiny")
    spec.topk_tokens = 4 * 64            # covers all 64 complete pools
    spec.q_rope_random = rope_random
    wl = KI.make(spec)
    pooled, _ = oracle.kpool_compress(KI.bits(wl.keys), KI.bits(wl.gates), KI.bits(wl.ape), 4)
    res = oracle.dsa_queries(wl.q_seq, wl.q_pos, np.zeros(1, np.int64), np.zeros(1, np.int64), 4,
                             64, 1, KI.bits(wl.q_idx), wl.w.numpy(), pooled, KI.bits(wl.q_lat),
                             KI.bits(wl.latent), spec.sm_scale)
    lat = oracle.bf16_to_double(KI.bits(wl.latent))
    ql = oracle.bf16_to_double(KI.bits(wl.q_lat))
    for i, t in enumerate(wl.q_pos):
        ref = _dense_reference(ql[i], lat, int(t), spec.sm_scale)
        np.testing.assert_allclose(res["out"][i], ref, rtol=1e-10, atol=1e-13)


def test_rope_columns_do_not_change_outputs():
    outs = []
    for rr in (False, True):
        spec = KI.named("tiny")
        spec.q_rope_random = rr
        wl = KI.make(spec)
        pooled, _ = oracle.kpool_compress(KI.bits(wl.keys), KI.bits(wl.gates), KI.bits(wl.ape), 4)
        outs.append(oracle.dsa_queries(wl.q_seq, wl.q_pos, np.zeros(1, np.int64), np.zeros(1, np.int64),
                                       4, 16, 1, KI.bits(wl.q_idx), wl.w.numpy(), pooled,
                                       KI.bits(wl.q_lat), KI.bits(wl.latent), spec.sm_scale))
    np.testing.assert_array_equal(outs[0]["out"], outs[1]["out"])
    np.testing.assert_array_equal(outs[0]["sel"], outs[1]["sel"])


def test_selection_budget_below_pools_is_active_on_tiny():
    wl = KI.make(KI.named("tiny"))
    pooled, _ = oracle.kpool_compress(KI.bits(wl.keys), KI.bits(wl.gates), KI.bits(wl.ape), 4)
    res = oracle.dsa_queries(wl.q_seq, wl.q_pos, np.zeros(1, np.int64), np.zeros(1, np.int64), 4,
                             16, 1, KI.bits(wl.q_idx), wl.w.numpy(), pooled, KI.bits(wl.q_lat),
                             KI.bits(wl.latent), 1 / 16, score_stride=64)
    assert res["n_sel"].tolist() == [16, 16, 16, 16]
    sc = res["scores"]
    for i, t in enumerate(wl.q_pos):
        nf = (int(t) + 1) // 4
        assert np.isneginf(sc[i, nf:]).all() and np.isfinite(sc[i, :nf]).all()
        sel = res["sel"][i]
        rest = np.setdiff1d(np.arange(nf), sel)
        assert sc[i, sel].min() >= sc[i, rest].max()


def test_kpool_one_reduces_to_per_token_selection():
    # kpool = 1: pooling is the identity, no tail exists, selection is over tokens
    L, dim = 40, 128
    keys = rand_bf16((L, dim), 1 / math.sqrt(128))
    pooled, _ = oracle.kpool_compress(keys, rand_bf16((L, dim)), rand_bf16((1, dim), 0.1), kpool=1)
    assert (pooled == keys).all()
    assert oracle.token_set(39, 1, np.array([1, 5], np.int32), 1).tolist() == [1, 5]


# ------------------------------------------------------------------ whole path


def _tiny_with_budget(k_pools):
    spec = KI.named("tiny")
    spec.topk_tokens = 4 * k_pools
    return KI.make(spec)


def test_whole_path_is_causal_per_query():
    # A query at position t sees only tokens 0..t: cutting every per-token array
    # (keys, gates, latent) after t leaves its selection, output and lse
    # unchanged.  A wrong pool count, tail bound or row offset breaks this.
    wl = _tiny_with_budget(16)
    keys, gates, ape, lat = KI.bits(wl.keys), KI.bits(wl.gates), KI.bits(wl.ape), KI.bits(wl.latent)
    pooled, _ = oracle.kpool_compress(keys, gates, ape, 4)
    z = np.zeros(1, np.int64)
    full = oracle.dsa_queries(wl.q_seq, wl.q_pos, z, z, 4, 16, 1, KI.bits(wl.q_idx), wl.w.numpy(), pooled,
                              KI.bits(wl.q_lat), lat, wl.spec.sm_scale)
    for qi, t in enumerate(wl.q_pos):
        n = int(t) + 1
        pooled_t, _ = oracle.kpool_compress(keys[:n], gates[:n], ape, 4)
        one = oracle.dsa_queries(np.zeros(1, np.int32), np.array([t], np.int32), z, z, 4, 16, 1,
                                 KI.bits(wl.q_idx)[qi:qi + 1], wl.w.numpy()[qi:qi + 1], pooled_t,
                                 KI.bits(wl.q_lat)[qi:qi + 1], lat[:n], wl.spec.sm_scale)
        assert one["n_sel"][0] == full["n_sel"][qi]
        assert np.array_equal(one["sel"][0], full["sel"][qi])
        assert np.array_equal(one["out"][0], full["out"][qi])
        assert np.array_equal(one["lse"][0], full["lse"][qi])


def test_ragged_batch_equals_sequences_run_singly():
    # Two sequences of different lengths packed back to back (row offsets)
    # give each query the same result as its sequence alone.
    wl = KI.make(KI.Spec("two", [130, 77], [2, 3], topk_tokens=64, seed=21))
    keys, gates, ape, lat = KI.bits(wl.keys), KI.bits(wl.gates), KI.bits(wl.ape), KI.bits(wl.latent)
    pooled_rows, pool_off = [], []
    for b in range(2):
        lo, hi = int(wl.tok_off[b]), int(wl.tok_off[b]) + int(wl.lens[b])
        p, _ = oracle.kpool_compress(keys[lo:hi], gates[lo:hi], ape, 4)
        pool_off.append(sum(r.shape[0] for r in pooled_rows))
        pooled_rows.append(p)
    pooled = np.concatenate(pooled_rows)
    both = oracle.dsa_queries(wl.q_seq, wl.q_pos, np.array(pool_off, np.int64), wl.tok_off.astype(np.int64), 4,
                              16, 1, KI.bits(wl.q_idx), wl.w.numpy(), pooled, KI.bits(wl.q_lat), lat,
                              wl.spec.sm_scale)
    z = np.zeros(1, np.int64)
    for qi in range(wl.NQ):
        b = int(wl.q_seq[qi])
        lo, hi = int(wl.tok_off[b]), int(wl.tok_off[b]) + int(wl.lens[b])
        one = oracle.dsa_queries(np.zeros(1, np.int32), wl.q_pos[qi:qi + 1], z, z, 4, 16, 1,
                                 KI.bits(wl.q_idx)[qi:qi + 1], wl.w.numpy()[qi:qi + 1], pooled_rows[b],
                                 KI.bits(wl.q_lat)[qi:qi + 1], lat[lo:hi], wl.spec.sm_scale)
        assert np.array_equal(one["sel"][0], both["sel"][qi])
        assert np.array_equal(one["out"][0], both["out"][qi])
        assert np.array_equal(one["lse"][0], both["lse"][qi])
