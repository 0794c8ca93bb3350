"""Pins of the oracle's dense steps either side of the DSA step (CPU only).

oracle.linear is the plain definition of a linear layer with weights stored
[out][in]; the compositions restate the indexer projections and the MLA
absorption.  Each is checked against something other than itself: a pure
Python triple loop, the identity matrix, and the absorption identities (an
absorbed logit equals the logit against the explicitly up-projected key; the
value up-projection commutes with the softmax-weighted sum), computed with
numpy einsum as an independent implementation.
"""
import numpy as np

import oracle

rng = np.random.default_rng(7)


def bf16(x):
    """bf16 bit patterns of float64 values (round to nearest even)."""
    return oracle.double_to_bf16(np.asarray(x, np.float64))


def val(bits):
    return oracle.bf16_to_double(bits)


def test_linear_matches_a_triple_loop():
    a, b = bf16(rng.standard_normal((3, 5))), bf16(rng.standard_normal((4, 5)))
    got = oracle.linear(a, b)
    A, B = val(a), val(b)
    for i in range(3):
        for j in range(4):
            ref = 0.0
            for k in range(5):
                ref += A[i, k] * B[j, k]
            assert abs(got[i, j] - ref) <= 1e-12 * max(1.0, abs(ref))


def test_linear_identity_and_abs_sums():
    a = bf16(rng.standard_normal((6, 64)))
    eye = bf16(np.eye(64))
    out, ab = oracle.linear(a, eye, with_abs=True)
    assert np.array_equal(out, val(a))
    assert np.array_equal(ab, np.abs(val(a)))


def test_absorbed_logit_equals_logit_against_up_projected_key():
    T, H, d, c_dim, S = 2, 3, 8, 16, 5
    q_nope = bf16(rng.standard_normal((T, H, d)))
    w_uk = bf16(rng.standard_normal((H, c_dim, d)))
    c = val(bf16(rng.standard_normal((S, c_dim))))
    q_lat = oracle.mla_absorb_q(q_nope, w_uk)                      # [T, H, c_dim]
    absorbed = np.einsum("thc,sc->ths", q_lat, c)
    k_nope = np.einsum("hcd,sc->shd", val(w_uk), c)                # the explicit key
    direct = np.einsum("thd,shd->ths", val(q_nope), k_nope)
    assert np.abs(absorbed - direct).max() <= 1e-12 * np.abs(direct).max()


def test_value_up_projection_commutes_with_the_weighted_sum():
    T, H, c_dim, v, S = 2, 3, 16, 8, 6
    c = val(bf16(rng.standard_normal((S, c_dim))))
    p = rng.random((T, H, S))
    p /= p.sum(-1, keepdims=True)
    out_lat = np.einsum("ths,sc->thc", p, c)
    w_uv = bf16(rng.standard_normal((H, v, c_dim)))
    o = oracle.mla_absorb_out_o(bf16(out_lat), w_uv)
    # the same up-projection applied per token before the weighted sum
    v_tok = np.einsum("hvc,sc->shv", val(w_uv), c)
    direct = np.einsum("ths,shv->thv", p, v_tok)
    # out_lat was rounded to bf16 before the product: allow that rounding
    bound = 2.0 ** -8 * np.einsum("hvc,thc->thv", np.abs(val(w_uv)), np.abs(out_lat))
    assert (np.abs(o - direct) <= bound + 1e-12).all()


def test_head_batching_follows_the_heads():
    T, H, d, c_dim = 2, 4, 8, 16
    q_nope = bf16(rng.standard_normal((T, H, d)))
    w_uk = bf16(rng.standard_normal((H, c_dim, d)))
    perm = np.array([2, 0, 3, 1])
    a = oracle.mla_absorb_q(q_nope, w_uk)
    b = oracle.mla_absorb_q(q_nope[:, perm], w_uk[perm])
    assert np.array_equal(a[:, perm], b)


def test_indexer_projection_shapes_and_definition():
    T = 3
    hidden = bf16(rng.standard_normal((T, 64)))
    q_lora = bf16(rng.standard_normal((T, 32)))
    w_iq = bf16(rng.standard_normal((32 * 128, 32)))
    w_ik, w_ig, w_iw = (bf16(rng.standard_normal((n, 64))) for n in (128, 128, 32))
    r = oracle.indexer_project(hidden, q_lora, w_iq, w_ik, w_ig, w_iw)
    assert r["q_idx"].shape == (T, 32, 128) and r["keys"].shape == (T, 128) and r["w"].shape == (T, 32)
    assert np.allclose(r["q_idx"][1, 5], val(w_iq)[5 * 128:6 * 128] @ val(q_lora)[1], rtol=0, atol=1e-12)
    assert np.allclose(r["w"][2], val(w_iw) @ val(hidden)[2], rtol=0, atol=1e-12)
