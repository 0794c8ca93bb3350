"""GPU parity of the dense steps either side of the DSA step: the tcgen05 GEMM
(kp_gemm_bf16) on several shapes and batch layouts, the indexer projections,
the absorbed query and the output side (W_UV, o_proj), and a layer step whose
indexer inputs and absorbed queries come from the projections.

Bound for one output element (fp32 accumulation of exact bf16 products, then
bf16 rounding when the output is bf16):
    |gpu - oracle| <= 2 * k * 2^-24 * sum_k |a b|  (+ 2^-8 * |oracle| for bf16)
"""
import numpy as np
import pytest
import torch

import kpool_inputs as KI
import oracle
import parity_lib as PL
import dsa_indexer_sparse_kpool_b300 as kp

pytestmark = pytest.mark.gpu

DEV = "cuda"


def bits(t):
    return t.detach().cpu().contiguous().view(torch.int16).numpy().view(np.uint16)


def check(gpu, ref, ab, k, bf16_out=True):
    g = gpu.detach().cpu().float().numpy().astype(np.float64) if bf16_out else gpu.detach().cpu().numpy()
    bound = 2.0 * k * 2.0 ** -24 * ab + (2.0 ** -8 * np.abs(ref) if bf16_out else 0.0) + 1e-30
    err = np.abs(g - ref)
    assert (err <= bound).all(), f"max excess {(err - bound).max():.3e}, max err {err.max():.3e}"
    return float(err.max())


def rnd(shape, gen, std=1.0):
    return (torch.randn(*shape, generator=gen) * std).to(torch.bfloat16)


@pytest.mark.parametrize("m,n,k,batch,f32", [
    (5, 32, 64, 1, True),          # tiny, fp32 out (the head weights w)
    (200, 128, 4096, 1, False),    # keys / gates shape, two row tiles with a ragged one
    (37, 512, 256, 64, False),     # per-head batch, the absorbed-query layout
    (129, 288, 192, 3, False),     # a column tile cut short, three batches
    (33, 4096, 16384, 1, False),   # the o_proj shape (32-column tiles: few rows)
    (50, 6400, 128, 1, False),     # 64-column tiles
])
def test_gemm_against_oracle(m, n, k, batch, f32):
    gen = torch.Generator().manual_seed(m * 7 + n)
    A = rnd((m, batch * k), gen)
    B = rnd((batch * n, k), gen, 1.0 / np.sqrt(k))
    out_dtype = torch.float32 if f32 else torch.bfloat16
    C = torch.full((m, batch * n + 8), float("nan"), dtype=out_dtype, device=DEV)   # 8 pad columns stay NaN
    kp.kp_gemm_bf16(A.to(DEV), B.to(DEV), C, m, n, k, batch=batch, lda=batch * k, a_batch_off=k, ldb=k,
                    b_batch_off=n, ldc=batch * n + 8, c_batch_off=n)
    torch.cuda.synchronize()
    Cc = C.cpu()
    assert torch.isnan(Cc[:, batch * n:].float()).all()
    for b in range(batch):
        ref, ab = oracle.linear(bits(A)[:, b * k:(b + 1) * k], bits(B)[b * n:(b + 1) * n], with_abs=True)
        check(Cc[:, b * n:(b + 1) * n], ref, ab, k, bf16_out=not f32)


def test_indexer_projections():
    T = 37
    pj = KI.make_projections(T, seed=1)
    d = {k: getattr(pj, k).to(DEV) for k in ("hidden", "q_lora", "w_iq", "w_ik", "w_ig", "w_iw")}
    q_idx = torch.empty(T, 32, 128, dtype=torch.bfloat16, device=DEV)
    keys = torch.empty(T, 128, dtype=torch.bfloat16, device=DEV)
    gates = torch.empty(T, 128, dtype=torch.bfloat16, device=DEV)
    w = torch.empty(T, 32, dtype=torch.float32, device=DEV)
    kp.kp_indexer_project(d["hidden"], d["q_lora"], d["w_iq"], d["w_ik"], d["w_ig"], d["w_iw"], q_idx, keys,
                          gates, w)
    torch.cuda.synchronize()
    ref, ab = oracle.indexer_project(bits(pj.hidden), bits(pj.q_lora), bits(pj.w_iq), bits(pj.w_ik),
                                     bits(pj.w_ig), bits(pj.w_iw), with_abs=True)
    check(q_idx, ref["q_idx"], ab["q_idx"], 1536)
    check(keys, ref["keys"], ab["keys"], 4096)
    check(gates, ref["gates"], ab["gates"], 4096)
    check(w, ref["w"], ab["w"], 4096, bf16_out=False)


def test_absorbed_query_leaves_rotary_columns():
    T = 37
    pj = KI.make_projections(T, seed=2)
    q_lat = torch.full((T, 64, 576), float("nan"), dtype=torch.bfloat16, device=DEV)
    kp.kp_mla_absorb_q(pj.q_nope.to(DEV), pj.w_uk.to(DEV), q_lat)
    torch.cuda.synchronize()
    ref, ab = oracle.mla_absorb_q(bits(pj.q_nope), bits(pj.w_uk), with_abs=True)
    got = q_lat.cpu()
    check(got[:, :, :512], ref, ab, 256)
    assert torch.isnan(got[:, :, 512:].float()).all(), "the rotary columns must be left as they were"


def test_output_side():
    T = 37
    pj = KI.make_projections(T, seed=3)
    o = torch.empty(T, 64, 256, dtype=torch.bfloat16, device=DEV)
    hid = torch.empty(T, 4096, dtype=torch.bfloat16, device=DEV)
    kp.kp_mla_absorb_out(pj.out_lat.to(DEV), pj.w_uv.to(DEV), pj.w_o.to(DEV), o, hid)
    torch.cuda.synchronize()
    ref_o, ab_o = oracle.mla_absorb_out_o(bits(pj.out_lat), bits(pj.w_uv), with_abs=True)
    check(o, ref_o, ab_o, 512)
    # o_proj on the GPU's own o (each stage checked on its own inputs)
    ref_h, ab_h = oracle.o_proj(bits(o), bits(pj.w_o), with_abs=True)
    check(hid, ref_h, ab_h, 16384)


def test_layer_step_from_projections():
    """A DSA layer step whose indexer keys, gates, queries and head weights come
    from kp_indexer_project and whose absorbed queries come from
    kp_mla_absorb_q, then the output side; every stage against the oracle on
    its own GPU inputs."""
    wl = KI.make(KI.Spec("layer", [600, 903], [2, 3], topk_tokens=256, seed=81))
    n_tok = int(wl.lens.sum())
    pj = KI.make_projections(n_tok, seed=4)
    d = {k: getattr(pj, k).to(DEV) for k in ("hidden", "q_lora", "w_iq", "w_ik", "w_ig", "w_iw", "q_nope", "w_uk")}
    q_idx = torch.empty(n_tok, 32, 128, dtype=torch.bfloat16, device=DEV)
    keys = torch.empty(n_tok, 128, dtype=torch.bfloat16, device=DEV)
    gates = torch.empty(n_tok, 128, dtype=torch.bfloat16, device=DEV)
    w = torch.empty(n_tok, 32, dtype=torch.float32, device=DEV)
    kp.kp_indexer_project(d["hidden"], d["q_lora"], d["w_iq"], d["w_ik"], d["w_ig"], d["w_iw"], q_idx, keys,
                          gates, w)
    q_lat = torch.zeros(n_tok, 64, 576, dtype=torch.bfloat16, device=DEV)
    kp.kp_mla_absorb_q(d["q_nope"], d["w_uk"], q_lat)
    torch.cuda.synchronize()
    # spot-check the projections of a few tokens
    sel = np.array([0, 17, n_tok - 1])
    ref = oracle.indexer_project(bits(pj.hidden)[sel], bits(pj.q_lora)[sel], bits(pj.w_iq), bits(pj.w_ik),
                                 bits(pj.w_ig), bits(pj.w_iw), with_abs=True)
    for name, gpu, kk in (("keys", keys, 4096), ("q_idx", q_idx, 1536)):
        check(gpu[torch.as_tensor(sel)], ref[0][name], ref[1][name], kk)
    # the step's inputs: projected per-token keys / gates, the query tokens' q_idx, w, q_lat
    rows = []
    for b in range(wl.B):
        rows += [int(wl.tok_off[b]) + int(p) for p in wl.q_pos[wl.q_seq == b]]
    rows = torch.as_tensor(rows)
    wl.keys, wl.gates = keys.cpu(), gates.cpu()
    wl.q_idx, wl.w, wl.q_lat = q_idx.cpu()[rows], w.cpu()[rows], q_lat.cpu()[rows]
    sess, step, rep = PL.full_check(wl)
    assert rep["checked"] == wl.NQ
    # output side on the step's latent-space output
    o = torch.empty(wl.NQ, 64, 256, dtype=torch.bfloat16, device=DEV)
    hid = torch.empty(wl.NQ, 4096, dtype=torch.bfloat16, device=DEV)
    w_uv, w_o = pj.w_uv.to(DEV), pj.w_o.to(DEV)
    kp.kp_mla_absorb_out(step.out, w_uv, w_o, o, hid)
    torch.cuda.synchronize()
    ref_o, ab_o = oracle.mla_absorb_out_o(bits(step.out), bits(pj.w_uv), with_abs=True)
    check(o, ref_o, ab_o, 512)
    ref_h, ab_h = oracle.o_proj(bits(o), bits(pj.w_o), with_abs=True)
    check(hid, ref_h, ab_h, 16384)
