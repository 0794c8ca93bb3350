"""fp64 CPU oracle of the KPool DSA step -- TEST INFRASTRUCTURE ONLY.

Only ``tests/``, ``__graft_entry__.smoke()`` and the CPU-baseline / reference
leg of ``bench.py`` may import this package.  The product path (the CUDA
library and its Python binding) never imports, links or runs it, and it
shares no code with them.

The arithmetic lives in ``kpool_oracle.c`` (plain C, double precision; see its
header for the pages and readings it follows).  This module compiles it with
gcc on first use and exposes thin numpy wrappers.  bf16 arrays are passed as
their raw 16-bit patterns (``numpy.uint16``).
"""
from __future__ import annotations

import ctypes
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kpool_oracle.c")
_BUILD = os.path.join(_HERE, "_build")
_SO = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the C oracle into ``oracle/_build/liboracle.so`` (gcc, -O2, OpenMP)."""
    os.makedirs(_BUILD, exist_ok=True)
    stale = force or (not os.path.exists(_SO)) or os.path.getmtime(_SO) < os.path.getmtime(_SRC)
    if stale:
        tmp = _SO + ".%d.tmp" % os.getpid()
        cmd = ["gcc", "-O2", "-std=c11", "-fopenmp", "-fPIC", "-shared", "-Wall",
               "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _SO)
    return _SO


def lib():
    global _lib
    with _lock:
        if _lib is None:
            L = ctypes.CDLL(build())
            P = ctypes.c_void_p
            i64, i32, dbl = ctypes.c_int64, ctypes.c_int, ctypes.c_double
            L.oracle_bf16_to_double.argtypes = [ctypes.c_uint16]
            L.oracle_bf16_to_double.restype = dbl
            L.oracle_double_to_bf16.argtypes = [dbl]
            L.oracle_double_to_bf16.restype = ctypes.c_uint16
            L.oracle_kpool_compress.argtypes = [i64, i32, i32, P, P, P, i32, P, P]
            L.oracle_kpool_compress.restype = None
            L.oracle_indexer_score.argtypes = [i32, i32, P, P, P, i64, P]
            L.oracle_indexer_score.restype = None
            L.oracle_topk_select.argtypes = [P, i64, i64, P]
            L.oracle_topk_select.restype = i64
            L.oracle_token_set.argtypes = [i64, i32, P, i64, i32, P]
            L.oracle_token_set.restype = i64
            L.oracle_attend.argtypes = [i32, i32, i32, P, P, P, i64, dbl, P, P]
            L.oracle_attend.restype = None
            L.oracle_dsa_queries.argtypes = [
                i32, P, P, P, P, i32, i64, i32,
                i32, i32, P, P, P,
                i32, i32, i32, P, P, dbl,
                P, i64, P, P, P, P, i32]
            L.oracle_dsa_queries.restype = None
            L.oracle_linear.argtypes = [i64, i64, i64, P, i64, P, i64, P, i64, P, i32]
            L.oracle_linear.restype = None
            L.oracle_has_openmp.argtypes = []
            L.oracle_has_openmp.restype = i32
            _lib = L
    return _lib


def _c(a, dtype):
    a = np.ascontiguousarray(a, dtype=dtype)
    return a, a.ctypes.data_as(ctypes.c_void_p)


# ---------------------------------------------------------------- bf16 helpers

def bf16_to_double(bits) -> np.ndarray:
    """Exact widening of bf16 bit patterns to float64."""
    b = np.ascontiguousarray(bits, dtype=np.uint16)
    return (b.astype(np.uint32) << 16).view(np.float32).astype(np.float64)


def double_to_bf16(x) -> np.ndarray:
    """Round float64 values to bf16 (nearest, ties to even) via the oracle's C routine."""
    L = lib()
    x = np.asarray(x, dtype=np.float64)
    flat = [L.oracle_double_to_bf16(float(v)) for v in x.ravel()]
    return np.array(flat, dtype=np.uint16).reshape(x.shape)


# ---------------------------------------------------------------- the four steps

def kpool_compress(keys, gates, ape, kpool: int = 4, mode: int = 0):
    """Pooled keys of one sequence's complete pools.

    keys, gates: [n_tokens, dim] bf16 bits; ape: [kpool, dim] bf16 bits.
    mode 0 = learned gate+ape softmax weights, 1 = plain mean.
    Returns (pooled bf16 bits [n_tokens//kpool, dim], exact float64 same shape).
    """
    keys, pk = _c(keys, np.uint16)
    gates, pg = _c(gates if gates is not None else np.zeros_like(keys), np.uint16)
    ape, pa = _c(ape if ape is not None else np.zeros((kpool, keys.shape[1]), np.uint16), np.uint16)
    n_tok, dim = keys.shape
    n_pool = n_tok // kpool
    pooled = np.zeros((n_pool, dim), np.uint16)
    exact = np.zeros((n_pool, dim), np.float64)
    lib().oracle_kpool_compress(n_tok, kpool, dim, pk, pg, pa, mode,
                                pooled.ctypes.data_as(ctypes.c_void_p),
                                exact.ctypes.data_as(ctypes.c_void_p))
    return pooled, exact


def indexer_score(q, w, pooled, n_visible: int) -> np.ndarray:
    """Scores of one query ([H, dim] bf16 bits, w [H] fp32) over the first n_visible pools."""
    q, pq = _c(q, np.uint16)
    w, pw = _c(w, np.float32)
    pooled, pp = _c(pooled, np.uint16)
    H, dim = q.shape
    assert pooled.shape[0] >= n_visible and pooled.shape[1] == dim
    out = np.zeros(max(n_visible, 0), np.float64)
    lib().oracle_indexer_score(H, dim, pq, pw, pp, n_visible, out.ctypes.data_as(ctypes.c_void_p))
    return out


def topk_select(scores, k: int) -> np.ndarray:
    """Indices (ascending) of the min(k, n) best scores; ties to the lower index."""
    s, ps = _c(scores, np.float64)
    idx = np.zeros(max(min(k, s.shape[0]), 1), np.int32)
    m = lib().oracle_topk_select(ps, s.shape[0], k, idx.ctypes.data_as(ctypes.c_void_p))
    return idx[:m].copy()


def token_set(t: int, kpool: int, sel, always_select_tail: int = 1) -> np.ndarray:
    """Positions attended by a query at position t given its selected pools."""
    sel, psel = _c(sel, np.int32)
    pos = np.zeros(sel.shape[0] * kpool + kpool, np.int64)
    n = lib().oracle_token_set(t, kpool, psel, sel.shape[0], always_select_tail,
                               pos.ctypes.data_as(ctypes.c_void_p))
    return pos[:n].copy()


def attend(q, latent, rows, scale: float, d_v: int = 512):
    """Softmax attention of one query's heads ([H, d_lat] bf16 bits) over latent rows."""
    q, pq = _c(q, np.uint16)
    latent, pl = _c(latent, np.uint16)
    rows, pr = _c(rows, np.int64)
    H, d_lat = q.shape
    assert latent.shape[1] == d_lat
    out = np.zeros((H, d_v), np.float64)
    lse = np.zeros(H, np.float64)
    lib().oracle_attend(H, d_lat, d_v, pq, pl, pr, rows.shape[0], float(scale),
                        out.ctypes.data_as(ctypes.c_void_p), lse.ctypes.data_as(ctypes.c_void_p))
    return out, lse


def dsa_queries(q_seq, q_pos, pool_row_off, latent_row_off, kpool, k_pools,
                always_select_tail, q_idx, w, pooled, q_lat, latent, scale,
                d_v: int = 512, score_stride: int = 0, threads: int = 1):
    """Steps 2-4 for a batch of queries given pooled caches (step 1 output).

    Returns dict(scores [nq, score_stride] or None, sel [nq, k_pools] (-1 padded),
    n_sel [nq], out [nq, H, d_v], lse [nq, H]).
    """
    q_seq, p_qs = _c(q_seq, np.int32)
    q_pos, p_qp = _c(q_pos, np.int32)
    pro, p_pro = _c(pool_row_off, np.int64)
    lro, p_lro = _c(latent_row_off, np.int64)
    q_idx, p_qi = _c(q_idx, np.uint16)
    w, p_w = _c(w, np.float32)
    pooled, p_pool = _c(pooled, np.uint16)
    q_lat, p_ql = _c(q_lat, np.uint16)
    latent, p_lat = _c(latent, np.uint16)
    nq = q_seq.shape[0]
    ih, idim = q_idx.shape[1], q_idx.shape[2]
    mh, d_lat = q_lat.shape[1], q_lat.shape[2]
    scores = np.zeros((nq, score_stride), np.float64) if score_stride > 0 else None
    sel = np.zeros((nq, k_pools), np.int32)
    n_sel = np.zeros(nq, np.int32)
    out = np.zeros((nq, mh, d_v), np.float64)
    lse = np.zeros((nq, mh), np.float64)
    V = ctypes.c_void_p
    lib().oracle_dsa_queries(
        nq, p_qs, p_qp, p_pro, p_lro, kpool, k_pools, int(always_select_tail),
        ih, idim, p_qi, p_w, p_pool,
        mh, d_lat, d_v, p_ql, p_lat, float(scale),
        scores.ctypes.data_as(V) if scores is not None else None, score_stride,
        sel.ctypes.data_as(V), n_sel.ctypes.data_as(V),
        out.ctypes.data_as(V), lse.ctypes.data_as(V), int(threads))
    return dict(scores=scores, sel=sel, n_sel=n_sel, out=out, lse=lse)


def has_openmp() -> bool:
    return bool(lib().oracle_has_openmp())


# ---------------------------------------------------------------- the steps either side

def linear(a, b, with_abs: bool = False, threads: int = 0):
    """out[i, j] = sum_k a[i, k] * b[j, k] in float64 for bf16 bit arrays a [m, k]
    and b [n, k] (a linear layer with weights stored [out][in]).  With
    with_abs, also returns sum_k |a[i, k] b[j, k]|."""
    a, pa = _c(a, np.uint16)
    b, pb = _c(b, np.uint16)
    m, k = a.shape
    n, kb = b.shape
    assert kb == k
    out = np.zeros((m, n), np.float64)
    ab = np.zeros((m, n), np.float64) if with_abs else None
    lib().oracle_linear(m, n, k, pa, k, pb, k, out.ctypes.data_as(ctypes.c_void_p), n,
                        ab.ctypes.data_as(ctypes.c_void_p) if ab is not None else None,
                        int(threads or (os.cpu_count() or 1)))
    return (out, ab) if with_abs else out


def indexer_project(hidden, q_lora, w_iq, w_ik, w_ig, w_iw, with_abs: bool = False):
    """The lightning indexer's inputs from the hidden state (linear layers):
    q_idx = W_iq q_lora [T, 32, 128]; keys = W_ik h; gates = W_ig h; w = W_iw h.
    Returns float64 arrays (and the |.| sums per output with with_abs)."""
    T = hidden.shape[0]
    res = {}
    for name, (x, W) in {"q_idx": (q_lora, w_iq), "keys": (hidden, w_ik), "gates": (hidden, w_ig),
                         "w": (hidden, w_iw)}.items():
        res[name] = linear(x, W, with_abs)
    if with_abs:
        out = {k: v[0] for k, v in res.items()}
        ab = {k: v[1] for k, v in res.items()}
        out["q_idx"] = out["q_idx"].reshape(T, 32, 128)
        ab["q_idx"] = ab["q_idx"].reshape(T, 32, 128)
        return out, ab
    res["q_idx"] = res["q_idx"].reshape(T, 32, 128)
    return res


def mla_absorb_q(q_nope, w_uk, with_abs: bool = False):
    """Absorbed query per head: q_lat[t, h, c] = sum_d W_UK[h, c, d] q_nope[t, h, d]
    (q_nope [T, H, 256], W_UK [H, 512, 256] bf16 bits) -> float64 [T, H, 512]."""
    T, H, _ = q_nope.shape
    outs, abss = [], []
    for h in range(H):
        r = linear(q_nope[:, h, :], w_uk[h], with_abs)
        outs.append(r[0] if with_abs else r)
        if with_abs:
            abss.append(r[1])
    out = np.stack(outs, axis=1)
    return (out, np.stack(abss, axis=1)) if with_abs else out


def mla_absorb_out_o(out_lat, w_uv, with_abs: bool = False):
    """Value up-projection per head: o[t, h, v] = sum_c W_UV[h, v, c] out[t, h, c]
    (out [T, H, 512], W_UV [H, 256, 512] bf16 bits) -> float64 [T, H, 256]."""
    return mla_absorb_q(out_lat, w_uv, with_abs)


def o_proj(o, w_o, with_abs: bool = False):
    """hidden_out[t] = W_O o[t] (o [T, H * 256] bf16 bits, W_O [4096, H * 256])."""
    return linear(o.reshape(o.shape[0], -1), w_o, with_abs)
