"""Seeded synthetic inputs for the KPool DSA step.

This module holds NO arithmetic of the method: it only draws random tensors
with the shapes, distributions and length mix of the workloads, and lays out
the per-sequence bookkeeping arrays.  Both the fp64 oracle harness and the
CUDA path consume what it returns; neither imports the other.

Workloads (GLM-5.3-Flash DSA layer shapes: indexer 32 heads x 128, kpool 4,
top-k budget 2048 tokens, MLA 64 heads over a 576-wide latent of which the
last 64 columns are zero):

  tiny      1 seq, ctx 258, 4 queries (t = 254..257), budget 64 tokens
  decode    32 seqs, ctx 32768, 1 query each (t = ctx-1)
  ragged    8 seqs, ctx ~ U[65537, 131071] (redrawn when a multiple of 4),
            2 queries each (decode + one MTP draft token: t = ctx-2, ctx-1)
  prefill   1 seq, 4096 new query tokens on top of 61440 cached (ctx 65536)
  long      1 seq, ctx 1,048,575, 4 queries (t = ctx-4 .. ctx-1)

Distributions: indexer q and k ~ N(0,1)/sqrt(128); gate ~ N(0,1);
ape ~ N(0, 0.1^2); head weights w ~ N(0,1)/sqrt(32); MLA q_lat and latent
columns 0..511 ~ N(0,1)/sqrt(576); latent columns 512..575 = 0; q_lat columns
512..575 = 0 unless ``q_rope_random``.  All draws come from seeded
numpy PCG64 streams (one SeedSequence per array, chunks spawned from it), then
round to bf16 (nearest even).
The queries of a sequence are its last n_q positions and are also the tokens
appended to the caches in this step (n_new = n_q).
"""
from __future__ import annotations

import dataclasses
import math
import os
from concurrent.futures import ThreadPoolExecutor
from typing import List, Optional

import numpy as np
import torch

INDEX_HEADS = 32
INDEX_DIM = 128
MLA_HEADS = 64
LATENT_DIM = 576
NOPE_DIM = 512
KPOOL = 4


@dataclasses.dataclass
class Spec:
    name: str
    lens: Optional[List[int]]       # per-sequence context length after the step
    n_q: List[int]                  # queries (= new tokens) per sequence
    topk_tokens: int = 2048
    seed: int = 0
    ragged_lo: int = 0              # when lens is None: draw B lengths in [lo, hi]
    ragged_hi: int = 0
    ragged_b: int = 0
    q_rope_random: bool = False
    q_scale: float = 1.0            # multiplies q_lat (a "peaked" softmax when > 1)
    kpool: int = KPOOL
    sm_scale: float = 1.0 / 16.0    # 1/sqrt(qk_head_dim = 256)


def named(name: str) -> Spec:
    """The five named workloads, seeded 0..4 in this order."""
    if name == "tiny":
        return Spec("tiny", [258], [4], topk_tokens=64, seed=0)
    if name == "decode":
        return Spec("decode", [32768] * 32, [1] * 32, seed=1)
    if name == "ragged":
        return Spec("ragged", None, [2] * 8, seed=2, ragged_lo=65537, ragged_hi=131071, ragged_b=8)
    if name == "prefill":
        return Spec("prefill", [65536], [4096], seed=3)
    if name == "long":
        return Spec("long", [1048575], [4], seed=4)
    raise KeyError(name)


NAMES = ("tiny", "decode", "ragged", "prefill", "long")


_THREADS = max(1, min(16, os.cpu_count() or 1))
_CHUNK = 1 << 22


def _normal_bf16_into(out_u16: np.ndarray, seed: int, tag: int, std: float) -> None:
    """Fills a 2-D uint16 array (or a column slice of one) with bf16 bit patterns of
    N(0, std^2) draws.  Each chunk of rows has its own PCG64 stream spawned from
    SeedSequence([seed, tag]), so the values do not depend on the thread count."""
    rows, cols = out_u16.shape
    rows_per = max(1, _CHUNK // max(cols, 1))
    starts = list(range(0, rows, rows_per))
    kids = np.random.SeedSequence([seed, tag]).spawn(len(starts))

    def work(i):
        a = starts[i]
        b = min(rows, a + rows_per)
        g = np.random.Generator(np.random.PCG64(kids[i]))
        x = g.standard_normal((b - a, cols), dtype=np.float32)
        x *= np.float32(std)
        u = x.view(np.uint32)
        u += ((u >> 16) & 1) + 0x7FFF          # round to nearest even at bit 16
        out_u16[a:b] = (u >> 16).astype(np.uint16)

    with ThreadPoolExecutor(_THREADS) as ex:
        list(ex.map(work, range(len(starts))))


def _bf16(u16: np.ndarray) -> torch.Tensor:
    return torch.from_numpy(u16.view(np.int16)).view(torch.bfloat16)


def _randn(seed: int, tag: int, shape, std: float) -> torch.Tensor:
    rows = int(np.prod(shape[:-1])) if len(shape) > 1 else 1
    u = np.empty((rows, shape[-1]), np.uint16)
    _normal_bf16_into(u, seed, tag, std)
    return _bf16(u).reshape(*shape)


def _round_up(x: int, m: int) -> int:
    return (x + m - 1) // m * m


@dataclasses.dataclass
class Workload:
    spec: Spec
    lens: np.ndarray            # [B] int32 context length after the step (L_b)
    prev_len: np.ndarray        # [B] int32 tokens already in the caches before the step
    new_off: np.ndarray         # [B+1] int32 CSR offsets of the new tokens
    tok_off: np.ndarray         # [B] int64 first row of each sequence in the per-token arrays
    pool_off: np.ndarray        # [B] int64 first row of each sequence in the pooled cache
    pool_rows: int              # pooled-cache capacity in rows
    q_seq: np.ndarray           # [NQ] int32
    q_pos: np.ndarray           # [NQ] int32
    keys: torch.Tensor          # [sum L, 128] bf16 raw per-token indexer keys
    gates: torch.Tensor         # [sum L, 128] bf16 per-token gate logits
    ape: torch.Tensor           # [kpool, 128] bf16 intra-pool position embedding
    latent: torch.Tensor        # [sum L, 576] bf16 MLA latent cache (cols 512.. = 0)
    q_idx: torch.Tensor         # [NQ, 32, 128] bf16 indexer queries
    w: torch.Tensor             # [NQ, 32] fp32 indexer head weights
    q_lat: torch.Tensor         # [NQ, 64, 576] bf16 absorbed MLA queries

    @property
    def B(self) -> int:
        return int(self.lens.shape[0])

    @property
    def NQ(self) -> int:
        return int(self.q_seq.shape[0])

    @property
    def k_pools(self) -> int:
        return self.spec.topk_tokens // self.spec.kpool

    @property
    def max_pools(self) -> int:
        """Largest number of complete pools any query sees."""
        return int(((self.q_pos.astype(np.int64) + 1) // self.spec.kpool).max())

    def new_rows(self) -> np.ndarray:
        """Per-token row numbers of this step's new tokens, in new-token order."""
        rows = []
        for b in range(self.B):
            rows.append(self.tok_off[b] + np.arange(self.prev_len[b], self.lens[b], dtype=np.int64))
        return np.concatenate(rows) if rows else np.zeros(0, np.int64)


def make(spec: Spec) -> Workload:
    if spec.lens is None:
        g = np.random.Generator(np.random.PCG64(np.random.SeedSequence([spec.seed, 0])))
        lens = []
        while len(lens) < spec.ragged_b:
            L = int(g.integers(spec.ragged_lo, spec.ragged_hi + 1))
            if L % spec.kpool != 0:
                lens.append(L)
    else:
        lens = list(spec.lens)
    B = len(lens)
    n_q = list(spec.n_q)
    assert len(n_q) == B
    lens_a = np.array(lens, np.int32)
    nq_a = np.array(n_q, np.int32)
    assert (nq_a <= lens_a).all()
    prev = lens_a - nq_a
    new_off = np.zeros(B + 1, np.int32)
    new_off[1:] = np.cumsum(nq_a)
    tok_off = np.zeros(B, np.int64)
    tok_off[1:] = np.cumsum(lens_a.astype(np.int64))[:-1]
    pool_cap = [_round_up(L // spec.kpool + 1, 8) for L in lens]
    pool_off = np.zeros(B, np.int64)
    pool_off[1:] = np.cumsum(np.array(pool_cap, np.int64))[:-1]
    pool_rows = int(sum(pool_cap))
    q_seq = np.concatenate([np.full(n, b, np.int32) for b, n in enumerate(n_q)])
    q_pos = np.concatenate([np.arange(L - n, L, dtype=np.int32) for L, n in zip(lens, n_q)])
    total = int(lens_a.astype(np.int64).sum())
    NQ = int(nq_a.sum())

    sd = spec.seed
    keys = _randn(sd, 1, (total, INDEX_DIM), 1.0 / math.sqrt(INDEX_DIM))
    gates = _randn(sd, 2, (total, INDEX_DIM), 1.0)
    ape = _randn(sd, 3, (spec.kpool, INDEX_DIM), 0.1)
    lat = np.zeros((total, LATENT_DIM), np.uint16)
    _normal_bf16_into(lat[:, :NOPE_DIM], sd, 4, 1.0 / math.sqrt(LATENT_DIM))
    latent = _bf16(lat)
    q_idx = _randn(sd, 5, (NQ, INDEX_HEADS, INDEX_DIM), 1.0 / math.sqrt(INDEX_DIM))
    w = torch.from_numpy(np.random.Generator(np.random.PCG64(np.random.SeedSequence([sd, 6])))
                         .standard_normal((NQ, INDEX_HEADS), dtype=np.float32) / np.float32(math.sqrt(INDEX_HEADS)))
    ql = np.zeros((NQ * MLA_HEADS, LATENT_DIM), np.uint16)
    _normal_bf16_into(ql[:, :NOPE_DIM], sd, 7, spec.q_scale / math.sqrt(LATENT_DIM))
    if spec.q_rope_random:
        _normal_bf16_into(ql[:, NOPE_DIM:], sd, 8, 1.0 / math.sqrt(LATENT_DIM))
    q_lat = _bf16(ql).reshape(NQ, MLA_HEADS, LATENT_DIM)
    return Workload(spec=spec, lens=lens_a, prev_len=prev, new_off=new_off, tok_off=tok_off,
                    pool_off=pool_off, pool_rows=pool_rows, q_seq=q_seq, q_pos=q_pos,
                    keys=keys, gates=gates, ape=ape, latent=latent, q_idx=q_idx, w=w, q_lat=q_lat)


def bits(t: torch.Tensor) -> np.ndarray:
    """Raw 16-bit patterns of a CPU bf16 tensor as numpy uint16 (no copy of values' meaning)."""
    assert t.dtype == torch.bfloat16
    return t.contiguous().view(torch.int16).numpy().view(np.uint16)


# ---------------------------------------------------------------- the steps either side

HIDDEN = 4096
Q_LORA = 1536
QK_NOPE = 256
V_HEAD = 256


@dataclasses.dataclass
class Projections:
    """Random-weight inputs of the dense steps around the DSA step, for T tokens.

    Activations ~ N(0, 1); every weight ~ N(0, 1) / sqrt(fan_in), times the
    width the DSA step's own synthetic inputs use for that output (so the
    projected q_idx, keys, w and q_lat have the distributions of the workloads
    above).  Weights are stored [out][in]."""
    hidden: torch.Tensor       # [T, 4096] bf16
    q_lora: torch.Tensor       # [T, 1536] bf16
    q_nope: torch.Tensor       # [T, 64, 256] bf16
    out_lat: torch.Tensor      # [T, 64, 512] bf16 (a stand-in attention output)
    w_iq: torch.Tensor         # [32 * 128, 1536]
    w_ik: torch.Tensor         # [128, 4096]
    w_ig: torch.Tensor         # [128, 4096]
    w_iw: torch.Tensor         # [32, 4096]
    w_uk: torch.Tensor         # [64, 512, 256]
    w_uv: torch.Tensor         # [64, 256, 512]
    w_o: torch.Tensor          # [4096, 64 * 256]


def make_projections(T: int, seed: int = 5, heads: int = MLA_HEADS) -> Projections:
    sd = 1000 + seed
    r = lambda tag, shape, std: _randn(sd, tag, shape, std)  # noqa: E731
    return Projections(
        hidden=r(1, (T, HIDDEN), 1.0),
        q_lora=r(2, (T, Q_LORA), 1.0),
        q_nope=r(3, (T, heads, QK_NOPE), 1.0),
        out_lat=r(4, (T, heads, NOPE_DIM), 1.0 / math.sqrt(NOPE_DIM)),
        w_iq=r(5, (INDEX_HEADS * INDEX_DIM, Q_LORA), 1.0 / math.sqrt(Q_LORA) / math.sqrt(INDEX_DIM)),
        w_ik=r(6, (INDEX_DIM, HIDDEN), 1.0 / math.sqrt(HIDDEN) / math.sqrt(INDEX_DIM)),
        w_ig=r(7, (INDEX_DIM, HIDDEN), 1.0 / math.sqrt(HIDDEN)),
        w_iw=r(8, (INDEX_HEADS, HIDDEN), 1.0 / math.sqrt(HIDDEN) / math.sqrt(INDEX_HEADS)),
        w_uk=r(9, (heads, NOPE_DIM, QK_NOPE), 1.0 / math.sqrt(QK_NOPE) / math.sqrt(LATENT_DIM)),
        w_uv=r(10, (heads, V_HEAD, NOPE_DIM), 1.0 / math.sqrt(NOPE_DIM)),
        w_o=r(11, (HIDDEN, heads * V_HEAD), 1.0 / math.sqrt(heads * V_HEAD)),
    )
