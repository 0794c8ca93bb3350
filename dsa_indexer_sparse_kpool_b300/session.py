"""Device state of one DSA layer for a batch of sequences, driven through the C ABI.

A ``Session`` owns the latent (MLA) cache, the pooled indexer cache, the tail
rings and the per-sequence bookkeeping on one CUDA device, and runs steps with
``kp_dsa_forward`` (or the four stage calls).  It moves data and fills the
argument structs; all arithmetic of the step runs in libkpool_dsa.so.
"""
from __future__ import annotations

from typing import Optional, Sequence

import torch

from . import (Config, Queries, Seqs, attend_args, forward_args, kp_dsa_forward, kp_indexer_score,
               kp_indexer_score_select, kp_kpool_compress, kp_score_workspace_size, kp_attend_workspace_size,
               kp_sparse_mla_attend, kp_sparse_mla_attend_args, kp_topk_select, kp_workspace_size, score_stride,
               FUSED_MAX_POOLS, SELECT_FUSED, INDEX_DIM, LATENT_DIM, MLA_HEADS, NOPE_DIM)


# Queries up to which the library's scorer builds its work plan in shared
# memory (4096 plan words: a 4-word header, four words per query, one more),
# and the same for the fused score-and-select kernel (2048 plan words).
SCORE_LOCAL_PLAN_MAX_QUERIES = (4096 - 5) // 4
SCORE_SELECT_LOCAL_PLAN_MAX_QUERIES = (2048 - 5) // 4

# Step.run_host pipelines batches of at least two chunks of this many queries:
# each chunk's q_lat copy, attention and output copy overlap the neighbouring
# chunks'.  From 128 queries on, a chunk and the whole batch alike attend
# with one CTA per query (no split of a query's tokens), so chunking changes
# no result bit.
HOST_CHUNK_QUERIES = 256
HOST_MIN_CHUNK_QUERIES = 128


def host_chunks(nq: int, chunk_queries: int):
    """Query ranges [a, b) of run_host's pipeline: nq // chunk_queries chunks
    as even as the count allows, so every chunk holds at least chunk_queries
    queries (one chunk, the whole batch, below two chunks' worth)."""
    n = max(1, nq // chunk_queries)
    return [(nq * c // n, nq * (c + 1) // n) for c in range(n)]


def _dev_i32(x, device):
    return torch.as_tensor(x, dtype=torch.int32).to(device).contiguous()


def _dev_i64(x, device):
    return torch.as_tensor(x, dtype=torch.int64).to(device).contiguous()


class Session:
    """Caches of B sequences.

    latent       [rows, 576] bf16
    pooled       [rows, 128] bf16, written by kp_kpool_compress
    Contiguous layout (page_tokens None): sequence b at latent rows
    latent_row_off[b] + position and pooled rows pool_row_off[b] + pool.
    Paged layout (page_tokens P): the caches are pages of P positions (P / 4
    pooled rows), handed to the sequences in a seeded random order, and a
    block table [B, blocks_per_seq] names each sequence's pages; `latent` is
    then given per token in the contiguous layout and scattered into pages.
    """

    def __init__(self, cfg: Config, lens: Sequence[int], latent_row_off: Sequence[int],
                 pool_row_off: Sequence[int], pool_rows: int, latent: torch.Tensor, ape: torch.Tensor,
                 device="cuda", page_tokens: Optional[int] = None, page_seed: int = 0):
        self.cfg = cfg
        self.device = torch.device(device)
        self.B = len(lens)
        self.lens = [int(x) for x in lens]
        self.latent_row_off_h = [int(x) for x in latent_row_off]
        self.pool_row_off_h = [int(x) for x in pool_row_off]
        self.page_tokens = page_tokens
        self.ape = ape.to(self.device).contiguous()
        if page_tokens is None:
            self.latent = latent.to(self.device).contiguous()
            self.pooled = torch.zeros(pool_rows, INDEX_DIM, dtype=torch.bfloat16, device=self.device)
            self.block_table = None
        else:
            P = int(page_tokens)
            need = [(L + P - 1) // P for L in self.lens]
            self.blocks_per_seq = max(need) + 1
            n_pages = sum(need) + max(1, sum(need) // 8)          # some pages stay free
            perm = torch.randperm(n_pages, generator=torch.Generator().manual_seed(page_seed))
            bt = torch.full((self.B, self.blocks_per_seq), -1, dtype=torch.int32)
            k = 0
            for b in range(self.B):
                bt[b, :need[b]] = perm[k:k + need[b]].to(torch.int32)
                k += need[b]
            self.block_table_h = bt
            self.block_table = bt.to(self.device).contiguous()
            self.latent = torch.zeros(n_pages * P, LATENT_DIM, dtype=torch.bfloat16, device=self.device)
            src = torch.cat([torch.arange(self.latent_row_off_h[b], self.latent_row_off_h[b] + self.lens[b])
                             for b in range(self.B)])
            dst = torch.cat([self.latent_rows_of(b, torch.arange(self.lens[b])) for b in range(self.B)])
            self.latent.index_copy_(0, dst.to(self.device), latent[src].to(self.device))
            self.pooled = torch.zeros(n_pages * (P // cfg.kpool), INDEX_DIM, dtype=torch.bfloat16,
                                      device=self.device)
        R = cfg.kpool - 1
        self.tail_keys = torch.zeros(self.B, R, INDEX_DIM, dtype=torch.bfloat16, device=self.device)
        self.tail_gates = torch.zeros(self.B, R, INDEX_DIM, dtype=torch.bfloat16, device=self.device)
        self.seq_len = _dev_i32(self.lens, self.device)
        self.latent_row_off = _dev_i64(self.latent_row_off_h, self.device) if page_tokens is None else None
        self.pool_row_off = _dev_i64(self.pool_row_off_h, self.device) if page_tokens is None else None
        self.status = torch.zeros(1, dtype=torch.int32, device=self.device)

    def latent_rows_of(self, b: int, pos: torch.Tensor) -> torch.Tensor:
        """Latent-cache rows of positions `pos` of sequence b (int64, host)."""
        pos = pos.to(torch.int64)
        if self.page_tokens is None:
            return pos + self.latent_row_off_h[b]
        P = int(self.page_tokens)
        return self.block_table_h[b, pos // P].to(torch.int64) * P + pos % P

    def pool_rows_of(self, b: int, pools: torch.Tensor) -> torch.Tensor:
        """Pooled-cache rows of pools `pools` of sequence b (int64, host)."""
        pools = pools.to(torch.int64)
        if self.page_tokens is None:
            return pools + self.pool_row_off_h[b]
        pp = int(self.page_tokens) // self.cfg.kpool
        return self.block_table_h[b, pools // pp].to(torch.int64) * pp + pools % pp

    def seqs(self) -> Seqs:
        return Seqs(self.seq_len, self.latent_row_off, self.pool_row_off, self.latent.shape[0],
                    self.pooled.shape[0], self.block_table, self.page_tokens or 0)

    def append(self, prev_len: Sequence[int], new_counts: Sequence[int], keys: torch.Tensor,
               gates: Optional[torch.Tensor], stream=None) -> None:
        """Appends new tokens' indexer keys (CSR by sequence) through kp_kpool_compress."""
        new_off = [0]
        for n in new_counts:
            new_off.append(new_off[-1] + int(n))
        keys = keys.to(self.device).contiguous()
        gates = gates.to(self.device).contiguous() if gates is not None else None
        kp_kpool_compress(self.cfg, self.seqs(), _dev_i32(list(prev_len), self.device),
                          _dev_i32(new_off, self.device), keys, gates, self.ape, self.tail_keys, self.tail_gates,
                          self.pooled, max(1, max(int(n) for n in new_counts)), d_status=self.status, stream=stream)


class Step:
    """Device buffers and argument struct of one kp_dsa_forward call."""

    def __init__(self, sess: Session, prev_len: Sequence[int], new_counts: Sequence[int], new_keys: torch.Tensor,
                 new_gates: torch.Tensor, q_seq: Sequence[int], q_pos: Sequence[int], q_idx: torch.Tensor,
                 w: torch.Tensor, q_lat: torch.Tensor, max_pools: Optional[int] = None):
        d = sess.device
        self.sess = sess
        cfg = sess.cfg
        NQ = len(q_seq)
        self.prev_len = _dev_i32(list(prev_len), d)
        off = [0]
        for n in new_counts:
            off.append(off[-1] + int(n))
        self.new_off = _dev_i32(off, d)
        self.max_new = max(1, max(int(n) for n in new_counts)) if len(new_counts) else 1
        self.keys = new_keys.to(d).contiguous()
        self.gates = new_gates.to(d).contiguous()
        if max_pools is None:
            max_pools = max((int(t) + 1) // cfg.kpool for t in q_pos) if NQ else 0
        self.queries = Queries(_dev_i32(list(q_seq), d), _dev_i32(list(q_pos), d), int(max_pools))
        self.q_idx = q_idx.to(d).contiguous()
        self.w = w.to(d).contiguous()
        self.q_lat = q_lat.to(d).contiguous()
        self.out = torch.empty(NQ, MLA_HEADS, NOPE_DIM, dtype=torch.bfloat16, device=d)
        self.lse = torch.empty(NQ, MLA_HEADS, dtype=torch.float32, device=d)
        self.pool_idx = torch.empty(NQ, cfg.k_pools, dtype=torch.int32, device=d)
        self.n_sel = torch.empty(NQ, dtype=torch.int32, device=d)
        self.seqs = sess.seqs()
        args = self._args(None)
        ws = kp_workspace_size(args)
        self.workspace = torch.empty(ws, dtype=torch.uint8, device=d)
        self.args = self._args(self.workspace)
        self._io = None          # (in_buf, out_buf, q_lat's byte offset in in_buf, lse's in out_buf)
        self._late_args = None   # the args with q_lat_ready set (run_host)
        self._chunked = None     # run_host's pipeline: chunk bounds, argument structs, streams, events

    def _args(self, workspace, q_lat_ready=None):
        s = self.sess
        return forward_args(s.cfg, self.seqs, self.queries, prev_len=self.prev_len, new_off=self.new_off,
                            max_new_per_seq=self.max_new, keys=self.keys, gates=self.gates, ape=s.ape,
                            tail_keys=s.tail_keys, tail_gates=s.tail_gates, pooled=s.pooled, q_idx=self.q_idx,
                            w=self.w, q_lat=self.q_lat, latent=s.latent, out=self.out, lse=self.lse,
                            pool_idx=self.pool_idx, n_sel=self.n_sel, workspace=workspace, d_status=s.status,
                            q_lat_ready=q_lat_ready)

    def run(self, stream=None) -> None:
        kp_dsa_forward(self.args, stream=stream)

    def set_share(self, share_src) -> None:
        """Shared selection: share_src[q] >= 0 makes query q attend that query's
        selection instead of selecting its own (None: every query selects).
        Call it before pack_io: the table is one of the step's inputs."""
        t = None if share_src is None else _dev_i32([int(x) for x in share_src], self.sess.device)
        self.queries = Queries(self.queries.q_seq, self.queries.q_pos, self.queries.max_pools, t)
        self.args = self._args(self.workspace)
        self._io = None
        self._late_args = None
        self._chunked = None

    def pack_io(self):
        """Moves the step's per-step inputs (positions, new keys and gates,
        queries) into one device buffer and its outputs (out, lse) into
        another, keeping their values, and re-points the step at them, so a
        caller moves each direction with one copy.  Returns the two buffers
        (uint8 device tensors, 256-byte aligned pieces).  q_lat is the last
        piece of the input buffer, so that it can cross separately
        (run_host).  A CUDA graph captured before the call still reads the
        old tensors."""
        d = self.sess.device
        share = self.queries.share_src
        ins = [self.prev_len, self.new_off, self.keys, self.gates, self.queries.q_seq, self.queries.q_pos,
               self.q_idx, self.w] + ([share] if share is not None else []) + [self.q_lat]
        outs = [self.out, self.lse]

        def carve(ts):
            offs, n = [], 0
            for t in ts:
                offs.append(n)
                n += (t.numel() * t.element_size() + 255) // 256 * 256
            buf = torch.empty(max(n, 256), dtype=torch.uint8, device=d)
            views = []
            for t, o in zip(ts, offs):
                v = buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
                v.copy_(t)
                views.append(v)
            return buf, views, offs

        in_buf, views, offs = carve(ins)
        (self.prev_len, self.new_off, self.keys, self.gates, q_seq, q_pos, self.q_idx, self.w) = views[:8]
        self.q_lat = views[-1]
        self.queries = Queries(q_seq, q_pos, self.queries.max_pools, views[8] if share is not None else None)
        out_buf, (self.out, self.lse), out_offs = carve(outs)
        self.args = self._args(self.workspace)
        self._io = (in_buf, out_buf, offs[-1], out_offs[1])
        self._late_args = None
        self._chunked = None
        return in_buf, out_buf

    def run_host(self, h_in: torch.Tensor, h_out: torch.Tensor, chunk_queries: Optional[int] = None) -> None:
        """One step from pinned host memory, asynchronous on the current
        stream (capturable in a CUDA graph): the inputs come from ``h_in``
        (laid out as the buffer pack_io returned) and out / lse go to
        ``h_out`` (laid out as pack_io's output buffer).

        q_lat, most of the input bytes and read only by the attention, crosses
        on a second stream while compression, scoring and selection run; the
        attention launch waits for it (kp_forward_args.q_lat_ready).  The
        second stream starts only once this stream's earlier work (the
        previous step's attention included) and the early inputs' copy are
        done.

        Batches of at least 2 * chunk_queries queries (default
        HOST_CHUNK_QUERIES; not with a shared selection) run as a pipeline
        instead: the selection for all queries (kp_dsa_forward with out =
        NULL), then per chunk of queries its q_lat copy, its attention
        (kp_sparse_mla_attend, in chunk order on this stream) and its out /
        lse copy back on a third stream, so the copies in both directions
        overlap the attention of other chunks.  Results are the same bits as
        the single call's."""
        if self._io is None:
            raise RuntimeError("run_host needs pack_io() first")
        in_buf, out_buf, late, _ = self._io
        if h_in.numel() != in_buf.numel() or h_out.numel() != out_buf.numel():
            raise ValueError("run_host: host buffers must match the sizes pack_io returned")
        main = torch.cuda.current_stream(self.sess.device)
        nq = self.queries.q_seq.numel()
        if nq == 0:          # no attention: nothing to overlap
            in_buf.copy_(h_in, non_blocking=True)
            kp_dsa_forward(self.args, stream=main)
            h_out.copy_(out_buf, non_blocking=True)
            return
        cq = HOST_CHUNK_QUERIES if chunk_queries is None else int(chunk_queries)
        if cq < HOST_MIN_CHUNK_QUERIES:
            raise ValueError(f"run_host: chunks of at least {HOST_MIN_CHUNK_QUERIES} queries")
        if self._late_args is None:
            self._copy_stream = torch.cuda.Stream(device=self.sess.device)
            self._fork = torch.cuda.Event()
            self._q_lat_ready = torch.cuda.Event()
        if nq >= 2 * cq and self.queries.share_src is None:
            self._run_host_chunked(h_in, h_out, host_chunks(nq, cq), main)
            return
        side = self._copy_stream
        # The early inputs first, alone on the bus: the compression and the
        # scorer wait for them, and two host-to-device copies in flight at once
        # finished later than the same copies one after the other.
        in_buf[:late].copy_(h_in[:late], non_blocking=True)
        self._fork.record(main)
        side.wait_event(self._fork)
        with torch.cuda.stream(side):
            in_buf[late:].copy_(h_in[late:], non_blocking=True)
        self._q_lat_ready.record(side)
        if self._late_args is None:              # the event exists once recorded
            self._late_args = self._args(self.workspace, q_lat_ready=self._q_lat_ready)
        kp_dsa_forward(self._late_args, stream=main)
        main.wait_event(self._q_lat_ready)       # rejoins the copy stream on every path
        h_out.copy_(out_buf, non_blocking=True)

    def _run_host_chunked(self, h_in, h_out, bounds, main) -> None:
        in_buf, out_buf, late, lse_off = self._io
        nq = self.queries.q_seq.numel()
        if self._chunked is None or self._chunked["bounds"] != bounds:
            s = self.sess
            sel = forward_args(s.cfg, self.seqs, self.queries, prev_len=self.prev_len, new_off=self.new_off,
                               max_new_per_seq=self.max_new, keys=self.keys, gates=self.gates, ape=s.ape,
                               tail_keys=s.tail_keys, tail_gates=s.tail_gates, pooled=s.pooled,
                               q_idx=self.q_idx, w=self.w, q_lat=None, latent=s.latent, out=None, lse=None,
                               pool_idx=self.pool_idx, n_sel=self.n_sel, workspace=self.workspace,
                               d_status=s.status)
            ws = torch.empty(kp_attend_workspace_size(s.cfg, nq), dtype=torch.uint8, device=s.device)
            att = [attend_args(s.cfg, self.seqs,
                               Queries(self.queries.q_seq[a:b], self.queries.q_pos[a:b], self.queries.max_pools),
                               self.q_lat[a:b], s.latent, self.pool_idx[a:b], self.n_sel[a:b], self.out[a:b],
                               self.lse[a:b], ws, s.status) for a, b in bounds]
            self._chunked = {"bounds": bounds, "sel": sel, "att": att, "ws": ws,
                             "d2h": torch.cuda.Stream(device=s.device),
                             "in": [torch.cuda.Event() for _ in bounds], "out": [torch.cuda.Event() for _ in bounds],
                             "done": torch.cuda.Event()}
        st = self._chunked
        side, d2h = self._copy_stream, st["d2h"]
        qb = self.q_lat[0].numel() * self.q_lat.element_size()      # q_lat bytes per query
        ob = self.out[0].numel() * self.out.element_size()          # out bytes per query
        lb = self.lse[0].numel() * self.lse.element_size()          # lse bytes per query
        in_buf[:late].copy_(h_in[:late], non_blocking=True)
        self._fork.record(main)
        side.wait_event(self._fork)
        with torch.cuda.stream(side):
            for (a, b), ev in zip(st["bounds"], st["in"]):
                in_buf[late + a * qb:late + b * qb].copy_(h_in[late + a * qb:late + b * qb], non_blocking=True)
                ev.record(side)
        kp_dsa_forward(st["sel"], stream=main)                     # the selection of every query
        for (a, b), args, ev_in, ev_out in zip(st["bounds"], st["att"], st["in"], st["out"]):
            main.wait_event(ev_in)
            kp_sparse_mla_attend_args(args, stream=main)
            ev_out.record(main)
            d2h.wait_event(ev_out)
            with torch.cuda.stream(d2h):
                h_out[a * ob:b * ob].copy_(out_buf[a * ob:b * ob], non_blocking=True)
                h_out[lse_off + a * lb:lse_off + b * lb].copy_(out_buf[lse_off + a * lb:lse_off + b * lb],
                                                                 non_blocking=True)
        st["done"].record(d2h)
        main.wait_event(st["in"][-1])            # rejoins both copy streams
        main.wait_event(st["done"])

    def fused(self) -> bool:
        """Whether ``run`` scores and selects in one kernel (SELECT_FUSED and
        rows short enough for it)."""
        return (self.sess.cfg.select_mode == SELECT_FUSED and self.queries.q_seq.numel() > 0
                and self.queries.max_pools <= FUSED_MAX_POOLS)

    def launches_per_step(self) -> int:
        """Kernels one ``run`` launches: compress, score, top-k and attention
        (score and top-k are one kernel when fused); no queries stops after
        compress.  The scorer builds its own work plan up to a query count
        (SCORE_LOCAL_PLAN_MAX_QUERIES, or SCORE_SELECT_LOCAL_PLAN_MAX_QUERIES
        fused); above that the plan rides in an extra grid row of the
        compression launch when there are new tokens, else it is one more
        kernel."""
        nq = self.queries.q_seq.numel()
        new = int(self.new_off[-1].item()) > 0
        if nq == 0:
            return 1 if new else 0
        local = SCORE_SELECT_LOCAL_PLAN_MAX_QUERIES if self.fused() else SCORE_LOCAL_PLAN_MAX_QUERIES
        plan_free = nq <= local or (new and self.seqs.seq_len.numel() < 65535)
        return (1 if new else 0) + (1 if plan_free else 2) + (1 if self.fused() else 2)

    def stage_calls(self, fused: bool = False):
        """The stage calls on persistent buffers (capturable one by one):
        [compress, score, topk, attend], or with fused [compress,
        score_select, attend]; returns (calls, scores tensor)."""
        s, cfg = self.sess, self.sess.cfg
        NQ = self.queries.q_seq.numel()
        if not hasattr(self, "_stage_bufs"):
            stride = score_stride(self.queries.max_pools)
            self._stage_bufs = (
                torch.empty(NQ, stride, dtype=torch.float32, device=s.device),
                torch.empty(kp_score_workspace_size(NQ), dtype=torch.uint8, device=s.device),
                torch.empty(max(256, kp_attend_workspace_size(cfg, NQ)), dtype=torch.uint8, device=s.device))
        scores, ws, aws = self._stage_bufs
        compress = lambda: kp_kpool_compress(cfg, self.seqs, self.prev_len, self.new_off, self.keys,  # noqa: E731
                                             self.gates, s.ape, s.tail_keys, s.tail_gates, s.pooled, self.max_new,
                                             d_status=s.status)
        attend = lambda: kp_sparse_mla_attend(cfg, self.seqs, self.queries, self.q_lat, s.latent,  # noqa: E731
                                              self.pool_idx, self.n_sel, self.out, self.lse, aws,
                                              d_status=s.status)
        if fused:
            select = lambda: kp_indexer_score_select(cfg, self.seqs, self.queries, self.q_idx,  # noqa: E731
                                                     self.w, s.pooled, self.pool_idx, self.n_sel, ws,
                                                     d_status=s.status)
            return [compress, select, attend], scores
        calls = [
            compress,
            lambda: kp_indexer_score(cfg, self.seqs, self.queries, self.q_idx, self.w, s.pooled, scores, ws,
                                     d_status=s.status),
            lambda: kp_topk_select(cfg, self.queries, scores, self.pool_idx, self.n_sel, d_status=s.status),
            attend,
        ]
        return calls, scores

    # ---- the four stages one by one (same buffers), for stage-level checks
    def run_stages(self, stream=None):
        s, cfg = self.sess, self.sess.cfg
        kp_kpool_compress(cfg, self.seqs, self.prev_len, self.new_off, self.keys, self.gates, s.ape, s.tail_keys,
                          s.tail_gates, s.pooled, self.max_new, d_status=s.status, stream=stream)
        NQ = self.queries.q_seq.numel()
        stride = score_stride(self.queries.max_pools)
        scores = torch.empty(NQ, stride, dtype=torch.float32, device=s.device)
        ws = torch.empty(kp_score_workspace_size(NQ), dtype=torch.uint8, device=s.device)
        kp_indexer_score(cfg, self.seqs, self.queries, self.q_idx, self.w, s.pooled, scores, ws,
                         d_status=s.status, stream=stream)
        kp_topk_select(cfg, self.queries, scores, self.pool_idx, self.n_sel, d_status=s.status, stream=stream)
        aws = torch.empty(max(256, kp_attend_workspace_size(cfg, NQ)), dtype=torch.uint8, device=s.device)
        kp_sparse_mla_attend(cfg, self.seqs, self.queries, self.q_lat, s.latent, self.pool_idx, self.n_sel,
                             self.out, self.lse, aws, d_status=s.status, stream=stream)
        return scores


def _ranges(starts, ends):
    parts = [torch.arange(int(s), int(e), dtype=torch.int64) for s, e in zip(starts, ends)]
    return torch.cat(parts) if parts else torch.zeros(0, dtype=torch.int64)


def build_session(cfg: Config, lens, prev_len, tok_off, pool_off, pool_rows: int, latent: torch.Tensor,
                  keys: torch.Tensor, gates: torch.Tensor, ape: torch.Tensor, device="cuda",
                  page_tokens: Optional[int] = None, page_seed: int = 0) -> Session:
    """Session whose caches hold positions [0, prev_len[b]) of each sequence.

    `keys`, `gates` and `latent` are per-token arrays laid out like the latent
    cache (sequence b at rows tok_off[b] + position).  The pooled cache and the
    tail rings are built on the device by kp_kpool_compress.  With page_tokens
    the caches are paged (block table, pages in a seeded random order)."""
    sess = Session(cfg, lens, tok_off, pool_off, pool_rows, latent, ape, device, page_tokens, page_seed)
    B = len(lens)
    idx = _ranges([tok_off[b] for b in range(B)], [tok_off[b] + prev_len[b] for b in range(B)])
    if idx.numel():
        sess.append([0] * B, [int(p) for p in prev_len], keys[idx], gates[idx])
    return sess


def build_step(sess: Session, lens, prev_len, tok_off, keys: torch.Tensor, gates: torch.Tensor, q_seq, q_pos,
               q_idx, w, q_lat, max_pools=None) -> Step:
    """Step that appends positions [prev_len[b], lens[b]) and runs the queries."""
    B = len(lens)
    idx = _ranges([tok_off[b] + prev_len[b] for b in range(B)], [tok_off[b] + lens[b] for b in range(B)])
    counts = [int(lens[b]) - int(prev_len[b]) for b in range(B)]
    return Step(sess, [int(p) for p in prev_len], counts, keys[idx], gates[idx], [int(x) for x in q_seq],
                [int(x) for x in q_pos], q_idx, w, q_lat, max_pools)
