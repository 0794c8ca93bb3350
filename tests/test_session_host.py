"""Host-side checks of the session helpers (no GPU, no library calls)."""
import types

import pytest

import torch

from dsa_indexer_sparse_kpool_b300 import Queries
from dsa_indexer_sparse_kpool_b300.session import SCORE_LOCAL_PLAN_MAX_QUERIES, Step, host_chunks


def _step_stub():
    st = Step.__new__(Step)
    st.sess = types.SimpleNamespace(device=torch.device("cpu"))
    g = torch.Generator().manual_seed(5)
    st.prev_len = torch.tensor([1, 2, 3], dtype=torch.int32)
    st.new_off = torch.tensor([0, 1, 2, 3], dtype=torch.int32)
    st.keys = torch.randn(3, 128, generator=g).to(torch.bfloat16)
    st.gates = torch.randn(3, 128, generator=g).to(torch.bfloat16)
    st.queries = Queries(torch.tensor([0, 1, 2], dtype=torch.int32), torch.tensor([5, 6, 7], dtype=torch.int32), 2)
    st.q_idx = torch.randn(3, 32, 128, generator=g).to(torch.bfloat16)
    st.w = torch.randn(3, 32, generator=g)
    st.q_lat = torch.randn(3, 64, 576, generator=g).to(torch.bfloat16)
    st.out = torch.randn(3, 64, 512, generator=g).to(torch.bfloat16)
    st.lse = torch.randn(3, 64, generator=g)
    st.workspace = None
    st._args = lambda ws: None
    return st


def test_pack_io_keeps_values_and_packs_into_two_buffers():
    st = _step_stub()
    names_in = ["prev_len", "new_off", "keys", "gates", "q_idx", "w", "q_lat"]
    old = {k: getattr(st, k).clone() for k in names_in + ["out", "lse"]}
    oq = (st.queries.q_seq.clone(), st.queries.q_pos.clone())
    in_buf, out_buf = st.pack_io()
    for k, v in old.items():
        t = getattr(st, k)
        assert t.dtype == v.dtype and t.shape == v.shape and torch.equal(t, v), k
        base = (out_buf if k in ("out", "lse") else in_buf).data_ptr()
        assert (t.data_ptr() - base) % 256 == 0, k
        span = out_buf if k in ("out", "lse") else in_buf
        assert base <= t.data_ptr() and t.data_ptr() + t.numel() * t.element_size() <= base + span.numel()
    assert torch.equal(st.queries.q_seq, oq[0]) and torch.equal(st.queries.q_pos, oq[1])
    assert st.queries.max_pools == 2
    # one copy per direction moves every byte of the step's inputs / outputs
    need_in = sum(old[k].numel() * old[k].element_size() for k in names_in) + 2 * 3 * 4
    assert in_buf.numel() >= need_in and out_buf.numel() >= 3 * 64 * 512 * 2 + 3 * 64 * 4
    # q_lat is the input buffer's last piece (run_host copies it on its own);
    # every other input ends before it
    _, _, late, lse_off = st._io
    assert st.q_lat.data_ptr() - in_buf.data_ptr() == late
    for k in ("prev_len", "new_off", "keys", "gates", "q_idx", "w"):
        t = getattr(st, k)
        assert t.data_ptr() + t.numel() * t.element_size() <= in_buf.data_ptr() + late, k
    assert st.out.data_ptr() == out_buf.data_ptr() and st.lse.data_ptr() - out_buf.data_ptr() == lse_off


@pytest.mark.parametrize("nq,cq", [(4096, 256), (600, 256), (530, 256), (511, 256), (512, 256), (300, 128),
                                   (10, 256)])
def test_host_chunks_cover_the_batch_with_full_chunks(nq, cq):
    ch = host_chunks(nq, cq)
    assert ch[0][0] == 0 and ch[-1][1] == nq
    assert all(a1 == b0 for (_, b0), (a1, _) in zip(ch, ch[1:]))
    assert len(ch) == max(1, nq // cq)
    if len(ch) > 1:
        assert min(b - a for a, b in ch) >= cq


def test_local_plan_threshold_matches_the_plan_layout():
    # 4 header words, four words per query and one closing word fit 4096 words
    assert 4 + 4 * SCORE_LOCAL_PLAN_MAX_QUERIES + 1 <= 4096 < 4 + 4 * (SCORE_LOCAL_PLAN_MAX_QUERIES + 1) + 1
