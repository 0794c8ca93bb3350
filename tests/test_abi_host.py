"""Host-side checks of the C ABI: the library builds, loads without a GPU, exports
every entry point the header declares, and rejects bad arguments before any
launch (these paths touch no device)."""
import ctypes
import os
import re

import pytest

import dsa_indexer_sparse_kpool_b300 as kp
from dsa_indexer_sparse_kpool_b300 import build as kbuild

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


@pytest.fixture(scope="module")
def L():
    kbuild.build()
    return kp.lib()


def header_functions():
    text = open(os.path.join(ROOT, "include", "kpool_dsa.h")).read()
    return re.findall(r"^KP_API\s+[\w\s\*]+?\b(kp_\w+)\s*\(", text, flags=re.M)


def test_exports_every_declared_entry_point(L):
    names = header_functions()
    assert len(names) >= 12
    for n in names:
        assert hasattr(L, n), n
    assert set(kp.EXPORTS) == set(names)
    assert L.kp_version() == 20400 == kp.ABI_VERSION


def test_status_strings(L):
    for code in range(7):
        assert L.kp_status_string(code).decode()
    assert L.kp_status_string(99).decode() == "unknown status"


def _cfg(**kw):
    c = kp.Config(**kw)
    return c.c()


def test_null_args_rejected(L):
    for name in ("kp_kpool_compress", "kp_indexer_score", "kp_topk_select", "kp_indexer_score_select",
                 "kp_sparse_mla_attend", "kp_dsa_forward"):
        assert getattr(L, name)(None, None) == 1


def test_unsupported_kpool_and_bad_budget(L):
    a = kp.kp_score_args()
    a.cfg = _cfg(kpool=8)                    # pools of 4 (the checkpoint) and 16 (NeMo's default) only
    assert L.kp_indexer_score(ctypes.byref(a), None) == 2
    a.cfg = _cfg(kpool=16, topk_tokens=2048)
    assert L.kp_indexer_score(ctypes.byref(a), None) == 1   # past the config check; no layout given
    a.cfg = _cfg(topk_tokens=6)
    assert L.kp_indexer_score(ctypes.byref(a), None) == 1
    a.cfg = _cfg(topk_tokens=4 * 2048)
    assert L.kp_indexer_score(ctypes.byref(a), None) == 2
    t = kp.kp_topk_args()
    t.cfg = _cfg(compress_mode=7)
    assert L.kp_topk_select(ctypes.byref(t), None) == 1
    t.cfg = _cfg(wait_limit_us=-1)
    assert L.kp_topk_select(ctypes.byref(t), None) == 1
    t.cfg = _cfg(debug_flags=2)
    assert L.kp_topk_select(ctypes.byref(t), None) == 1
    t.cfg = _cfg(select_mode=3)
    assert L.kp_topk_select(ctypes.byref(t), None) == 1


def test_score_rejects_small_workspace_and_stride(L):
    a = kp.kp_score_args()
    a.cfg = _cfg()
    a.seqs = kp.kp_seqs(1, 0x1000, 0x1000, 0x1000, 100, 100)
    a.q = kp.kp_queries(4, 0x1000, 0x1000, 64)
    a.q_idx = a.w = a.pooled = a.scores = 0x10000
    a.score_stride = 64                      # must be >= 128 (64 pools rounded up)
    a.workspace = 0x10000
    a.workspace_bytes = 1 << 20
    assert L.kp_indexer_score(ctypes.byref(a), None) == 1
    a.score_stride = 128
    a.workspace_bytes = 8                    # too small
    assert L.kp_indexer_score(ctypes.byref(a), None) == 6
    a.q = kp.kp_queries(4, 0x1000, 0x1000, kp.MAX_SCORE_POOLS + 1)
    assert L.kp_indexer_score(ctypes.byref(a), None) == 2
    a.q = kp.kp_queries(4, 0x1000, 0x1000, 64)
    a.workspace_bytes = 1 << 20
    a.seqs = kp.kp_seqs(1, 0x1000, 0x1000, 0x1000, 100, 1 << 31)   # pooled rows beyond TMA's int32 rows
    assert L.kp_indexer_score(ctypes.byref(a), None) == 1


def test_compress_rejects_inconsistent_sizes(L):
    c = kp.kp_compress_args()
    c.cfg = _cfg()
    c.num_seqs = 2
    c.num_new = 5
    c.max_new_per_seq = 9                    # larger than num_new
    assert L.kp_kpool_compress(ctypes.byref(c), None) == 1
    c.num_new = 0                             # nothing to do: OK without touching the device
    assert L.kp_kpool_compress(ctypes.byref(c), None) == 0


def test_workspace_size_queries_need_no_gpu(L):
    cfg = kp.Config()
    assert kp.kp_score_workspace_size(4096) >= 4 * (4 * 4096 + 5)
    assert kp.kp_attend_workspace_size(cfg, 32) > 0
    args = kp.kp_forward_args()
    args.cfg = cfg.c()
    args.q = kp.kp_queries(32, 0, 0, 8192)
    ws = L.kp_workspace_size(ctypes.byref(args))
    assert ws >= 32 * 8192 * 4 + 32 * 512 * 4


def test_noalloc_score_rejects_too_many_queries_before_any_launch(L):
    a = kp.kp_score_args()
    a.cfg = _cfg()
    a.seqs = kp.kp_seqs(1, 0x1000, 0x1000, 0x1000, 100, 100)
    a.q = kp.kp_queries(kp.NOALLOC_MAX_QUERIES + 1, 0x1000, 0x1000, 64)
    assert L.kp_indexer_score_noalloc(ctypes.byref(a), None) == 2
    assert "KP_NOALLOC_MAX_QUERIES" in L.kp_last_error().decode()
    assert L.kp_indexer_score_noalloc(None, None) == 1


def test_fused_score_select_checks_before_any_launch(L):
    a = kp.kp_score_select_args()
    a.cfg = _cfg()
    a.seqs = kp.kp_seqs(1, 0x1000, 0x1000, 0x1000, 100, 100)
    a.q = kp.kp_queries(4, 0x1000, 0x1000, kp.FUSED_MAX_POOLS + 1)   # longer rows: the staged calls
    a.q_idx = a.w = a.pooled = a.pool_idx = a.n_sel = 0x10000
    a.workspace = 0x10000
    a.workspace_bytes = 1 << 20
    assert L.kp_indexer_score_select(ctypes.byref(a), None) == 2
    a.q = kp.kp_queries(4, 0x1000, 0x1000, kp.FUSED_MAX_POOLS)
    a.workspace_bytes = 8
    assert L.kp_indexer_score_select(ctypes.byref(a), None) == 6
    a.workspace_bytes = 1 << 20
    a.n_sel = None
    assert L.kp_indexer_score_select(ctypes.byref(a), None) == 1
    a.q = kp.kp_queries(0, None, None, 0)                          # nothing to do
    assert L.kp_indexer_score_select(ctypes.byref(a), None) == 0


def test_fused_mode_workspace_holds_no_score_matrix(L):
    args = kp.kp_forward_args()
    args.q = kp.kp_queries(32, 0, 0, 8192)
    args.cfg = kp.Config(select_mode=kp.SELECT_STAGED).c()
    staged = L.kp_workspace_size(ctypes.byref(args))
    args.cfg = kp.Config(select_mode=kp.SELECT_FUSED).c()
    fused = L.kp_workspace_size(ctypes.byref(args))
    assert staged - fused >= 32 * 8192 * 4
    args.q = kp.kp_queries(32, 0, 0, kp.FUSED_MAX_POOLS + 128)    # too long for the fused kernel: staged
    fused_long = L.kp_workspace_size(ctypes.byref(args))
    args.cfg = kp.Config(select_mode=kp.SELECT_STAGED).c()
    assert fused_long == L.kp_workspace_size(ctypes.byref(args))


def test_forward_select_only_needs_the_selection_buffers(L):
    # out = NULL with queries: the selection only, into the caller's pool_idx
    # and n_sel, which must then be given
    a = kp.kp_forward_args()
    a.cfg = _cfg()
    a.seqs = kp.kp_seqs(1, 0x1000, 0x1000, 0x1000, 100, 100)
    a.q = kp.kp_queries(4, 0x1000, 0x1000, 16)
    a.prev_len = a.new_off = 0x1000
    a.q_idx = a.w = a.pooled = a.latent = 0x10000
    a.workspace = 0x10000
    a.workspace_bytes = 1 << 30
    assert L.kp_dsa_forward(ctypes.byref(a), None) == 1
    a.pool_idx = a.n_sel = 0x10000
    # past the argument checks: the next step asks for the device (none here)
    assert L.kp_dsa_forward(ctypes.byref(a), None) == 3
