"""Python binding of libkpool_dsa.so -- the KPool DSA sparse-attention step on B300.

Argument marshalling only: every step runs in the library's CUDA kernels.
PyTorch provides device memory and the current stream.  The functions carry
the C-ABI names (``kp_kpool_compress``, ``kp_indexer_score``,
``kp_topk_select``, ``kp_sparse_mla_attend``, ``kp_dsa_forward``) and take
``torch.Tensor`` arguments on the CUDA device; bf16 tensors are passed as
their storage.  Loading fails loudly when the compiled library is missing.
"""
from __future__ import annotations

import ctypes
import dataclasses
import os
from typing import Optional

import torch

_PKG = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_PKG, "libkpool_dsa.so")

INDEX_HEADS, INDEX_DIM, MLA_HEADS, LATENT_DIM, NOPE_DIM, KPOOL = 32, 128, 64, 576, 512, 4
MAX_TOPK_POOLS, MAX_SCORE_POOLS, NOALLOC_MAX_QUERIES = 1024, 262144, 8192
COMPRESS_LEARNED, COMPRESS_MEAN = 0, 1
DEBUG_STALL_FIRST_WAIT = 1
SELECT_AUTO, SELECT_STAGED, SELECT_FUSED = 0, 1, 2
FUSED_MAX_POOLS = 16384

STATUS = {0: "KP_OK", 1: "KP_ERR_INVALID_ARG", 2: "KP_ERR_UNSUPPORTED", 3: "KP_ERR_CUDA",
          4: "KP_ERR_DEVICE_TIMEOUT", 5: "KP_ERR_DEVICE_BOUNDS", 6: "KP_ERR_WORKSPACE"}

_i32, _i64, _f32, _vp, _sz = ctypes.c_int32, ctypes.c_int64, ctypes.c_float, ctypes.c_void_p, ctypes.c_size_t


class kp_config(ctypes.Structure):
    _fields_ = [("kpool", _i32), ("topk_tokens", _i32), ("compress_mode", _i32),
                ("always_select_tail", _i32), ("sm_scale", _f32), ("wait_limit_us", _i32),
                ("debug_flags", _i32), ("select_mode", _i32)]


class kp_seqs(ctypes.Structure):
    _fields_ = [("num_seqs", _i32), ("seq_len", _vp), ("latent_row_off", _vp), ("pool_row_off", _vp),
                ("latent_rows", _i64), ("pool_rows", _i64), ("block_table", _vp), ("page_tokens", _i32),
                ("blocks_per_seq", _i32)]


class kp_queries(ctypes.Structure):
    _fields_ = [("num_queries", _i32), ("q_seq", _vp), ("q_pos", _vp), ("max_pools", _i32), ("share_src", _vp)]


class kp_compress_args(ctypes.Structure):
    _fields_ = [("cfg", kp_config), ("num_seqs", _i32), ("prev_len", _vp), ("new_off", _vp),
                ("num_new", _i32), ("max_new_per_seq", _i32), ("keys", _vp), ("gates", _vp), ("ape", _vp),
                ("tail_keys", _vp), ("tail_gates", _vp), ("pooled", _vp), ("seqs", kp_seqs),
                ("d_status", _vp)]


class kp_score_args(ctypes.Structure):
    _fields_ = [("cfg", kp_config), ("seqs", kp_seqs), ("q", kp_queries), ("q_idx", _vp), ("w", _vp),
                ("pooled", _vp), ("scores", _vp), ("score_stride", _i64), ("workspace", _vp),
                ("workspace_bytes", _sz), ("d_status", _vp)]


class kp_topk_args(ctypes.Structure):
    _fields_ = [("cfg", kp_config), ("q", kp_queries), ("scores", _vp), ("score_stride", _i64),
                ("pool_idx", _vp), ("n_sel", _vp), ("d_status", _vp)]


class kp_score_select_args(ctypes.Structure):
    _fields_ = [("cfg", kp_config), ("seqs", kp_seqs), ("q", kp_queries), ("q_idx", _vp), ("w", _vp),
                ("pooled", _vp), ("pool_idx", _vp), ("n_sel", _vp), ("workspace", _vp),
                ("workspace_bytes", _sz), ("d_status", _vp)]


class kp_attend_args(ctypes.Structure):
    _fields_ = [("cfg", kp_config), ("seqs", kp_seqs), ("q", kp_queries), ("q_lat", _vp), ("latent", _vp),
                ("pool_idx", _vp), ("n_sel", _vp), ("out", _vp), ("lse", _vp), ("workspace", _vp),
                ("workspace_bytes", _sz), ("d_status", _vp)]


class kp_forward_args(ctypes.Structure):
    _fields_ = [("cfg", kp_config), ("seqs", kp_seqs), ("q", kp_queries),
                ("prev_len", _vp), ("new_off", _vp), ("num_new", _i32), ("max_new_per_seq", _i32),
                ("keys", _vp), ("gates", _vp), ("ape", _vp), ("tail_keys", _vp), ("tail_gates", _vp),
                ("pooled", _vp), ("q_idx", _vp), ("w", _vp), ("q_lat", _vp), ("latent", _vp),
                ("out", _vp), ("lse", _vp), ("pool_idx", _vp), ("n_sel", _vp),
                ("workspace", _vp), ("workspace_bytes", _sz), ("d_status", _vp), ("q_lat_ready", _vp)]


class kp_gemm_args(ctypes.Structure):
    _fields_ = [("m", _i32), ("n", _i32), ("k", _i32), ("batch", _i32), ("a", _vp), ("lda", _i64),
                ("a_batch_off", _i64), ("b", _vp), ("ldb", _i64), ("b_batch_off", _i64), ("c", _vp),
                ("ldc", _i64), ("c_batch_off", _i64), ("c_dtype", _i32), ("wait_limit_us", _i32),
                ("d_status", _vp)]


class kp_indexer_project_args(ctypes.Structure):
    _fields_ = [("num_tokens", _i32), ("hidden", _vp), ("q_lora", _vp), ("w_iq", _vp), ("w_ik", _vp),
                ("w_ig", _vp), ("w_iw", _vp), ("q_idx", _vp), ("keys", _vp), ("gates", _vp), ("w", _vp),
                ("wait_limit_us", _i32), ("d_status", _vp)]


class kp_mla_absorb_q_args(ctypes.Structure):
    _fields_ = [("num_tokens", _i32), ("q_nope", _vp), ("w_uk", _vp), ("q_lat", _vp), ("wait_limit_us", _i32),
                ("d_status", _vp)]


class kp_mla_absorb_out_args(ctypes.Structure):
    _fields_ = [("num_tokens", _i32), ("out", _vp), ("w_uv", _vp), ("w_o", _vp), ("o", _vp),
                ("hidden_out", _vp), ("wait_limit_us", _i32), ("d_status", _vp)]


EXPORTS = ("kp_kpool_compress", "kp_indexer_score", "kp_topk_select", "kp_indexer_score_select",
           "kp_sparse_mla_attend",
           "kp_dsa_forward", "kp_indexer_score_noalloc", "kp_score_workspace_size", "kp_attend_workspace_size",
           "kp_workspace_size", "kp_gemm_bf16", "kp_indexer_project", "kp_mla_absorb_q", "kp_mla_absorb_out",
           "kp_status_string", "kp_last_error", "kp_read_device_status", "kp_version")
DTYPE_BF16, DTYPE_F32 = 0, 1

ABI_VERSION = 20400   # kp_version() of the library whose structs the classes above mirror
_lib = None


def lib() -> ctypes.CDLL:
    """The loaded C library (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise RuntimeError("libkpool_dsa.so is not built: run `python -m dsa_indexer_sparse_kpool_b300.build`")
        L = ctypes.CDLL(LIB_PATH)
        for name, argt in (("kp_kpool_compress", kp_compress_args), ("kp_indexer_score", kp_score_args),
                           ("kp_indexer_score_noalloc", kp_score_args),
                           ("kp_topk_select", kp_topk_args), ("kp_sparse_mla_attend", kp_attend_args),
                           ("kp_indexer_score_select", kp_score_select_args),
                           ("kp_dsa_forward", kp_forward_args), ("kp_gemm_bf16", kp_gemm_args),
                           ("kp_indexer_project", kp_indexer_project_args),
                           ("kp_mla_absorb_q", kp_mla_absorb_q_args),
                           ("kp_mla_absorb_out", kp_mla_absorb_out_args)):
            f = getattr(L, name)
            f.argtypes = [ctypes.POINTER(argt), _vp]
            f.restype = ctypes.c_int
        L.kp_score_workspace_size.argtypes = [_i32]
        L.kp_score_workspace_size.restype = _sz
        L.kp_attend_workspace_size.argtypes = [ctypes.POINTER(kp_config), _i32]
        L.kp_attend_workspace_size.restype = _sz
        L.kp_workspace_size.argtypes = [ctypes.POINTER(kp_forward_args)]
        L.kp_workspace_size.restype = _sz
        L.kp_status_string.argtypes = [ctypes.c_int]
        L.kp_status_string.restype = ctypes.c_char_p
        L.kp_last_error.argtypes = []
        L.kp_last_error.restype = ctypes.c_char_p
        L.kp_read_device_status.argtypes = [_vp, _vp]
        L.kp_read_device_status.restype = ctypes.c_int
        L.kp_version.argtypes = []
        L.kp_version.restype = ctypes.c_int
        if L.kp_version() != ABI_VERSION:   # the structs above must match the library's
            raise RuntimeError(f"{LIB_PATH} is version {L.kp_version()}, the binding expects {ABI_VERSION}: "
                               "rebuild with `python -m dsa_indexer_sparse_kpool_b300.build`")
        _lib = L
    return _lib


class KPError(RuntimeError):
    def __init__(self, code: int, where: str):
        L = lib()
        msg = L.kp_status_string(code).decode()
        if code == 3:
            msg += ": " + L.kp_last_error().decode()
        super().__init__(f"{where}: {STATUS.get(code, code)} ({msg})")
        self.code = code


def _check(code: int, where: str) -> None:
    if code != 0:
        raise KPError(code, where)


def _p(t: Optional[torch.Tensor]):
    """Device address of a tensor (None -> NULL)."""
    if t is None:
        return None
    assert t.is_cuda and t.is_contiguous(), "expected a contiguous CUDA tensor"
    return t.data_ptr()


def _stream(stream) -> int:
    if stream is None:
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


@dataclasses.dataclass
class Config:
    topk_tokens: int = 2048
    kpool: int = KPOOL
    compress_mode: int = COMPRESS_LEARNED
    always_select_tail: bool = True
    sm_scale: float = 1.0 / 16.0
    wait_limit_us: int = 0          # 0: each device-side wait gives up after 1 s
    debug_flags: int = 0            # DEBUG_* bits (failure-path tests only)
    select_mode: int = SELECT_AUTO  # how kp_dsa_forward scores and selects (SELECT_*)

    def c(self) -> kp_config:
        return kp_config(self.kpool, self.topk_tokens, self.compress_mode, int(self.always_select_tail),
                         float(self.sm_scale), int(self.wait_limit_us), int(self.debug_flags),
                         int(self.select_mode))

    @property
    def k_pools(self) -> int:
        return self.topk_tokens // self.kpool


@dataclasses.dataclass
class Seqs:
    """Per-sequence cache layout (device int tensors): contiguous rows per
    sequence (row offsets), or pages of page_tokens positions named by a block
    table [B, blocks_per_seq] (int32 physical page ids)."""
    seq_len: torch.Tensor           # [B] int32
    latent_row_off: Optional[torch.Tensor]    # [B] int64 (contiguous)
    pool_row_off: Optional[torch.Tensor]      # [B] int64 (contiguous)
    latent_rows: int
    pool_rows: int
    block_table: Optional[torch.Tensor] = None   # [B, blocks_per_seq] int32 (paged)
    page_tokens: int = 0

    def c(self) -> kp_seqs:
        bt = self.block_table
        return kp_seqs(self.seq_len.numel(), _p(self.seq_len), _p(self.latent_row_off), _p(self.pool_row_off),
                       self.latent_rows, self.pool_rows, _p(bt), int(self.page_tokens) if bt is not None else 0,
                       int(bt.shape[1]) if bt is not None else 0)


@dataclasses.dataclass
class Queries:
    q_seq: torch.Tensor     # [NQ] int32
    q_pos: torch.Tensor     # [NQ] int32
    max_pools: int          # upper bound of floor((q_pos + 1) / kpool)
    share_src: Optional[torch.Tensor] = None   # [NQ] int32: query whose selection each query attends (-1: its own)

    def c(self) -> kp_queries:
        return kp_queries(self.q_seq.numel(), _p(self.q_seq), _p(self.q_pos), int(self.max_pools),
                          _p(self.share_src))


def score_stride(max_pools: int) -> int:
    return max(1, (max_pools + 127) // 128) * 128


def kp_kpool_compress(cfg: Config, seqs: Seqs, prev_len, new_off, keys, gates, ape, tail_keys, tail_gates, pooled,
                      max_new_per_seq: int, d_status=None, stream=None) -> None:
    a = kp_compress_args(cfg.c(), prev_len.numel(), _p(prev_len), _p(new_off), keys.shape[0], int(max_new_per_seq),
                         _p(keys), _p(gates), _p(ape), _p(tail_keys), _p(tail_gates), _p(pooled), seqs.c(),
                         _p(d_status))
    _check(lib().kp_kpool_compress(ctypes.byref(a), _stream(stream)), "kp_kpool_compress")


def kp_score_workspace_size(num_queries: int) -> int:
    return int(lib().kp_score_workspace_size(num_queries))


def kp_attend_workspace_size(cfg: Config, num_queries: int) -> int:
    c = cfg.c()
    return int(lib().kp_attend_workspace_size(ctypes.byref(c), num_queries))


def kp_indexer_score(cfg: Config, seqs: Seqs, queries: Queries, q_idx, w, pooled, scores, workspace,
                     d_status=None, stream=None) -> None:
    a = kp_score_args(cfg.c(), seqs.c(), queries.c(), _p(q_idx), _p(w), _p(pooled), _p(scores), scores.shape[1],
                      _p(workspace), workspace.numel() * workspace.element_size(), _p(d_status))
    _check(lib().kp_indexer_score(ctypes.byref(a), _stream(stream)), "kp_indexer_score")


def kp_indexer_score_noalloc(cfg: Config, seqs: Seqs, queries: Queries, q_idx, w, pooled, scores,
                             d_status=None, stream=None) -> None:
    """kp_indexer_score without a workspace argument, for callers that cannot
    allocate device memory: the work plan lives in a device array inside the
    library (at most NOALLOC_MAX_QUERIES queries per call; calls that overlap
    on the GPU share that array and race)."""
    a = kp_score_args(cfg.c(), seqs.c(), queries.c(), _p(q_idx), _p(w), _p(pooled), _p(scores), scores.shape[1],
                      None, 0, _p(d_status))
    _check(lib().kp_indexer_score_noalloc(ctypes.byref(a), _stream(stream)), "kp_indexer_score_noalloc")


def kp_topk_select(cfg: Config, queries: Queries, scores, pool_idx, n_sel, d_status=None, stream=None) -> None:
    a = kp_topk_args(cfg.c(), queries.c(), _p(scores), scores.shape[1], _p(pool_idx), _p(n_sel), _p(d_status))
    _check(lib().kp_topk_select(ctypes.byref(a), _stream(stream)), "kp_topk_select")


def kp_indexer_score_select(cfg: Config, seqs: Seqs, queries: Queries, q_idx, w, pooled, pool_idx, n_sel,
                            workspace, d_status=None, stream=None) -> None:
    """kp_indexer_score then kp_topk_select in one kernel, the scores kept on
    chip (queries.max_pools <= FUSED_MAX_POOLS)."""
    a = kp_score_select_args(cfg.c(), seqs.c(), queries.c(), _p(q_idx), _p(w), _p(pooled), _p(pool_idx),
                             _p(n_sel), _p(workspace), workspace.numel() * workspace.element_size(), _p(d_status))
    _check(lib().kp_indexer_score_select(ctypes.byref(a), _stream(stream)), "kp_indexer_score_select")


def attend_args(cfg: Config, seqs: Seqs, queries: Queries, q_lat, latent, pool_idx, n_sel, out, lse,
                workspace, d_status=None) -> kp_attend_args:
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    return kp_attend_args(cfg.c(), seqs.c(), queries.c(), _p(q_lat), _p(latent), _p(pool_idx), _p(n_sel), _p(out),
                          _p(lse), _p(workspace), ws_bytes, _p(d_status))


def kp_sparse_mla_attend_args(args: kp_attend_args, stream=None) -> None:
    _check(lib().kp_sparse_mla_attend(ctypes.byref(args), _stream(stream)), "kp_sparse_mla_attend")


def kp_sparse_mla_attend(cfg: Config, seqs: Seqs, queries: Queries, q_lat, latent, pool_idx, n_sel, out, lse,
                         workspace, d_status=None, stream=None) -> None:
    kp_sparse_mla_attend_args(attend_args(cfg, seqs, queries, q_lat, latent, pool_idx, n_sel, out, lse, workspace,
                                          d_status), stream)


def forward_args(cfg: Config, seqs: Seqs, queries: Queries, *, prev_len, new_off, max_new_per_seq, keys, gates,
                 ape, tail_keys, tail_gates, pooled, q_idx, w, q_lat, latent, out, lse=None, pool_idx=None,
                 n_sel=None, workspace=None, d_status=None, q_lat_ready=None) -> kp_forward_args:
    """q_lat_ready: None, or a recorded torch.cuda.Event that the attention
    launch waits for (kp_forward_args.q_lat_ready)."""
    ws_bytes = 0 if workspace is None else workspace.numel() * workspace.element_size()
    ev = None
    if q_lat_ready is not None:
        ev = q_lat_ready.cuda_event
        if not ev:
            raise ValueError("q_lat_ready: the event has not been recorded")
    return kp_forward_args(cfg.c(), seqs.c(), queries.c(), _p(prev_len), _p(new_off), keys.shape[0],
                           int(max_new_per_seq), _p(keys), _p(gates), _p(ape), _p(tail_keys), _p(tail_gates),
                           _p(pooled), _p(q_idx), _p(w), _p(q_lat), _p(latent), _p(out), _p(lse), _p(pool_idx),
                           _p(n_sel), _p(workspace), ws_bytes, _p(d_status), ev)


def kp_workspace_size(args: kp_forward_args) -> int:
    return int(lib().kp_workspace_size(ctypes.byref(args)))


def kp_dsa_forward(args: kp_forward_args, stream=None) -> None:
    _check(lib().kp_dsa_forward(ctypes.byref(args), _stream(stream)), "kp_dsa_forward")


def kp_read_device_status(d_status: torch.Tensor, stream=None) -> int:
    return int(lib().kp_read_device_status(_p(d_status), _stream(stream)))


def kp_version() -> int:
    return int(lib().kp_version())


# ---------------------------------------------------------------- the steps either side

def kp_gemm_bf16(a, b, c, m, n, k, batch=1, lda=None, a_batch_off=0, ldb=None, b_batch_off=0, ldc=None,
                 c_batch_off=0, d_status=None, stream=None, wait_limit_us=0) -> None:
    """C[b][m][n] = sum_k A[b][m][k] B[b][n][k] (bf16 tensors A, B; C bf16 or fp32)."""
    c_dtype = DTYPE_F32 if c.dtype == torch.float32 else DTYPE_BF16
    g = kp_gemm_args(m, n, k, batch, _p(a), lda if lda is not None else k, a_batch_off, _p(b),
                     ldb if ldb is not None else k, b_batch_off, _p(c), ldc if ldc is not None else n, c_batch_off,
                     c_dtype, int(wait_limit_us), _p(d_status))
    _check(lib().kp_gemm_bf16(ctypes.byref(g), _stream(stream)), "kp_gemm_bf16")


def kp_indexer_project(hidden, q_lora, w_iq, w_ik, w_ig, w_iw, q_idx, keys, gates, w, d_status=None,
                       stream=None) -> None:
    a = kp_indexer_project_args(hidden.shape[0], _p(hidden), _p(q_lora), _p(w_iq), _p(w_ik), _p(w_ig), _p(w_iw),
                                _p(q_idx), _p(keys), _p(gates), _p(w), 0, _p(d_status))
    _check(lib().kp_indexer_project(ctypes.byref(a), _stream(stream)), "kp_indexer_project")


def kp_mla_absorb_q(q_nope, w_uk, q_lat, d_status=None, stream=None) -> None:
    a = kp_mla_absorb_q_args(q_nope.shape[0], _p(q_nope), _p(w_uk), _p(q_lat), 0, _p(d_status))
    _check(lib().kp_mla_absorb_q(ctypes.byref(a), _stream(stream)), "kp_mla_absorb_q")


def kp_mla_absorb_out(out, w_uv, w_o, o, hidden_out, d_status=None, stream=None) -> None:
    a = kp_mla_absorb_out_args(out.shape[0], _p(out), _p(w_uv), _p(w_o), _p(o), _p(hidden_out), 0, _p(d_status))
    _check(lib().kp_mla_absorb_out(ctypes.byref(a), _stream(stream)), "kp_mla_absorb_out")
