// api.cu -- the extern "C" entry points of libkpool_dsa.so: argument checks,
// workspace carving and the fused step.  No allocation, no synchronisation
// (except kp_read_device_status), everything on the caller's stream.
#include <cmath>
#include <cstdio>
#include <cstring>
#include <string>

#include "kp_common.cuh"
#include "kp_internal.h"

namespace kp {

namespace {
thread_local std::string g_last_error;

bool aligned(const void *p, size_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

kp_status check_config(const kp_config &c) {
    if (c.kpool != 4 && c.kpool != 16) return KP_ERR_UNSUPPORTED;
    if (c.topk_tokens <= 0 || c.topk_tokens % c.kpool != 0) return KP_ERR_INVALID_ARG;
    if (c.topk_tokens / c.kpool > KP_MAX_TOPK_POOLS) return KP_ERR_UNSUPPORTED;
    if (c.compress_mode != KP_COMPRESS_LEARNED && c.compress_mode != KP_COMPRESS_MEAN)
        return KP_ERR_INVALID_ARG;
    if (c.always_select_tail != 0 && c.always_select_tail != 1) return KP_ERR_INVALID_ARG;
    if (!std::isfinite(c.sm_scale)) return KP_ERR_INVALID_ARG;
    if (c.wait_limit_us < 0) return KP_ERR_INVALID_ARG;
    if ((c.debug_flags & ~KP_DEBUG_STALL_FIRST_WAIT) != 0) return KP_ERR_INVALID_ARG;
    if (c.select_mode != KP_SELECT_AUTO && c.select_mode != KP_SELECT_STAGED && c.select_mode != KP_SELECT_FUSED)
        return KP_ERR_INVALID_ARG;
    return KP_OK;
}

kp_status check_queries(const kp_queries &q) {
    if (q.num_queries < 0) return KP_ERR_INVALID_ARG;
    if (q.num_queries > 0 && (!q.q_seq || !q.q_pos)) return KP_ERR_INVALID_ARG;
    if (q.max_pools < 0) return KP_ERR_INVALID_ARG;
    if (q.max_pools > KP_MAX_SCORE_POOLS) return KP_ERR_UNSUPPORTED;
    if (q.num_queries > (1 << 24)) return KP_ERR_UNSUPPORTED;
    return KP_OK;
}

bool is_pow2(int64_t x) { return x > 0 && (x & (x - 1)) == 0; }

// Layout checks: latent / pooled say which cache the call reads or writes.
// Paged mode: page_tokens a power of two in 16 .. 65536 holding at least 4
// pools, the latent cache a whole number of at least one page, the pooled
// cache as many pages of page_tokens / kpool rows, and valid page ids that
// fit a TMA row coordinate.
kp_status check_seqs(const kp_seqs &s, int kpool, bool latent, bool pooled, bool need_seq_len = true) {
    if (s.num_seqs < 1 || s.num_seqs > 65535 || (need_seq_len && !s.seq_len)) return KP_ERR_INVALID_ARG;
    if (s.latent_rows <= 0 && (latent || s.block_table)) return KP_ERR_INVALID_ARG;
    if (latent && s.latent_rows >= (int64_t(1) << 40)) return KP_ERR_INVALID_ARG;
    if (pooled && (s.pool_rows <= 0 || s.pool_rows >= (int64_t(1) << 31))) return KP_ERR_INVALID_ARG;
    if (!s.block_table) {
        if ((latent && !s.latent_row_off) || (pooled && !s.pool_row_off)) return KP_ERR_INVALID_ARG;
        return KP_OK;
    }
    if (!is_pow2(s.page_tokens) || s.page_tokens < 16 || s.page_tokens > 65536 || s.blocks_per_seq < 1 ||
        s.page_tokens < 4 * kpool)
        return KP_ERR_INVALID_ARG;
    const int64_t pages = s.latent_rows / s.page_tokens;
    if (pages < 1 || pages > INT32_MAX) return KP_ERR_INVALID_ARG;
    if (pooled && s.pool_rows < pages * (s.page_tokens / kpool)) return KP_ERR_INVALID_ARG;
    return KP_OK;
}

int64_t score_stride_for(int32_t max_pools) {
    const int64_t p = max_pools > 0 ? max_pools : 1;
    return (p + 127) / 128 * 128;
}

// Forward workspace layout: [scores][pool_idx][n_sel][step scratch].
// Whether the step scores and selects in one kernel (no score matrix).
bool forward_fused(const kp_forward_args &a) {
    return a.cfg.select_mode == KP_SELECT_FUSED && a.q.num_queries > 0 && score_select_fits(a.cfg, a.q);
}

struct ForwardLayout {
    size_t scores, pool_idx, n_sel, scratch, total;
};
ForwardLayout forward_layout(const kp_forward_args &a, int sm_count) {
    ForwardLayout L;
    const size_t nq = static_cast<size_t>(a.q.num_queries > 0 ? a.q.num_queries : 0);
    const size_t K = static_cast<size_t>(a.cfg.topk_tokens / (a.cfg.kpool > 0 ? a.cfg.kpool : 1));
    L.scores = 0;
    const size_t score_bytes = forward_fused(a) ? 0 : nq * score_stride_for(a.q.max_pools) * 4;
    L.pool_idx = L.scores + align_up(score_bytes, 256);
    L.n_sel = L.pool_idx + align_up(nq * K * 4, 256);
    L.scratch = L.n_sel + align_up(nq * 4, 256);
    const size_t plan = score_plan_bytes(static_cast<int32_t>(nq));
    const size_t att = attend_ws_bytes(a.cfg, static_cast<int32_t>(nq),
                                       attend_splits(a.cfg, static_cast<int32_t>(nq), sm_count));
    L.total = L.scratch + (plan > att ? plan : att);
    return L;
}
}  // namespace

CacheMap cache_map(const kp_seqs &s, int kpool) {
    CacheMap m;
    m.pool_shift = kpool_shift(kpool);
    m.latent_row_off = s.latent_row_off;
    m.pool_row_off = s.pool_row_off;
    m.block_table = s.block_table;
    m.page_shift = 0;
    m.blocks_per_seq = s.block_table ? s.blocks_per_seq : 0;
    m.num_pages = 0;
    if (s.block_table) {
        while ((1 << m.page_shift) < s.page_tokens) ++m.page_shift;
        m.num_pages = static_cast<int>(s.latent_rows / s.page_tokens);
    }
    m.latent_rows = s.latent_rows;
    m.pool_rows = s.pool_rows;
    return m;
}

void record_cuda_error(const char *where, cudaError_t err) {
    g_last_error = std::string(where) + ": " + cudaGetErrorName(err) + " (" + cudaGetErrorString(err) + ")";
}
void record_error_text(const char *text) { g_last_error = text; }

kp_status check_launch(const char *where) {
    cudaError_t e = cudaGetLastError();
    if (e != cudaSuccess) {
        record_cuda_error(where, e);
        return KP_ERR_CUDA;
    }
    return KP_OK;
}

namespace {
typedef CUresult (*EncodeTiledFn)(CUtensorMap *, CUtensorMapDataType, cuuint32_t, void *,
                                  const cuuint64_t *, const cuuint64_t *, const cuuint32_t *,
                                  const cuuint32_t *, CUtensorMapInterleave, CUtensorMapSwizzle,
                                  CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

// cuTensorMapEncodeTiled through the runtime's driver entry point, so the
// library needs no link-time dependency on libcuda.
EncodeTiledFn encode_fn() {
    static EncodeTiledFn fn = []() -> EncodeTiledFn {
        void *p = nullptr;
        cudaDriverEntryPointQueryResult q;
        if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &p, 12000, cudaEnableDefault,
                                             &q) != cudaSuccess ||
            q != cudaDriverEntryPointSuccess)
            return nullptr;
        return reinterpret_cast<EncodeTiledFn>(p);
    }();
    return fn;
}
}  // namespace

bool make_tmap_bf16_sw128(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows,
                          uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) {
        record_error_text("cuTensorMapEncodeTiled is not available");
        return false;
    }
    cuuint64_t dims[2] = {static_cast<cuuint64_t>(inner), static_cast<cuuint64_t>(rows)};
    cuuint64_t strides[1] = {static_cast<cuuint64_t>(row_bytes)};
    cuuint32_t box[2] = {box_inner, box_rows};
    cuuint32_t estr[2] = {1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void *>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        record_error_text("cuTensorMapEncodeTiled failed");
        return false;
    }
    return true;
}

bool make_tmap_bf16_sw128_kblocks(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows,
                                  uint64_t row_bytes, uint32_t box_rows, uint32_t kblocks) {
    EncodeTiledFn fn = encode_fn();
    if (!fn) {
        record_error_text("cuTensorMapEncodeTiled is not available");
        return false;
    }
    if (cols % 64 != 0) return false;
    // (64 columns, rows, column blocks of 64): a box of kblocks blocks lands as
    // kblocks consecutive [box_rows][128 B] slabs
    cuuint64_t dims[3] = {64, static_cast<cuuint64_t>(rows), static_cast<cuuint64_t>(cols / 64)};
    cuuint64_t strides[2] = {static_cast<cuuint64_t>(row_bytes), 128};
    cuuint32_t box[3] = {64, box_rows, kblocks};
    cuuint32_t estr[3] = {1, 1, 1};
    const CUresult r = fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void *>(base), dims, strides, box,
                          estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                          CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
    if (r != CUDA_SUCCESS) {
        record_error_text("cuTensorMapEncodeTiled (column blocks) failed");
        return false;
    }
    return true;
}

int device_sm_count() {
    int dev = 0, n = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess) return 0;
    return n;
}

}  // namespace kp

using namespace kp;

extern "C" {

namespace {
// Argument checks of the four stages (no launch).  KP_OK with nothing to do
// (no new tokens, no queries) is left to the launchers.
kp_status validate_compress(const kp_compress_args *a) {
    if (!a) return KP_ERR_INVALID_ARG;
    kp_status st = check_config(a->cfg);
    if (st != KP_OK) return st;
    if (a->num_seqs < 1 || a->num_seqs > 65535 || a->num_new < 0 || a->max_new_per_seq < 0)
        return KP_ERR_INVALID_ARG;
    if (a->num_new == 0) return KP_OK;
    if (a->max_new_per_seq == 0 || a->max_new_per_seq > a->num_new) return KP_ERR_INVALID_ARG;
    if (!a->prev_len || !a->new_off || !a->keys || !a->tail_keys || !a->pooled) return KP_ERR_INVALID_ARG;
    if (a->seqs.num_seqs != a->num_seqs) return KP_ERR_INVALID_ARG;
    const kp_status sst = check_seqs(a->seqs, a->cfg.kpool, false, true, false);
    if (sst != KP_OK) return sst;
    if (a->cfg.compress_mode == KP_COMPRESS_LEARNED && (!a->gates || !a->ape || !a->tail_gates))
        return KP_ERR_INVALID_ARG;
    if (!aligned(a->keys, 8) || !aligned(a->pooled, 8) || !aligned(a->tail_keys, 8) ||
        (a->gates && !aligned(a->gates, 8)) || (a->ape && !aligned(a->ape, 8)) ||
        (a->tail_gates && !aligned(a->tail_gates, 8)))
        return KP_ERR_INVALID_ARG;
    return KP_OK;
}

kp_status validate_score(const kp_score_args *a) {
    if (!a) return KP_ERR_INVALID_ARG;
    kp_status st = check_config(a->cfg);
    if (st != KP_OK) return st;
    if ((st = check_queries(a->q)) != KP_OK) return st;
    if ((st = check_seqs(a->seqs, a->cfg.kpool, false, true)) != KP_OK) return st;
    if (a->q.num_queries == 0) return KP_OK;
    if (!a->q_idx || !a->w || !a->pooled || !a->scores) return KP_ERR_INVALID_ARG;
    if (!aligned(a->q_idx, 16) || !aligned(a->pooled, 16) || !aligned(a->w, 4) || !aligned(a->scores, 4))
        return KP_ERR_INVALID_ARG;
    if (a->score_stride < score_stride_for(a->q.max_pools)) return KP_ERR_INVALID_ARG;
    if (!a->workspace || a->workspace_bytes < score_plan_bytes(a->q.num_queries) ||
        !aligned(a->workspace, 256))
        return KP_ERR_WORKSPACE;
    return KP_OK;
}

kp_status validate_topk(const kp_topk_args *a) {
    if (!a) return KP_ERR_INVALID_ARG;
    kp_status st = check_config(a->cfg);
    if (st != KP_OK) return st;
    if ((st = check_queries(a->q)) != KP_OK) return st;
    if (a->q.num_queries == 0) return KP_OK;
    if (!a->scores || !a->pool_idx || !a->n_sel) return KP_ERR_INVALID_ARG;
    if (a->score_stride < (a->q.max_pools > 0 ? a->q.max_pools : 1)) return KP_ERR_INVALID_ARG;
    return KP_OK;
}

size_t attend_ws_need(const kp_config &cfg, int32_t num_queries) {
    if (cfg.kpool <= 0 || cfg.topk_tokens <= 0) return 256;
    int sms = device_sm_count();
    if (sms <= 0) sms = 148;
    return attend_ws_bytes(cfg, num_queries, attend_splits(cfg, num_queries, sms));
}

kp_status validate_attend(const kp_attend_args *a) {
    if (!a) return KP_ERR_INVALID_ARG;
    kp_status st = check_config(a->cfg);
    if (st != KP_OK) return st;
    if ((st = check_queries(a->q)) != KP_OK) return st;
    if ((st = check_seqs(a->seqs, a->cfg.kpool, true, false)) != KP_OK) return st;
    if (a->q.num_queries == 0) return KP_OK;
    if (!a->q_lat || !a->latent || !a->pool_idx || !a->n_sel || !a->out) return KP_ERR_INVALID_ARG;
    if (!aligned(a->q_lat, 16) || !aligned(a->latent, 16) || !aligned(a->out, 4)) return KP_ERR_INVALID_ARG;
    if (a->seqs.latent_rows > INT32_MAX) return KP_ERR_UNSUPPORTED;  // TMA row coordinates are int32
    const size_t need = attend_ws_need(a->cfg, a->q.num_queries);
    if (need > 256 && (!a->workspace || a->workspace_bytes < need || !aligned(a->workspace, 256)))
        return KP_ERR_WORKSPACE;
    return KP_OK;
}
}  // namespace

kp_status kp_kpool_compress(const kp_compress_args *a, kp_stream_t stream) {
    const kp_status st = validate_compress(a);
    if (st != KP_OK || a->num_new == 0) return st;
    return launch_compress(*a, reinterpret_cast<cudaStream_t>(stream));
}

size_t kp_score_workspace_size(int32_t num_queries) {
    return score_plan_bytes(num_queries > 0 ? num_queries : 0);
}

kp_status kp_indexer_score(const kp_score_args *a, kp_stream_t stream) {
    const kp_status st = validate_score(a);
    if (st != KP_OK || a->q.num_queries == 0) return st;
    return launch_score(*a, reinterpret_cast<cudaStream_t>(stream));
}

kp_status kp_topk_select(const kp_topk_args *a, kp_stream_t stream) {
    const kp_status st = validate_topk(a);
    if (st != KP_OK || a->q.num_queries == 0) return st;
    return launch_topk(*a, reinterpret_cast<cudaStream_t>(stream));
}

kp_status kp_indexer_score_select(const kp_score_select_args *a, kp_stream_t stream) {
    if (!a) return KP_ERR_INVALID_ARG;
    kp_status st = check_config(a->cfg);
    if (st != KP_OK) return st;
    if ((st = check_queries(a->q)) != KP_OK) return st;
    if ((st = check_seqs(a->seqs, a->cfg.kpool, false, true)) != KP_OK) return st;
    if (a->q.num_queries == 0) return KP_OK;
    if (!score_select_fits(a->cfg, a->q)) return KP_ERR_UNSUPPORTED;
    if (!a->q_idx || !a->w || !a->pooled || !a->pool_idx || !a->n_sel) return KP_ERR_INVALID_ARG;
    if (!aligned(a->q_idx, 16) || !aligned(a->pooled, 16) || !aligned(a->w, 4)) return KP_ERR_INVALID_ARG;
    if (!a->workspace || a->workspace_bytes < score_plan_bytes(a->q.num_queries) || !aligned(a->workspace, 256))
        return KP_ERR_WORKSPACE;
    kp_score_args sc;
    std::memset(&sc, 0, sizeof sc);
    sc.cfg = a->cfg;
    sc.seqs = a->seqs;
    sc.q = a->q;
    sc.q_idx = a->q_idx;
    sc.w = a->w;
    sc.pooled = a->pooled;
    sc.workspace = a->workspace;
    sc.workspace_bytes = a->workspace_bytes;
    sc.d_status = a->d_status;
    kp_topk_args tk;
    std::memset(&tk, 0, sizeof tk);
    tk.cfg = a->cfg;
    tk.q = a->q;
    tk.pool_idx = a->pool_idx;
    tk.n_sel = a->n_sel;
    tk.d_status = a->d_status;
    return launch_score_select(sc, tk, reinterpret_cast<cudaStream_t>(stream), false, nullptr);
}

size_t kp_attend_workspace_size(const kp_config *cfg, int32_t num_queries) {
    if (!cfg) return 256;
    return attend_ws_need(*cfg, num_queries);
}

kp_status kp_sparse_mla_attend(const kp_attend_args *a, kp_stream_t stream) {
    const kp_status st = validate_attend(a);
    if (st != KP_OK || a->q.num_queries == 0) return st;
    return launch_attend(*a, reinterpret_cast<cudaStream_t>(stream));
}

size_t kp_workspace_size(const kp_forward_args *a) {
    if (!a) return 0;
    int sms = device_sm_count();
    if (sms <= 0) sms = 148;
    return forward_layout(*a, sms).total;
}

// The attention is the only stage that reads q_lat: when the caller's copy of
// q_lat may still be in flight, the stream waits for it here, after the
// earlier stages were launched.
static kp_status wait_for_q_lat(const kp_forward_args &a, cudaStream_t s) {
    if (!a.q_lat_ready) return KP_OK;
    const cudaError_t e = cudaStreamWaitEvent(s, reinterpret_cast<cudaEvent_t>(a.q_lat_ready), 0);
    if (e != cudaSuccess) {
        record_cuda_error("cudaStreamWaitEvent(q_lat_ready)", e);
        return KP_ERR_CUDA;
    }
    return KP_OK;
}

kp_status kp_dsa_forward(const kp_forward_args *a, kp_stream_t stream) {
    if (!a) return KP_ERR_INVALID_ARG;
    kp_status st = check_config(a->cfg);
    if (st != KP_OK) return st;
    if ((st = check_queries(a->q)) != KP_OK) return st;
    if ((st = check_seqs(a->seqs, a->cfg.kpool, true, true)) != KP_OK) return st;
    // No out with queries: the selection only (stages 1-3), into the caller's
    // pool_idx and n_sel; the attention is left to kp_sparse_mla_attend.
    const bool select_only = a->q.num_queries > 0 && !a->out;
    if (select_only && (!a->pool_idx || !a->n_sel)) return KP_ERR_INVALID_ARG;
    const int sms = device_sm_count();
    if (sms <= 0) {
        record_error_text("cannot query the current CUDA device");
        return KP_ERR_CUDA;
    }
    const ForwardLayout L = forward_layout(*a, sms);
    if (!a->workspace || a->workspace_bytes < L.total || !aligned(a->workspace, 256)) return KP_ERR_WORKSPACE;
    uint8_t *ws = static_cast<uint8_t *>(a->workspace);

    kp_compress_args c;
    std::memset(&c, 0, sizeof c);
    c.cfg = a->cfg;
    c.num_seqs = a->seqs.num_seqs;
    c.prev_len = a->prev_len;
    c.new_off = a->new_off;
    c.num_new = a->num_new;
    c.max_new_per_seq = a->max_new_per_seq;
    c.keys = a->keys;
    c.gates = a->gates;
    c.ape = a->ape;
    c.tail_keys = a->tail_keys;
    c.tail_gates = a->tail_gates;
    c.pooled = a->pooled;
    c.seqs = a->seqs;
    c.d_status = a->d_status;

    kp_score_args sc;
    std::memset(&sc, 0, sizeof sc);
    sc.cfg = a->cfg;
    sc.seqs = a->seqs;
    sc.q = a->q;
    sc.q_idx = a->q_idx;
    sc.w = a->w;
    sc.pooled = a->pooled;
    sc.scores = reinterpret_cast<float *>(ws + L.scores);
    sc.score_stride = score_stride_for(a->q.max_pools);
    sc.workspace = ws + L.scratch;
    sc.workspace_bytes = L.total - L.scratch;
    sc.d_status = a->d_status;

    kp_topk_args tk;
    std::memset(&tk, 0, sizeof tk);
    tk.cfg = a->cfg;
    tk.q = a->q;
    tk.scores = sc.scores;
    tk.score_stride = sc.score_stride;
    tk.pool_idx = a->pool_idx ? a->pool_idx : reinterpret_cast<int32_t *>(ws + L.pool_idx);
    tk.n_sel = a->n_sel ? a->n_sel : reinterpret_cast<int32_t *>(ws + L.n_sel);
    tk.d_status = a->d_status;

    kp_attend_args at;
    std::memset(&at, 0, sizeof at);
    at.cfg = a->cfg;
    at.seqs = a->seqs;
    at.q = a->q;
    at.q_lat = a->q_lat;
    at.latent = a->latent;
    at.pool_idx = tk.pool_idx;
    at.n_sel = tk.n_sel;
    at.out = a->out;
    at.lse = a->lse;
    at.workspace = ws + L.scratch;
    at.workspace_bytes = L.total - L.scratch;
    at.d_status = a->d_status;

    if ((st = validate_compress(&c)) != KP_OK) return st;
    if ((st = validate_score(&sc)) != KP_OK) return st;
    if ((st = validate_topk(&tk)) != KP_OK) return st;
    if (!select_only && (st = validate_attend(&at)) != KP_OK) return st;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    const bool queries = a->q.num_queries > 0;
    if (forward_fused(*a)) {
        // Scores and top-k in one kernel, the scores kept on chip.  Its plan
        // (groups of up to 4 queries) is built in that kernel when small
        // enough, else by an extra grid row of the compression launch, else
        // by the plan kernel.
        if (c.num_new > 0 && score_select_plan_is_local(a->q.num_queries)) {
            if ((st = launch_compress(c, s)) != KP_OK) return st;
            if ((st = launch_score_select(sc, tk, s, false, c.prev_len)) != KP_OK) return st;
        } else if (c.num_new > 0 && c.num_seqs < 65535) {
            const ScorePlanArgs pa = score_select_plan_args(sc);
            if ((st = launch_compress(c, s, &pa)) != KP_OK) return st;
            if ((st = launch_score_select(sc, tk, s, true, nullptr)) != KP_OK) return st;
        } else {
            if (c.num_new > 0 && (st = launch_compress(c, s)) != KP_OK) return st;
            if ((st = launch_score_select(sc, tk, s, false, nullptr)) != KP_OK) return st;
        }
        if (select_only) return KP_OK;
        if ((st = wait_for_q_lat(*a, s)) != KP_OK) return st;
        return launch_attend(at, s);
    }
    // The scorer's plan: built by the scorer itself in shared memory when it
    // fits (then the scorer also starts on the older pooled keys during the
    // compression); otherwise by an extra CTA of the compression launch (one
    // launch fewer), except when there is nothing to compress or no room for
    // one more row of CTAs in gridDim.y, where the scorer's own plan kernel runs.
    if (c.num_new > 0 && queries && score_plan_is_local(a->q.num_queries)) {
        // The scorer builds its plan itself and loads the pooled keys older than
        // this step while the compression runs.
        if ((st = launch_compress(c, s)) != KP_OK) return st;
        if ((st = launch_score(sc, s, false, c.prev_len)) != KP_OK) return st;
    } else if (c.num_new > 0 && queries && c.num_seqs < 65535) {
        const ScorePlanArgs pa = score_plan_args(sc);
        if ((st = launch_compress(c, s, &pa)) != KP_OK) return st;
        if ((st = launch_score(sc, s, true)) != KP_OK) return st;
    } else {
        if (c.num_new > 0 && (st = launch_compress(c, s)) != KP_OK) return st;
        if (queries && (st = launch_score(sc, s)) != KP_OK) return st;
    }
    if (!queries) return KP_OK;
    if ((st = launch_topk(tk, s)) != KP_OK) return st;
    if (select_only) return KP_OK;
    if ((st = wait_for_q_lat(*a, s)) != KP_OK) return st;
    return launch_attend(at, s);
}

// ---- the steps either side: dense products -------------------------------

namespace {
kp_status validate_gemm(const kp_gemm_args *g) {
    if (!g) return KP_ERR_INVALID_ARG;
    if (g->m < 0 || g->n < 0 || g->k <= 0 || g->k % 64 != 0 || g->batch < 1) return KP_ERR_INVALID_ARG;
    if (g->c_dtype != KP_DTYPE_BF16 && g->c_dtype != KP_DTYPE_F32) return KP_ERR_INVALID_ARG;
    if (g->wait_limit_us < 0) return KP_ERR_INVALID_ARG;
    if (g->m == 0 || g->n == 0) return KP_OK;
    if (!g->a || !g->b || !g->c) return KP_ERR_INVALID_ARG;
    if (!aligned(g->a, 16) || !aligned(g->b, 16) || !aligned(g->c, g->c_dtype == KP_DTYPE_F32 ? 4 : 2))
        return KP_ERR_INVALID_ARG;
    if (g->lda % 8 != 0 || g->ldb % 8 != 0 || g->ldb < g->k || g->ldc < 1) return KP_ERR_INVALID_ARG;
    if (g->a_batch_off < 0 || g->b_batch_off < 0 || g->c_batch_off < 0) return KP_ERR_INVALID_ARG;
    if (g->batch > 1 && (g->a_batch_off % 64 != 0 || g->b_batch_off < g->n)) return KP_ERR_INVALID_ARG;
    // every batch's K slice inside A's rows, and TMA row coordinates in int32
    if (g->a_batch_off * (g->batch - 1) + g->k > g->lda) return KP_ERR_INVALID_ARG;
    if (g->b_batch_off * (g->batch - 1) + g->n > INT32_MAX || g->m > INT32_MAX - 128) return KP_ERR_UNSUPPORTED;
    if (g->ldc < g->c_batch_off * (g->batch - 1) + g->n) return KP_ERR_INVALID_ARG;
    return KP_OK;
}

kp_gemm_args gemm_args(int m, int n, int k, int batch, const uint16_t *a, int64_t lda, int64_t a_off,
                       const uint16_t *b, int64_t ldb, int64_t b_off, void *c, int64_t ldc, int64_t c_off,
                       int32_t c_dtype, int32_t wait_limit_us, int32_t *d_status) {
    kp_gemm_args g;
    std::memset(&g, 0, sizeof g);
    g.m = m;
    g.n = n;
    g.k = k;
    g.batch = batch;
    g.a = a;
    g.lda = lda;
    g.a_batch_off = a_off;
    g.b = b;
    g.ldb = ldb;
    g.b_batch_off = b_off;
    g.c = c;
    g.ldc = ldc;
    g.c_batch_off = c_off;
    g.c_dtype = c_dtype;
    g.wait_limit_us = wait_limit_us;
    g.d_status = d_status;
    return g;
}

kp_status run_gemms(const kp_gemm_args *gs, int n, cudaStream_t s) {
    for (int i = 0; i < n; ++i) {
        const kp_status st = validate_gemm(&gs[i]);
        if (st != KP_OK) return st;
    }
    for (int i = 0; i < n; ++i) {
        const kp_status st = launch_gemm(gs[i], s);
        if (st != KP_OK) return st;
    }
    return KP_OK;
}
}  // namespace

kp_status kp_gemm_bf16(const kp_gemm_args *g, kp_stream_t stream) {
    const kp_status st = validate_gemm(g);
    if (st != KP_OK || g->m == 0 || g->n == 0) return st;
    return launch_gemm(*g, reinterpret_cast<cudaStream_t>(stream));
}

kp_status kp_indexer_project(const kp_indexer_project_args *a, kp_stream_t stream) {
    if (!a || a->num_tokens < 0) return KP_ERR_INVALID_ARG;
    if (a->num_tokens == 0) return KP_OK;
    const int T = a->num_tokens;
    const kp_gemm_args gs[4] = {
        gemm_args(T, KP_INDEX_HEADS * KP_INDEX_DIM, KP_Q_LORA, 1, a->q_lora, KP_Q_LORA, 0, a->w_iq, KP_Q_LORA, 0,
                  a->q_idx, KP_INDEX_HEADS * KP_INDEX_DIM, 0, KP_DTYPE_BF16, a->wait_limit_us, a->d_status),
        gemm_args(T, KP_INDEX_DIM, KP_HIDDEN, 1, a->hidden, KP_HIDDEN, 0, a->w_ik, KP_HIDDEN, 0, a->keys,
                  KP_INDEX_DIM, 0, KP_DTYPE_BF16, a->wait_limit_us, a->d_status),
        gemm_args(T, KP_INDEX_DIM, KP_HIDDEN, 1, a->hidden, KP_HIDDEN, 0, a->w_ig, KP_HIDDEN, 0, a->gates,
                  KP_INDEX_DIM, 0, KP_DTYPE_BF16, a->wait_limit_us, a->d_status),
        gemm_args(T, KP_INDEX_HEADS, KP_HIDDEN, 1, a->hidden, KP_HIDDEN, 0, a->w_iw, KP_HIDDEN, 0, a->w,
                  KP_INDEX_HEADS, 0, KP_DTYPE_F32, a->wait_limit_us, a->d_status)};
    for (const kp_gemm_args &g : gs) {
        const kp_status st = validate_gemm(&g);
        if (st != KP_OK) return st;
    }
    // four independent products: one launch, side by side
    return launch_gemm_group(gs, 4, reinterpret_cast<cudaStream_t>(stream));
}

kp_status kp_mla_absorb_q(const kp_mla_absorb_q_args *a, kp_stream_t stream) {
    if (!a || a->num_tokens < 0) return KP_ERR_INVALID_ARG;
    if (a->num_tokens == 0) return KP_OK;
    // batch = head: A = q_nope [T][64 * 256] (head h at column 256 h), B = W_UK
    // [64 * 512][256] (head h at row 512 h), C = q_lat [T][64 * 576] (head h at column 576 h)
    const kp_gemm_args g = gemm_args(a->num_tokens, KP_NOPE_DIM, KP_QK_NOPE, KP_MLA_HEADS, a->q_nope,
                                     KP_MLA_HEADS * KP_QK_NOPE, KP_QK_NOPE, a->w_uk, KP_QK_NOPE, KP_NOPE_DIM,
                                     a->q_lat, KP_MLA_HEADS * KP_LATENT_DIM, KP_LATENT_DIM, KP_DTYPE_BF16,
                                     a->wait_limit_us, a->d_status);
    return run_gemms(&g, 1, reinterpret_cast<cudaStream_t>(stream));
}

kp_status kp_mla_absorb_out(const kp_mla_absorb_out_args *a, kp_stream_t stream) {
    if (!a || a->num_tokens < 0) return KP_ERR_INVALID_ARG;
    if (a->num_tokens == 0) return KP_OK;
    const int T = a->num_tokens;
    const kp_gemm_args gs[2] = {
        // batch = head: A = out [T][64 * 512], B = W_UV [64 * 256][512], C = o [T][64 * 256]
        gemm_args(T, KP_V_HEAD, KP_NOPE_DIM, KP_MLA_HEADS, a->out, KP_MLA_HEADS * KP_NOPE_DIM, KP_NOPE_DIM, a->w_uv,
                  KP_NOPE_DIM, KP_V_HEAD, a->o, KP_MLA_HEADS * KP_V_HEAD, KP_V_HEAD, KP_DTYPE_BF16,
                  a->wait_limit_us, a->d_status),
        // o_proj: A = o [T][16384], B = W_O [4096][16384], C = hidden_out [T][4096]
        gemm_args(T, KP_HIDDEN, KP_MLA_HEADS * KP_V_HEAD, 1, a->o, KP_MLA_HEADS * KP_V_HEAD, 0, a->w_o,
                  KP_MLA_HEADS * KP_V_HEAD, 0, a->hidden_out, KP_HIDDEN, 0, KP_DTYPE_BF16, a->wait_limit_us,
                  a->d_status)};
    return run_gemms(gs, 2, reinterpret_cast<cudaStream_t>(stream));
}

const char *kp_status_string(kp_status s) {
    switch (s) {
        case KP_OK: return "ok";
        case KP_ERR_INVALID_ARG: return "invalid argument";
        case KP_ERR_UNSUPPORTED: return "unsupported shape or option";
        case KP_ERR_CUDA: return "CUDA error";
        case KP_ERR_DEVICE_TIMEOUT: return "device wait timed out";
        case KP_ERR_DEVICE_BOUNDS: return "device index out of range";
        case KP_ERR_WORKSPACE: return "workspace missing or too small";
    }
    return "unknown status";
}

const char *kp_last_error(void) { return g_last_error.c_str(); }

kp_status kp_read_device_status(const int32_t *d_status, kp_stream_t stream) {
    if (!d_status) return KP_ERR_INVALID_ARG;
    cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
    int32_t v = 0;
    cudaError_t e = cudaMemcpyAsync(&v, d_status, sizeof v, cudaMemcpyDeviceToHost, s);
    if (e == cudaSuccess) e = cudaStreamSynchronize(s);
    if (e != cudaSuccess) {
        record_cuda_error("kp_read_device_status", e);
        return KP_ERR_CUDA;
    }
    return static_cast<kp_status>(v);
}

int kp_version(void) { return 20400; }

}  // extern "C"

namespace kp {
kp_status score_with_workspace_plan(const kp_score_args *a, cudaStream_t stream) {
    const kp_status st = validate_score(a);
    if (st != KP_OK || a->q.num_queries == 0) return st;
    return launch_score(*a, stream, false, nullptr, false);
}
}  // namespace kp
