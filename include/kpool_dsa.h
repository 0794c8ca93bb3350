/*
 * kpool_dsa.h -- C ABI of the KPool DSA sparse-attention step (sm_103a).
 *
 * One DSA layer step of the GLM-5.3-Flash hybrid decoder, in four stages:
 *
 *   1. kp_kpool_compress     pool every run of `kpool` (4 or 16) consecutive indexer
 *                            keys into one pooled key and append it to the
 *                            pooled indexer cache; keep the rows of the
 *                            still-incomplete pool in a per-sequence tail ring.
 *                            (MAX docs, max.pipelines.architectures.glm5_next,
 *                            Glm5NextConfig.index_kpool / index_kpool_compress;
 *                            llama.cpp PR "add GLM-5.3-Flash (GLM5-Next)
 *                            support", Overview: pools of 4 consecutive tokens,
 *                            per-token key | gate.)
 *   2. kp_indexer_score      lightning-indexer score of every complete pool a
 *                            query can see: s = sum_h w_h * ReLU(q_h . k_pool),
 *                            32 heads x 128 dims (llm-atlas GLM-5.3-Flash card,
 *                            raw config index_n_heads / index_head_dim).
 *   3. kp_topk_select        the index_topk / kpool best pools per query
 *                            (2048 tokens = 512 pools; llm-atlas card,
 *                            index_topk), ascending pool order.
 *   4. kp_sparse_mla_attend  nope-only MLA in latent space over the selected
 *                            pools' rows plus the query's incomplete tail pool
 *                            (MAX docs Glm5NextConfig.index_kpool_always_select_tail,
 *                            mla_use_nope; Glm5Next.build_layers: 576-wide
 *                            latent rows whose last 64 columns are zero).
 *
 *   kp_indexer_score_select  2 and 3 in one kernel, the scores kept on chip.
 *
 *   kp_dsa_forward runs 1-4 in order on one stream.
 *
 * Conventions shared by every entry point
 * ---------------------------------------
 *  - Every pointer in an args struct is a DEVICE pointer unless marked
 *    "host".  The args struct itself is read on the host during the call
 *    and may be freed when the call returns.
 *  - bf16 tensors are passed as `uint16_t*` holding bf16 bit patterns.
 *  - The caller owns every buffer.  The library allocates no device or host
 *    memory per call (a tensor-map descriptor is built on the host stack),
 *    frees nothing, and never synchronises the stream, except
 *    kp_read_device_status.
 *  - All work is enqueued on `stream` (a cudaStream_t; NULL = legacy default
 *    stream) in order.  Calls are graph-capturable.  Calls on different
 *    streams that share output or workspace buffers race.
 *  - Host-side validation runs before any launch.  A call that returns an
 *    error other than KP_ERR_CUDA has enqueued nothing.
 *  - `d_status` (optional, may be NULL) is a device int32 the kernels set to
 *    a kp_status code when they detect bad data (an out-of-range pool index
 *    or cache row); the offending element is skipped, never dereferenced.
 *    The library never clears it: zero it before the calls you want to check.
 *  - Fixed shapes (compile-time): indexer 32 heads x 128 dims; MLA 64 heads
 *    over latent rows of 576 bf16 of which the first 512 are read; kpool 4
 *    (the llm-atlas card's index_kpool) or 16 (the NeMo AutoModel
 *    Glm5NextTextConfig default).  Anything else returns KP_ERR_UNSUPPORTED.
 *
 * Query positions and visibility
 * ------------------------------
 *  A query q belongs to sequence q_seq[q] and sits at absolute position
 *  t = q_pos[q] (0-based, t < seq_len of that sequence).  It sees the
 *  n_full(t) = floor((t + 1) / kpool) complete pools of its sequence; its tail
 *  is positions kpool * n_full(t) .. t (empty when (t + 1) % kpool == 0),
 *  always attended when always_select_tail, and never scored.  Decode, MTP
 *  verification and chunked causal prefill differ only in these arrays.
 */
#ifndef KPOOL_DSA_H
#define KPOOL_DSA_H

#include <stddef.h>
#include <stdint.h>

#if defined(__GNUC__)
#define KP_API __attribute__((visibility("default")))
#else
#define KP_API
#endif

#ifdef __cplusplus
extern "C" {
#endif

/* cudaStream_t and cudaEvent_t without including the CUDA headers. */
typedef struct CUstream_st *kp_stream_t;
typedef struct CUevent_st *kp_event_t;

typedef enum kp_status {
    KP_OK = 0,
    KP_ERR_INVALID_ARG = 1,     /* null pointer, negative size, inconsistent sizes */
    KP_ERR_UNSUPPORTED = 2,     /* shape or option this build does not implement */
    KP_ERR_CUDA = 3,            /* a CUDA runtime or driver call failed (see kp_last_error) */
    KP_ERR_DEVICE_TIMEOUT = 4,  /* a kernel's bounded wait ran out (device status) */
    KP_ERR_DEVICE_BOUNDS = 5,   /* a kernel met an out-of-range index (device status) */
    KP_ERR_WORKSPACE = 6        /* workspace missing or smaller than required */
} kp_status;

enum {
    KP_INDEX_HEADS = 32,   /* lightning-indexer heads */
    KP_INDEX_DIM = 128,    /* indexer key / query width */
    KP_MLA_HEADS = 64,     /* attention heads */
    KP_LATENT_DIM = 576,   /* latent cache row width (bf16) */
    KP_NOPE_DIM = 512,     /* latent columns read (kv_lora_rank); 512..575 are zero */
    KP_KPOOL = 4,          /* tokens per pool (16 is supported too) */
    KP_MAX_TOPK_POOLS = 1024,    /* largest supported topk_tokens / kpool */
    KP_MAX_SCORE_POOLS = 262144, /* largest supported pools per query (1,048,576 tokens) */
    KP_NOALLOC_MAX_QUERIES = 8192, /* largest num_queries of kp_indexer_score_noalloc */
    KP_FUSED_MAX_POOLS = 16384    /* largest max_pools of kp_indexer_score_select */
};

enum { KP_COMPRESS_LEARNED = 0, KP_COMPRESS_MEAN = 1 };

/* debug_flags bits (tests of the failure paths; 0 in normal use). */
enum {
    /* The first pipeline wait of the scoring and attention kernels waits on a
     * barrier that nothing completes, so it gives up after wait_limit_us: the
     * kernel sets KP_ERR_DEVICE_TIMEOUT in d_status, lets every copy and MMA
     * it issued finish, frees its tensor memory and returns (outputs of the
     * call are then undefined).  Host-side only: no fault, no trap. */
    KP_DEBUG_STALL_FIRST_WAIT = 1
};

/* select_mode values: how kp_dsa_forward scores and selects. */
enum {
    /* The faster path for the call's shape on B300.  At present that is the
     * staged kernels (kp_indexer_score then kp_topk_select) on every shape. */
    KP_SELECT_AUTO = 0,
    /* kp_indexer_score then kp_topk_select: the fp32 score matrix
     * [NQ][max_pools rounded up to 128] lives in the workspace. */
    KP_SELECT_STAGED = 1,
    /* kp_indexer_score_select: scores kept on chip, no score matrix in the
     * workspace, when max_pools <= KP_FUSED_MAX_POOLS (else staged).  Same
     * results, bit for bit. */
    KP_SELECT_FUSED = 2
};

/* Method and execution options. */
typedef struct kp_config {
    int32_t kpool;              /* tokens per pool: 4, or 16 */
    int32_t topk_tokens;        /* token budget of the top-k (index_topk, 2048); a
                                   positive multiple of kpool, <= 4 * KP_MAX_TOPK_POOLS */
    int32_t compress_mode;      /* KP_COMPRESS_LEARNED (gate + ape softmax) or _MEAN */
    int32_t always_select_tail; /* 1: the query's incomplete pool is always attended */
    float sm_scale;             /* attention logit scale (1/16 = 1/sqrt(qk_head_dim 256)) */
    int32_t wait_limit_us;      /* limit of any one device-side wait in microseconds; 0 =
                                   1 s.  A wait that runs out sets KP_ERR_DEVICE_TIMEOUT
                                   in d_status and the kernel returns early */
    int32_t debug_flags;        /* KP_DEBUG_* bits; 0 in normal use */
    int32_t select_mode;        /* KP_SELECT_*: how kp_dsa_forward runs stages 2-3 */
} kp_config;

/* Per-sequence cache layout, in one of two modes.
 *
 * Contiguous (block_table == NULL): sequence b's latent rows are rows
 * latent_row_off[b] .. + seq_len[b] - 1 of the latent cache (row i = token
 * position i), and its pooled keys are rows pool_row_off[b] + p of the pooled
 * cache (p = pool index).
 *
 * Paged (block_table != NULL): both caches are split into pages of
 * page_tokens token positions; the latent cache holds page j at rows
 * j * page_tokens .. + page_tokens - 1 and the pooled cache holds the same
 * page's pooled keys at rows j * (page_tokens / kpool) .. + page_tokens /
 * kpool - 1, so one physical page id addresses both (the KV-pool pages of the
 * MAX docs, Glm5NextConfig.infer_optimal_batch_size; the persistent block
 * table of the Rust loader's Mixer::Dsa).  Position i of sequence b lives in
 * physical page block_table[b * blocks_per_seq + i / page_tokens], pool p in
 * page block_table[b * blocks_per_seq + p / (page_tokens / kpool)].  A pool
 * never straddles two pages.  latent_row_off / pool_row_off are unused.  The
 * valid page ids are 0 .. latent_rows / page_tokens - 1, and the pooled cache
 * needs at least that many pages of rows; a page id out of range, or a
 * position past blocks_per_seq pages, is skipped and reported as
 * KP_ERR_DEVICE_BOUNDS.  Entries of pages past a sequence's length are never
 * read. */
typedef struct kp_seqs {
    int32_t num_seqs;                /* host: B >= 1 */
    const int32_t *seq_len;          /* [B] tokens in the caches, after this step's appends; a
                                        query at or past its sequence's length is skipped
                                        (no scores, out 0, lse -inf) with KP_ERR_DEVICE_BOUNDS */
    const int64_t *latent_row_off;   /* [B] (contiguous mode) */
    const int64_t *pool_row_off;     /* [B] (contiguous mode) */
    int64_t latent_rows;             /* host: rows allocated in the latent cache */
    int64_t pool_rows;               /* host: rows allocated in the pooled cache (< 2^31:
                                        TMA row coordinates are signed 32-bit) */
    const int32_t *block_table;      /* [B][blocks_per_seq] physical page ids (paged mode), or NULL */
    int32_t page_tokens;             /* host, paged mode: tokens per page, a power of two in
                                        16 .. 65536 */
    int32_t blocks_per_seq;          /* host, paged mode: row length of block_table, >= 1 */
} kp_seqs;

/* The query tokens of this step, flattened over sequences.  Queries of one
 * sequence should be adjacent (any order is correct; adjacency lets the
 * scorer share pooled-key tiles between them). */
typedef struct kp_queries {
    int32_t num_queries;        /* host: NQ >= 0 */
    const int32_t *q_seq;       /* [NQ] sequence of each query */
    const int32_t *q_pos;       /* [NQ] absolute position of each query */
    int32_t max_pools;          /* host: an upper bound of n_full(q_pos) over the queries,
                                   <= KP_MAX_SCORE_POOLS */
    const int32_t *share_src;   /* [NQ] or NULL: shared selection (below) */
} kp_queries;

/* Shared selection (MAX docs, Glm5NextConfig.index_share_for_mtp_iteration,
 * read for the MTP verification query of a step): share_src[q] >= 0 names the
 * query whose selection query q attends, instead of its own.  The source must
 * be a query of the same sequence that is not itself shared.  Then:
 *  - kp_topk_select and kp_indexer_score_select skip query q: pool_idx[q] and
 *    n_sel[q] are left as they were (kp_indexer_score still scores it);
 *  - kp_sparse_mla_attend attends the source's pool_idx row and n_sel (pools
 *    past q's own n_full are skipped and reported) plus q's own tail.
 * A source out of range, in another sequence or itself shared is reported as
 * KP_ERR_DEVICE_BOUNDS, and query q then attends its tail alone.
 * share_src[q] < 0, or share_src NULL: q selects for itself. */

/* ---- 1. pooled-key compression (fused into the indexer-cache write) ---- */
/* For sequence b the new tokens are positions prev_len[b] .. prev_len[b] +
 * n_b - 1 with n_b = new_off[b+1] - new_off[b]; their raw indexer key and gate
 * rows are rows new_off[b] .. new_off[b+1]-1 of `keys` / `gates`.  Every pool
 * the new tokens complete is written to the pooled cache:
 *   logit_i[d] = gate[kpool*p + i][d] + ape[i][d],  alpha = softmax_i(logit)
 *   pooled[p][d] = bf16_rne( sum_i alpha_i[d] * key[kpool*p + i][d] )
 * (mean mode: alpha_i = 1/kpool), fp32 arithmetic.  Rows of a pool that is
 * still incomplete after the step go to the tail ring, slot = position %
 * kpool; rows of older positions of a completing pool are read from there.
 * The ring must hold the rows of positions kpool*floor(prev_len/kpool) ..
 * prev_len-1 on entry (any content when that range is empty). */
typedef struct kp_compress_args {
    kp_config cfg;
    int32_t num_seqs;             /* host: B */
    const int32_t *prev_len;      /* [B] tokens already appended before this call */
    const int32_t *new_off;       /* [B+1] CSR offsets into keys/gates; new_off[0] = 0 */
    int32_t num_new;              /* host: total new tokens = new_off[B] */
    int32_t max_new_per_seq;      /* host: an upper bound of n_b */
    const uint16_t *keys;         /* [num_new][128] bf16 */
    const uint16_t *gates;        /* [num_new][128] bf16 (unused in mean mode, may be NULL) */
    const uint16_t *ape;          /* [kpool][128] bf16 (unused in mean mode, may be NULL) */
    uint16_t *tail_keys;          /* [B][kpool-1][128] bf16, in/out */
    uint16_t *tail_gates;         /* [B][kpool-1][128] bf16, in/out */
    uint16_t *pooled;             /* [pool_rows][128] bf16, out (completed pools only) */
    kp_seqs seqs;                 /* pooled-cache addressing: uses num_seqs (== num_seqs above),
                                     pool_row_off and pool_rows, or the block table */
    int32_t *d_status;            /* optional */
} kp_compress_args;

/* ---- 2. indexer scores ---- */
/* scores[q][p] = sum_h w[q][h] * max(0, sum_d q_idx[q][h][d] * pooled[row(p)][d])
 * for p < n_full(q_pos[q]), fp32 (bf16 products, fp32 accumulation).  Entries
 * n_full .. the next multiple of 128 are set to -inf; later entries of the
 * row are left as they were. */
typedef struct kp_score_args {
    kp_config cfg;
    kp_seqs seqs;                 /* uses num_seqs, seq_len, pool_row_off, pool_rows or the block table */
    kp_queries q;
    const uint16_t *q_idx;        /* [NQ][32][128] bf16 */
    const float *w;               /* [NQ][32] fp32 head weights */
    const uint16_t *pooled;       /* [pool_rows][128] bf16 */
    float *scores;                /* [NQ][score_stride] fp32, out */
    int64_t score_stride;         /* host: >= max_pools rounded up to 128 */
    void *workspace;              /* >= kp_score_workspace_size(NQ) bytes, 256-aligned */
    size_t workspace_bytes;
    int32_t *d_status;
} kp_score_args;

/* ---- 3. top-k pool selection ---- */
/* For each query with n = n_full(q_pos[q]) and K = topk_tokens / kpool:
 * n_sel[q] = min(K, n); pool_idx[q][0 .. n_sel) = the selected pools in
 * ascending order (all pools when n <= K, else the K largest scores, ties to
 * the lower index; -0 equals +0; NaN ranks lowest); pool_idx[q][n_sel .. K)
 * = -1. */
typedef struct kp_topk_args {
    kp_config cfg;
    kp_queries q;
    const float *scores;          /* [NQ][score_stride] */
    int64_t score_stride;         /* host */
    int32_t *pool_idx;            /* [NQ][K] out */
    int32_t *n_sel;               /* [NQ] out */
    int32_t *d_status;
} kp_topk_args;

/* ---- 2+3 in one kernel ---- */
/* The pool_idx and n_sel of kp_indexer_score followed by kp_topk_select, bit
 * for bit, with every score kept in on-chip memory: no score matrix is
 * written (the llama.cpp PR "add GLM-5.3-Flash (GLM5-Next) support", review
 * comments: re-materialised pooled intermediates are what slow the graph).
 * A group of up to 4 adjacent queries of one sequence is scored by a cluster
 * of C CTAs (C * 2048 >= max_pools), each CTA holding its 2048-pool slice's
 * scores in shared memory; one CTA per query then gathers the row and selects.
 * max_pools above KP_FUSED_MAX_POOLS returns KP_ERR_UNSUPPORTED (use the
 * staged calls).  A query whose visible pools exceed max_pools is cut at
 * the cluster's capacity and reported as KP_ERR_DEVICE_BOUNDS. */
typedef struct kp_score_select_args {
    kp_config cfg;
    kp_seqs seqs;                 /* as kp_score_args */
    kp_queries q;
    const uint16_t *q_idx;        /* [NQ][32][128] bf16 */
    const float *w;               /* [NQ][32] fp32 */
    const uint16_t *pooled;       /* [pool_rows][128] bf16 */
    int32_t *pool_idx;            /* [NQ][K] out, as kp_topk_args */
    int32_t *n_sel;               /* [NQ] out */
    void *workspace;              /* >= kp_score_workspace_size(NQ) bytes, 256-aligned */
    size_t workspace_bytes;
    int32_t *d_status;
} kp_score_select_args;

/* ---- 4. sparse MLA over the selected pools + tail ---- */
/* Token set of query q: rows kpool*p .. kpool*p + kpool-1 of every selected
 * pool p, then the tail positions (when always_select_tail).  For head h:
 *   z_s = sm_scale * sum_{d<512} q_lat[q][h][d] * latent[row_s][d]
 *   out[q][h][:] = sum_s softmax(z)_s * latent[row_s][0..512)   (bf16, RNE)
 *   lse[q][h] = ln sum_s exp(z_s)                                (fp32)
 * An empty token set gives out = 0 and lse = -inf.
 * latent_rows above 2^31 - 1 returns KP_ERR_UNSUPPORTED (rows are gathered
 * by TMA, whose coordinates are signed 32-bit). */
typedef struct kp_attend_args {
    kp_config cfg;
    kp_seqs seqs;                 /* uses seq_len, latent_row_off, latent_rows or the block table */
    kp_queries q;
    const uint16_t *q_lat;        /* [NQ][64][576] bf16 (columns 512.. ignored) */
    const uint16_t *latent;       /* [latent_rows][576] bf16 */
    const int32_t *pool_idx;      /* [NQ][K] */
    const int32_t *n_sel;         /* [NQ] */
    uint16_t *out;                /* [NQ][64][512] bf16 out */
    float *lse;                   /* [NQ][64] fp32 out (may be NULL) */
    void *workspace;              /* >= kp_attend_workspace_size(...) bytes */
    size_t workspace_bytes;
    int32_t *d_status;
} kp_attend_args;

/* ---- the whole step ---- */
typedef struct kp_forward_args {
    kp_config cfg;
    kp_seqs seqs;
    kp_queries q;
    /* stage 1 inputs (see kp_compress_args) */
    const int32_t *prev_len;
    const int32_t *new_off;
    int32_t num_new;
    int32_t max_new_per_seq;
    const uint16_t *keys;
    const uint16_t *gates;
    const uint16_t *ape;
    uint16_t *tail_keys;
    uint16_t *tail_gates;
    uint16_t *pooled;             /* pooled cache, in/out */
    /* stage 2-4 inputs */
    const uint16_t *q_idx;
    const float *w;
    const uint16_t *q_lat;
    const uint16_t *latent;
    /* outputs */
    uint16_t *out;                /* [NQ][64][512] bf16; NULL with queries: the call stops
                                     after the selection (stages 1-3), which it writes to
                                     pool_idx and n_sel (both required then); q_lat is not
                                     read, and kp_sparse_mla_attend runs the attention
                                     (for instance over chunks of the queries) */
    float *lse;                   /* [NQ][64] fp32 (may be NULL) */
    int32_t *pool_idx;            /* [NQ][K] (may be NULL: kept in the workspace) */
    int32_t *n_sel;               /* [NQ]    (may be NULL: kept in the workspace) */
    void *workspace;              /* >= kp_workspace_size(args) bytes */
    size_t workspace_bytes;
    int32_t *d_status;
    /* May be NULL.  An event that completes once q_lat holds this step's
     * queries, e.g. one recorded after an asynchronous host-to-device copy of
     * q_lat on another stream.  The call makes `stream` wait for it just
     * before the attention launch (cudaStreamWaitEvent), so compression,
     * scoring and selection run while q_lat is still in transit: no stage
     * before the attention reads q_lat.  Record the event before the call.
     * A failed wait returns KP_ERR_CUDA with the first stages already
     * launched and out / lse not written. */
    kp_event_t q_lat_ready;
} kp_forward_args;

KP_API kp_status kp_kpool_compress(const kp_compress_args *args, kp_stream_t stream);
KP_API kp_status kp_indexer_score(const kp_score_args *args, kp_stream_t stream);
KP_API kp_status kp_topk_select(const kp_topk_args *args, kp_stream_t stream);
KP_API kp_status kp_indexer_score_select(const kp_score_select_args *args, kp_stream_t stream);
KP_API kp_status kp_sparse_mla_attend(const kp_attend_args *args, kp_stream_t stream);
KP_API kp_status kp_dsa_forward(const kp_forward_args *args, kp_stream_t stream);

/* ---- the steps either side: projections and MLA absorption ----
 * Dense bf16 products around the DSA step, with the GLM-5.3-Flash widths
 * (llm-atlas GLM-5.3-Flash card, raw config: hidden_size 4096, q_lora_rank
 * 1536, qk_nope_head_dim 256, kv_lora_rank 512, num_attention_heads 64,
 * index_n_heads 32, index_head_dim 128; v_head_dim 256 from the NeMo
 * AutoModel Glm5NextTextConfig defaults).  fp32 accumulation; bf16 outputs
 * are rounded to nearest even. */
enum {
    KP_HIDDEN = 4096,       /* hidden size */
    KP_Q_LORA = 1536,       /* compressed query width (q_lora_rank) */
    KP_QK_NOPE = 256,       /* per-head query / key width (qk_nope_head_dim) */
    KP_V_HEAD = 256         /* per-head value width (v_head_dim) */
};
enum { KP_DTYPE_BF16 = 0, KP_DTYPE_F32 = 1 };

/* C[b][m][n] = sum_k A[b][m][k] * B[b][n][k] for b < batch (both operands
 * K-contiguous, "A times B transposed").  Batch b reads columns
 * b * a_batch_off .. + k - 1 of A's rows, rows b * b_batch_off .. + n - 1 of
 * B, and writes columns b * c_batch_off .. + n - 1 of C's rows. */
typedef struct kp_gemm_args {
    int32_t m, n, k;              /* host: per-batch sizes; m, n >= 0, k a positive multiple of 64 */
    int32_t batch;                /* host: >= 1 */
    const uint16_t *a;            /* bf16, row r at a + r * lda (16-byte aligned) */
    int64_t lda, a_batch_off;     /* host: elements; lda a multiple of 8 */
    const uint16_t *b;            /* bf16, row r at b + r * ldb (16-byte aligned) */
    int64_t ldb, b_batch_off;     /* host: elements; ldb a multiple of 8, >= k */
    void *c;                      /* bf16 or fp32, row r of batch b at c + r * ldc + b * c_batch_off */
    int64_t ldc, c_batch_off;     /* host: elements */
    int32_t c_dtype;              /* KP_DTYPE_BF16 or KP_DTYPE_F32 */
    int32_t wait_limit_us;        /* as kp_config.wait_limit_us */
    int32_t *d_status;            /* optional */
} kp_gemm_args;

/* The lightning indexer's inputs from a layer's hidden state, for T tokens
 * (DeepSeek-V3.2 lineage of Glm5NextConfig; the gate feeds the pooled-key
 * compression, index_kpool_compress):
 *   q_idx[t] = W_iq . q_lora[t]      [T][32][128] bf16   (W_iq  [32 * 128][1536])
 *   keys[t]  = W_ik . hidden[t]      [T][128] bf16       (W_ik  [128][4096])
 *   gates[t] = W_ig . hidden[t]      [T][128] bf16       (W_ig  [128][4096])
 *   w[t]     = W_iw . hidden[t]      [T][32] fp32        (W_iw  [32][4096])
 * Any scale of the score is folded into W_iw.  Weights are row-major [out][in]
 * bf16. */
typedef struct kp_indexer_project_args {
    int32_t num_tokens;           /* host: T >= 0 */
    const uint16_t *hidden;       /* [T][4096] */
    const uint16_t *q_lora;       /* [T][1536] */
    const uint16_t *w_iq, *w_ik, *w_ig, *w_iw;
    uint16_t *q_idx;              /* [T][32][128] out */
    uint16_t *keys;               /* [T][128] out */
    uint16_t *gates;              /* [T][128] out */
    float *w;                     /* [T][32] out */
    int32_t wait_limit_us;
    int32_t *d_status;
} kp_indexer_project_args;

/* Absorbed query: the key up-projection W_UK folded into the query, so the
 * attention runs on the latent cache (MAX docs Glm5NextConfig mla_use_nope,
 * kv_lora_rank; the cache stores the latent width):
 *   q_lat[t][h][c] = sum_d W_UK[h][c][d] * q_nope[t][h][d],  c < 512
 * q_nope [T][64][256] bf16, W_UK [64][512][256] bf16, q_lat [T][64][576] bf16
 * (columns 512..575 are left as they are: the attention does not read them). */
typedef struct kp_mla_absorb_q_args {
    int32_t num_tokens;
    const uint16_t *q_nope;
    const uint16_t *w_uk;
    uint16_t *q_lat;
    int32_t wait_limit_us;
    int32_t *d_status;
} kp_mla_absorb_q_args;

/* Output side: the value up-projection W_UV applied to the latent-space
 * attention output, then o_proj:
 *   o[t][h][v]      = sum_c W_UV[h][v][c] * out[t][h][c]       v < 256 (bf16)
 *   hidden_out[t]   = W_O . o[t]                               [T][4096] bf16
 * out [T][64][512] bf16 (kp_sparse_mla_attend's output), W_UV [64][256][512]
 * bf16, W_O [4096][64 * 256] bf16; o [T][64][256] bf16 is a caller buffer
 * (also an output). */
typedef struct kp_mla_absorb_out_args {
    int32_t num_tokens;
    const uint16_t *out;
    const uint16_t *w_uv;
    const uint16_t *w_o;
    uint16_t *o;
    uint16_t *hidden_out;
    int32_t wait_limit_us;
    int32_t *d_status;
} kp_mla_absorb_out_args;

KP_API kp_status kp_gemm_bf16(const kp_gemm_args *args, kp_stream_t stream);
KP_API kp_status kp_indexer_project(const kp_indexer_project_args *args, kp_stream_t stream);
KP_API kp_status kp_mla_absorb_q(const kp_mla_absorb_q_args *args, kp_stream_t stream);
KP_API kp_status kp_mla_absorb_out(const kp_mla_absorb_out_args *args, kp_stream_t stream);

/* ---- scoring without a caller workspace ----
 * The pages describe no such call: it exists for callers that cannot
 * allocate device memory when they score (a host framework whose allocator
 * forbids raw cudaMalloc, a plugin handed only its input and output buffers,
 * a process whose memory budget is fixed before the first step).
 * Same contract and results as kp_indexer_score, except that args->workspace
 * and args->workspace_bytes are ignored: the work plan lives in a device
 * array compiled into the library (about 128 KB, held by every GPU that loads
 * the library until the process exits).  The call allocates nothing.
 *  - num_queries > KP_NOALLOC_MAX_QUERIES returns KP_ERR_UNSUPPORTED and
 *    launches nothing.
 *  - Every call made outside stream capture looks up the array's device
 *    address with the current device (cudaGetSymbolAddress) and caches it
 *    per device; a call made while its stream is being captured uses that
 *    cache, so make one call on the device outside capture first (a capture
 *    before any such call returns KP_ERR_CUDA).  After cudaDeviceReset, make
 *    one call outside capture again before capturing.
 *  - Every call shares the one array: calls whose kernels overlap on the GPU
 *    (different streams, or different host threads, without ordering between
 *    them) race and may produce wrong scores.  Calls in one stream are fine. */
KP_API kp_status kp_indexer_score_noalloc(const kp_score_args *args, kp_stream_t stream);

/* Workspace sizes in bytes (0 never returned; sizes depend only on host fields). */
KP_API size_t kp_score_workspace_size(int32_t num_queries);
KP_API size_t kp_attend_workspace_size(const kp_config *cfg, int32_t num_queries);
KP_API size_t kp_workspace_size(const kp_forward_args *args);

/* Static text for a status code. */
KP_API const char *kp_status_string(kp_status s);
/* Text of the last KP_ERR_CUDA raised on the calling host thread ("" if none). */
KP_API const char *kp_last_error(void);
/* Synchronises `stream`, reads *d_status and returns it as a kp_status
 * (debug / tests only). */
KP_API kp_status kp_read_device_status(const int32_t *d_status, kp_stream_t stream);
/* Library version: major * 10000 + minor * 100 + patch. */
KP_API int kp_version(void);

#ifdef __cplusplus
}
#endif
#endif /* KPOOL_DSA_H */
