/*
 * kpool_oracle.c -- plain, slow, fp64 CPU oracle of the KPool DSA step.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path links, loads or
 * calls this file; only the tests, the smoke check and the bench's CPU
 * baseline leg do.  It shares no source, header, table or helper with the
 * CUDA library.
 *
 * What it follows (pages about GLM-5.3-Flash / "GLM5-Next"):
 *   - MAX API docs, max.pipelines.architectures.glm5_next, Glm5NextConfig:
 *       index_kpool            ("tokens per indexer scoring pool")
 *       index_kpool_compress   (pooled key = learned weighted average of the
 *                               pool's tokens: gate logits plus a learned
 *                               intra-pool position embedding; else a mean)
 *       index_kpool_always_select_tail (the incomplete trailing pool is
 *                               always visible)
 *       mla_use_nope / build_layers (no rotary; the 576-wide latent carries
 *                               64 rotary columns that are all zero)
 *   - llama.cpp PR "add GLM-5.3-Flash (GLM5-Next) support", Overview and the
 *     soft_max bug report: pools of 4 consecutive tokens, the incomplete tail
 *     always kept, per-token key|gate, the pooling softmax over a
 *     [4, 128, n_pool] tensor (softmax over the 4 in-pool positions, one per
 *     dimension and pool).
 *   - llm-atlas GLM-5.3-Flash card, "Raw config fields": index_n_heads 32,
 *     index_head_dim 128, index_kpool 4, index_topk 2048, kv_lora_rank 512,
 *     num_attention_heads 64, qk_head_dim 256.
 *   - The lightning-indexer score  s = sum_h w_h * ReLU(q_h . k_pool)  of the
 *     DeepSeek-V3.2 family that Glm5NextConfig derives from.
 *
 * Precision: every product and sum is in double.  bf16 inputs are widened
 * exactly.  The one rounding the method defines is the storage of pooled
 * keys in the bf16 indexer cache; it is done here round-to-nearest-even
 * straight from the double result.
 *
 * Readings of the pages (where they are silent) used here:
 *   - the gate is per token AND per dimension ([n_tok, 128]); the position
 *     embedding (ape) is [kpool, 128]; the softmax runs over the kpool
 *     positions of a pool, separately for every dimension;
 *   - n_full(t) = floor((t+1)/kpool) complete pools are visible to a query
 *     at position t; its tail is positions kpool*n_full(t) .. t (empty when
 *     (t+1) is a multiple of kpool);
 *   - the tail is added on top of the top-k budget; budget = topk_tokens /
 *     kpool pools; when n_full <= budget every complete pool is selected;
 *   - top-k order: larger score first, ties to the lower pool index, NaN
 *     below -inf; the selected indices are returned in ascending order;
 *   - attention logits use all 576 latent columns, the output only the first
 *     512 (the latent part); lse is the natural-log log-sum-exp of the
 *     scaled logits; an empty token set gives out = 0, lse = -inf.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* ---- bf16 <-> double ------------------------------------------------ */

double oracle_bf16_to_double(uint16_t b) {
    uint32_t u = ((uint32_t)b) << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Round a double to the nearest bf16 (ties to even), directly from the
 * double value (no intermediate float rounding).  bf16 = 1 sign, 8 exponent,
 * 7 stored mantissa bits: a normal value has 8 significant bits. */
uint16_t oracle_double_to_bf16(double x) {
    if (isnan(x)) return 0x7fc0;
    uint16_t sign = signbit(x) ? 0x8000 : 0;
    double a = fabs(x);
    if (isinf(a)) return sign | 0x7f80;
    if (a == 0.0) return sign;
    int e;
    (void)frexp(a, &e);            /* a = m * 2^e, m in [0.5, 1) */
    int q = e - 8;                 /* quantum of an 8-significant-bit value */
    if (q < -133) q = -133;        /* subnormal bf16 quantum is 2^-133 */
    double scaled = ldexp(a, -q);  /* exact: only the exponent changes */
    double r = nearbyint(scaled);  /* default mode: round half to even */
    double y = ldexp(r, q);
    if (y >= ldexp(1.0, 128)) return sign | 0x7f80;
    float f = (float)y;            /* exact: y has <= 8 significant bits */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

/* ---- step 1: pooled-key compression --------------------------------- */

/* Pools every complete run of kpool consecutive tokens of ONE sequence.
 *   keys, gates : [n_tokens][dim] bf16 (raw per-token indexer key and gate)
 *   ape         : [kpool][dim] bf16 (intra-pool position embedding)
 *   mode        : 0 = learned (gate + ape softmax weights), 1 = plain mean
 *   pooled      : [n_tokens / kpool][dim] bf16 out (RNE of the exact value)
 *   pooled_exact: same shape in double before rounding (may be NULL)
 * For pool p and dimension d:
 *   logit_i = gate[kpool*p+i][d] + ape[i][d]            i = 0..kpool-1
 *   alpha_i = exp(logit_i - max_j logit_j) / sum_j exp(logit_j - max)
 *   k_pool[p][d] = sum_i alpha_i * key[kpool*p+i][d]
 * Mean mode: alpha_i = 1/kpool. */
void oracle_kpool_compress(int64_t n_tokens, int kpool, int dim,
                           const uint16_t *keys, const uint16_t *gates,
                           const uint16_t *ape, int mode,
                           uint16_t *pooled, double *pooled_exact) {
    int64_t n_pools = n_tokens / kpool;
    double *logit = (double *)malloc(sizeof(double) * (size_t)kpool);
    for (int64_t p = 0; p < n_pools; ++p) {
        for (int d = 0; d < dim; ++d) {
            double acc = 0.0;
            if (mode == 1) {
                for (int i = 0; i < kpool; ++i)
                    acc += oracle_bf16_to_double(keys[(p * kpool + i) * dim + d]);
                acc /= (double)kpool;
            } else {
                double mx = -INFINITY;
                for (int i = 0; i < kpool; ++i) {
                    logit[i] = oracle_bf16_to_double(gates[(p * kpool + i) * dim + d]) +
                               oracle_bf16_to_double(ape[i * dim + d]);
                    if (logit[i] > mx) mx = logit[i];
                }
                double den = 0.0;
                for (int i = 0; i < kpool; ++i) den += exp(logit[i] - mx);
                for (int i = 0; i < kpool; ++i) {
                    double alpha = exp(logit[i] - mx) / den;
                    acc += alpha * oracle_bf16_to_double(keys[(p * kpool + i) * dim + d]);
                }
            }
            if (pooled_exact) pooled_exact[p * dim + d] = acc;
            pooled[p * dim + d] = oracle_double_to_bf16(acc);
        }
    }
    free(logit);
}

/* ---- step 2: lightning-indexer scores over pooled keys -------------- */

/* One query against the first n_visible pooled keys of its sequence:
 *   s[p] = sum_h w[h] * max(0, sum_d q[h][d] * k_pool[p][d]).
 *   q      : [n_heads][dim] bf16,   w : [n_heads] fp32
 *   pooled : [>= n_visible][dim] bf16
 *   scores : [n_visible] out */
void oracle_indexer_score(int n_heads, int dim, const uint16_t *q, const float *w,
                          const uint16_t *pooled, int64_t n_visible, double *scores) {
    for (int64_t p = 0; p < n_visible; ++p) {
        double s = 0.0;
        for (int h = 0; h < n_heads; ++h) {
            double dot = 0.0;
            for (int d = 0; d < dim; ++d)
                dot += oracle_bf16_to_double(q[h * dim + d]) *
                       oracle_bf16_to_double(pooled[p * dim + d]);
            double relu = dot > 0.0 ? dot : 0.0;
            s += (double)w[h] * relu;
        }
        scores[p] = s;
    }
}

/* ---- step 3: top-k pool selection ------------------------------------ */

typedef struct { double s; int64_t i; } scored_t;

/* Larger score first; NaN ranks below every number (including -inf);
 * equal scores: lower index first. */
static int cmp_scored(const void *a, const void *b) {
    const scored_t *x = (const scored_t *)a, *y = (const scored_t *)b;
    int xn = isnan(x->s), yn = isnan(y->s);
    if (xn != yn) return xn ? 1 : -1;
    if (!xn) {
        if (x->s > y->s) return -1;
        if (x->s < y->s) return 1;
    }
    return (x->i < y->i) ? -1 : (x->i > y->i) ? 1 : 0;
}

static int cmp_i32(const void *a, const void *b) {
    int32_t x = *(const int32_t *)a, y = *(const int32_t *)b;
    return (x > y) - (x < y);
}

/* Selects min(k, n) of the n scores by full sort; writes the selected pool
 * indices in ascending order to idx_out and returns how many. */
int64_t oracle_topk_select(const double *scores, int64_t n, int64_t k, int32_t *idx_out) {
    if (n <= 0 || k <= 0) return 0;
    scored_t *v = (scored_t *)malloc(sizeof(scored_t) * (size_t)n);
    for (int64_t i = 0; i < n; ++i) { v[i].s = scores[i]; v[i].i = i; }
    qsort(v, (size_t)n, sizeof(scored_t), cmp_scored);
    int64_t m = n < k ? n : k;
    for (int64_t j = 0; j < m; ++j) idx_out[j] = (int32_t)v[j].i;
    qsort(idx_out, (size_t)m, sizeof(int32_t), cmp_i32);
    free(v);
    return m;
}

/* ---- the token set a query attends to -------------------------------- */

/* Positions (within the sequence) a query at position t attends to: the
 * kpool rows of every selected pool (in the order given), then the tail
 * kpool*floor((t+1)/kpool) .. t when always_select_tail.  Returns the count;
 * pos_out must hold n_sel*kpool + kpool - 1 entries. */
int64_t oracle_token_set(int64_t t, int kpool, const int32_t *sel, int64_t n_sel,
                         int always_select_tail, int64_t *pos_out) {
    int64_t n = 0;
    for (int64_t j = 0; j < n_sel; ++j)
        for (int i = 0; i < kpool; ++i) pos_out[n++] = (int64_t)sel[j] * kpool + i;
    if (always_select_tail) {
        int64_t n_full = (t + 1) / kpool;
        for (int64_t s = n_full * kpool; s <= t; ++s) pos_out[n++] = s;
    }
    return n;
}

/* ---- step 4: softmax attention over a token set in latent space ------ */

/* For every head h:
 *   z_s   = scale * sum_{d < d_lat} q[h][d] * c[row_s][d]
 *   out_h = sum_s softmax(z)_s * c[row_s][0 .. d_v)
 *   lse_h = log sum_s exp(z_s)
 *   q      : [n_heads][d_lat] bf16
 *   latent : rows of d_lat bf16 (row r at latent + r*d_lat)
 *   rows   : [n_rows] row numbers of the token set
 *   out    : [n_heads][d_v],  lse : [n_heads] */
void oracle_attend(int n_heads, int d_lat, int d_v, const uint16_t *q,
                   const uint16_t *latent, const int64_t *rows, int64_t n_rows,
                   double scale, double *out, double *lse) {
    double *z = (double *)malloc(sizeof(double) * (size_t)(n_rows > 0 ? n_rows : 1));
    for (int h = 0; h < n_heads; ++h) {
        double *o = out + (int64_t)h * d_v;
        for (int d = 0; d < d_v; ++d) o[d] = 0.0;
        if (n_rows == 0) { lse[h] = -INFINITY; continue; }
        double mx = -INFINITY;
        for (int64_t s = 0; s < n_rows; ++s) {
            const uint16_t *c = latent + rows[s] * (int64_t)d_lat;
            double dot = 0.0;
            for (int d = 0; d < d_lat; ++d)
                dot += oracle_bf16_to_double(q[h * d_lat + d]) * oracle_bf16_to_double(c[d]);
            z[s] = scale * dot;
            if (z[s] > mx) mx = z[s];
        }
        double den = 0.0;
        for (int64_t s = 0; s < n_rows; ++s) {
            double e = exp(z[s] - mx);
            den += e;
            const uint16_t *c = latent + rows[s] * (int64_t)d_lat;
            for (int d = 0; d < d_v; ++d) o[d] += e * oracle_bf16_to_double(c[d]);
        }
        for (int d = 0; d < d_v; ++d) o[d] /= den;
        lse[h] = mx + log(den);
    }
    free(z);
}

/* ---- one whole step for a batch of queries --------------------------- */

/* All queries of a batch, steps 2-4, given the pooled caches (from step 1):
 *   q_seq, q_pos      : [nq] sequence and absolute position of each query
 *   pool_row_off      : [B] first pooled-cache row of each sequence
 *   latent_row_off    : [B] first latent-cache row of each sequence
 *   q_idx [nq][ih][idim] bf16, w [nq][ih] fp32, pooled rows [*][idim] bf16
 *   q_lat [nq][mh][d_lat] bf16, latent rows [*][d_lat] bf16
 *   scores_out        : [nq][score_stride] (may be NULL); -inf beyond n_full
 *   sel_out [nq][k_pools] int32 (-1 padded), n_sel_out [nq]
 *   out [nq][mh][d_v], lse [nq][mh]
 * Queries are independent; `threads` > 1 splits them over OpenMP threads. */
void oracle_dsa_queries(int nq, const int32_t *q_seq, const int32_t *q_pos,
                        const int64_t *pool_row_off, const int64_t *latent_row_off,
                        int kpool, int64_t k_pools, int always_select_tail,
                        int ih, int idim, const uint16_t *q_idx, const float *w,
                        const uint16_t *pooled,
                        int mh, int d_lat, int d_v, const uint16_t *q_lat,
                        const uint16_t *latent, double scale,
                        double *scores_out, int64_t score_stride,
                        int32_t *sel_out, int32_t *n_sel_out,
                        double *out, double *lse, int threads) {
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads > 0 ? threads : 1)
#endif
    for (int qi = 0; qi < nq; ++qi) {
        int b = q_seq[qi];
        int64_t t = q_pos[qi];
        int64_t n_full = (t + 1) / kpool;
        double *sc = (double *)malloc(sizeof(double) * (size_t)(n_full > 0 ? n_full : 1));
        oracle_indexer_score(ih, idim, q_idx + (int64_t)qi * ih * idim, w + (int64_t)qi * ih,
                             pooled + pool_row_off[b] * idim, n_full, sc);
        if (scores_out) {
            for (int64_t p = 0; p < score_stride; ++p)
                scores_out[(int64_t)qi * score_stride + p] = p < n_full ? sc[p] : -INFINITY;
        }
        int32_t *sel = sel_out + (int64_t)qi * k_pools;
        int64_t ns = oracle_topk_select(sc, n_full, k_pools, sel);
        for (int64_t j = ns; j < k_pools; ++j) sel[j] = -1;
        n_sel_out[qi] = (int32_t)ns;
        int64_t *pos = (int64_t *)malloc(sizeof(int64_t) * (size_t)(ns * kpool + kpool));
        int64_t n_tok = oracle_token_set(t, kpool, sel, ns, always_select_tail, pos);
        for (int64_t s = 0; s < n_tok; ++s) pos[s] += latent_row_off[b];
        oracle_attend(mh, d_lat, d_v, q_lat + (int64_t)qi * mh * d_lat, latent, pos, n_tok,
                      scale, out + (int64_t)qi * mh * d_v, lse + (int64_t)qi * mh);
        free(pos);
        free(sc);
    }
}

/* ---- the steps either side: dense products ---------------------------
 * out[i][j] = sum_k a[i][k] * b[j][k] in double (bf16 inputs widened
 * exactly), the plain definition of a linear layer y = W x with W stored
 * [out][in].  Used for the indexer projections from the hidden state
 * (q_idx, keys, gates, w), the absorbed query q_lat[h] = W_UK[h]^T q_nope[h]
 * and the output side (W_UV per head, then o_proj).  When abs_out is given,
 * it receives sum_k |a[i][k] * b[j][k]| (for error bounds of the GPU's fp32
 * accumulation). */
void oracle_linear(int64_t m, int64_t n, int64_t k, const uint16_t *a, int64_t lda, const uint16_t *b,
                   int64_t ldb, double *out, int64_t ldo, double *abs_out, int threads) {
#ifdef _OPENMP
#pragma omp parallel for schedule(dynamic, 1) num_threads(threads > 0 ? threads : 1)
#endif
    for (int64_t i = 0; i < m; ++i) {
        double *arow = (double *)malloc(sizeof(double) * (size_t)k);
        for (int64_t kk = 0; kk < k; ++kk) arow[kk] = oracle_bf16_to_double(a[i * lda + kk]);
        for (int64_t j = 0; j < n; ++j) {
            double acc = 0.0, aacc = 0.0;
            const uint16_t *brow = b + j * ldb;
            for (int64_t kk = 0; kk < k; ++kk) {
                const double pr = arow[kk] * oracle_bf16_to_double(brow[kk]);
                acc += pr;
                aacc += fabs(pr);
            }
            out[i * ldo + j] = acc;
            if (abs_out) abs_out[i * ldo + j] = aacc;
        }
        free(arow);
    }
    (void)threads;
}

/* Reports whether the library was built with OpenMP (threads it can use). */
int oracle_has_openmp(void) {
#ifdef _OPENMP
    return 1;
#else
    return 0;
#endif
}
