// score_select.cu -- the lightning-indexer scores fused with the top-k pool
// selection: the scores of a query never leave the chip.
//
// Method: s[q,p] = sum_h w[q,h] * ReLU(q_idx[q,h,:] . k_pool[p,:]) over the
// n_full(t) complete pools a query sees (the DeepSeek-V3.2 lightning indexer
// that MAX docs' Glm5NextConfig derives from; 32 heads x 128 dims, llm-atlas
// GLM-5.3-Flash card), then the index_topk / kpool best pools, ties to the
// lower index, in ascending order.  The llama.cpp PR "add GLM-5.3-Flash
// (GLM5-Next) support" names re-materialising pooled intermediates every
// graph as what slows decode; here the fp32 score matrix is never written.
//
// B300 design.  A group of up to 4 adjacent queries of one sequence belongs to
// a thread-block cluster of C CTAs; CTA r scores the pools r * chunk ..
// (r + 1) * chunk - 1 of all the group's queries with the same tcgen05
// pipeline as the scorer (TMA-fed 128-pool tiles, queries x heads as N, two
// TMEM accumulators, eight epilogue warps) and keeps the results as
// order-preserving keys in shared memory.  Then CTA r % C gathers query row r
// (rows r >= C in later rounds) from every CTA's slice over distributed shared
// memory into its own shared memory, runs the exact radix select of the top-k
// kernel on the whole row and writes the selection.  The clusters are
// persistent over the groups.
//
// Warp roles (512 threads, one CTA per SM):
//   warp 0      TMA producer (the whole warp walks the tiles; lane 0 waits)
//   warp 1      TMEM allocation, MMA issue (one lane)
//   warps 2-9   epilogue: TMEM -> registers -> keys in shared memory
//   all         the row exchange and the selection
#include <cuda.h>

#include <algorithm>

#include "kp_common.cuh"
#include "kp_internal.h"
#include "score_plan.cuh"
#include "topk_select.cuh"

namespace kp {

namespace {

constexpr int kSsQ = 4;                                    // queries per group
constexpr int kSsN = kSsQ * kIndexHeads;                   // 128: MMA N max
constexpr int kSsChunk = 2048;                             // pools per CTA and group (multiple of 128)
constexpr int kSsMaxCluster = 8;                           // rows up to 16,384 pools
constexpr int kSsStages = 4;
constexpr int kSsABlock = kScM * 128;                      // 16 KB: 128 pools x 64 dims
constexpr int kSsAStage = 2 * kSsABlock;                   // 32 KB
constexpr int kSsBBlock = kSsN * 128;                      // 16 KB: 128 (query, head) rows x 64 dims
constexpr int kSsBBytes = 2 * kSsBBlock;
constexpr int kSsQBox = kIndexHeads * 128;                 // one query, one K block: 4 KB
constexpr int kSsKeysBytes = kSsQ * kSsChunk * 4;          // 32 KB
constexpr int kSsThreads = 512;
constexpr int kSsEpiThreads = 256;
constexpr int kSsNumBars = 2 * kSsStages + 4 + 2 + 2;      // full, empty, acc x 4, B x 2, drain, never
constexpr int kSsPlanWords = 2048;                         // the plan in shared memory (local plans)
constexpr int kSsLocalMaxQ = (kSsPlanWords - 5) / 4;
constexpr int kSsOffB = kSsStages * kSsAStage;
constexpr int kSsOffKeys = kSsOffB + kSsBBytes;
constexpr int kSsOffBars = kSsOffKeys + kSsKeysBytes;
constexpr int kSsOffPlan = kSsOffBars + kSsNumBars * 8;
constexpr int kSsSmemBytes = kSsOffPlan + kSsPlanWords * 4 + 1024;
static_assert(kSsMaxCluster * kSsChunk * 4 + 16 <= kSsStages * kSsAStage, "a whole row fits the tile stages");
static_assert(kSsEpiThreads == 256, "named barrier 1 spans the eight epilogue warps");
static_assert(kSsMaxCluster * kSsChunk == KP_FUSED_MAX_POOLS, "the header's bound is the kernel's capacity");

struct SsParams {
    const int32_t *plan;       // the plan in global memory (when not built here)
    int nq;
    bool local_plan;
    int num_seqs;
    int max_tiles;
    const int32_t *q_seq;
    const int32_t *prev_len;   // tokens of each sequence before this step (nullptr: no early loads)
    const int32_t *q_pos;
    const int32_t *share;      // [nq] shared selection (nullptr: none): shared rows are skipped
    const int32_t *seq_len;
    int kshift;
    const float *w;
    CacheMap cmap;
    int seg;                   // pooled rows per TMA box
    int chunk;                 // pools per CTA and group (multiple of 128)
    int K;
    int32_t *pool_idx;
    int32_t *n_sel;
    int32_t *status;
    unsigned long long wait_ns;
    int stall;
};

__device__ __forceinline__ bool ss_epi_bar_all(bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, 1, 256, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v))
        : "memory");
    return r != 0;
}
// Block-wide AND of a flag (all 512 threads).
__device__ __forceinline__ bool block_all(bool v) { return __syncthreads_and(v ? 1 : 0) != 0; }

// Bytes of CTA c's slice of a row of n keys, rounded up to whole 16-byte
// units (the copy reads a few stale keys past n, which the select ignores).
__device__ __forceinline__ uint32_t slice_bytes(int n, int c, int chunk) {
    const int m = min(chunk, n - c * chunk);
    return m > 0 ? static_cast<uint32_t>((m + 3) & ~3) * 4u : 0u;
}

__global__ void __launch_bounds__(kSsThreads, 1)
    score_select_kernel(const __grid_constant__ CUtensorMap tm_pool, const __grid_constant__ CUtensorMap tm_q,
                        SsParams P) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;
    __shared__ __align__(16) float w_s[kSsQ * kIndexHeads];
    __shared__ __align__(16) TopkShared sh;

    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t sA = smem_u32(smem);
    const uint32_t sB = sA + kSsOffB;
    uint32_t *keys_s = reinterpret_cast<uint32_t *>(smem + kSsOffKeys);
    uint32_t *row_s = reinterpret_cast<uint32_t *>(smem);   // the tile stages, between groups
    const uint32_t bar0 = sA + kSsOffBars;
    int32_t *plan_s = reinterpret_cast<int32_t *>(smem + kSsOffPlan);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kSsStages + s); };
    auto accf_bar = [&](int a) { return bar0 + 8u * (2 * kSsStages + a); };
    auto acce_bar = [&](int a) { return bar0 + 8u * (2 * kSsStages + 2 + a); };
    const uint32_t bfull_bar = bar0 + 8u * (2 * kSsStages + 4);
    const uint32_t bempty_bar = bar0 + 8u * (2 * kSsStages + 5);
    const uint32_t drain_bar = bar0 + 8u * (2 * kSsStages + 6);
    const uint32_t never_bar = bar0 + 8u * (2 * kSsStages + 7);

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int rank = static_cast<int>(cluster_ctarank());
    const int C = static_cast<int>(cluster_size());
    const int cluster_id = blockIdx.x / C, n_clusters = gridDim.x / C;
    volatile int *abort_flag = &abort_s;

    if (tid == 0) {
        for (int s = 0; s < kSsStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(accf_bar(a), 1);
            mbar_init(acce_bar(a), kSsEpiThreads);
        }
        mbar_init(bfull_bar, 1);
        mbar_init(bempty_bar, 1);
        mbar_init(drain_bar, 1);
        mbar_init(never_bar, 1);
        fence_mbar_init();
        abort_s = 0;
        tma_prefetch_desc(&tm_pool);
        tma_prefetch_desc(&tm_q);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&tmem_base_s), 256);
        tmem_relinquish();
    }
    // The plan: built here from the query positions (inputs) when it fits,
    // else built by the previous kernel (read after the grid dependency).
    __shared__ int plan_scratch[33];
    bool dep_done = false;
    const int32_t *plan_base;
    if (P.local_plan) {
        build_score_plan(P.nq, P.num_seqs, P.q_seq, P.q_pos, P.seq_len, P.kshift, P.max_tiles, plan_s, P.status,
                         plan_scratch, kSsQ);
        plan_base = plan_s;
    } else {
        pdl_wait_then_release();
        dep_done = true;
        plan_base = P.plan;
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    const PlanView plan(const_cast<int32_t *>(plan_base), P.nq);
    const int ng = plan.hdr[0];

    // state carried across groups
    int stage = 0, acc = 0, b_loads = 0;
    uint32_t phase = 0, acc_phase = 0;
    bool first_mma = true;

    for (int g = cluster_id; g < ng; g += n_clusters) {  // the same groups for every CTA of the cluster
        const int q0 = plan.q0[g], nqg = plan.nq[g], bseq = plan.seq[g];
        // A group the plan gave no tiles although its queries see pools has a bad
        // sequence or position (the plan has reported it): nothing of it is read.
        const bool size_ok = nqg >= 1 && nqg <= kSsQ;
        if (!size_ok && tid == 0) set_status(P.status, KP_ERR_DEVICE_BOUNDS);
        const bool gvalid = size_ok && plan.unit0[g + 1] > plan.unit0[g];
        const int cap = C * P.chunk;   // pools a row may have here
        const int nf_mine = (gvalid && lane < nqg) ? (P.q_pos[q0 + lane] + 1) >> P.kshift : 0;
        int n_max = __reduce_max_sync(0xffffffffu, nf_mine);  // pools the group's queries see
        if (n_max > cap) {                                     // max_pools was not an upper bound
            if (tid == 0) set_status(P.status, KP_ERR_DEVICE_BOUNDS);
            n_max = cap;
        }
        const int p_begin = rank * P.chunk;
        const int p_end = min(n_max, p_begin + P.chunk);
        const int tiles = p_end > p_begin ? (p_end - p_begin + kScM - 1) / kScM : 0;
        // Every thread takes the same view of the abort flag (the roles below
        // meet at named and block barriers, which all of them must reach).
        const bool live = block_all(*abort_flag == 0);

        if (live && warp == 0) {
            // ---- producer
            const unsigned full = 0xffffffffu;
            const bool paged = P.cmap.paged();
            const int nseg = kScM / P.seg;
            const int old_pools = (P.prev_len && tiles > 0) ? P.prev_len[bseq] >> P.kshift : 0;
            int a_phase[kSsStages];
#pragma unroll
            for (int i = 0; i < kSsStages; ++i) a_phase[i] = -1;
            bool ok = true;
            if (tiles > 0) {
                bool w_ok = true;
                if (lane == 0 && b_loads > 0)
                    w_ok = mbar_wait(bempty_bar, (b_loads - 1) & 1, abort_flag, P.status, P.wait_ns);
                ok = __shfl_sync(full, w_ok, 0);
                if (ok && lane == 0) {
                    mbar_expect_tx(bfull_bar, nqg * 2 * kSsQBox);
                    for (int qi = 0; qi < nqg; ++qi)
                        for (int kb = 0; kb < 2; ++kb)
                            tma_load_2d(sB + kb * kSsBBlock + qi * kSsQBox, &tm_q, bfull_bar, kb * 64,
                                        (q0 + qi) * kIndexHeads);
                }
                if (ok) ++b_loads;
            }
            for (int t = 0; ok && t < tiles; ++t) {
                bool w_ok = true;
                if (lane == 0) w_ok = mbar_wait(empty_bar(stage), phase ^ 1, abort_flag, P.status, P.wait_ns);
                if (!__shfl_sync(full, w_ok, 0)) {
                    ok = false;
                    break;
                }
                const int p0 = p_begin + t * kScM;
                if (!dep_done && p0 + kScM > old_pools) {  // may hold pools written this step
                    pdl_wait_then_release();
                    dep_done = true;
                }
                const uint32_t dst = sA + stage * kSsAStage;
                if (lane == 0) mbar_expect_tx(full_bar(stage), kSsAStage);
                if (!paged) {
                    if (lane == 0) {
                        const int row = static_cast<int>(P.cmap.pool_row_off[bseq] + p0);
                        tma_load_2d(dst, &tm_pool, full_bar(stage), 0, row);
                        tma_load_2d(dst + kSsABlock, &tm_pool, full_bar(stage), 64, row);
                    }
                } else if (lane < nseg) {
                    const int p = p0 + lane * P.seg;
                    int y = -P.seg;
                    if (p < n_max) {
                        const int64_t r = P.cmap.pool_row(bseq, p);
                        if (r >= 0) y = static_cast<int>(r);
                        else set_status(P.status, KP_ERR_DEVICE_BOUNDS);
                    }
                    const uint32_t off = static_cast<uint32_t>(lane * P.seg * 128);
                    tma_load_2d(dst + off, &tm_pool, full_bar(stage), 0, y);
                    tma_load_2d(dst + kSsABlock + off, &tm_pool, full_bar(stage), 64, y);
                }
                a_phase[stage] = static_cast<int>(phase);
                if (++stage == kSsStages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
            if (!ok && lane == 0) {  // gave up: every load issued lands before the stages are reused
                if (b_loads > 0) mbar_wait(bfull_bar, (b_loads - 1) & 1, nullptr, P.status);
#pragma unroll
                for (int i = 0; i < kSsStages; ++i)
                    if (a_phase[i] >= 0) mbar_wait(full_bar(i), static_cast<uint32_t>(a_phase[i]), nullptr, P.status);
            }
        } else if (live && warp == 1) {
            // ---- MMA issuer
            if (lane == 0 && tiles > 0) {
                bool ok = true;
                if (first_mma && P.stall) ok = mbar_wait(never_bar, 0, abort_flag, P.status, P.wait_ns);
                ok = ok && mbar_wait(bfull_bar, (b_loads) & 1, abort_flag, P.status, P.wait_ns);
                const uint32_t idesc = idesc_bf16_f32(kScM, kIndexHeads * nqg);
                for (int t = 0; ok && t < tiles; ++t) {
                    if (!(ok = mbar_wait(acce_bar(acc), acc_phase ^ 1, abort_flag, P.status, P.wait_ns))) break;
                    if (!(ok = mbar_wait(full_bar(stage), phase, abort_flag, P.status, P.wait_ns))) break;
                    tc_fence_after();
                    const uint32_t a_base = sA + stage * kSsAStage;
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const uint32_t koff = (kk & 3) * 32;
                        const uint64_t ad = desc_kmajor_sw128(a_base + (kk >> 2) * kSsABlock + koff);
                        const uint64_t bd = desc_kmajor_sw128(sB + (kk >> 2) * kSsBBlock + koff);
                        tc_mma_bf16(tmem + acc * kSsN, ad, bd, idesc, kk > 0 ? 1u : 0u);
                    }
                    tc_commit(empty_bar(stage));
                    tc_commit(accf_bar(acc));
                    if (++stage == kSsStages) {
                        stage = 0;
                        phase ^= 1;
                    }
                    if (++acc == 2) {
                        acc = 0;
                        acc_phase ^= 1;
                    }
                }
                if (ok) {
                    tc_commit(bempty_bar);
                } else {  // gave up: every MMA issued completes before the TMEM is reused or freed
                    tc_commit(drain_bar);
                    mbar_wait(drain_bar, 0, nullptr, P.status);
                }
            }
            first_mma = false;
            if (tiles > 0) ++b_loads;
        } else if (live && warp >= 2 && warp < 10) {
            // ---- epilogue: warp w reads TMEM lanes 32*(w%4) .. +31; the two warps
            // of a lane quadrant take the even / odd queries of the group.
            const int quad = warp & 3, et = tid - 64, half = et >> 7;
            if (tiles > 0) {
                for (int k = et; k < nqg * kIndexHeads; k += kSsEpiThreads)
                    w_s[k] = P.w[static_cast<int64_t>(q0) * kIndexHeads + k];
                ss_epi_bar_all(true);
            }
            auto reduce = [&](const uint32_t (&r)[32], int qi) -> float {
                const uint64_t *wq = reinterpret_cast<const uint64_t *>(w_s + qi * kIndexHeads);
                uint64_t a[4] = {0ull, 0ull, 0ull, 0ull};
#pragma unroll
                for (int h2 = 0; h2 < kIndexHeads / 2; ++h2)
                    a[h2 & 3] = fma_f32x2(wq[h2], pack_f32x2(fmaxf(__uint_as_float(r[2 * h2]), 0.f),
                                                               fmaxf(__uint_as_float(r[2 * h2 + 1]), 0.f)),
                                          a[h2 & 3]);
                const float2 s0 = unpack_f32x2(a[0]), s1 = unpack_f32x2(a[1]), s2 = unpack_f32x2(a[2]),
                             s3 = unpack_f32x2(a[3]);
                return ((s0.x + s0.y) + (s1.x + s1.y)) + ((s2.x + s2.y) + (s3.x + s3.y));
            };
            for (int t = 0; t < tiles; ++t) {
                if (!ss_epi_bar_all(mbar_wait(accf_bar(acc), acc_phase, abort_flag, P.status, P.wait_ns))) break;
                tc_fence_after();
                const int pl = t * kScM + quad * 32 + lane;   // pool index inside this CTA's slice
                const uint32_t tbase = tmem + acc * kSsN + (static_cast<uint32_t>(quad * 32) << 16);
                if (half < nqg && t * kScM + quad * 32 < kSsChunk) {   // warp-uniform
                    const int qi = half, qj = half + 2;
                    uint32_t r0[32], r1[32];
                    tmem_ld_32x32b_x32(tbase + qi * kIndexHeads, r0);
                    if (qj < nqg) tmem_ld_32x32b_x32(tbase + qj * kIndexHeads, r1);
                    tmem_ld_wait();
                    keys_s[qi * kSsChunk + pl] = score_key(reduce(r0, qi));
                    if (qj < nqg) keys_s[qj * kSsChunk + pl] = score_key(reduce(r1, qj));
                }
                tc_fence_before();
                mbar_arrive(acce_bar(acc));
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1;
                }
            }
        }

        // ---- the row exchange, in rounds: in round j, CTA r of the cluster owns
        // row j * C + r of the group (rows past the group's queries: nobody)
        // and pulls every CTA's slice of it into its tile stages (16-byte
        // loads from distributed shared memory; its own slice locally), then
        // selects.  A cluster barrier before (every CTA's keys are complete) and
        // after (every owner has read them) each round.
        const int rounds = (nqg + C - 1) / C;
        for (int j = 0; j < rounds; ++j) {
            const int rr = j * C + rank;
            const int row_q = q0 + rr;
            const int row_n = (gvalid && rr < nqg) ? min(cap, (P.q_pos[row_q] + 1) >> P.kshift) : 0;
            __syncthreads();
            if (C > 1) cluster_barrier();
            // read after the barrier: nothing sets the flag during the rounds; a
            // shared query's row is left as it was
            const bool own = rr < nqg && *abort_flag == 0 && !(P.share && P.share[row_q] >= 0);
            if (own) {
                int32_t *out = P.pool_idx + static_cast<int64_t>(row_q) * P.K;
                if (row_n > P.K) {
                    // the row's keys and their range, in one pass
                    uint32_t kmin = 0xffffffffu, kmax = 0u;
                    auto take = [&](const uint4 &v, int j) {  // j: row position of v.x
                        const uint32_t k[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
                        for (int u = 0; u < 4; ++u)
                            if (j + u < row_n) {
                                kmin = min(kmin, k[u]);
                                kmax = max(kmax, k[u]);
                            }
                    };
                    // 16-byte pieces of CTA c's slice (the bounds are checked, not assumed)
                    auto pieces = [&](int c) {
                        const int m4 = static_cast<int>(slice_bytes(row_n, c, P.chunk) / 16);
                        if (c * P.chunk + 4 * m4 > kSsMaxCluster * kSsChunk || 4 * m4 > kSsChunk) {
                            set_status(P.status, KP_ERR_DEVICE_BOUNDS);
                            return 0;
                        }
                        return m4;
                    };
                    const uint32_t src_off = smem_u32(keys_s + rr * kSsChunk);
                    const uint4 *own_src = reinterpret_cast<const uint4 *>(keys_s + rr * kSsChunk);
                    for (int c0 = 0; c0 < C; c0 += 4) {      // four slices' loads in flight per thread
                        int m4[4];
#pragma unroll
                        for (int u = 0; u < 4; ++u) m4[u] = c0 + u < C ? pieces(c0 + u) : 0;
                        for (int i = tid; i < kSsChunk / 4; i += kSsThreads) {
                            uint4 v[4];
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const int c = c0 + u;
                                if (i < m4[u])
                                    v[u] = c == rank ? own_src[i]
                                                     : ld_cluster_u32x4(dsmem_addr(src_off, static_cast<uint32_t>(c)) + 16u * i);
                            }
#pragma unroll
                            for (int u = 0; u < 4; ++u) {
                                const int c = c0 + u;
                                if (i < m4[u]) {
                                    reinterpret_cast<uint4 *>(row_s + c * P.chunk)[i] = v[u];
                                    take(v[u], c * P.chunk + 4 * i);
                                }
                            }
                        }
                    }
                    if (tid == 0) {
                        sh.kmin = 0xffffffffu;
                        sh.kmax = 0u;
                    }
                    for (int i = tid; i < kTkBins; i += kSsThreads) sh.hist[0][i] = 0u;
                    __syncthreads();
                    radix_select_slice<kSsThreads, true>(row_s, row_n, 0, 1u, 0u, P.K, out, kmin, kmax, sh, P.status);
                    if (tid == 0) P.n_sel[row_q] = P.K;
                } else {
                    for (int i = tid; i < P.K; i += kSsThreads) out[i] = i < row_n ? i : -1;
                    if (tid == 0) P.n_sel[row_q] = row_n;
                }
            }
            __syncthreads();
            if (C > 1) cluster_barrier();  // every owner has read the round's keys
        }
    }

    // This grid completes only after the previous one: kernels that wait on it
    // may rely on everything before it.
    if (!dep_done) pdl_wait_then_release();
    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, 256);
    }
}

}  // namespace

bool score_select_fits(const kp_config &cfg, const kp_queries &q) {
    (void)cfg;
    return q.num_queries > 0 && q.max_pools <= kSsMaxCluster * kSsChunk;
}

bool score_select_plan_is_local(int32_t num_queries) { return num_queries <= kSsLocalMaxQ; }

ScorePlanArgs score_select_plan_args(const kp_score_args &a) {
    ScorePlanArgs p = score_plan_args(a);
    p.max_q = kSsQ;
    return p;
}

kp_status launch_score_select(const kp_score_args &sc, const kp_topk_args &tk, cudaStream_t s, bool plan_ready,
                              const int32_t *prev_len) {
    const int nq = sc.q.num_queries;
    if (nq == 0) return KP_OK;
    const int sms = device_sm_count();
    if (sms <= 0) return KP_ERR_CUDA;
    const int maxp = sc.q.max_pools > 0 ? sc.q.max_pools : 1;
    int C = 1;
    while (C < kSsMaxCluster && static_cast<int64_t>(C) * kSsChunk < maxp) C *= 2;
    const int chunk = ((maxp + C - 1) / C + kScM - 1) / kScM * kScM;
    const bool local_plan = score_select_plan_is_local(nq);
    int32_t *plan = static_cast<int32_t *>(sc.workspace);
    if (!plan_ready && !local_plan) {
        const kp_status st = launch_score_plan(score_select_plan_args(sc), s);
        if (st != KP_OK) return st;
    }
    const int pool_page = sc.seqs.block_table ? sc.seqs.page_tokens / sc.cfg.kpool : kScM;
    const int seg = pool_page < kScM ? pool_page : kScM;
    CUtensorMap tm_pool, tm_q;
    if (!make_tmap_bf16_sw128(&tm_pool, sc.pooled, kIndexDim, static_cast<uint64_t>(sc.seqs.pool_rows),
                              kIndexDim * 2, 64, static_cast<uint32_t>(seg)) ||
        !make_tmap_bf16_sw128(&tm_q, sc.q_idx, kIndexDim, static_cast<uint64_t>(nq) * kIndexHeads, kIndexDim * 2,
                              64, kIndexHeads))
        return KP_ERR_CUDA;
    cudaError_t e = cudaFuncSetAttribute(score_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kSsSmemBytes);
    if (e != cudaSuccess) {
        record_cuda_error("cudaFuncSetAttribute(score_select_kernel)", e);
        return KP_ERR_CUDA;
    }
    // clusters: one per group at most (groups <= queries), as many as fit at once
    int n_clusters = std::min(nq, sms / C);
    if (C > 1) {
        cudaLaunchConfig_t cfg = {};
        cfg.gridDim = dim3(C * n_clusters);
        cfg.blockDim = dim3(kSsThreads);
        cfg.dynamicSmemBytes = kSsSmemBytes;
        cudaLaunchAttribute attr[1];
        attr[0].id = cudaLaunchAttributeClusterDimension;
        attr[0].val.clusterDim.x = C;
        attr[0].val.clusterDim.y = 1;
        attr[0].val.clusterDim.z = 1;
        cfg.attrs = attr;
        cfg.numAttrs = 1;
        int fit = 0;
        if (cudaOccupancyMaxActiveClusters(&fit, score_select_kernel, &cfg) == cudaSuccess && fit > 0)
            n_clusters = std::min(n_clusters, fit);
        else
            cudaGetLastError();
    }
    if (n_clusters < 1) n_clusters = 1;
    SsParams P;
    P.plan = plan;
    P.nq = nq;
    P.local_plan = local_plan;
    P.num_seqs = sc.seqs.num_seqs;
    P.max_tiles = (sc.q.max_pools + kScM - 1) / kScM;
    P.q_seq = sc.q.q_seq;
    P.prev_len = local_plan ? prev_len : nullptr;
    P.q_pos = sc.q.q_pos;
    P.share = tk.q.share_src;
    P.seq_len = sc.seqs.seq_len;
    P.kshift = kpool_shift(sc.cfg.kpool);
    P.w = sc.w;
    P.cmap = cache_map(sc.seqs, sc.cfg.kpool);
    P.seg = seg;
    P.chunk = chunk;
    P.K = tk.cfg.topk_tokens / tk.cfg.kpool;
    P.pool_idx = tk.pool_idx;
    P.n_sel = tk.n_sel;
    P.status = sc.d_status;
    P.wait_ns = wait_limit_ns(sc.cfg.wait_limit_us);
    P.stall = (sc.cfg.debug_flags & KP_DEBUG_STALL_FIRST_WAIT) ? 1 : 0;
    return launch_kernel("score_select_kernel", score_select_kernel,
                         LaunchCfg(dim3(static_cast<unsigned>(C * n_clusters)), dim3(kSsThreads), kSsSmemBytes, s, C),
                         tm_pool, tm_q, P);
}

}  // namespace kp
