// score.cu -- lightning-indexer scores over pooled keys on tcgen05 tensor cores.
//
// Method: s[q,p] = sum_h w[q,h] * ReLU(q_idx[q,h,:] . k_pool[p,:]) with 32
// heads x 128 dims (llm-atlas GLM-5.3-Flash card, raw config index_n_heads /
// index_head_dim; the DeepSeek-V3.2 lightning indexer that Glm5NextConfig
// derives from, MAX docs glm5_next), over the n_full(t) = floor((t+1)/4)
// complete pools a query at position t can see.
//
// B300 design.  The contraction is [pools x 128] . [128 x (queries*32 heads)]:
//   A = 128 pooled keys of one sequence (TMA, 128-byte swizzle, 32 KB / tile)
//   B = up to 8 queries x 32 heads of the same sequence (TMA, resident while
//       the CTA works on that query group)
//   D = 128 x (32 * nq) fp32 in TMEM (two 256-column accumulators, so the
//       epilogue of one tile overlaps the MMAs of the next).
// Pools are the MMA's M dimension, so after tcgen05.ld each epilogue thread
// owns one pool row and reduces ReLU(.) * w over its 32 head columns in
// registers -- no cross-thread reduction.  Decode (1-4 queries per sequence)
// and chunked prefill (8 queries per group) run the same kernel: decode is
// bound by streaming pooled keys from HBM, prefill by the tensor pipe.
//
// Warp roles (192 threads, one CTA per SM, persistent):
//   warp 0     TMA producer (one elected lane)
//   warp 1     TMEM allocator + MMA issuer (one elected lane)
//   warps 2-5  epilogue: TMEM -> registers -> masked scores -> global
// Work units are (query group, 128-pool tile) pairs laid out by a tiny plan
// kernel; each CTA takes a contiguous range of units.
#include <cuda.h>

#include "kp_common.cuh"
#include "kp_internal.h"

namespace kp {

namespace {

constexpr int kScM = 128;                                 // pools per tile (MMA M)
constexpr int kScMaxQ = 8;                                // queries per group
constexpr int kScMaxN = kScMaxQ * kIndexHeads;            // 256 (MMA N max)
constexpr int kScStages = 4;
constexpr int kScABlockBytes = kScM * 128;                // [128 rows][64 bf16] = 16 KB
constexpr int kScAStageBytes = 2 * kScABlockBytes;        // K = 128 -> two swizzle blocks
constexpr int kScBBlockBytes = kScMaxN * 128;             // [256 rows][64 bf16] = 32 KB
constexpr int kScBBytes = 2 * kScBBlockBytes;
constexpr int kScQBoxBytes = kIndexHeads * 128;           // one query, one K block: 4 KB
constexpr int kScThreads = 192;
constexpr int kScTmemCols = 512;
constexpr int kScAccCols = 256;
constexpr int kScNumBars = 2 * kScStages + 4 + 2;
constexpr int kScSmemBytes = kScStages * kScAStageBytes + kScBBytes + kScNumBars * 8 + 1024;

// Plan layout (int32 words) inside the score workspace.
struct PlanView {
    int32_t *hdr;      // [0] groups, [1] units
    int32_t *q0;       // [NQ] first query of each group
    int32_t *nq;       // [NQ] queries in each group
    int32_t *seq;      // [NQ] sequence of each group
    int32_t *unit0;    // [NQ + 1] first unit of each group (exclusive scan of tiles)
    __host__ __device__ PlanView(int32_t *base, int n)
        : hdr(base), q0(base + 4), nq(base + 4 + n), seq(base + 4 + 2 * n), unit0(base + 4 + 3 * n) {}
};

// Groups runs of up to 8 adjacent queries of the same sequence and counts the
// 128-pool tiles each group needs (the largest n_full among its queries).
__global__ void __launch_bounds__(1024) score_plan_kernel(int nq, int num_seqs,
                                                          const int32_t *__restrict__ q_seq,
                                                          const int32_t *__restrict__ q_pos,
                                                          int max_tiles, int32_t *plan_base,
                                                          int32_t *status) {
    __shared__ int scratch[33];
    PlanView plan(plan_base, nq);
    int carry_run = -1, carry_groups = 0;
    for (int base = 0; base < nq; base += blockDim.x) {
        const int i = base + threadIdx.x;
        const bool in = i < nq;
        const int sq = in ? q_seq[i] : 0;
        const bool run_start = in && (i == 0 || q_seq[i - 1] != sq);
        int tot;
        int rs = block_inclusive_scan<1>(run_start ? i : -1, scratch, &tot);
        rs = max(rs, carry_run);
        carry_run = max(carry_run, tot);
        const bool gs = in && ((i - rs) % kScMaxQ == 0);
        const int incl = block_inclusive_scan<0>(gs ? 1 : 0, scratch, &tot);
        if (gs) {
            const int gid = carry_groups + incl - 1;
            plan.q0[gid] = i;
            plan.seq[gid] = sq;
        }
        carry_groups += tot;
    }
    __syncthreads();
    const int ng = carry_groups;
    for (int g = threadIdx.x; g < ng; g += blockDim.x) {
        const int q0 = plan.q0[g];
        const int q1 = (g + 1 < ng) ? plan.q0[g + 1] : nq;
        int mx = 0;
        for (int q = q0; q < q1; ++q) mx = max(mx, (q_pos[q] + 1) / kKpool);
        int tiles = (mx + kScM - 1) / kScM;
        const int sq = plan.seq[g];
        if (sq < 0 || sq >= num_seqs) {
            set_status(status, KP_ERR_DEVICE_BOUNDS);
            tiles = 0;
        }
        if (tiles > max_tiles) {
            set_status(status, KP_ERR_DEVICE_BOUNDS);
            tiles = max_tiles;
        }
        plan.nq[g] = q1 - q0;
        plan.unit0[g] = tiles;
    }
    __syncthreads();
    int carry_units = 0;
    for (int base = 0; base < ng; base += blockDim.x) {
        const int g = base + threadIdx.x;
        const int v = g < ng ? plan.unit0[g] : 0;
        int tot;
        const int incl = block_inclusive_scan<0>(v, scratch, &tot);
        if (g < ng) plan.unit0[g] = carry_units + incl - v;
        carry_units += tot;
    }
    if (threadIdx.x == 0) {
        plan.unit0[ng] = carry_units;
        plan.hdr[0] = ng;
        plan.hdr[1] = carry_units;
    }
}

struct ScoreParams {
    const int32_t *plan;
    int nq;
    const int32_t *q_pos;
    const float *w;
    const int64_t *pool_row_off;
    float *scores;
    int64_t stride;
    int32_t *status;
};

// Largest group whose first unit is <= u (skips empty groups correctly).
__device__ __forceinline__ int find_group(const int32_t *unit0, int ng, int u) {
    int lo = 0, hi = ng - 1;
    while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (unit0[mid] <= u) lo = mid;
        else hi = mid - 1;
    }
    return lo;
}

__global__ void __launch_bounds__(kScThreads, 1)
    indexer_score_kernel(const __grid_constant__ CUtensorMap tm_pool,
                         const __grid_constant__ CUtensorMap tm_q, ScoreParams P) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;

    PlanView plan(const_cast<int32_t *>(P.plan), P.nq);
    const int ng = plan.hdr[0];
    const long long n_units = plan.hdr[1];
    const int u_begin = static_cast<int>(n_units * blockIdx.x / gridDim.x);
    const int u_end = static_cast<int>(n_units * (blockIdx.x + 1) / gridDim.x);
    if (u_begin >= u_end) return;

    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t sA = smem_u32(smem);
    const uint32_t sB = sA + kScStages * kScAStageBytes;
    const uint32_t bar0 = sB + kScBBytes;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kScStages + s); };
    auto accf_bar = [&](int a) { return bar0 + 8u * (2 * kScStages + a); };
    auto acce_bar = [&](int a) { return bar0 + 8u * (2 * kScStages + 2 + a); };
    const uint32_t bfull_bar = bar0 + 8u * (2 * kScStages + 4);
    const uint32_t bempty_bar = bar0 + 8u * (2 * kScStages + 5);

    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kScStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(accf_bar(a), 1);
            mbar_init(acce_bar(a), 128);
        }
        mbar_init(bfull_bar, 1);
        mbar_init(bempty_bar, 1);
        fence_mbar_init();
        abort_s = 0;
        tma_prefetch_desc(&tm_pool);
        tma_prefetch_desc(&tm_q);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&tmem_base_s), kScTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = tmem_base_s;
    volatile int *abort_flag = &abort_s;

    if (warp == 0) {
        if (lane == 0) {
            int g = find_group(plan.unit0, ng, u_begin), cur_g = -1, b_loads = 0, stage = 0;
            uint32_t phase = 0;
            for (int u = u_begin; u < u_end; ++u) {
                while (plan.unit0[g + 1] <= u) ++g;
                if (g != cur_g) {
                    if (b_loads > 0 &&
                        !mbar_wait(bempty_bar, (b_loads - 1) & 1, abort_flag, P.status))
                        break;
                    const int q0 = plan.q0[g], nq = plan.nq[g];
                    mbar_expect_tx(bfull_bar, nq * 2 * kScQBoxBytes);
                    for (int qi = 0; qi < nq; ++qi)
                        for (int kb = 0; kb < 2; ++kb)
                            tma_load_2d(sB + kb * kScBBlockBytes + qi * kScQBoxBytes, &tm_q,
                                        bfull_bar, kb * 64, (q0 + qi) * kIndexHeads);
                    ++b_loads;
                    cur_g = g;
                }
                if (!mbar_wait(empty_bar(stage), phase ^ 1, abort_flag, P.status)) break;
                mbar_expect_tx(full_bar(stage), kScAStageBytes);
                const int row = static_cast<int>(P.pool_row_off[plan.seq[g]] +
                                                 static_cast<int64_t>(u - plan.unit0[g]) * kScM);
                const uint32_t dst = sA + stage * kScAStageBytes;
                tma_load_2d(dst, &tm_pool, full_bar(stage), 0, row);
                tma_load_2d(dst + kScABlockBytes, &tm_pool, full_bar(stage), 64, row);
                if (++stage == kScStages) {
                    stage = 0;
                    phase ^= 1;
                }
            }
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int g = find_group(plan.unit0, ng, u_begin), cur_g = -1, b_loads = 0, stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0, idesc = 0;
            for (int u = u_begin; u < u_end; ++u) {
                while (plan.unit0[g + 1] <= u) ++g;
                if (g != cur_g) {
                    if (b_loads > 0) tc_commit(bempty_bar);
                    if (!mbar_wait(bfull_bar, b_loads & 1, abort_flag, P.status)) break;
                    ++b_loads;
                    cur_g = g;
                    idesc = idesc_bf16_f32(kScM, kIndexHeads * plan.nq[g]);
                }
                if (!mbar_wait(acce_bar(acc), acc_phase ^ 1, abort_flag, P.status)) break;
                if (!mbar_wait(full_bar(stage), phase, abort_flag, P.status)) break;
                tc_fence_after();
                const uint32_t a_base = sA + stage * kScAStageBytes;
                const uint32_t d_tmem = tmem + acc * kScAccCols;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t koff = (kk & 3) * 32;  // 16 bf16 = 32 B inside the swizzled row
                    const uint64_t ad = desc_kmajor_sw128(a_base + (kk >> 2) * kScABlockBytes + koff);
                    const uint64_t bd = desc_kmajor_sw128(sB + (kk >> 2) * kScBBlockBytes + koff);
                    tc_mma_bf16(d_tmem, ad, bd, idesc, kk > 0 ? 1u : 0u);
                }
                tc_commit(empty_bar(stage));
                tc_commit(accf_bar(acc));
                if (++stage == kScStages) {
                    stage = 0;
                    phase ^= 1;
                }
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1;
                }
            }
        }
    } else {
        // Epilogue: warp w may only touch TMEM lanes 32*(w%4) .. +31.
        const int quad = warp & 3;
        int g = find_group(plan.unit0, ng, u_begin), acc = 0;
        uint32_t acc_phase = 0;
        for (int u = u_begin; u < u_end; ++u) {
            while (plan.unit0[g + 1] <= u) ++g;
            if (!mbar_wait(accf_bar(acc), acc_phase, abort_flag, P.status)) break;
            tc_fence_after();
            const int p = (u - plan.unit0[g]) * kScM + quad * 32 + lane;
            const int q0 = plan.q0[g], nq = plan.nq[g];
            for (int qi = 0; qi < nq; ++qi) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tmem + acc * kScAccCols + qi * kIndexHeads +
                                       (static_cast<uint32_t>(quad * 32) << 16),
                                   r);
                tmem_ld_wait();
                const int q = q0 + qi;
                const float *wq = P.w + static_cast<int64_t>(q) * kIndexHeads;
                float s = 0.f;
#pragma unroll
                for (int h = 0; h < kIndexHeads; ++h)
                    s = fmaf(__ldg(wq + h), fmaxf(__uint_as_float(r[h]), 0.f), s);
                const int nf = (P.q_pos[q] + 1) / kKpool;
                if (p < P.stride) P.scores[static_cast<int64_t>(q) * P.stride + p] = p < nf ? s : -INFINITY;
            }
            tc_fence_before();
            mbar_arrive(acce_bar(acc));
            if (++acc == 2) {
                acc = 0;
                acc_phase ^= 1;
            }
        }
    }

    tc_fence_before();
    __syncthreads();
    if (warp == 1) {
        tc_fence_after();
        tmem_dealloc(tmem, kScTmemCols);
    }
}

}  // namespace

size_t score_plan_bytes(int32_t num_queries) {
    return align_up(sizeof(int32_t) * (4 + 4 * static_cast<size_t>(num_queries) + 1), 256);
}

kp_status launch_score(const kp_score_args &a, cudaStream_t s) {
    const int nq = a.q.num_queries;
    if (nq == 0) return KP_OK;
    const int sms = device_sm_count();
    if (sms <= 0) return KP_ERR_CUDA;
    int32_t *plan = static_cast<int32_t *>(a.workspace);
    const int max_tiles = (a.q.max_pools + kScM - 1) / kScM;
    score_plan_kernel<<<1, 1024, 0, s>>>(nq, a.seqs.num_seqs, a.q.q_seq, a.q.q_pos, max_tiles, plan,
                                         a.d_status);
    kp_status st = check_launch("score_plan_kernel");
    if (st != KP_OK) return st;
    if (max_tiles == 0) return KP_OK;

    CUtensorMap tm_pool, tm_q;
    if (!make_tmap_bf16_sw128(&tm_pool, a.pooled, kIndexDim, static_cast<uint64_t>(a.seqs.pool_rows),
                              kIndexDim * 2, 64, kScM) ||
        !make_tmap_bf16_sw128(&tm_q, a.q_idx, kIndexDim, static_cast<uint64_t>(nq) * kIndexHeads,
                              kIndexDim * 2, 64, kIndexHeads))
        return KP_ERR_CUDA;
    cudaError_t e = cudaFuncSetAttribute(indexer_score_kernel,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, kScSmemBytes);
    if (e != cudaSuccess) {
        record_cuda_error("cudaFuncSetAttribute(indexer_score_kernel)", e);
        return KP_ERR_CUDA;
    }
    ScoreParams P;
    P.plan = plan;
    P.nq = nq;
    P.q_pos = a.q.q_pos;
    P.w = a.w;
    P.pool_row_off = a.seqs.pool_row_off;
    P.scores = a.scores;
    P.stride = a.score_stride;
    P.status = a.d_status;
    indexer_score_kernel<<<sms, kScThreads, kScSmemBytes, s>>>(tm_pool, tm_q, P);
    return check_launch("indexer_score_kernel");
}

}  // namespace kp
