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
// Warp roles (320 threads, one CTA per SM, persistent):
//   warp 0     TMA producer (one elected lane)
//   warp 1     TMEM allocator + MMA issuer (one elected lane)
//   warps 2-9  epilogue: TMEM -> registers -> masked scores -> global (two per lane quadrant)
// Work units are (query group, 128-pool tile) pairs laid out by a work plan:
// built by every CTA in shared memory for up to 1,022 queries, else by a plan
// kernel or an extra row of the compression launch; each CTA takes a
// contiguous range of units.
#include <cuda.h>

#include "kp_common.cuh"
#include "kp_internal.h"
#include "score_plan.cuh"

namespace kp {

namespace {

constexpr int kScMaxN = kScMaxQ * kIndexHeads;            // 256 (MMA N max)
constexpr int kScStages = 4;
constexpr int kScABlockBytes = kScM * 128;                // [128 rows][64 bf16] = 16 KB
constexpr int kScAStageBytes = 2 * kScABlockBytes;        // K = 128 -> two swizzle blocks
constexpr int kScBBlockBytes = kScMaxN * 128;             // [256 rows][64 bf16] = 32 KB
constexpr int kScBBytes = 2 * kScBBlockBytes;
constexpr int kScQBoxBytes = kIndexHeads * 128;           // one query, one K block: 4 KB
constexpr int kScEpiThreads = 256;                       // 8 epilogue warps, two per TMEM lane quadrant
constexpr int kScThreads = 64 + kScEpiThreads;
constexpr int kScTmemCols = 512;
constexpr int kScAccCols = 256;
constexpr int kScNumBars = 2 * kScStages + 4 + 4 + 2;  // full, empty, acc x 4, queries full/empty x 2, drain, never
// The queries' buffer: one 64 KB region for groups of up to 8 queries, or,
// when no group has more than 4, two 32 KB slots used in turn, so that the next
// group's queries load while the current group's MMAs still read its own.
constexpr int kScBSlotBytes = kScBBytes / 2;                  // 32 KB
constexpr int kScBSlotBlockBytes = kScBSlotBytes / 2;         // [128 rows][64 bf16] = 16 KB
constexpr int kScPlanStage = 4096;                        // plan words held in shared memory
constexpr int kScLocalPlanMaxQ = (kScPlanStage - 5) / 4;  // queries whose whole plan fits there
constexpr int kScSmemBytes = kScStages * kScAStageBytes + kScBBytes + kScNumBars * 8 + kScPlanStage * 4 + 1024;

// The plan as its own one-CTA kernel (the standalone scoring call).
__global__ void __launch_bounds__(1024) score_plan_kernel(int nq, int num_seqs,
                                                          const int32_t *__restrict__ q_seq,
                                                          const int32_t *__restrict__ q_pos,
                                                          const int32_t *__restrict__ seq_len, int kshift,
                                                          int max_tiles, int32_t *plan_base,
                                                          int32_t *status, int max_q) {
    __shared__ int scratch[33];
    pdl_wait_then_release();
    build_score_plan(nq, num_seqs, q_seq, q_pos, seq_len, kshift, max_tiles, plan_base, status, scratch, max_q);
}

struct ScoreParams {
    const int32_t *plan;       // the plan in global memory (when not built here)
    int nq;
    bool local_plan;           // build the plan in shared memory from q_seq / q_pos
    int num_seqs;
    int max_tiles;
    const int32_t *q_seq;
    const int32_t *prev_len;   // tokens of each sequence before this step (nullptr: no early loads)
    const int32_t *q_pos;
    const int32_t *seq_len;
    int kshift;                // log2(tokens per pool)
    const float *w;
    CacheMap cmap;             // where each sequence's pooled keys live
    int seg;                   // pooled rows per TMA box: 128, or a page's pools when pages are shorter
    float *scores;
    int64_t stride;
    int32_t *status;
    unsigned long long wait_ns;  // limit of one pipeline wait
    int stall;                   // KP_DEBUG_STALL_FIRST_WAIT: the MMA warp's first wait never completes
};

// Barrier over the 4 epilogue warps (named barrier 1) that also ANDs a flag,
// so a failed wait in any of them makes all of them leave together.
__device__ __forceinline__ bool epi_bar_all(bool v) {
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

// Walks the plan's groups alongside a CTA's units: one global read per group
// change instead of several dependent reads per unit.
struct GroupCursor {
    const int32_t *unit0;
    int g, u0, u1;
    __device__ void init(const int32_t *unit0_, int g0) {
        unit0 = unit0_;
        g = g0;
        u0 = unit0[g];
        u1 = unit0[g + 1];
    }
    // Advances to the group containing unit u; true when the group changed.
    __device__ bool seek(int u) {
        bool moved = false;
        while (u >= u1) {
            ++g;
            u0 = u1;
            u1 = unit0[g + 1];
            moved = true;
        }
        return moved;
    }
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
    __shared__ __align__(16) float w_s[kScMaxQ * kIndexHeads];  // head weights of the current group
    __shared__ int nf_s[kScMaxQ];                                 // complete pools each query sees

    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t sA = smem_u32(smem);
    const uint32_t sB = sA + kScStages * kScAStageBytes;
    const uint32_t bar0 = sB + kScBBytes;
    int32_t *unit0_s = reinterpret_cast<int32_t *>(smem + kScStages * kScAStageBytes + kScBBytes + kScNumBars * 8);
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kScStages + s); };
    auto accf_bar = [&](int a) { return bar0 + 8u * (2 * kScStages + a); };
    auto acce_bar = [&](int a) { return bar0 + 8u * (2 * kScStages + 2 + a); };
    auto bfull_bar = [&](int s) { return bar0 + 8u * (2 * kScStages + 4 + s); };   // queries slot s landed
    auto bempty_bar = [&](int s) { return bar0 + 8u * (2 * kScStages + 6 + s); };  // slot s's MMAs done
    const uint32_t drain_bar = bar0 + 8u * (2 * kScStages + 8);  // MMAs issued before a give-up are done
    const uint32_t never_bar = bar0 + 8u * (2 * kScStages + 9);  // nothing arrives (failure-path tests)

    // Set-up that reads nothing an earlier kernel writes: before the grid
    // dependency resolves.  The query sequences and positions the local plan
    // is built from are fetched first, so their latency hides behind the rest.
    const int plan_words = 4 + 4 * P.nq + 1;
    const bool stage_q = P.local_plan && plan_words + 2 * P.nq <= kScPlanStage;
    int32_t *qseq_s = unit0_s + plan_words, *qpos_s = qseq_s + P.nq;
    if (stage_q)
        for (int i = threadIdx.x; i < P.nq; i += kScThreads) {
            qseq_s[i] = P.q_seq[i];
            qpos_s[i] = P.q_pos[i];
        }
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    if (threadIdx.x == 0) {
        for (int s = 0; s < kScStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(accf_bar(a), 1);
            mbar_init(acce_bar(a), kScEpiThreads);
        }
        for (int b = 0; b < 2; ++b) {
            mbar_init(bfull_bar(b), 1);
            mbar_init(bempty_bar(b), 1);
        }
        mbar_init(drain_bar, 1);
        mbar_init(never_bar, 1);
        fence_mbar_init();
        abort_s = 0;
        tma_prefetch_desc(&tm_pool);
        tma_prefetch_desc(&tm_q);
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&tmem_base_s), kScTmemCols);
        tmem_relinquish();
    }

    // ---- the plan.  Built right here from the query positions when it fits
    // in shared memory (it depends only on inputs, so this overlaps the
    // previous kernel); otherwise it comes from the previous kernel, and its
    // header and group table are read in one round trip (the table has at
    // most nq + 1 entries), so finding a unit's group is a search in shared
    // memory.  Only reads of pooled keys that this step's compression may have
    // written need the grid dependency: with prev_len given, the producer
    // loads tiles wholly below each sequence's first new pool before waiting.
    __shared__ int plan_scratch[33];
    int32_t *plan_base;
    bool dep_done = false;
    if (P.local_plan) {
        if (stage_q) __syncthreads();
        build_score_plan(P.nq, P.num_seqs, stage_q ? qseq_s : P.q_seq, stage_q ? qpos_s : P.q_pos, P.seq_len,
                         P.kshift, P.max_tiles, unit0_s, P.status, plan_scratch);
        plan_base = unit0_s;
    } else {
        pdl_wait_then_release();
        dep_done = true;
        const PlanView gplan(const_cast<int32_t *>(P.plan), P.nq);
        if (P.nq + 1 <= kScPlanStage)
            for (int i = threadIdx.x; i <= P.nq; i += kScThreads) unit0_s[i] = gplan.unit0[i];
        plan_base = const_cast<int32_t *>(P.plan);
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const PlanView plan(plan_base, P.nq);
    const int ng = plan.hdr[0];
    const long long n_units = plan.hdr[1];
    const bool b_dbl = plan.hdr[2] <= kScMaxQ / 2;   // every group fits one queries slot
    const int32_t *unit0 = (P.local_plan || P.nq + 1 > kScPlanStage) ? plan.unit0 : unit0_s;
    const int u_begin = static_cast<int>(n_units * blockIdx.x / gridDim.x);
    const int u_end = static_cast<int>(n_units * (blockIdx.x + 1) / gridDim.x);
    const uint32_t tmem = tmem_base_s;
    volatile int *abort_flag = &abort_s;
    if (u_begin >= u_end || ng <= 0) {  // no work: release the TMEM and leave
        if (!dep_done && threadIdx.x == 0) pdl_wait_then_release();
        __syncthreads();
        if (warp == 1) tmem_dealloc(tmem, kScTmemCols);
        return;
    }

    if (warp == 0) {
        // TMA producer.  The whole warp walks the units (its control flow is
        // uniform); lane 0 waits on the barriers and loads the queries, and the
        // pooled-key tile is one box per K block (contiguous caches) or one box
        // per page segment per K block, issued by lanes 0 .. segments - 1 (paged
        // caches: a 128-pool tile spans 128 / (page_tokens / 4) pages when pages
        // are shorter than 512 tokens).  Segments wholly past the group's last
        // visible pool are zero-filled (negative row coordinate) instead of read
        // through the block table.
        const unsigned full = 0xffffffffu;
        GroupCursor gc;
        gc.init(unit0, find_group(unit0, ng, u_begin));
        int b_loads0 = 0, b_loads1 = 0, b_slot = 1, stage = 0;   // queries loads per slot, last slot used
        int64_t row_base = 0;
        uint32_t phase = 0;
        int old_pools = 0;  // pools of the group's sequence complete before this step
        int need = 0;       // pools the group's queries can see
        int bseq = 0;
        int a_phase[kScStages];  // phase of the last load issued into each stage (-1: none)
#pragma unroll
        for (int i = 0; i < kScStages; ++i) a_phase[i] = -1;
        bool ok = true;
        const bool paged = P.cmap.paged();
        const int nseg = kScM / P.seg;
        for (int u = u_begin; u < u_end; ++u) {
            if (gc.seek(u) || b_loads0 + b_loads1 == 0) {
                const int g = gc.g;
                const int bs = b_dbl ? (b_slot ^ 1) : 0;
                const int nb = bs ? b_loads1 : b_loads0;
                bool w_ok = true;
                if (lane == 0 && nb > 0)   // the slot's previous group's MMAs are done
                    w_ok = mbar_wait(bempty_bar(bs), (nb - 1) & 1, abort_flag, P.status, P.wait_ns);
                if (!__shfl_sync(full, w_ok, 0)) {
                    ok = false;
                    break;
                }
                const int q0 = plan.q0[g], nq = plan.nq[g];
                bseq = plan.seq[g];
                if (!paged) row_base = P.cmap.pool_row_off[bseq];
                old_pools = P.prev_len ? P.prev_len[bseq] >> P.kshift : 0;
                if (paged) need = __reduce_max_sync(full, lane < nq ? (P.q_pos[q0 + lane] + 1) >> P.kshift : 0);
                if (lane == 0) {
                    const uint32_t b_base = sB + bs * kScBSlotBytes;
                    const int kb_bytes = b_dbl ? kScBSlotBlockBytes : kScBBlockBytes;
                    mbar_expect_tx(bfull_bar(bs), nq * 2 * kScQBoxBytes);
                    for (int qi = 0; qi < nq; ++qi)
                        for (int kb = 0; kb < 2; ++kb)
                            tma_load_2d(b_base + kb * kb_bytes + qi * kScQBoxBytes, &tm_q, bfull_bar(bs), kb * 64,
                                        (q0 + qi) * kIndexHeads);
                }
                if (bs) ++b_loads1;
                else ++b_loads0;
                b_slot = bs;
            }
            bool w_ok = true;
            if (lane == 0) w_ok = mbar_wait(empty_bar(stage), phase ^ 1, abort_flag, P.status, P.wait_ns);
            if (!__shfl_sync(full, w_ok, 0)) {
                ok = false;
                break;
            }
            if (!dep_done && (u - gc.u0 + 1) * kScM > old_pools) {  // may hold pools written this step
                pdl_wait_then_release();
                dep_done = true;
            }
            const uint32_t dst = sA + stage * kScAStageBytes;
            const int p0 = (u - gc.u0) * kScM;
            if (lane == 0) mbar_expect_tx(full_bar(stage), kScAStageBytes);
            if (!paged) {
                if (lane == 0) {
                    const int row = static_cast<int>(row_base + p0);
                    tma_load_2d(dst, &tm_pool, full_bar(stage), 0, row);
                    tma_load_2d(dst + kScABlockBytes, &tm_pool, full_bar(stage), 64, row);
                }
            } else if (lane < nseg) {
                const int p = p0 + lane * P.seg;
                int y = -P.seg;
                if (p < need) {
                    const int64_t r = P.cmap.pool_row(bseq, p);
                    if (r >= 0) y = static_cast<int>(r);
                    else set_status(P.status, KP_ERR_DEVICE_BOUNDS);
                }
                const uint32_t off = static_cast<uint32_t>(lane * P.seg * 128);
                tma_load_2d(dst + off, &tm_pool, full_bar(stage), 0, y);
                tma_load_2d(dst + kScABlockBytes + off, &tm_pool, full_bar(stage), 64, y);
            }
            a_phase[stage] = static_cast<int>(phase);
            if (++stage == kScStages) {
                stage = 0;
                phase ^= 1;
            }
        }
        // This grid completes only after the previous one: kernels that wait
        // on this one may rely on everything before it.
        if (!dep_done) pdl_wait_then_release();
        if (!ok && lane == 0) {
            // Gave up: every load the warp issued lands before the shared memory
            // and the CTA go away (the latest phase of each barrier it armed;
            // bounded by the default limit).
            if (b_loads0 > 0) mbar_wait(bfull_bar(0), (b_loads0 - 1) & 1, nullptr, P.status);
            if (b_loads1 > 0) mbar_wait(bfull_bar(1), (b_loads1 - 1) & 1, nullptr, P.status);
#pragma unroll
            for (int i = 0; i < kScStages; ++i)
                if (a_phase[i] >= 0) mbar_wait(full_bar(i), static_cast<uint32_t>(a_phase[i]), nullptr, P.status);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            GroupCursor gc;
            gc.init(unit0, find_group(unit0, ng, u_begin));
            int b_uses0 = 0, b_uses1 = 0, b_slot = 1, b_cur = -1, stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0, idesc = 0, b_base = sB;
            int kb_bytes = kScBBlockBytes;
            bool ok = !P.stall || mbar_wait(never_bar, 0, abort_flag, P.status, P.wait_ns);
            for (int u = u_begin; ok && u < u_end; ++u) {
                if (gc.seek(u) || b_cur < 0) {
                    if (b_cur >= 0) tc_commit(bempty_bar(b_cur));   // the previous group's queries are free
                    const int bs = b_dbl ? (b_slot ^ 1) : 0;
                    if (!(ok = mbar_wait(bfull_bar(bs), (bs ? b_uses1 : b_uses0) & 1, abort_flag, P.status,
                                         P.wait_ns)))
                        break;
                    if (bs) ++b_uses1;
                    else ++b_uses0;
                    b_slot = b_cur = bs;
                    b_base = sB + bs * kScBSlotBytes;
                    kb_bytes = b_dbl ? kScBSlotBlockBytes : kScBBlockBytes;
                    idesc = idesc_bf16_f32(kScM, kIndexHeads * plan.nq[gc.g]);
                }
                if (!(ok = mbar_wait(acce_bar(acc), acc_phase ^ 1, abort_flag, P.status, P.wait_ns))) break;
                if (!(ok = mbar_wait(full_bar(stage), phase, abort_flag, P.status, P.wait_ns))) break;
                tc_fence_after();
                const uint32_t a_base = sA + stage * kScAStageBytes;
                const uint32_t d_tmem = tmem + acc * kScAccCols;
#pragma unroll
                for (int kk = 0; kk < 8; ++kk) {
                    const uint32_t koff = (kk & 3) * 32;  // 16 bf16 = 32 B inside the swizzled row
                    const uint64_t ad = desc_kmajor_sw128(a_base + (kk >> 2) * kScABlockBytes + koff);
                    const uint64_t bd = desc_kmajor_sw128(b_base + (kk >> 2) * kb_bytes + koff);
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
            if (!ok) {
                // Gave up: every MMA already issued completes before the TMEM is freed.
                tc_commit(drain_bar);
                mbar_wait(drain_bar, 0, nullptr, P.status);
            }
        }
    } else {
        // Epilogue: warp w may only touch TMEM lanes 32*(w%4) .. +31.  Two warps
        // share each lane quadrant and split the group's queries (even / odd),
        // so each scheduler has two epilogue warps to interleave.  A thread owns
        // one pool row: it loads two queries' 32 head columns before waiting,
        // then reduces ReLU(.) * w over the heads with packed fp32x2 FMAs into
        // eight independent partial sums (fp32, round to nearest).  The head
        // weights and causal limits of the current query group are staged in
        // shared memory when the group changes.
        const int quad = warp & 3, et = threadIdx.x - 64, half = et >> 7;
        GroupCursor gc;
        gc.init(unit0, find_group(unit0, ng, u_begin));
        int acc = 0, q0 = 0, nq = 0;
        bool first = true;
        uint32_t acc_phase = 0;
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
        for (int u = u_begin; u < u_end; ++u) {
            const bool moved = gc.seek(u) || first;
            // every epilogue thread leaves together if any wait failed
            if (!epi_bar_all(mbar_wait(accf_bar(acc), acc_phase, abort_flag, P.status, P.wait_ns))) break;
            tc_fence_after();
            if (moved) {
                q0 = plan.q0[gc.g];
                nq = plan.nq[gc.g];
                for (int k = et; k < nq * kIndexHeads; k += kScEpiThreads)
                    w_s[k] = P.w[static_cast<int64_t>(q0) * kIndexHeads + k];
                if (et < nq) nf_s[et] = (P.q_pos[q0 + et] + 1) >> P.kshift;
                epi_bar_all(true);
                first = false;
            }
            const int p = (u - gc.u0) * kScM + quad * 32 + lane;
            const uint32_t tbase = tmem + acc * kScAccCols + (static_cast<uint32_t>(quad * 32) << 16);
            for (int qi = half; qi < nq; qi += 4) {
                const int qj = qi + 2;                   // the warp's next query, if any
                uint32_t r0[32], r1[32];
                tmem_ld_32x32b_x32(tbase + qi * kIndexHeads, r0);
                if (qj < nq) tmem_ld_32x32b_x32(tbase + qj * kIndexHeads, r1);
                tmem_ld_wait();
                const float v0 = reduce(r0, qi);
                if (p < P.stride)
                    P.scores[static_cast<int64_t>(q0 + qi) * P.stride + p] = p < nf_s[qi] ? v0 : -INFINITY;
                if (qj < nq) {
                    const float v1 = reduce(r1, qj);
                    if (p < P.stride)
                        P.scores[static_cast<int64_t>(q0 + qj) * P.stride + p] = p < nf_s[qj] ? v1 : -INFINITY;
                }
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

ScorePlanArgs score_plan_args(const kp_score_args &a) {
    ScorePlanArgs p;
    p.nq = a.q.num_queries;
    p.num_seqs = a.seqs.num_seqs;
    p.q_seq = a.q.q_seq;
    p.q_pos = a.q.q_pos;
    p.seq_len = a.seqs.seq_len;
    p.kshift = kpool_shift(a.cfg.kpool);
    p.max_q = kScMaxQ;
    p.max_tiles = (a.q.max_pools + kScM - 1) / kScM;
    p.plan = static_cast<int32_t *>(a.workspace);
    p.status = a.d_status;
    return p;
}

bool score_plan_is_local(int32_t num_queries) { return num_queries <= kScLocalPlanMaxQ; }

kp_status launch_score_plan(const ScorePlanArgs &p, cudaStream_t s) {
    return launch_kernel("score_plan_kernel", score_plan_kernel, LaunchCfg(dim3(1), dim3(1024), 0, s), p.nq,
                         p.num_seqs, p.q_seq, p.q_pos, p.seq_len, p.kshift, p.max_tiles, p.plan, p.status, p.max_q);
}

kp_status launch_score(const kp_score_args &a, cudaStream_t s, bool plan_ready, const int32_t *prev_len,
                       bool allow_local_plan) {
    const int nq = a.q.num_queries;
    if (nq == 0) return KP_OK;
    const int sms = device_sm_count();
    if (sms <= 0) return KP_ERR_CUDA;
    int32_t *plan = static_cast<int32_t *>(a.workspace);
    const int max_tiles = (a.q.max_pools + kScM - 1) / kScM;
    const bool local_plan = allow_local_plan && score_plan_is_local(nq);
    if (!plan_ready && !local_plan) {
        const kp_status st = launch_kernel("score_plan_kernel", score_plan_kernel,
                                           LaunchCfg(dim3(1), dim3(1024), 0, s), nq, a.seqs.num_seqs, a.q.q_seq,
                                           a.q.q_pos, a.seqs.seq_len, kpool_shift(a.cfg.kpool), max_tiles, plan,
                                           a.d_status, kScMaxQ);
        if (st != KP_OK) return st;
    }
    if (max_tiles == 0) return KP_OK;

    const int pool_page = a.seqs.block_table ? a.seqs.page_tokens / a.cfg.kpool : kScM;  // pools per page
    const int seg = pool_page < kScM ? pool_page : kScM;
    CUtensorMap tm_pool, tm_q;
    if (!make_tmap_bf16_sw128(&tm_pool, a.pooled, kIndexDim, static_cast<uint64_t>(a.seqs.pool_rows),
                              kIndexDim * 2, 64, static_cast<uint32_t>(seg)) ||
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
    P.local_plan = local_plan;
    P.num_seqs = a.seqs.num_seqs;
    P.max_tiles = max_tiles;
    P.q_seq = a.q.q_seq;
    P.prev_len = local_plan ? prev_len : nullptr;
    P.q_pos = a.q.q_pos;
    P.seq_len = a.seqs.seq_len;
    P.kshift = kpool_shift(a.cfg.kpool);
    P.w = a.w;
    P.cmap = cache_map(a.seqs, a.cfg.kpool);
    P.seg = seg;
    P.scores = a.scores;
    P.stride = a.score_stride;
    P.status = a.d_status;
    P.wait_ns = wait_limit_ns(a.cfg.wait_limit_us);
    P.stall = (a.cfg.debug_flags & KP_DEBUG_STALL_FIRST_WAIT) ? 1 : 0;
    return launch_kernel("indexer_score_kernel", indexer_score_kernel,
                         LaunchCfg(dim3(sms), dim3(kScThreads), kScSmemBytes, s), tm_pool, tm_q, P);
}

}  // namespace kp
