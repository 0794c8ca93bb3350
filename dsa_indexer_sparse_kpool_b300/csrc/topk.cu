// topk.cu -- top-k pool selection: exact radix select on order-preserving
// keys, then an order-preserving compaction.
//
// Method: each query keeps index_topk / kpool pools (2048 tokens / 4 = 512;
// llm-atlas GLM-5.3-Flash card, raw config index_topk / index_kpool); when it
// sees no more complete pools than that, it keeps them all.  Ties go to the
// lower pool index and the kept pools are written in ascending order.
//
// B300 design.  A query's row of n = n_full(t) scores is split over a
// thread-block cluster of C CTAs (one CTA for rows up to 16K keys; longer
// rows over as many CTAs as hold them in shared memory, and more while every
// CTA keeps over 16K keys and all rows' CTAs still fit one wave; up to 8),
// each holding its slice in shared memory as order-preserving uint32 keys.
// A CTA has 1024 threads when every row's CTAs fit one wave on the SMs (few
// rows: shorter passes cut the latency) and 512 otherwise (many rows: the SMs
// are full either way and block barriers are cheaper).
//  1. The cluster's smallest key and key span fix a shift s with at most 2048
//     bins of width 2^s.  Each level histograms the keys inside the current
//     range into its bins, finds the bin holding the K-th largest key and
//     narrows the range to that bin, split next into bins of width
//     2^max(0, s - 11).  After at most three
//     levels the range is one key value: the threshold T, with the number of
//     keys equal to T that are taken (the lowest indices first).  A level
//     costs one pass over the keys and one cluster barrier: every CTA reads
//     every peer's histogram through distributed shared memory (two buffers,
//     so a level never waits for the previous one to be read).  When the
//     K-th largest key's bin is taken whole (it holds exactly the keys still
//     needed, typically one key at the second level) the selection is every
//     key >= the bin's lower edge and the search stops there; otherwise, once
//     the chosen bin holds at most 32 keys of the row, those keys are collected
//     and one warp ranks them against each other, which gives T directly.
//  2. Counts of keys above / equal to T, per warp and per CTA, give every
//     selected key its output position; each warp walks its own contiguous
//     range of keys with lanes interleaved (no shared-memory bank conflicts),
//     so the selection is written in ascending pool order with no sort.
// Cluster barriers are hardware barriers (all CTAs of a cluster are
// co-resident): no spin loop anywhere.
#include "kp_common.cuh"
#include "kp_internal.h"

namespace kp {

namespace {

constexpr int kTkMaxThreads = 1024;    // CTA size when every row's CTAs fit one wave (latency)
constexpr int kTkMinThreads = 512;     // otherwise (many rows: throughput)
constexpr int kTkMaxWarps = kTkMaxThreads / 32;
constexpr int kTkChunkMax = 32768;    // keys per CTA (128 KB of shared memory)
constexpr int kTkMaxCluster = 8;
constexpr int kTkBins = 2048;
constexpr int kTkDigit = 11;           // log2(kTkBins)
constexpr int kTkKeysPerCta = 16384;   // a row this long stays in one CTA (cluster rounds cost more than the pass)
constexpr int kTkSmall = 32;           // a chosen bin this small is resolved by ranking
constexpr int kTkLoadUnroll = 8;       // float4 loads a thread has in flight

__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ uint4 ld_cluster_u32x4(uint32_t addr) {
    uint4 v;
    asm volatile("ld.shared::cluster.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "r"(addr)
                 : "memory");
    return v;
}
__device__ __forceinline__ uint2 ld_cluster_u32x2(uint32_t addr) {
    uint2 v;
    asm volatile("ld.shared::cluster.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr) : "memory");
    return v;
}

// Order-preserving key: larger float -> larger key; -0 == +0; NaN lowest.
__device__ __forceinline__ uint32_t score_key(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7fffffffu) > 0x7f800000u) return 0u;
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Exclusive block-wide scan of an unsigned 32-bit value (blockDim.x a multiple of 32).
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t *warp_tot, uint32_t *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
    uint32_t incl = v;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const uint32_t n = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) warp_tot[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        uint32_t w = lane < static_cast<int>(blockDim.x >> 5) ? warp_tot[lane] : 0u;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t n = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w += n;
        }
        warp_tot[lane] = w;  // inclusive over warps
    }
    __syncthreads();
    const uint32_t before = (warp > 0 ? warp_tot[warp - 1] : 0u) + incl - v;
    *total = warp_tot[(blockDim.x >> 5) - 1];
    __syncthreads();
    return before;
}

struct TopkShared {
    uint32_t hist[2][kTkBins];        // this CTA's histogram of a level (two buffers)
    uint32_t warp_tot[32];
    uint32_t wgt[kTkMaxWarps], weq[kTkMaxWarps];  // per-warp counts above / equal to T
    uint32_t wgt_before[kTkMaxWarps], weq_before[kTkMaxWarps];  // the same summed over earlier warps
    uint32_t kmin, kmax;              // this CTA's key range
    uint32_t gmin, gmax;              // the cluster's key range
    uint32_t out_base, eq_before;     // output offset and equal keys of earlier CTAs
    uint32_t cnt_gt, cnt_eq;          // this CTA's keys above / equal to T
    int pick_bin, pick_need;
    uint32_t pick_cnt;                // keys of the row in the chosen bin
    uint32_t small_n;                 // this CTA's keys in a small chosen bin
    uint32_t small[kTkSmall];
    uint32_t res_T, res_need;
};

template <int kTkThreads>
__global__ void __launch_bounds__(kTkThreads, 1)
    topk_select_kernel(const float *__restrict__ scores, int64_t stride,
                       const int32_t *__restrict__ q_pos, int kshift, int K, int32_t *__restrict__ pool_idx,
                       int32_t *__restrict__ n_sel, int chunk_cap, int32_t *status) {
    constexpr int kTkWarps = kTkThreads / 32;
    extern __shared__ uint32_t keys[];
    __shared__ __align__(16) TopkShared sh;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t rank = cluster_ctarank(), C = cluster_size();
    const int q = blockIdx.x / C;
    // A one-CTA row needs only block barriers.
    auto cbar = [&]() {
        if (C > 1) cluster_barrier();
        else __syncthreads();
    };
    // Inputs and shared-memory set-up first: the scores come from the previous
    // kernel, so only their reads wait for the grid dependency.
    const int t = q_pos[q];
    const int n = t >= 0 ? (t + 1) >> kshift : 0;
    int32_t *out = pool_idx + static_cast<int64_t>(q) * K;
    if (tid == 0) {
        sh.kmin = 0xffffffffu;
        sh.kmax = 0u;
    }
    for (int i = tid; i < kTkBins; i += kTkThreads) sh.hist[0][i] = 0u;
    pdl_wait_then_release();

    if (n <= K) {  // every visible pool is kept
        for (int i = rank * kTkThreads + tid; i < K; i += C * kTkThreads) out[i] = i < n ? i : -1;
        if (rank == 0 && tid == 0) n_sel[q] = n;
        return;
    }

    const int cs = static_cast<int>(static_cast<int64_t>(n) * rank / C);
    int len = static_cast<int>(static_cast<int64_t>(n) * (rank + 1) / C) - cs;
    if (len > chunk_cap) {  // the caller's max_pools bound was too small
        if (tid == 0) set_status(status, KP_ERR_DEVICE_BOUNDS);
        len = chunk_cap;
    }

    // ---- keys, key range
    const float *row = scores + static_cast<int64_t>(q) * stride + cs;
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    if ((reinterpret_cast<uintptr_t>(row) & 15) == 0) {
        const int n4 = len >> 2;
        for (int i0 = tid; i0 < n4; i0 += kTkLoadUnroll * kTkThreads) {
            float4 v[kTkLoadUnroll];  // every load issued before the first is used
#pragma unroll
            for (int u = 0; u < kTkLoadUnroll; ++u) {
                const int i = i0 + u * kTkThreads;
                if (i < n4) v[u] = __ldcs(reinterpret_cast<const float4 *>(row) + i);
            }
#pragma unroll
            for (int u = 0; u < kTkLoadUnroll; ++u) {
                const int i = i0 + u * kTkThreads;
                if (i < n4) {
                    const uint32_t a = score_key(v[u].x), b = score_key(v[u].y), c = score_key(v[u].z),
                                   d = score_key(v[u].w);
                    reinterpret_cast<uint4 *>(keys)[i] = make_uint4(a, b, c, d);
                    kmin = min(kmin, min(min(a, b), min(c, d)));
                    kmax = max(kmax, max(max(a, b), max(c, d)));
                }
            }
        }
        for (int i = 4 * n4 + tid; i < len; i += kTkThreads) {
            const uint32_t k = score_key(row[i]);
            keys[i] = k;
            kmin = min(kmin, k);
            kmax = max(kmax, k);
        }
    } else {
        for (int i = tid; i < len; i += kTkThreads) {
            const uint32_t k = score_key(row[i]);
            keys[i] = k;
            kmin = min(kmin, k);
            kmax = max(kmax, k);
        }
    }
    kmin = __reduce_min_sync(0xffffffffu, kmin);
    kmax = __reduce_max_sync(0xffffffffu, kmax);
    __syncthreads();
    if (lane == 0) {
        atomicMin(&sh.kmin, kmin);
        atomicMax(&sh.kmax, kmax);
    }
    cbar();
    // One warp gathers the cluster's key range (every thread reading the same
    // remote words would serialise on them) and broadcasts it.
    if (warp == 0) {
        uint32_t mn = 0xffffffffu, mx = 0u;
        if (static_cast<uint32_t>(lane) < C) {
            mn = ld_cluster_u32(dsmem_addr(smem_u32(&sh.kmin), lane));
            mx = ld_cluster_u32(dsmem_addr(smem_u32(&sh.kmax), lane));
        }
        mn = __reduce_min_sync(0xffffffffu, mn);
        mx = __reduce_max_sync(0xffffffffu, mx);
        if (lane == 0) {
            sh.gmin = mn;
            sh.gmax = mx;
        }
    }
    __syncthreads();
    const uint32_t gmin = sh.gmin, gmax = sh.gmax;

    // ---- radix select: the range [base, base + 2^wb) holds the K-th largest key;
    // a level splits it into bins of width 2^s (at most 2048 of them).
    const uint64_t span = static_cast<uint64_t>(gmax) - gmin + 1;
    int s = 0;
    while (((span - 1) >> s) >= static_cast<uint64_t>(kTkBins)) ++s;
    int wb = s + kTkDigit;
    uint32_t base = gmin;
    int need = K;
    constexpr int kPer = kTkBins / kTkThreads;  // bins per thread in the scan
    static_assert(kPer == 2 || kPer == 4, "the histogram scan reads two or four bins per thread");
    for (int level = 0;; ++level) {
        uint32_t *hist = sh.hist[level & 1];
        if (level > 0) {  // this buffer was last read by peers two levels ago
            for (int i = tid; i < kTkBins; i += kTkThreads) hist[i] = 0u;
            __syncthreads();
        }
        const uint64_t range = static_cast<uint64_t>(1) << wb;
        for (int i = tid; i < len; i += kTkThreads) {
            const uint32_t k = keys[i];
            if (k >= base && static_cast<uint64_t>(k - base) < range) atomicAdd(&hist[(k - base) >> s], 1u);
        }
        cbar();  // every CTA's histogram of this level is complete
        // Cluster totals of this thread's kPer bins, read from every CTA; the
        // thread holds bins b0+kPer-1 .. b0 (descending key order across threads).
        const int b0 = kTkBins - kPer * (tid + 1);
        uint32_t c[kPer], sum = 0;
#pragma unroll
        for (int j = 0; j < kPer; ++j) c[j] = 0u;
        for (uint32_t r = 0; r < C; ++r) {
            if constexpr (kPer == 4) {
                const uint4 v = C == 1 ? *reinterpret_cast<const uint4 *>(hist + b0)
                                       : ld_cluster_u32x4(dsmem_addr(smem_u32(hist + b0), r));
                c[0] += v.w;
                c[1] += v.z;
                c[2] += v.y;
                c[3] += v.x;
            } else {
                const uint2 v = C == 1 ? *reinterpret_cast<const uint2 *>(hist + b0)
                                       : ld_cluster_u32x2(dsmem_addr(smem_u32(hist + b0), r));
                c[0] += v.y;
                c[1] += v.x;
            }
        }
#pragma unroll
        for (int j = 0; j < kPer; ++j) sum += c[j];
        uint32_t tot;
        uint32_t above = block_excl_scan(sum, sh.warp_tot, &tot);
        if (tid == 0 && tot < static_cast<uint32_t>(need)) {  // counts lost: cannot happen with consistent data
            set_status(status, KP_ERR_DEVICE_BOUNDS);
            sh.pick_bin = kTkBins - 1;
            sh.pick_need = 1;
            sh.pick_cnt = 0xffffffffu;
        }
        if (above < static_cast<uint32_t>(need) && static_cast<uint32_t>(need) <= above + sum) {
#pragma unroll
            for (int j = 0; j < kPer; ++j) {
                if (above < static_cast<uint32_t>(need) && above + c[j] >= static_cast<uint32_t>(need)) {
                    sh.pick_bin = b0 + kPer - 1 - j;
                    sh.pick_need = need - static_cast<int>(above);
                    sh.pick_cnt = c[j];
                }
                above += c[j];
            }
        }
        __syncthreads();
        base += static_cast<uint32_t>(sh.pick_bin) << s;
        need = sh.pick_need;
        const uint32_t bin_cnt = sh.pick_cnt;
        __syncthreads();  // pick_* is rewritten by the next level
        if (s == 0) break;
        if (static_cast<uint32_t>(need) == bin_cnt && base > 0u) {
            // Every key of the chosen bin is taken (usual once a bin holds one
            // key): the selection is the keys >= base, i.e. above base - 1.
            base -= 1u;
            need = 0;
            break;
        }
        if (bin_cnt <= static_cast<uint32_t>(kTkSmall)) {
            // The chosen bin [base, base + 2^s) holds at most 32 keys of the row:
            // collect them (every CTA) and rank them in one warp.
            if (tid == 0) sh.small_n = 0u;
            __syncthreads();
            const uint64_t brange = static_cast<uint64_t>(1) << s;
            for (int i = tid; i < len; i += kTkThreads) {
                const uint32_t k = keys[i];
                if (k >= base && static_cast<uint64_t>(k - base) < brange) {
                    const uint32_t slot = atomicAdd(&sh.small_n, 1u);
                    if (slot < static_cast<uint32_t>(kTkSmall)) sh.small[slot] = k;
                }
            }
            cbar();  // every CTA's list is complete
            if (warp == 0) {
                uint32_t key = 0u, off = 0u;
                bool has = false;
                for (uint32_t r = 0; r < C; ++r) {
                    const uint32_t nr = min(static_cast<uint32_t>(kTkSmall),
                                            ld_cluster_u32(dsmem_addr(smem_u32(&sh.small_n), r)));
                    if (!has && static_cast<uint32_t>(lane) >= off && static_cast<uint32_t>(lane) < off + nr) {
                        key = ld_cluster_u32(dsmem_addr(smem_u32(&sh.small[lane - off]), r));
                        has = true;
                    }
                    off += nr;
                }
                uint32_t gtk = 0, eqk = 0;  // keys of the bin above / equal to mine
#pragma unroll 8
                for (int j = 0; j < 32; ++j) {
                    const uint32_t kj = __shfl_sync(0xffffffffu, key, j);
                    const bool hj = __shfl_sync(0xffffffffu, has, j);
                    gtk += hj && kj > key;
                    eqk += hj && kj == key;
                }
                const bool mine = has && gtk < static_cast<uint32_t>(need) && static_cast<uint32_t>(need) <= gtk + eqk;
                const uint32_t who = __ballot_sync(0xffffffffu, mine);
                if (lane == 0) {
                    if (who == 0u) {  // counts lost: cannot happen with consistent data
                        set_status(status, KP_ERR_DEVICE_BOUNDS);
                        sh.res_T = base;
                        sh.res_need = 1u;
                    }
                }
                if (who != 0u) {
                    const int src = __ffs(who) - 1;
                    const uint32_t T0 = __shfl_sync(0xffffffffu, key, src);
                    const uint32_t g0 = __shfl_sync(0xffffffffu, gtk, src);
                    if (lane == 0) {
                        sh.res_T = T0;
                        sh.res_need = static_cast<uint32_t>(need) - g0;
                    }
                }
            }
            __syncthreads();
            base = sh.res_T;
            need = static_cast<int>(sh.res_need);
            break;
        }
        wb = s;  // the chosen bin is the next range
        s = wb > kTkDigit ? wb - kTkDigit : 0;
    }
    const uint32_t T = base;                               // the K-th largest key
    const uint32_t eq_take = static_cast<uint32_t>(need);  // keys equal to T that are taken

    // ---- per-warp and per-CTA counts above / equal to T
    const int wlen = ((len + kTkWarps - 1) / kTkWarps + 31) & ~31;  // contiguous keys per warp
    const int w0 = min(len, warp * wlen), w1 = min(len, w0 + wlen);
    uint32_t gt = 0, eq = 0;
    for (int i = w0 + lane; i < w1; i += 32) {
        const uint32_t k = keys[i];
        gt += k > T;
        eq += k == T;
    }
    gt = __reduce_add_sync(0xffffffffu, gt);
    eq = __reduce_add_sync(0xffffffffu, eq);
    if (lane == 0) {
        sh.wgt[warp] = gt;
        sh.weq[warp] = eq;
    }
    __syncthreads();
    // Warp 0 turns the per-warp counts into exclusive prefixes (a shuffle scan)
    // and the CTA's totals.
    if (warp == 0) {
        const uint32_t g = lane < kTkWarps ? sh.wgt[lane] : 0u, e = lane < kTkWarps ? sh.weq[lane] : 0u;
        uint32_t gi = g, ei = e;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const uint32_t gu = __shfl_up_sync(0xffffffffu, gi, o), eu = __shfl_up_sync(0xffffffffu, ei, o);
            if (lane >= o) {
                gi += gu;
                ei += eu;
            }
        }
        if (lane < kTkWarps) {
            sh.wgt_before[lane] = gi - g;
            sh.weq_before[lane] = ei - e;
        }
        if (lane == 31) {
            sh.cnt_gt = gi;
            sh.cnt_eq = ei;
        }
    }
    cbar();
    // This CTA's first output position and share of the keys equal to T, from
    // the counts of the CTAs before it (one thread reads them, then broadcasts).
    if (C > 1) {
        if (tid == 0) {
            uint32_t ob = 0, eb = 0;
            for (uint32_t r = 0; r < rank; ++r) {
                const uint32_t gt_r = ld_cluster_u32(dsmem_addr(smem_u32(&sh.cnt_gt), r));
                const uint32_t eq_r = ld_cluster_u32(dsmem_addr(smem_u32(&sh.cnt_eq), r));
                const uint32_t rem = eq_take > eb ? eq_take - eb : 0u;
                ob += gt_r + min(rem, eq_r);
                eb += eq_r;
            }
            sh.out_base = ob;
            sh.eq_before = eb;
        }
        __syncthreads();
    }
    const uint32_t out_base = C > 1 ? sh.out_base : 0u, eq_before = C > 1 ? sh.eq_before : 0u;
    const uint32_t my_take = min(eq_take > eq_before ? eq_take - eq_before : 0u, sh.cnt_eq);

    // ---- order-preserving compaction: a selected key's position is the number of
    // keys above T before it plus min(keys equal to T before it, my_take).
    uint32_t gt_run = sh.wgt_before[warp], eq_run = sh.weq_before[warp];
    const uint32_t lane_lt = (1u << lane) - 1u;
    for (int i0 = w0; i0 < w1; i0 += 32) {
        const int i = i0 + lane;
        const uint32_t k = i < w1 ? keys[i] : 0u;
        const bool isgt = i < w1 && k > T;
        const bool iseq = i < w1 && k == T;
        const uint32_t bgt = __ballot_sync(0xffffffffu, isgt), beq = __ballot_sync(0xffffffffu, iseq);
        const uint32_t eq_b = eq_run + __popc(beq & lane_lt);
        if (isgt || (iseq && eq_b < my_take)) {
            const uint32_t pos = out_base + gt_run + __popc(bgt & lane_lt) + min(eq_b, my_take);
            if (pos < static_cast<uint32_t>(K)) out[pos] = cs + i;
        }
        gt_run += __popc(bgt);
        eq_run += __popc(beq);
    }
    if (rank == 0 && tid == 0) n_sel[q] = K;
    cbar();  // keep this CTA's shared memory alive until every peer is done reading it
}

}  // namespace

kp_status launch_topk(const kp_topk_args &a, cudaStream_t s) {
    const int nq = a.q.num_queries;
    if (nq == 0) return KP_OK;
    const int K = a.cfg.topk_tokens / a.cfg.kpool;
    const int maxp = a.q.max_pools;
    // A row is latency-bound work and every cluster round costs more than a
    // pass over 16K keys in shared memory.  The cluster is as small as shared
    // memory allows (<= 32768 keys per CTA), then grows while every CTA keeps
    // more than 16K keys and all rows' CTAs still fit one wave on the SMs.
    int C = 1;
    while (C < kTkMaxCluster && (maxp + C - 1) / C > kTkChunkMax) C *= 2;
    const int64_t sms = device_sm_count() > 0 ? device_sm_count() : 1;
    while (C < kTkMaxCluster && (maxp + C - 1) / C > kTkKeysPerCta &&
           static_cast<int64_t>(nq) * C * 2 <= sms)
        C *= 2;
    const int chunk_cap = (maxp + C - 1) / C;
    if (chunk_cap > kTkChunkMax) return KP_ERR_UNSUPPORTED;
    const size_t smem = static_cast<size_t>(chunk_cap > 0 ? chunk_cap : 1) * sizeof(uint32_t);
    // Few rows (every CTA in one wave): the wider CTA shortens each pass.  Many
    // rows: the narrower one, since the SMs are full either way.
    const bool wide = static_cast<int64_t>(nq) * C <= sms;
    auto kern = wide ? topk_select_kernel<kTkMaxThreads> : topk_select_kernel<kTkMinThreads>;
    cudaError_t e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kTkChunkMax * static_cast<int>(sizeof(uint32_t)));
    if (e != cudaSuccess) {
        record_cuda_error("cudaFuncSetAttribute(topk_select_kernel)", e);
        return KP_ERR_CUDA;
    }
    return launch_kernel("topk_select_kernel", kern,
                         LaunchCfg(dim3(static_cast<unsigned>(nq) * C), dim3(wide ? kTkMaxThreads : kTkMinThreads),
                                   smem, s, C),
                         a.scores, a.score_stride, a.q.q_pos, kpool_shift(a.cfg.kpool), K, a.pool_idx, a.n_sel,
                         chunk_cap, a.d_status);
}

}  // namespace kp
