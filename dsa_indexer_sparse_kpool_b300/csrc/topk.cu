// topk.cu -- top-k pool selection by radix select in shared memory.
//
// Method: each query keeps index_topk / kpool pools (2048 tokens / 4 = 512;
// llm-atlas GLM-5.3-Flash card, raw config index_topk / index_kpool); when it
// sees no more complete pools than that, it keeps them all.  Ties go to the
// lower pool index and the kept pools are written in ascending order.
//
// B300 design.  A query's row of n = n_full(t) scores is split over a
// thread-block cluster of C CTAs (C = 1 for rows up to 32K pools, up to 8 for
// the 262,143-pool rows of a 1M-token context), each holding its slice as
// order-preserving uint32 keys in shared memory (<= 128 KB).  Four 8-bit radix
// passes find the K-th largest key exactly: per pass every CTA builds a
// warp-aggregated histogram and adds it into the cluster leader's shared
// histogram through distributed shared memory; after a cluster barrier each
// CTA reads the combined histogram and picks the same digit.  The selected
// indices are then emitted by an order-preserving compaction (block scans of
// ballots) at offsets given by the lower-ranked CTAs' counts, so the output
// is ascending with no sort.  Cluster barriers are hardware barriers (all
// CTAs of a cluster are co-resident): no spin loop anywhere.
#include "kp_common.cuh"
#include "kp_internal.h"

namespace kp {

namespace {

constexpr int kTkThreads = 1024;
constexpr int kTkChunkMax = 32768;  // keys per CTA (128 KB of shared memory)
constexpr int kTkMaxCluster = 8;

__device__ __forceinline__ uint32_t cluster_rank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_sync_all() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}
__device__ __forceinline__ uint32_t map_rank(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
__device__ __forceinline__ void red_add_cluster(uint32_t addr, uint32_t v) {
    asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t ld_cluster(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}

// Order-preserving key: larger float -> larger key; -0 == +0; NaN lowest.
__device__ __forceinline__ uint32_t score_key(float f) {
    uint32_t u = __float_as_uint(f);
    if ((u & 0x7fffffffu) > 0x7f800000u) return 0u;
    if (u == 0x80000000u) u = 0u;
    return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

__global__ void __launch_bounds__(kTkThreads, 1)
    topk_select_kernel(const float *__restrict__ scores, int64_t stride,
                       const int32_t *__restrict__ q_pos, int K, int32_t *__restrict__ pool_idx,
                       int32_t *__restrict__ n_sel, int chunk_cap, int32_t *status) {
    extern __shared__ uint32_t keys[];
    __shared__ uint32_t hist[4][256];  // the leader's copy holds the cluster totals
    __shared__ uint32_t lhist[256];
    __shared__ int wsum[2][32];
    __shared__ int cnt[2];
    __shared__ int pick[2];

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint32_t rank = cluster_rank(), C = cluster_size();
    const int q = blockIdx.x / C;
    const int t = q_pos[q];
    const int n = t >= 0 ? (t + 1) / kKpool : 0;
    int32_t *out = pool_idx + static_cast<int64_t>(q) * K;

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
    const float *row = scores + static_cast<int64_t>(q) * stride + cs;
    for (int i = tid; i < len; i += kTkThreads) keys[i] = score_key(row[i]);
    for (int i = tid; i < 4 * 256; i += kTkThreads) (&hist[0][0])[i] = 0u;
    cluster_sync_all();

    const uint32_t lane_lt = (1u << lane) - 1u;
    uint32_t prefix = 0, mask = 0;
    int krem = K;  // how many still to take among keys matching `prefix` on `mask`
    for (int pass = 0; pass < 4; ++pass) {
        const int shift = 24 - 8 * pass;
        if (tid < 256) lhist[tid] = 0u;
        __syncthreads();
        for (int base = 0; base < len; base += kTkThreads) {
            const int i = base + tid;
            const uint32_t k = i < len ? keys[i] : 0u;
            const bool m = i < len && (k & mask) == prefix;
            const uint32_t act = __ballot_sync(0xffffffffu, m);
            if (m) {
                const uint32_t bin = (k >> shift) & 255u;
                const uint32_t peers = __match_any_sync(act, bin);
                if (lane == __ffs(peers) - 1) atomicAdd(&lhist[bin], __popc(peers));
            }
        }
        __syncthreads();
        if (tid < 256 && lhist[tid]) red_add_cluster(map_rank(smem_u32(&hist[pass][tid]), 0), lhist[tid]);
        cluster_sync_all();
        if (warp == 0) {
            // lane l covers bins 255-8l .. 248-8l (descending key order)
            uint32_t c[8], sum = 0;
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                c[j] = ld_cluster(map_rank(smem_u32(&hist[pass][255 - (lane * 8 + j)]), 0));
                sum += c[j];
            }
            uint32_t incl = sum;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t v = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += v;
            }
            const uint32_t excl = incl - sum;
            const bool hit = excl < static_cast<uint32_t>(krem) && static_cast<uint32_t>(krem) <= incl;
            const uint32_t hb = __ballot_sync(0xffffffffu, hit);
            if (hb == 0u && lane == 0) {  // histogram lost counts: cannot happen with sane data
                set_status(status, KP_ERR_DEVICE_BOUNDS);
                pick[0] = 0;
                pick[1] = 1;
            }
            if (lane == __ffs(hb) - 1) {
                uint32_t above = excl;
                for (int j = 0; j < 8; ++j) {
                    if (above + c[j] >= static_cast<uint32_t>(krem)) {
                        pick[0] = 255 - (lane * 8 + j);
                        pick[1] = krem - static_cast<int>(above);
                        break;
                    }
                    above += c[j];
                }
            }
        }
        __syncthreads();
        prefix |= static_cast<uint32_t>(pick[0]) << shift;
        mask |= 255u << shift;
        krem = pick[1];
        __syncthreads();
    }
    const uint32_t T = prefix;  // the K-th largest key; krem ties of it are taken

    // Per-CTA counts of keys above / equal to the threshold.
    if (tid < 2) cnt[tid] = 0;
    __syncthreads();
    {
        int gt = 0, eq = 0;
        for (int i = tid; i < len; i += kTkThreads) {
            gt += keys[i] > T;
            eq += keys[i] == T;
        }
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) {
            gt += __shfl_xor_sync(0xffffffffu, gt, o);
            eq += __shfl_xor_sync(0xffffffffu, eq, o);
        }
        if (lane == 0) {
            atomicAdd(&cnt[0], gt);
            atomicAdd(&cnt[1], eq);
        }
    }
    cluster_sync_all();
    int out_base = 0, eq_before = 0;
    for (uint32_t r = 0; r < rank; ++r) {
        const int gt_r = static_cast<int>(ld_cluster(map_rank(smem_u32(&cnt[0]), r)));
        const int eq_r = static_cast<int>(ld_cluster(map_rank(smem_u32(&cnt[1]), r)));
        const int take_r = min(max(krem - eq_before, 0), eq_r);
        out_base += gt_r + take_r;
        eq_before += eq_r;
    }
    const int my_take = min(max(krem - eq_before, 0), cnt[1]);

    // Order-preserving compaction of this CTA's slice.
    int sel_carry = 0, eq_carry = 0;
    for (int base = 0; base < len; base += kTkThreads) {
        const int i = base + tid;
        const uint32_t k = i < len ? keys[i] : 0u;
        const bool gt = i < len && k > T;
        const bool eq = i < len && k == T;
        const uint32_t beq = __ballot_sync(0xffffffffu, eq);
        if (lane == 0) wsum[0][warp] = __popc(beq);
        __syncthreads();
        int eq_rank = eq_carry + __popc(beq & lane_lt), eq_tot = 0;
        for (int w = 0; w < kTkThreads / 32; ++w) {
            const int v = wsum[0][w];
            if (w < warp) eq_rank += v;
            eq_tot += v;
        }
        const bool take = gt || (eq && eq_rank < my_take);
        const uint32_t bt = __ballot_sync(0xffffffffu, take);
        if (lane == 0) wsum[1][warp] = __popc(bt);
        __syncthreads();
        int pos = sel_carry + __popc(bt & lane_lt), sel_tot = 0;
        for (int w = 0; w < kTkThreads / 32; ++w) {
            const int v = wsum[1][w];
            if (w < warp) pos += v;
            sel_tot += v;
        }
        if (take && out_base + pos < K) out[out_base + pos] = cs + i;
        eq_carry += eq_tot;
        sel_carry += sel_tot;
        __syncthreads();
    }
    if (rank == 0 && tid == 0) n_sel[q] = K;
    cluster_sync_all();  // keep this CTA's shared memory alive until every peer is done reading it
}

}  // namespace

kp_status launch_topk(const kp_topk_args &a, cudaStream_t s) {
    const int nq = a.q.num_queries;
    if (nq == 0) return KP_OK;
    const int K = a.cfg.topk_tokens / a.cfg.kpool;
    const int maxp = a.q.max_pools;
    int C = 1;
    while (C < kTkMaxCluster && (maxp + C - 1) / C > kTkChunkMax) C *= 2;
    const int chunk_cap = (maxp + C - 1) / C;
    if (chunk_cap > kTkChunkMax) return KP_ERR_UNSUPPORTED;
    const size_t smem = static_cast<size_t>(chunk_cap) * sizeof(uint32_t);
    cudaError_t e = cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kTkChunkMax * static_cast<int>(sizeof(uint32_t)));
    if (e != cudaSuccess) {
        record_cuda_error("cudaFuncSetAttribute(topk_select_kernel)", e);
        return KP_ERR_CUDA;
    }
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(nq) * C);
    cfg.blockDim = dim3(kTkThreads);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    e = cudaLaunchKernelEx(&cfg, topk_select_kernel, a.scores, a.score_stride, a.q.q_pos, K,
                           a.pool_idx, a.n_sel, chunk_cap, a.d_status);
    if (e != cudaSuccess) {
        record_cuda_error("cudaLaunchKernelEx(topk_select_kernel)", e);
        return KP_ERR_CUDA;
    }
    return check_launch("topk_select_kernel");
}

}  // namespace kp
