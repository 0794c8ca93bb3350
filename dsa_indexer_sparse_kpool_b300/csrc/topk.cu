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
#include "topk_select.cuh"

namespace kp {

namespace {

template <int kTkThreads>
__global__ void __launch_bounds__(kTkThreads, 1)
    topk_select_kernel(const float *__restrict__ scores, int64_t stride,
                       const int32_t *__restrict__ q_pos, const int32_t *__restrict__ share, int kshift, int K,
                       int32_t *__restrict__ pool_idx, int32_t *__restrict__ n_sel, int chunk_cap, int32_t *status) {
    extern __shared__ __align__(16) uint32_t keys[];
    __shared__ __align__(16) TopkShared sh;

    const int tid = threadIdx.x;
    const uint32_t rank = cluster_ctarank(), C = cluster_size();
    const int q = blockIdx.x / C;
    if (share && share[q] >= 0) {  // a shared query: its row is left as it was (every CTA of its cluster)
        pdl_wait_then_release();
        return;
    }
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
    radix_select_slice<kTkThreads, false>(keys, len, cs, C, rank, K, out, kmin, kmax, sh, status);
    if (rank == 0 && tid == 0) n_sel[q] = K;
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
                         a.scores, a.score_stride, a.q.q_pos, a.q.share_src, kpool_shift(a.cfg.kpool), K, a.pool_idx,
                         a.n_sel,
                         chunk_cap, a.d_status);
}

}  // namespace kp
