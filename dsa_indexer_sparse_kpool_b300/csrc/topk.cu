// topk.cu -- top-k pool selection: one histogram pass, exact resolution of
// the threshold bin, order-preserving compaction.
//
// Method: each query keeps index_topk / kpool pools (2048 tokens / 4 = 512;
// llm-atlas GLM-5.3-Flash card, raw config index_topk / index_kpool); when it
// sees no more complete pools than that, it keeps them all.  Ties go to the
// lower pool index and the kept pools are written in ascending order.
//
// B300 design.  A query's row of n = n_full(t) scores is split over a
// thread-block cluster of C CTAs (C = 1 up to 16K pools; up to 8 for the
// 262,143-pool rows of a 1M-token context), each holding its slice as
// order-preserving uint32 keys.
//  1. The cluster's smallest and largest keys fix up to 2048 bins of equal
//     width (a power of two) in key space (monotone, so the K-th largest key
//     lies in exactly one bin, B).  One histogram pass, summed into the leader CTA through
//     distributed shared memory, gives B and how many of its keys are needed.
//  2. The keys of bin B (typically a few dozen) are gathered into the
//     leader, sorted (key descending, index ascending) and give the exact
//     threshold key T and how many keys equal to T are taken.  If bin B holds
//     more than 4096 keys (heavy ties), 8-bit radix passes restricted to bin B
//     find T instead.
//  3. Every CTA counts its keys above / equal to T; one packed block scan
//     turns the counts into output positions, so the selected pools are
//     written in ascending order with no sort.
// Cluster barriers are hardware barriers (all CTAs of a cluster are
// co-resident): no spin loop anywhere.
#include "kp_common.cuh"
#include "kp_internal.h"

namespace kp {

namespace {

constexpr int kTkThreads = 512;
constexpr int kTkChunkMax = 32768;  // keys per CTA (128 KB of shared memory)
constexpr int kTkMaxCluster = 8;
constexpr int kTkBins = 2048;
constexpr int kTkCandMax = 4096;
constexpr int kTkKeysPerCta = 16384;  // preferred largest slice per CTA

__device__ __forceinline__ uint32_t cluster_size() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_nctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void red_add_cluster(uint32_t addr, uint32_t v) {
    asm volatile("red.shared::cluster.add.u32 [%0], %1;" ::"r"(addr), "r"(v) : "memory");
}
__device__ __forceinline__ uint32_t atom_add_cluster(uint32_t addr, uint32_t v) {
    uint32_t old;
    asm volatile("atom.shared::cluster.add.u32 %0, [%1], %2;" : "=r"(old) : "r"(addr), "r"(v) : "memory");
    return old;
}
__device__ __forceinline__ uint32_t ld_cluster_u32(uint32_t addr) {
    uint32_t v;
    asm volatile("ld.shared::cluster.u32 %0, [%1];" : "=r"(v) : "r"(addr) : "memory");
    return v;
}
__device__ __forceinline__ void st_cluster_u64(uint32_t addr, uint64_t v) {
    asm volatile("st.shared::cluster.u64 [%0], %1;" ::"r"(addr), "l"(v) : "memory");
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
    uint32_t hist[kTkBins];           // leader: cluster totals
    uint64_t cand[kTkCandMax];        // leader: (key << 32) | ~index of bin-B keys
    uint32_t warp_tot[32];
    uint32_t kmin, kmax;              // this CTA's key range
    uint32_t n_cand;                  // leader: candidates gathered
    uint32_t thr_key, eq_take;        // leader: threshold key and how many of its ties to take
    uint32_t cnt_gt, cnt_eq;          // this CTA's keys above / equal to the threshold
    int pick_bin, pick_need;
};

__global__ void __launch_bounds__(kTkThreads, 1)
    topk_select_kernel(const float *__restrict__ scores, int64_t stride,
                       const int32_t *__restrict__ q_pos, int K, int32_t *__restrict__ pool_idx,
                       int32_t *__restrict__ n_sel, int chunk_cap, int32_t *status) {
    extern __shared__ uint32_t keys[];
    __shared__ TopkShared sh;

    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    pdl_wait_then_release();
    const uint32_t rank = cluster_ctarank(), C = cluster_size();
    const int q = blockIdx.x / C;
    // A one-CTA row needs only block barriers.
    auto cbar = [&]() {
        if (C > 1) cluster_barrier();
        else __syncthreads();
    };
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

    // ---- keys, key range
    const float *row = scores + static_cast<int64_t>(q) * stride + cs;
    uint32_t kmin = 0xffffffffu, kmax = 0u;
    if ((reinterpret_cast<uintptr_t>(row) & 15) == 0) {
        const int n4 = len >> 2;
        for (int i = tid; i < n4; i += kTkThreads) {
            const float4 v = __ldcs(reinterpret_cast<const float4 *>(row) + i);
            const uint32_t a = score_key(v.x), b = score_key(v.y), c = score_key(v.z), d = score_key(v.w);
            reinterpret_cast<uint4 *>(keys)[i] = make_uint4(a, b, c, d);
            kmin = min(kmin, min(min(a, b), min(c, d)));
            kmax = max(kmax, max(max(a, b), max(c, d)));
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
    if (tid == 0) {
        sh.kmin = 0xffffffffu;
        sh.kmax = 0u;
        sh.n_cand = 0u;
    }
    for (int i = tid; i < kTkBins; i += kTkThreads) sh.hist[i] = 0u;
    __syncthreads();
    if (lane == 0) {
        atomicMin(&sh.kmin, kmin);
        atomicMax(&sh.kmax, kmax);
    }
    cbar();
    uint32_t gmin = 0xffffffffu, gmax = 0u;
    for (uint32_t r = 0; r < C; ++r) {
        gmin = min(gmin, ld_cluster_u32(dsmem_addr(smem_u32(&sh.kmin), r)));
        gmax = max(gmax, ld_cluster_u32(dsmem_addr(smem_u32(&sh.kmax), r)));
    }
    // bin(k) = (k - gmin) >> sh with the smallest sh that maps the key span into
    // 2048 bins: monotone in k, one shift per key.
    const uint64_t span = static_cast<uint64_t>(gmax) - gmin + 1;
    int bsh = 0;
    while ((span - 1) >> bsh >= static_cast<uint64_t>(kTkBins)) ++bsh;
    auto bin_of = [&](uint32_t k) -> uint32_t { return (k - gmin) >> bsh; };

    // ---- histogram into the leader
    {
        // Private per-CTA histogram first (in this CTA's own hist, zeroed above),
        // then one remote add per non-empty bin.
        for (int i = tid; i < len; i += kTkThreads) atomicAdd(&sh.hist[bin_of(keys[i])], 1u);
        __syncthreads();
        if (rank != 0) {
            for (int i = tid; i < kTkBins; i += kTkThreads) {
                const uint32_t v = sh.hist[i];
                if (v) red_add_cluster(dsmem_addr(smem_u32(&sh.hist[i]), 0), v);
            }
        }
    }
    cbar();

    // ---- threshold bin: the K-th largest key lies in bin B
    if (rank != 0) {  // local copy of the cluster totals
        for (int i = tid; i < kTkBins; i += kTkThreads) sh.hist[i] = ld_cluster_u32(dsmem_addr(smem_u32(&sh.hist[i]), 0));
    }
    __syncthreads();
    {
        // Thread i holds bins 2047-4i .. 2044-4i (descending); one block scan
        // gives the count above its group, and the group containing the K-th
        // largest key names B.
        constexpr int kPer = kTkBins / kTkThreads;
        uint32_t c[kPer], sum = 0;
#pragma unroll
        for (int j = 0; j < kPer; ++j) {
            c[j] = sh.hist[kTkBins - 1 - (tid * kPer + j)];
            sum += c[j];
        }
        uint32_t tot;
        uint32_t above = block_excl_scan(sum, sh.warp_tot, &tot);
        if (tid == 0 && tot < static_cast<uint32_t>(K)) {  // counts lost: cannot happen with consistent data
            set_status(status, KP_ERR_DEVICE_BOUNDS);
            sh.pick_bin = kTkBins - 1;
            sh.pick_need = 1;
        }
        if (above < static_cast<uint32_t>(K) && static_cast<uint32_t>(K) <= above + sum) {
#pragma unroll
            for (int j = 0; j < kPer; ++j) {
                if (above < static_cast<uint32_t>(K) && above + c[j] >= static_cast<uint32_t>(K)) {
                    sh.pick_bin = kTkBins - 1 - (tid * kPer + j);
                    sh.pick_need = K - static_cast<int>(above);
                }
                above += c[j];
            }
        }
    }
    __syncthreads();
    const uint32_t B = static_cast<uint32_t>(sh.pick_bin);
    const int need = sh.pick_need;
    const uint32_t cnt_b = sh.hist[B];

    uint32_t T;         // threshold key
    uint32_t eq_take;   // keys equal to T that are taken (lowest indices first)
    if (cnt_b <= static_cast<uint32_t>(kTkCandMax)) {
        // ---- gather bin B into the leader, sort, read off T
        const uint32_t cnt_addr = dsmem_addr(smem_u32(&sh.n_cand), 0);
        const uint32_t cand_addr = dsmem_addr(smem_u32(&sh.cand[0]), 0);
        for (int base = 0; base < len; base += kTkThreads) {
            const int i = base + tid;
            const bool m = i < len && bin_of(keys[i]) == B;
            const uint32_t bal = __ballot_sync(0xffffffffu, m);
            if (bal) {
                uint32_t slot0 = 0;
                if (lane == __ffs(bal) - 1) slot0 = atom_add_cluster(cnt_addr, __popc(bal));
                slot0 = __shfl_sync(0xffffffffu, slot0, __ffs(bal) - 1);
                if (m) {
                    const uint32_t slot = slot0 + __popc(bal & ((1u << lane) - 1u));
                    const uint64_t v = (static_cast<uint64_t>(keys[i]) << 32) |
                                       static_cast<uint32_t>(~static_cast<uint32_t>(cs + i));
                    if (slot < static_cast<uint32_t>(kTkCandMax)) st_cluster_u64(cand_addr + 8u * slot, v);
                }
            }
        }
        cbar();
        if (rank == 0) {
            const int m = static_cast<int>(min(sh.n_cand, static_cast<uint32_t>(kTkCandMax)));
            const bool need_ok = need >= 1 && need <= m;
            if (!need_ok && tid == 0) set_status(status, KP_ERR_DEVICE_BOUNDS);
            const int nd = need_ok ? need : (m > 0 ? m : 1);
            if (m <= kTkThreads) {
                // Rank every candidate against all others (values are distinct: the
                // low half holds the inverted index); the one of rank nd-1 is T.
                uint64_t v = 0;
                int rk = m;
                if (tid < m) {
                    v = sh.cand[tid];
                    rk = 0;
                    for (int j = 0; j < m; ++j) rk += sh.cand[j] > v;
                    if (rk == nd - 1) sh.thr_key = static_cast<uint32_t>(v >> 32);
                }
                __syncthreads();
                const uint32_t tk = sh.thr_key;
                const int e = __syncthreads_count(tid < m && rk < nd && static_cast<uint32_t>(v >> 32) == tk);
                if (tid == 0) sh.eq_take = static_cast<uint32_t>(e);
            } else {
                int m2 = 1;
                while (m2 < m) m2 <<= 1;
                for (int i = m + tid; i < m2; i += kTkThreads) sh.cand[i] = 0ull;  // sorts last
                __syncthreads();
                // bitonic sort, descending
                for (int kk = 2; kk <= m2; kk <<= 1) {
                    for (int j = kk >> 1; j > 0; j >>= 1) {
                        for (int i = tid; i < (m2 >> 1); i += kTkThreads) {
                            const int lo = 2 * i - (i & (j - 1));
                            const int hi = lo + j;
                            const bool desc = (lo & kk) == 0;
                            const uint64_t a = sh.cand[lo], b = sh.cand[hi];
                            if ((a < b) == desc) {
                                sh.cand[lo] = b;
                                sh.cand[hi] = a;
                            }
                        }
                        __syncthreads();
                    }
                }
                if (tid == 0) {
                    const uint32_t tk = static_cast<uint32_t>(sh.cand[nd - 1] >> 32);
                    uint32_t e = 0;
                    for (int j = nd - 1; j >= 0 && static_cast<uint32_t>(sh.cand[j] >> 32) == tk; --j) ++e;
                    sh.thr_key = tk;
                    sh.eq_take = e;
                }
            }
        }
        cbar();
        T = ld_cluster_u32(dsmem_addr(smem_u32(&sh.thr_key), 0));
        eq_take = ld_cluster_u32(dsmem_addr(smem_u32(&sh.eq_take), 0));
    } else {
        // ---- heavy ties: 8-bit radix passes over the keys of bin B
        uint32_t prefix = 0, mask = 0;
        int krem = need;
        for (int pass = 0; pass < 4; ++pass) {
            const int shift = 24 - 8 * pass;
            cbar();  // every CTA is done reading the leader's previous totals
            for (int i = tid; i < 256; i += kTkThreads) sh.hist[i] = 0u;
            cbar();  // ... and every histogram is cleared
            for (int i = tid; i < len; i += kTkThreads) {
                const uint32_t k = keys[i];
                if (bin_of(k) == B && (k & mask) == prefix) atomicAdd(&sh.hist[(k >> shift) & 255u], 1u);
            }
            __syncthreads();
            if (rank != 0 && tid < 256 && sh.hist[tid]) red_add_cluster(dsmem_addr(smem_u32(&sh.hist[tid]), 0), sh.hist[tid]);
            cbar();
            if (warp == 0) {
                uint32_t c[8], sum = 0;
#pragma unroll
                for (int j = 0; j < 8; ++j) {
                    c[j] = ld_cluster_u32(dsmem_addr(smem_u32(&sh.hist[255 - (lane * 8 + j)]), 0));
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
                if (hb == 0u && lane == 0) {
                    set_status(status, KP_ERR_DEVICE_BOUNDS);
                    sh.pick_bin = 0;
                    sh.pick_need = 1;
                }
                if (lane == __ffs(hb) - 1) {
                    uint32_t above = excl;
                    for (int j = 0; j < 8; ++j) {
                        if (above + c[j] >= static_cast<uint32_t>(krem)) {
                            sh.pick_bin = 255 - (lane * 8 + j);
                            sh.pick_need = krem - static_cast<int>(above);
                            break;
                        }
                        above += c[j];
                    }
                }
            }
            __syncthreads();
            prefix |= static_cast<uint32_t>(sh.pick_bin) << shift;
            mask |= 255u << shift;
            krem = sh.pick_need;
            __syncthreads();
        }
        T = prefix;
        eq_take = static_cast<uint32_t>(krem);
    }

    // ---- per-CTA counts above / equal to T, output offsets
    if (tid == 0) {
        sh.cnt_gt = 0u;
        sh.cnt_eq = 0u;
    }
    __syncthreads();
    const int per = (len + kTkThreads - 1) / kTkThreads;
    const int i0 = min(len, tid * per), i1 = min(len, i0 + per);
    uint32_t gt = 0, eq = 0;
    for (int i = i0; i < i1; ++i) {
        gt += keys[i] > T;
        eq += keys[i] == T;
    }
    {
        const uint32_t g = __reduce_add_sync(0xffffffffu, gt), e = __reduce_add_sync(0xffffffffu, eq);
        if (lane == 0) {
            atomicAdd(&sh.cnt_gt, g);
            atomicAdd(&sh.cnt_eq, e);
        }
    }
    cbar();
    uint32_t out_base = 0, eq_before = 0;
    for (uint32_t r = 0; r < rank; ++r) {
        const uint32_t gt_r = ld_cluster_u32(dsmem_addr(smem_u32(&sh.cnt_gt), r));
        const uint32_t eq_r = ld_cluster_u32(dsmem_addr(smem_u32(&sh.cnt_eq), r));
        const uint32_t rem = eq_take > eq_before ? eq_take - eq_before : 0u;
        out_base += gt_r + min(rem, eq_r);
        eq_before += eq_r;
    }
    const uint32_t my_take = min(eq_take > eq_before ? eq_take - eq_before : 0u, sh.cnt_eq);

    // ---- order-preserving compaction: one packed scan (ties in the high half)
    uint32_t tot;
    const uint32_t pre = block_excl_scan((eq << 16) | gt, sh.warp_tot, &tot);
    uint32_t gt_pre = pre & 0xffffu, eq_pre = pre >> 16;
    for (int i = i0; i < i1; ++i) {
        const uint32_t k = keys[i];
        if (k > T) {
            const uint32_t pos = out_base + gt_pre + min(eq_pre, my_take);
            if (pos < static_cast<uint32_t>(K)) out[pos] = cs + i;
            ++gt_pre;
        } else if (k == T) {
            if (eq_pre < my_take) {
                const uint32_t pos = out_base + gt_pre + eq_pre;
                if (pos < static_cast<uint32_t>(K)) out[pos] = cs + i;
            }
            ++eq_pre;
        }
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
    const int sms = device_sm_count();
    if (sms <= 0) return KP_ERR_CUDA;
    // Enough CTAs per row to hold it in shared memory; more (up to 8) while the
    // grid is smaller than the GPU and every CTA keeps >= 2048 keys.
    // A row is latency-bound work: one CTA per row while it fits comfortably,
    // a cluster only for long rows (up to 8 CTAs of <= 32768 keys).
    int C = 1;
    while (C < kTkMaxCluster && (maxp + C - 1) / C > kTkKeysPerCta) C *= 2;
    const int chunk_cap = (maxp + C - 1) / C;
    if (chunk_cap > kTkChunkMax) return KP_ERR_UNSUPPORTED;
    if (static_cast<int64_t>(chunk_cap) + 16 >= 65536) return KP_ERR_UNSUPPORTED;  // packed 16-bit scan
    const size_t smem = static_cast<size_t>(chunk_cap > 0 ? chunk_cap : 1) * sizeof(uint32_t);
    cudaError_t e = cudaFuncSetAttribute(topk_select_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kTkChunkMax * static_cast<int>(sizeof(uint32_t)));
    if (e != cudaSuccess) {
        record_cuda_error("cudaFuncSetAttribute(topk_select_kernel)", e);
        return KP_ERR_CUDA;
    }
    return launch_kernel("topk_select_kernel", topk_select_kernel,
                         LaunchCfg(dim3(static_cast<unsigned>(nq) * C), dim3(kTkThreads), smem, s, C), a.scores,
                         a.score_stride, a.q.q_pos, K, a.pool_idx, a.n_sel, chunk_cap, a.d_status);
}

}  // namespace kp
