// topk_select.cuh -- the exact radix select over order-preserving score keys
// held in shared memory, by one CTA or split over the CTAs of a cluster.
// Used by the top-k kernel (keys loaded from a score matrix) and by the fused
// score-and-select kernel (keys written by its own epilogue).
//
// Method: each query keeps its index_topk / kpool best pools (llm-atlas
// GLM-5.3-Flash card, raw config index_topk / index_kpool); ties go to the
// lower pool index; the kept pools are written in ascending order.
#pragma once

#include "kp_common.cuh"

namespace kp {

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
// The caller passes a block barrier before its next call.
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
    // warp_tot is written again only after the caller's next barrier
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


// Selects the K largest keys of a row of n keys and writes their row positions
// in ascending order to out[0 .. K).  The row is split over the C CTAs of a
// cluster (C == 1: one CTA holds it all): this CTA holds keys[0 .. len), row
// positions cs .. cs + len - 1.  kmin / kmax are the calling thread's partial
// key range over its share of keys[].  Every thread of every CTA of the
// cluster calls it, with sh.hist[0] zero and sh.kmin = ~0u, sh.kmax = 0 on
// entry.  The CTA's shared memory stays valid for its peers until it returns.
// kVec reads the keys as 16-byte groups (keys 16-byte aligned and readable up
// to the next multiple of 4 past len; those words are ignored): fewer, wider
// passes, which pay off where one CTA per SM runs the select and its
// latency is exposed; the one-key passes issue fewer instructions, which
// pays off where several CTAs share an SM.
template <int kTkThreads, bool kVec>
__device__ __forceinline__ void radix_select_slice(const uint32_t *keys, int len, int cs, uint32_t C,
                                                   uint32_t rank, int K, int32_t *out, uint32_t kmin,
                                                   uint32_t kmax, TopkShared &sh, int32_t *status) {
    constexpr int kTkWarps = kTkThreads / 32;
    const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
    const uint4 *keys4 = reinterpret_cast<const uint4 *>(keys);
    const int len4 = (len + 3) >> 2;  // 16-byte groups, the last one possibly partial
    auto cbar = [&]() {
        if (C > 1) cluster_barrier();
        else __syncthreads();
    };
    kmin = __reduce_min_sync(0xffffffffu, kmin);
    kmax = __reduce_max_sync(0xffffffffu, kmax);
    __syncthreads();
    if (lane == 0) {
        atomicMin(&sh.kmin, kmin);
        atomicMax(&sh.kmax, kmax);
    }
    cbar();
    // One warp gathers the cluster's key range (every thread reading the same
    // remote words would serialise on them) and broadcasts it.  A CTA that
    // holds the whole row (C == 1) reads its own words: it may be one CTA of a
    // larger cluster, whose rank 0 is another CTA.
    if (C == 1) {
        if (tid == 0) {
            sh.gmin = sh.kmin;
            sh.gmax = sh.kmax;
        }
    } else if (warp == 0) {
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
        if constexpr (kVec) {
        auto bin_add = [&](uint32_t k, bool valid) {
            if (valid && k >= base && static_cast<uint64_t>(k - base) < range) atomicAdd(&hist[(k - base) >> s], 1u);
        };
        for (int i = tid; i < len4; i += 2 * kTkThreads) {  // two 16-byte loads in flight
            const bool has_b = i + kTkThreads < len4;
            const uint4 a = keys4[i];
            const uint4 b = has_b ? keys4[i + kTkThreads] : make_uint4(0u, 0u, 0u, 0u);
            const int ja = 4 * i, jb = 4 * (i + kTkThreads);
            bin_add(a.x, ja < len);
            bin_add(a.y, ja + 1 < len);
            bin_add(a.z, ja + 2 < len);
            bin_add(a.w, ja + 3 < len);
            if (has_b) {
                bin_add(b.x, jb < len);
                bin_add(b.y, jb + 1 < len);
                bin_add(b.z, jb + 2 < len);
                bin_add(b.w, jb + 3 < len);
            }
        }
        } else {
        for (int i = tid; i < len; i += kTkThreads) {
            const uint32_t k = keys[i];
            if (k >= base && static_cast<uint64_t>(k - base) < range) atomicAdd(&hist[(k - base) >> s], 1u);
        }
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
        // pick_* is written again only after the next level's histogram barrier
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
            if constexpr (kVec) {
            auto collect = [&](uint32_t k, bool valid) {
                if (valid && k >= base && static_cast<uint64_t>(k - base) < brange) {
                    const uint32_t slot = atomicAdd(&sh.small_n, 1u);
                    if (slot < static_cast<uint32_t>(kTkSmall)) sh.small[slot] = k;
                }
            };
            for (int i = tid; i < len4; i += kTkThreads) {
                const uint4 v = keys4[i];
                const int j = 4 * i;
                collect(v.x, j < len);
                collect(v.y, j + 1 < len);
                collect(v.z, j + 2 < len);
                collect(v.w, j + 3 < len);
            }
            } else {
            for (int i = tid; i < len; i += kTkThreads) {
                const uint32_t k = keys[i];
                if (k >= base && static_cast<uint64_t>(k - base) < brange) {
                    const uint32_t slot = atomicAdd(&sh.small_n, 1u);
                    if (slot < static_cast<uint32_t>(kTkSmall)) sh.small[slot] = k;
                }
            }
            }
            cbar();  // every CTA's list is complete
            if (warp == 0) {
                uint32_t key = 0u, off = 0u;
                bool has = false;
                for (uint32_t r = 0; r < C; ++r) {
                    const uint32_t nr = min(static_cast<uint32_t>(kTkSmall),
                                            C == 1 ? sh.small_n : ld_cluster_u32(dsmem_addr(smem_u32(&sh.small_n), r)));
                    if (!has && static_cast<uint32_t>(lane) >= off && static_cast<uint32_t>(lane) < off + nr) {
                        key = C == 1 ? sh.small[lane - off]
                                     : ld_cluster_u32(dsmem_addr(smem_u32(&sh.small[lane - off]), r));
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

    // ---- per-warp and per-CTA counts above / equal to T.  Warp w owns the
    // contiguous units w0 .. w1 - 1 (a unit: one key, or with kVec a 16-byte
    // group of four consecutive keys), so lane order is key order.
    const int n_units = kVec ? len4 : len;
    const int wlen = ((n_units + kTkWarps - 1) / kTkWarps + 31) & ~31;  // units per warp
    const int w0 = min(n_units, warp * wlen), w1 = min(n_units, w0 + wlen);
    // masks of the unit's keys above / equal to T (keys past len: neither)
    auto masks = [&](int i, uint32_t &mg, uint32_t &me) {
        if constexpr (kVec) {
            const uint4 v = keys4[i];
            const int j = 4 * i;
            const uint32_t k[4] = {v.x, v.y, v.z, v.w};
            mg = 0u;
            me = 0u;
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const bool valid = j + u < len;
                mg |= static_cast<uint32_t>(valid && k[u] > T) << u;
                me |= static_cast<uint32_t>(valid && k[u] == T) << u;
            }
        } else {
            const uint32_t k = keys[i];
            mg = k > T;
            me = k == T;
        }
    };
    uint32_t gt = 0, eq = 0;
    for (int i = w0 + lane; i < w1; i += 32) {
        uint32_t mg, me;
        masks(i, mg, me);
        gt += __popc(mg);
        eq += __popc(me);
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
    if constexpr (kVec) {
        // the lanes' counts (above in the low half, equal in the high half: at
        // most 4 each) are scanned across the warp in one pass
        for (int i0 = w0; i0 < w1; i0 += 32) {
            const int i = i0 + lane;
            uint32_t mg = 0u, me = 0u;
            if (i < w1) masks(i, mg, me);
            const uint32_t cnt = static_cast<uint32_t>(__popc(mg)) | (static_cast<uint32_t>(__popc(me)) << 16);
            uint32_t incl = cnt;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const uint32_t nb = __shfl_up_sync(0xffffffffu, incl, o);
                if (lane >= o) incl += nb;
            }
            const uint32_t tot = __shfl_sync(0xffffffffu, incl, 31);
            const uint32_t excl = incl - cnt;
            uint32_t g_b = gt_run + (excl & 0xffffu), e_b = eq_run + (excl >> 16);
#pragma unroll
            for (int u = 0; u < 4; ++u) {
                const bool isgt = (mg >> u) & 1u, iseq = (me >> u) & 1u;
                if (isgt || (iseq && e_b < my_take)) {
                    const uint32_t pos = out_base + g_b + min(e_b, my_take);
                    if (pos < static_cast<uint32_t>(K)) out[pos] = cs + 4 * i + u;
                }
                g_b += isgt;
                e_b += iseq;
            }
            gt_run += tot & 0xffffu;
            eq_run += tot >> 16;
        }
    } else {
        const uint32_t lane_lt = (1u << lane) - 1u;
        for (int i0 = w0; i0 < w1; i0 += 32) {
            const int i = i0 + lane;
            uint32_t mg = 0u, me = 0u;
            if (i < w1) masks(i, mg, me);
            const bool isgt = mg != 0u, iseq = me != 0u;
            const uint32_t bgt = __ballot_sync(0xffffffffu, isgt), beq = __ballot_sync(0xffffffffu, iseq);
            const uint32_t eq_b = eq_run + __popc(beq & lane_lt);
            if (isgt || (iseq && eq_b < my_take)) {
                const uint32_t pos = out_base + gt_run + __popc(bgt & lane_lt) + min(eq_b, my_take);
                if (pos < static_cast<uint32_t>(K)) out[pos] = cs + i;
            }
            gt_run += __popc(bgt);
            eq_run += __popc(beq);
        }
    }
    cbar();  // keep this CTA's shared memory alive until every peer is done reading it
}

}  // namespace kp
