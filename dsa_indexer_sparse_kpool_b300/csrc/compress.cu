// compress.cu -- pooled-key compression fused into the indexer-cache write.
//
// Method: MAX docs (max.pipelines.architectures.glm5_next), Glm5NextConfig
// index_kpool / index_kpool_compress: a pooled key is a learned weighted
// average of the pool's kpool tokens, the weights coming from per-token gate
// logits plus a learned intra-pool position embedding (ape); the softmax runs
// over the kpool positions separately for each of the 128 dimensions (the
// [4, 128, n_pool] pooling softmax of the llama.cpp PR "add GLM-5.3-Flash
// (GLM5-Next) support").  Mean mode uses equal weights.
//
// B300 design: instead of re-pooling every pool from a per-token key|gate
// cache each step (the llama.cpp graph), only pools completed by this step's
// new tokens are computed, straight from the new rows plus a tiny per-sequence
// tail ring holding the rows of the still-incomplete pool.  One warp per
// completed pool, each lane owning 4 of the 128 dimensions (8-byte loads and
// stores, fp32 math, bf16 round-to-nearest-even store).  Pools sit on
// gridDim.x, sequences on gridDim.y: no launch dimension scales with the
// number of pools beyond gridDim.x's 2^31 limit.
//
// The pooled row of a pool comes from the sequence's row offset, or from its
// block table when the caches are paged.
//
// Ring ownership: for sequence b, item 0 (the warp of the first pool touched)
// is the only reader of the old ring rows AND the only writer of the new
// ring rows; it reads before it writes, so no other warp can race with it.
#include "kp_common.cuh"
#include "kp_internal.h"
#include "score_plan.cuh"

namespace kp {

namespace {

constexpr int kCompressWarps = 4;

struct Row4 {
    float v[4];
};

__device__ __forceinline__ Row4 load_bf16x4(const uint16_t *p) {
    uint2 raw = *reinterpret_cast<const uint2 *>(p);
    Row4 r;
    r.v[0] = __uint_as_float(raw.x << 16);
    r.v[1] = __uint_as_float(raw.x & 0xffff0000u);
    r.v[2] = __uint_as_float(raw.y << 16);
    r.v[3] = __uint_as_float(raw.y & 0xffff0000u);
    return r;
}

template <int KP>
__global__ void __launch_bounds__(kCompressWarps * 32)
    kpool_compress_kernel(int32_t mode, const int32_t *__restrict__ prev_len,
                          const int32_t *__restrict__ new_off, const uint16_t *__restrict__ keys,
                          const uint16_t *__restrict__ gates, const uint16_t *__restrict__ ape,
                          uint16_t *__restrict__ tail_keys, uint16_t *__restrict__ tail_gates,
                          uint16_t *__restrict__ pooled, CacheMap cmap, int32_t *status, ScorePlanArgs plan) {
    constexpr int R = KP - 1;  // ring slots per sequence
    __shared__ int scratch[33];
    pdl_wait_then_release();
    if (plan.plan && blockIdx.y == gridDim.y - 1) {  // the extra row of CTAs: the scorer's plan
        if (blockIdx.x == 0)
            build_score_plan(plan.nq, plan.num_seqs, plan.q_seq, plan.q_pos, plan.seq_len, plan.kshift,
                             plan.max_tiles, plan.plan, plan.status, scratch, plan.max_q);
        return;
    }
    const int b = blockIdx.y;
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int item = blockIdx.x * kCompressWarps + warp;
    const int prev = prev_len[b];
    const int n0 = new_off[b];
    const int n_new = new_off[b + 1] - n0;
    if (n_new <= 0 || prev < 0) return;
    const int len = prev + n_new;
    const int p_first = prev / KP;             // first pool touched
    const int n_complete = len / KP - p_first;  // pools completed by this step
    const int n_items = n_complete > 0 ? n_complete : 1;
    if (item >= n_items) return;
    const int d0 = lane * 4;

    if (item < n_complete) {
        const int p = p_first + item;
        Row4 k[KP], g[KP];
#pragma unroll
        for (int i = 0; i < KP; ++i) {
            const int pos = p * KP + i;
            const uint16_t *ksrc, *gsrc;
            if (pos < prev) {  // only possible for item 0: row held in the ring
                const size_t off = (static_cast<size_t>(b) * R + (pos % KP)) * kIndexDim + d0;
                ksrc = tail_keys + off;
                gsrc = tail_gates + off;
            } else {
                const size_t off = static_cast<size_t>(n0 + pos - prev) * kIndexDim + d0;
                ksrc = keys + off;
                gsrc = gates + off;
            }
            k[i] = load_bf16x4(ksrc);
            if (mode == KP_COMPRESS_LEARNED) g[i] = load_bf16x4(gsrc);
        }
        float out[4];
        if (mode == KP_COMPRESS_LEARNED) {
#pragma unroll
            for (int i = 0; i < KP; ++i) {
                Row4 a = load_bf16x4(ape + i * kIndexDim + d0);
#pragma unroll
                for (int j = 0; j < 4; ++j) g[i].v[j] += a.v[j];
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float m = g[0].v[j];
#pragma unroll
                for (int i = 1; i < KP; ++i) m = fmaxf(m, g[i].v[j]);
                float den = 0.f, num = 0.f;
#pragma unroll
                for (int i = 0; i < KP; ++i) {
                    const float e = expf(g[i].v[j] - m);
                    den += e;
                    num += e * k[i].v[j];
                }
                out[j] = num / den;
            }
        } else {
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                float s = 0.f;
#pragma unroll
                for (int i = 0; i < KP; ++i) s += k[i].v[j];
                out[j] = s * (1.0f / KP);
            }
        }
        const int64_t row = cmap.pool_row(b, p);
        if (row < 0) {
            if (lane == 0) set_status(status, KP_ERR_DEVICE_BOUNDS);
        } else {
            uint2 packed;
            packed.x = pack_bf16x2(out[0], out[1]);
            packed.y = pack_bf16x2(out[2], out[3]);
            *reinterpret_cast<uint2 *>(pooled + row * kIndexDim + d0) = packed;
        }
    }

    if (item == 0) {
        // Rows of the pool left incomplete go to the ring (slot = position % kpool).
        // This warp already holds the old ring rows it needed in registers.
        __syncwarp();
        const int tail_start = (len / KP) * KP;
        for (int pos = max(prev, tail_start); pos < len; ++pos) {
            const size_t src = static_cast<size_t>(n0 + pos - prev) * kIndexDim + d0;
            const size_t dst = (static_cast<size_t>(b) * R + (pos % KP)) * kIndexDim + d0;
            *reinterpret_cast<uint2 *>(tail_keys + dst) = *reinterpret_cast<const uint2 *>(keys + src);
            if (mode == KP_COMPRESS_LEARNED)
                *reinterpret_cast<uint2 *>(tail_gates + dst) =
                    *reinterpret_cast<const uint2 *>(gates + src);
        }
    }
}

}  // namespace

kp_status launch_compress(const kp_compress_args &a, cudaStream_t s, const ScorePlanArgs *plan) {
    if (a.num_new == 0) return KP_OK;
    const int kp = a.cfg.kpool;
    const int max_items = (a.max_new_per_seq + kp - 1) / kp + 1;
    ScorePlanArgs pa{};
    if (plan) pa = *plan;
    dim3 grid((max_items + kCompressWarps - 1) / kCompressWarps, a.num_seqs + (pa.plan ? 1 : 0));
    return launch_kernel("kpool_compress_kernel", kp == 16 ? kpool_compress_kernel<16> : kpool_compress_kernel<4>,
                         LaunchCfg(grid, dim3(kCompressWarps * 32), 0, s), a.cfg.compress_mode, a.prev_len,
                         a.new_off, a.keys, a.gates, a.ape, a.tail_keys, a.tail_gates, a.pooled,
                         cache_map(a.seqs, kp),
                         a.d_status, pa);
}

}  // namespace kp
