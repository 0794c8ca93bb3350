// attend.cu -- nope-only sparse MLA in latent space over the selected pools.
//
// Method (MAX docs, max.pipelines.architectures.glm5_next: Glm5NextConfig
// mla_use_nope -- no rotary embedding anywhere in the text decoder;
// Glm5Next.build_layers -- the 576-wide latent row carries 64 rotary columns
// that are all zero; index_kpool_always_select_tail -- the incomplete
// trailing pool is always visible): the token set of a query is the kpool
// rows of every selected pool plus its tail; for each of the 64 heads
//   out_h = softmax_s(scale * q_lat_h . c_s) . c_s[:512],  lse_h = ln sum exp
// with q_lat the absorbed query (latent space) and c the latent cache rows.
// Only the 512 latent columns are read: the 64 rotary columns are zero by
// the cache's contract, so they add nothing to the logits.
//
// Design (first version, legacy tensor-core path): one CTA = one query x one
// split of its token list.  64-token tiles of latent rows are gathered with
// cp.async (16 B chunks, XOR-swizzled rows) into a double-buffered ring;
// 8 warps = 4 head groups (16 heads) x 2 halves of the 512 latent columns.
// QK^T partial sums over each half are exchanged through shared memory,
// online softmax in registers, P.V with the P fragments reused from the QK
// accumulators.  Splits of one query write (o, lse) partials; the last CTA
// to finish (atomic ticket, no waiting) merges them.
#include "kp_common.cuh"
#include "kp_internal.h"

namespace kp {

namespace {

constexpr int kAtTile = 64;
constexpr int kAtThreads = 256;
constexpr int kAtRowBytes = kNopeDim * 2;             // 1024
constexpr int kAtQBytes = kMlaHeads * kAtRowBytes;    // 64 KB
constexpr int kAtKVBytes = kAtTile * kAtRowBytes;     // 64 KB per stage
constexpr int kAtXBytes = 8 * 32 * 32 * 4;            // QK partial exchange, 32 KB
constexpr int kAtRowsBytes = 2 * kAtTile * 8;
constexpr int kAtSmemBytes = kAtQBytes + 2 * kAtKVBytes + kAtXBytes + kAtRowsBytes;
constexpr float kLn2 = 0.69314718055994530942f;
constexpr float kLog2e = 1.44269504088896340736f;

struct AttendParams {
    const uint16_t *q_lat;
    const uint16_t *latent;
    int64_t latent_rows;
    const int32_t *q_seq;
    const int32_t *q_pos;
    const int64_t *latent_row_off;
    int num_seqs;
    const int32_t *pool_idx;
    const int32_t *n_sel;
    int K;
    int tail;
    float scale_log2;
    uint16_t *out;
    float *lse;
    float *ws_o;
    float *ws_lse;
    int32_t *ws_cnt;
    int splits;
    int32_t *status;
};

__device__ __forceinline__ uint32_t swz(int row, int chunk) {
    return static_cast<uint32_t>(row * kAtRowBytes + ((chunk ^ (row & 7)) << 4));
}

__device__ __forceinline__ void named_bar(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}

__global__ void __launch_bounds__(kAtThreads, 1) sparse_mla_mma_kernel(AttendParams P) {
    extern __shared__ __align__(128) uint8_t sm[];
    __shared__ int s_last;
    uint8_t *sQ = sm;
    uint8_t *sKV = sm + kAtQBytes;
    float *sX = reinterpret_cast<float *>(sm + kAtQBytes + 2 * kAtKVBytes);
    int64_t *sRows = reinterpret_cast<int64_t *>(sm + kAtQBytes + 2 * kAtKVBytes + kAtXBytes);

    const int q = blockIdx.x / P.splits, split = blockIdx.x % P.splits;
    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int hg = warp & 3, dh = warp >> 2;
    const int g = lane >> 2, c4 = lane & 3, mi = lane >> 3, rr = lane & 7;

    const int b = P.q_seq[q];
    const int t = P.q_pos[q];
    int n_tok = 0, ns = 0, nf = 0;
    int64_t base_row = 0;
    if (b < 0 || b >= P.num_seqs || t < 0) {
        if (tid == 0) set_status(P.status, KP_ERR_DEVICE_BOUNDS);
    } else {
        nf = (t + 1) / kKpool;
        ns = P.n_sel[q];
        const int ns_max = min(P.K, nf);
        if (ns < 0 || ns > ns_max) {
            if (tid == 0) set_status(P.status, KP_ERR_DEVICE_BOUNDS);
            ns = max(0, min(ns, ns_max));
        }
        const int tail = P.tail ? (t + 1) - nf * kKpool : 0;
        n_tok = ns * kKpool + tail;
        base_row = P.latent_row_off[b];
    }
    const int n_tiles = (n_tok + kAtTile - 1) / kAtTile;
    const int tb = n_tiles * split / P.splits, te = n_tiles * (split + 1) / P.splits;

    // Q: 64 heads x 512 columns (the rotary columns 512..575 are never read).
    for (int i = tid; i < kMlaHeads * 64; i += kAtThreads) {
        const int h = i >> 6, c = i & 63;
        cp_async_16(smem_u32(sQ) + swz(h, c),
                    P.q_lat + (static_cast<int64_t>(q) * kMlaHeads + h) * kLatentDim + c * 8, 16);
    }
    cp_async_commit();

    auto compute_rows = [&](int k, int slot) {
        if (tid < kAtTile) {
            const int i = k * kAtTile + tid;
            int64_t row = -1;
            if (i < n_tok) {
                if (i < ns * kKpool) {
                    const int p = P.pool_idx[static_cast<int64_t>(q) * P.K + i / kKpool];
                    if (p >= 0 && p < nf) row = base_row + static_cast<int64_t>(p) * kKpool + (i % kKpool);
                    else set_status(P.status, KP_ERR_DEVICE_BOUNDS);
                } else {
                    row = base_row + static_cast<int64_t>(nf) * kKpool + (i - ns * kKpool);
                }
                if (row >= P.latent_rows) {
                    set_status(P.status, KP_ERR_DEVICE_BOUNDS);
                    row = -1;
                }
            }
            sRows[slot * kAtTile + tid] = row;
        }
    };
    auto issue_tile = [&](int slot) {
        const int c = tid & 63, r0 = tid >> 6;
        const uint32_t dst0 = smem_u32(sKV + slot * kAtKVBytes);
#pragma unroll
        for (int j = 0; j < kAtTile / 4; ++j) {
            const int r = r0 + 4 * j;
            const int64_t row = sRows[slot * kAtTile + r];
            const uint16_t *src = P.latent + (row < 0 ? 0 : row) * kLatentDim + c * 8;
            cp_async_16(dst0 + swz(r, c), src, row < 0 ? 0u : 16u);
        }
    };

    float O[32][4];
#pragma unroll
    for (int i = 0; i < 32; ++i) O[i][0] = O[i][1] = O[i][2] = O[i][3] = 0.f;
    float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};

    if (tb < te) {
        compute_rows(tb, 0);
        __syncthreads();
        issue_tile(0);
        cp_async_commit();
    }
    for (int k = tb; k < te; ++k) {
        const int slot = (k - tb) & 1;
        if (k + 1 < te) {
            compute_rows(k + 1, slot ^ 1);
            __syncthreads();
            issue_tile(slot ^ 1);
            cp_async_commit();
            cp_async_wait<1>();
        } else {
            cp_async_wait<0>();
        }
        __syncthreads();
        const uint32_t kv = smem_u32(sKV + slot * kAtKVBytes);
        const uint32_t qs = smem_u32(sQ);

        // S_partial[16 heads x 64 tokens] over this warp's 256 latent columns.
        float S[8][4];
#pragma unroll
        for (int i = 0; i < 8; ++i) S[i][0] = S[i][1] = S[i][2] = S[i][3] = 0.f;
#pragma unroll 4
        for (int ks = 0; ks < 16; ++ks) {
            const int kc = dh * 32 + ks * 2;
            uint32_t a0, a1, a2, a3;
            const int arow = 16 * hg + rr + 8 * (mi & 1);
            ldsm_x4(qs + swz(arow, kc + (mi >> 1)), a0, a1, a2, a3);
#pragma unroll
            for (int nt2 = 0; nt2 < 4; ++nt2) {
                uint32_t b0, b1, b2, b3;
                const int brow = 16 * nt2 + rr + 8 * (mi >> 1);
                ldsm_x4(kv + swz(brow, kc + (mi & 1)), b0, b1, b2, b3);
                mma_bf16_16816(S[2 * nt2], a0, a1, a2, a3, b0, b1);
                mma_bf16_16816(S[2 * nt2 + 1], a0, a1, a2, a3, b2, b3);
            }
        }
        // Add the other column half's partial sums (same value in both warps).
        float *myX = sX + warp * 1024;
        const float *otX = sX + (warp ^ 4) * 1024;
#pragma unroll
        for (int j = 0; j < 32; ++j) myX[j * 32 + lane] = S[j >> 2][j & 3];
        named_bar(1 + hg, 64);
#pragma unroll
        for (int j = 0; j < 32; ++j) S[j >> 2][j & 3] += otX[j * 32 + lane];

        // Online softmax (log2 domain).  Row r = 0: head 16hg+g, r = 1: +8.
        float mx[2] = {-INFINITY, -INFINITY};
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int col = 8 * nt + 2 * c4 + (e & 1);
                const bool valid = sRows[slot * kAtTile + col] >= 0;
                const float v = valid ? S[nt][e] * P.scale_log2 : -INFINITY;
                S[nt][e] = v;
                mx[e >> 1] = fmaxf(mx[e >> 1], v);
            }
        float alpha[2], rsum[2] = {0.f, 0.f};
#pragma unroll
        for (int r = 0; r < 2; ++r) {
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 1));
            mx[r] = fmaxf(mx[r], __shfl_xor_sync(0xffffffffu, mx[r], 2));
            const float m_new = fmaxf(m_run[r], mx[r]);
            alpha[r] = (m_new == -INFINITY) ? 1.f : exp2f(m_run[r] - m_new);
            m_run[r] = m_new;
        }
#pragma unroll
        for (int nt = 0; nt < 8; ++nt)
#pragma unroll
            for (int e = 0; e < 4; ++e) {
                const int r = e >> 1;
                const float p = (m_run[r] == -INFINITY) ? 0.f : exp2f(S[nt][e] - m_run[r]);
                S[nt][e] = p;
                rsum[r] += p;
            }
#pragma unroll
        for (int r = 0; r < 2; ++r) l_run[r] = l_run[r] * alpha[r] + rsum[r];
#pragma unroll
        for (int i = 0; i < 32; ++i) {
            O[i][0] *= alpha[0];
            O[i][1] *= alpha[0];
            O[i][2] *= alpha[1];
            O[i][3] *= alpha[1];
        }
        uint32_t pa[4][4];
#pragma unroll
        for (int k2 = 0; k2 < 4; ++k2) {
            pa[k2][0] = pack_bf16x2(S[2 * k2][0], S[2 * k2][1]);
            pa[k2][1] = pack_bf16x2(S[2 * k2][2], S[2 * k2][3]);
            pa[k2][2] = pack_bf16x2(S[2 * k2 + 1][0], S[2 * k2 + 1][1]);
            pa[k2][3] = pack_bf16x2(S[2 * k2 + 1][2], S[2 * k2 + 1][3]);
        }
        // O[16 heads x 256 cols] += P[16 x 64] . V[64 x 256]
#pragma unroll
        for (int k2 = 0; k2 < 4; ++k2) {
            const int vrow = 16 * k2 + rr + 8 * (mi & 1);
#pragma unroll
            for (int nd2 = 0; nd2 < 16; ++nd2) {
                uint32_t b0, b1, b2, b3;
                ldsm_x4_t(kv + swz(vrow, dh * 32 + 2 * nd2 + (mi >> 1)), b0, b1, b2, b3);
                mma_bf16_16816(O[2 * nd2], pa[k2][0], pa[k2][1], pa[k2][2], pa[k2][3], b0, b1);
                mma_bf16_16816(O[2 * nd2 + 1], pa[k2][0], pa[k2][1], pa[k2][2], pa[k2][3], b2, b3);
            }
        }
        __syncthreads();
    }
    cp_async_wait<0>();

    // Finalise this split.
    float inv[2], lse_v[2];
#pragma unroll
    for (int r = 0; r < 2; ++r) {
        l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 1);
        l_run[r] += __shfl_xor_sync(0xffffffffu, l_run[r], 2);
        if (l_run[r] > 0.f) {
            inv[r] = 1.f / l_run[r];
            lse_v[r] = (m_run[r] + log2f(l_run[r])) * kLn2;
        } else {
            inv[r] = 0.f;
            lse_v[r] = -INFINITY;
        }
    }
    const int h0 = 16 * hg + g, h1 = h0 + 8;
    if (P.splits == 1) {
        uint16_t *o0 = P.out + (static_cast<int64_t>(q) * kMlaHeads + h0) * kNopeDim;
        uint16_t *o1 = P.out + (static_cast<int64_t>(q) * kMlaHeads + h1) * kNopeDim;
#pragma unroll
        for (int nd = 0; nd < 32; ++nd) {
            const int d = dh * 256 + 8 * nd + 2 * c4;
            *reinterpret_cast<uint32_t *>(o0 + d) = pack_bf16x2(O[nd][0] * inv[0], O[nd][1] * inv[0]);
            *reinterpret_cast<uint32_t *>(o1 + d) = pack_bf16x2(O[nd][2] * inv[1], O[nd][3] * inv[1]);
        }
        if (P.lse && dh == 0 && c4 == 0) {
            P.lse[static_cast<int64_t>(q) * kMlaHeads + h0] = lse_v[0];
            P.lse[static_cast<int64_t>(q) * kMlaHeads + h1] = lse_v[1];
        }
        return;
    }
    const int64_t wi = static_cast<int64_t>(q) * P.splits + split;
    float *wo = P.ws_o + wi * kMlaHeads * kNopeDim;
#pragma unroll
    for (int nd = 0; nd < 32; ++nd) {
        const int d = dh * 256 + 8 * nd + 2 * c4;
        *reinterpret_cast<float2 *>(wo + h0 * kNopeDim + d) = make_float2(O[nd][0] * inv[0], O[nd][1] * inv[0]);
        *reinterpret_cast<float2 *>(wo + h1 * kNopeDim + d) = make_float2(O[nd][2] * inv[1], O[nd][3] * inv[1]);
    }
    if (dh == 0 && c4 == 0) {
        P.ws_lse[wi * kMlaHeads + h0] = lse_v[0];
        P.ws_lse[wi * kMlaHeads + h1] = lse_v[1];
    }
    __threadfence();
    __syncthreads();
    if (tid == 0) s_last = atomicAdd(&P.ws_cnt[q], 1) == P.splits - 1;
    __syncthreads();
    if (!s_last) return;
    __threadfence();
    // Last split of this query: merge the partials, lse-weighted.
    const float *base_o = P.ws_o + static_cast<int64_t>(q) * P.splits * kMlaHeads * kNopeDim;
    const float *base_l = P.ws_lse + static_cast<int64_t>(q) * P.splits * kMlaHeads;
    for (int idx = tid; idx < kMlaHeads * (kNopeDim / 2); idx += kAtThreads) {
        const int h = idx / (kNopeDim / 2), d = 2 * (idx % (kNopeDim / 2));
        float mx = -INFINITY;
        for (int s = 0; s < P.splits; ++s) mx = fmaxf(mx, __ldcg(base_l + s * kMlaHeads + h));
        float a0 = 0.f, a1 = 0.f, den = 0.f;
        if (mx > -INFINITY) {
            for (int s = 0; s < P.splits; ++s) {
                const float wgt = expf(__ldcg(base_l + s * kMlaHeads + h) - mx);
                const float2 v = __ldcg(reinterpret_cast<const float2 *>(
                    base_o + (static_cast<int64_t>(s) * kMlaHeads + h) * kNopeDim + d));
                den += wgt;
                a0 += wgt * v.x;
                a1 += wgt * v.y;
            }
        }
        const float iv = den > 0.f ? 1.f / den : 0.f;
        *reinterpret_cast<uint32_t *>(P.out + (static_cast<int64_t>(q) * kMlaHeads + h) * kNopeDim + d) =
            pack_bf16x2(a0 * iv, a1 * iv);
        if (P.lse && d == 0) P.lse[static_cast<int64_t>(q) * kMlaHeads + h] = den > 0.f ? mx + logf(den) : -INFINITY;
    }
    if (tid == 0) P.ws_cnt[q] = 0;  // ready for the next call
}

}  // namespace

int attend_splits(const kp_config &cfg, int32_t num_queries, int sm_count) {
    if (num_queries <= 0) return 1;
    const int K = cfg.topk_tokens / cfg.kpool;
    const int max_tiles = (K * cfg.kpool + cfg.kpool - 1 + kAtTile - 1) / kAtTile;
    int s = sm_count / num_queries;
    if (s > max_tiles) s = max_tiles;
    return s < 1 ? 1 : s;
}

size_t attend_ws_bytes(const kp_config &cfg, int32_t num_queries, int splits) {
    (void)cfg;
    if (splits <= 1) return 256;
    const size_t n = static_cast<size_t>(num_queries) * splits;
    return align_up(n * kMlaHeads * kNopeDim * 4, 256) + align_up(n * kMlaHeads * 4, 256) +
           align_up(static_cast<size_t>(num_queries) * 4, 256);
}

kp_status launch_attend(const kp_attend_args &a, cudaStream_t s) {
    const int nq = a.q.num_queries;
    if (nq == 0) return KP_OK;
    const int sms = device_sm_count();
    if (sms <= 0) return KP_ERR_CUDA;
    const int splits = attend_splits(a.cfg, nq, sms);
    AttendParams P;
    P.q_lat = a.q_lat;
    P.latent = a.latent;
    P.latent_rows = a.seqs.latent_rows;
    P.q_seq = a.q.q_seq;
    P.q_pos = a.q.q_pos;
    P.latent_row_off = a.seqs.latent_row_off;
    P.num_seqs = a.seqs.num_seqs;
    P.pool_idx = a.pool_idx;
    P.n_sel = a.n_sel;
    P.K = a.cfg.topk_tokens / a.cfg.kpool;
    P.tail = a.cfg.always_select_tail ? 1 : 0;
    P.scale_log2 = a.cfg.sm_scale * kLog2e;
    P.out = a.out;
    P.lse = a.lse;
    P.splits = splits;
    P.status = a.d_status;
    P.ws_o = nullptr;
    P.ws_lse = nullptr;
    P.ws_cnt = nullptr;
    if (splits > 1) {
        const size_t n = static_cast<size_t>(nq) * splits;
        uint8_t *w = static_cast<uint8_t *>(a.workspace);
        P.ws_o = reinterpret_cast<float *>(w);
        w += align_up(n * kMlaHeads * kNopeDim * 4, 256);
        P.ws_lse = reinterpret_cast<float *>(w);
        w += align_up(n * kMlaHeads * 4, 256);
        P.ws_cnt = reinterpret_cast<int32_t *>(w);
        cudaError_t e = cudaMemsetAsync(P.ws_cnt, 0, static_cast<size_t>(nq) * 4, s);
        if (e != cudaSuccess) {
            record_cuda_error("cudaMemsetAsync(attend tickets)", e);
            return KP_ERR_CUDA;
        }
    }
    cudaError_t e = cudaFuncSetAttribute(sparse_mla_mma_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kAtSmemBytes);
    if (e != cudaSuccess) {
        record_cuda_error("cudaFuncSetAttribute(sparse_mla_mma_kernel)", e);
        return KP_ERR_CUDA;
    }
    sparse_mla_mma_kernel<<<static_cast<unsigned>(nq) * splits, kAtThreads, kAtSmemBytes, s>>>(P);
    return check_launch("sparse_mla_mma_kernel");
}

}  // namespace kp
