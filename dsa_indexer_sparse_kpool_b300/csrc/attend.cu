// attend.cu -- nope-only sparse MLA in latent space over the selected pools,
// on tcgen05 tensor cores with TMEM accumulators.
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
// B300 design.  The 64 heads of a query share every latent row (MQA-like),
// so heads are the natural N of the tensor-core products and the gathered
// tokens their M:
//   S^T[tok, h] = C[tok, :512] . Q[h, :512]^T     M = 128 tokens, N = 64, K = 512
//   O^T[d, h]  += C[tok, d]^T . P[tok, h]          M = 128 latent columns (x4), N = 64, K = 128 tokens
// One 128-token tile of latent rows (128 KB) is gathered into shared memory
// in the 128-byte-swizzle layout; the S product reads it K-major, the P.V
// product reads the same bytes M-major, so each latent row crosses HBM once.
// S (64 TMEM columns) and O^T (4 x 64 columns) live in TMEM.  Each softmax
// thread owns one token (one TMEM lane): per-head tile maxima come from one
// warp redux per head plus a 4-warp exchange; the running max is raised only
// when a tile's max exceeds it by 2^8 (then O^T and the row sums are rescaled),
// so the correction pass almost never runs.
//
// A query's token list is split over the CTAs of a thread-block cluster
// (up to 8).  After its tiles, each CTA dumps its unnormalised O^T, running
// max and row sums to its own shared memory; after a cluster barrier, CTA r
// merges heads [64r/S, 64(r+1)/S) across the cluster through distributed
// shared memory, adds the <= 3 tail tokens (computed on CUDA cores, so the
// tail never costs a tensor-core tile), normalises and writes bf16 out and
// fp32 lse.  No global scratch, no second launch.
//
// Warp roles (384 threads, one CTA per SM):
//   warps 0-7  softmax: warp w owns TMEM lane quadrant w % 4 (32 tokens) and
//              heads 32 * (w / 4) .. +31; then the O^T dump
//   warp 8     TMEM allocation, Q TMA, MMA issue (one lane)
//   warps 9-11 gather: cp.async 16-byte pieces of the selected rows into the
//              swizzled tile (each warp instruction moves two whole 256-byte
//              row segments; warp g takes token pairs g, g+3, g+6, ...)
//   all        cluster merge and output
#include "kp_common.cuh"
#include "kp_internal.h"

namespace kp {

namespace {

constexpr int kAtTok = 128;                               // tokens per tile
constexpr int kAtChunks = 4;                              // 128-column chunks of a latent row
constexpr int kAtBlockBytes = kAtTok * 128;               // [128 rows][64 bf16] swizzle block
constexpr int kAtChunkBytes = 2 * kAtBlockBytes;          // 32 KB
constexpr int kAtTileBytes = kAtChunks * kAtChunkBytes;   // 128 KB
constexpr int kAtQBlockBytes = kMlaHeads * 128;           // [64 heads][64 bf16] = 8 KB
constexpr int kAtQBytes = 8 * kAtQBlockBytes;             // 64 KB
constexpr int kAtPBytes = kAtTok * kMlaHeads * 2;         // 16 KB
constexpr int kAtMaxSplits = 8;
constexpr int kAtMaxTail = kKpool - 1;
constexpr int kAtSoftWarps = 8;
constexpr int kAtSoftThreads = 32 * kAtSoftWarps;
constexpr int kAtMmaWarp = 8;
constexpr int kAtProdWarp0 = 9;
constexpr int kAtProdWarps = 3;
constexpr int kAtProdThreads = 32 * kAtProdWarps;
constexpr int kAtThreads = 384;
constexpr int kAtTmemCols = 512;
constexpr uint32_t kAtOCol = 0;                           // O^T: chunk c at columns 64c .. 64c+63
constexpr uint32_t kAtSCol = 256;                         // S^T: 64 columns
constexpr float kAtRescaleLog2 = 8.f;                     // raise the running max only past 2^8

// Shared memory (offsets from a 1024-aligned base).
constexpr int kOffQ = 0;
constexpr int kOffTile = kOffQ + kAtQBytes;               // also the O dump [64][512] fp32
constexpr int kOffP = kOffTile + kAtTileBytes;
constexpr int kOffMisc = kOffP + kAtPBytes;
constexpr int kMiscRed = 0;                               // [4][64] f32
constexpr int kMiscMUsed = kMiscRed + 4 * 64 * 4;         // [64] f32 running max (log2 units)
constexpr int kMiscFac = kMiscMUsed + 64 * 4;             // [64] f32 rescale factors of this tile
constexpr int kMiscLSum = kMiscFac + 64 * 4;              // [64] f32 row sums
constexpr int kMiscTail = kMiscLSum + 64 * 4;             // [3][512] bf16 tail rows
constexpr int kMiscZTail = kMiscTail + kAtMaxTail * kNopeDim * 2;   // [64][4] f32 tail logits
constexpr int kMiscW = kMiscZTail + 64 * 4 * 4;           // [64][16] f32 merge weights
constexpr int kMiscBars = kMiscW + 64 * 16 * 4;           // mbarriers
constexpr int kNumBars = 13;
constexpr int kMiscTmem = kMiscBars + kNumBars * 8;
constexpr int kMiscAbort = kMiscTmem + 4;
constexpr int kMiscBytes = kMiscAbort + 12;
constexpr int kAtSmemBytes = kOffMisc + kMiscBytes + 1024;  // + alignment slack
static_assert(kAtSmemBytes <= 232448, "attention shared memory over the per-CTA limit");
static_assert(kAtTileBytes >= kMlaHeads * kNopeDim * 4, "O dump must fit in the tile region");

// mbarrier indices
constexpr int kBarFull = 0;    // [4] chunk gathered (96 producer arrivals)
constexpr int kBarFree = 4;    // [4] chunk consumed by P.V (tcgen05.commit)
constexpr int kBarQ = 8;       // Q landed (TMA)
constexpr int kBarS = 9;       // S^T ready (commit)
constexpr int kBarP = 10;      // P written and O^T rescaled (256 softmax arrivals)
constexpr int kBarO = 11;      // every MMA of the CTA done (commit)
constexpr int kBarDrain = 12;  // teardown after an abort

struct AttendParams {
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
    int splits;
    int32_t *status;
};

__device__ __forceinline__ void named_bar(int id, int count) {
    asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(count) : "memory");
}
// Named barrier that also ANDs a flag over the participating threads, so a
// failed wait in any of them makes all of them leave together.
__device__ __forceinline__ bool named_bar_all(int id, int count, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.and.pred p, %2, %3, q;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(r)
        : "r"(static_cast<uint32_t>(v)), "r"(id), "r"(count)
        : "memory");
    return r != 0;
}

// Byte offset of element (row, col) of a [rows][64 bf16] 128-byte-swizzled block.
__device__ __forceinline__ uint32_t sw128_off(int row, int col) {
    return static_cast<uint32_t>(row * 128 + ((((col >> 3) ^ row) & 7) << 4) + (col & 7) * 2);
}

__device__ __forceinline__ float bf16_lo(uint32_t v) { return __uint_as_float(v << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t v) { return __uint_as_float(v & 0xffff0000u); }

__global__ void __launch_bounds__(kAtThreads, 1)
    sparse_mla_tc_kernel(const __grid_constant__ CUtensorMap tm_q, AttendParams P) {
    extern __shared__ uint8_t smem_raw[];
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t sbase = smem_u32(smem);
    const uint32_t sQ = sbase + kOffQ, sTile = sbase + kOffTile, sP = sbase + kOffP;
    uint8_t *misc = smem + kOffMisc;
    float *red_s = reinterpret_cast<float *>(misc + kMiscRed);
    float *mused_s = reinterpret_cast<float *>(misc + kMiscMUsed);
    float *fac_s = reinterpret_cast<float *>(misc + kMiscFac);
    float *lsum_s = reinterpret_cast<float *>(misc + kMiscLSum);
    uint16_t *tail_s = reinterpret_cast<uint16_t *>(misc + kMiscTail);
    float *ztail_s = reinterpret_cast<float *>(misc + kMiscZTail);
    float *wm_s = reinterpret_cast<float *>(misc + kMiscW);
    const uint32_t bar0 = sbase + kOffMisc + kMiscBars;
    auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    uint32_t *tmem_s = reinterpret_cast<uint32_t *>(misc + kMiscTmem);
    int *abort_s = reinterpret_cast<int *>(misc + kMiscAbort);
    volatile int *abort_flag = abort_s;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = P.splits;
    const int q = blockIdx.x / S, split = blockIdx.x % S;

    // ---- what this query attends to
    const int b = P.q_seq[q];
    const int t = P.q_pos[q];
    bool qvalid = true;
    int nf = 0, ns = 0, n_tail = 0;
    int64_t base_row = 0;
    if (b < 0 || b >= P.num_seqs || t < 0) {
        if (tid == 0) set_status(P.status, KP_ERR_DEVICE_BOUNDS);
        qvalid = false;
    } else {
        nf = (t + 1) / kKpool;
        ns = P.n_sel[q];
        const int ns_max = min(P.K, nf);
        if (ns < 0 || ns > ns_max) {
            if (tid == 0) set_status(P.status, KP_ERR_DEVICE_BOUNDS);
            ns = max(0, min(ns, ns_max));
        }
        n_tail = P.tail ? (t + 1) - nf * kKpool : 0;
        base_row = P.latent_row_off[b];
        if (base_row < 0 || base_row + t >= P.latent_rows) {
            if (tid == 0) set_status(P.status, KP_ERR_DEVICE_BOUNDS);
            qvalid = false;
            ns = 0;
            n_tail = 0;
        }
    }
    const int n_pool_tok = ns * kKpool;
    const int n_tiles = (n_pool_tok + kAtTok - 1) / kAtTok;
    const int tb = n_tiles * split / S, te = n_tiles * (split + 1) / S;
    const int nt = te - tb;

    // ---- set-up
    if (tid == 0) {
        for (int c = 0; c < kAtChunks; ++c) {
            mbar_init(bar(kBarFull + c), kAtProdThreads);
            mbar_init(bar(kBarFree + c), 1);
        }
        mbar_init(bar(kBarQ), 1);
        mbar_init(bar(kBarS), 1);
        mbar_init(bar(kBarP), kAtSoftThreads);
        mbar_init(bar(kBarO), 1);
        mbar_init(bar(kBarDrain), 1);
        fence_mbar_init();
        *abort_s = 0;
        tma_prefetch_desc(&tm_q);
    }
    if (tid < kMlaHeads) {
        mused_s[tid] = -INFINITY;
        lsum_s[tid] = 0.f;
    }
    if (warp == kAtMmaWarp) {
        tmem_alloc(smem_u32(tmem_s), kAtTmemCols);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_s;

    if (warp == kAtMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        if (lane == 0) {
            if (qvalid) {
                mbar_expect_tx(bar(kBarQ), kAtQBytes);
                for (int blk = 0; blk < 8; ++blk)
                    tma_load_2d(sQ + blk * kAtQBlockBytes, &tm_q, bar(kBarQ), blk * 64, q * kMlaHeads);
            }
            bool ok = true;
            if (nt > 0) ok = mbar_wait(bar(kBarQ), 0, abort_flag, P.status);
            const uint32_t idesc_s = idesc_bf16_f32(kAtTok, kMlaHeads);
            const uint32_t idesc_pv = idesc_bf16_f32(kAtTok, kMlaHeads, true, true);
            for (int jj = 0; ok && jj < nt; ++jj) {
                const uint32_t par = jj & 1;
                for (int c = 0; ok && c < kAtChunks; ++c) {
                    if (!(ok = mbar_wait(bar(kBarFull + c), par, abort_flag, P.status))) break;
                    tc_fence_after();
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        const int blk = 2 * c + (kk >> 2);
                        const uint32_t koff = (kk & 3) * 32;
                        const uint64_t ad = desc_sw128(sTile + blk * kAtBlockBytes + koff, 16, 1024);
                        const uint64_t bd = desc_sw128(sQ + blk * kAtQBlockBytes + koff, 16, 1024);
                        tc_mma_bf16(tmem + kAtSCol, ad, bd, idesc_s, (c | kk) ? 1u : 0u);
                    }
                }
                if (!ok) break;
                tc_commit(bar(kBarS));
                if (!(ok = mbar_wait(bar(kBarP), par, abort_flag, P.status))) break;
                tc_fence_after();
                for (int c = 0; c < kAtChunks; ++c) {
#pragma unroll
                    for (int kk = 0; kk < 8; ++kk) {
                        // A = C^T (latent columns x tokens), M-major: 64-column groups 16 KB
                        // apart, 8-token groups 1 KB apart.  B = P (tokens x heads), N-major.
                        const uint64_t ad = desc_sw128(sTile + 2 * c * kAtBlockBytes + kk * 2048,
                                                       kAtBlockBytes, 1024);
                        // (B is one 64-head group wide, so its LBO is never stepped.)
                        const uint64_t bd = desc_sw128(sP + kk * 2048, 8192, 1024);
                        tc_mma_bf16(tmem + kAtOCol + 64 * c, ad, bd, idesc_pv, (jj | kk) ? 1u : 0u);
                    }
                    tc_commit(bar(kBarFree + c));
                }
            }
            if (ok) {
                if (nt > 0) tc_commit(bar(kBarO));
                else mbar_arrive(bar(kBarO));
            } else {
                // Let every MMA already issued finish before the TMEM is freed.
                tc_commit(bar(kBarDrain));
                mbar_wait(bar(kBarDrain), 0, nullptr, P.status);
                mbar_arrive(bar(kBarO));
            }
        }
    } else if (warp >= kAtProdWarp0) {
        // ------------------------------------------------------------ gather
        const int pw = warp - kAtProdWarp0;
        const int piece = lane & 15, sub = lane >> 4;
        // Token pairs (2k, 2k+1), k = pw + 3m, m < n_pairs; list index j = 2m + sub.
        const int n_pairs = (64 - pw + kAtProdWarps - 1) / kAtProdWarps;
        auto row_of = [&](int tile, int j) -> int64_t {
            if (j >= 2 * n_pairs) return -1;
            const int tok = tile * kAtTok + 2 * (pw + kAtProdWarps * (j >> 1)) + (j & 1);
            if (tok >= n_pool_tok) return -1;
            const int p = P.pool_idx[static_cast<int64_t>(q) * P.K + tok / kKpool];
            if (p < 0 || p >= nf) {
                set_status(P.status, KP_ERR_DEVICE_BOUNDS);
                return -1;
            }
            return base_row + static_cast<int64_t>(p) * kKpool + (tok % kKpool);
        };
        for (int jj = 0; jj < nt; ++jj) {
            const int tile = tb + jj;
            const int64_t row0 = row_of(tile, lane), row1 = row_of(tile, lane + 32);
            bool ok = true;
            for (int c = 0; c < kAtChunks; ++c) {
                if (jj > 0 && !(ok = mbar_wait(bar(kBarFree + c), (jj - 1) & 1, abort_flag, P.status)))
                    break;
                for (int m = 0; m < n_pairs; ++m) {
                    const int tk = 2 * (pw + kAtProdWarps * m) + sub;
                    const int64_t r = __shfl_sync(0xffffffffu, m < 16 ? row0 : row1, (2 * m + sub) & 31);
                    const uint16_t *src = P.latent + (r < 0 ? 0 : r) * kLatentDim + c * 128 + piece * 8;
                    const uint32_t dst = sTile + (2 * c + (piece >> 3)) * kAtBlockBytes + tk * 128 +
                                         (((piece & 7) ^ (tk & 7)) << 4);
                    cp_async_16(dst, src, r < 0 ? 0u : 16u);
                }
                cp_async_commit();
            }
            if (!ok) {
                cp_async_wait<0>();
                break;
            }
            // Chunk c is complete once at most 3 - c newer groups are pending.
            cp_async_wait<3>();
            fence_proxy_async_smem();
            mbar_arrive(bar(kBarFull + 0));
            cp_async_wait<2>();
            fence_proxy_async_smem();
            mbar_arrive(bar(kBarFull + 1));
            cp_async_wait<1>();
            fence_proxy_async_smem();
            mbar_arrive(bar(kBarFull + 2));
            cp_async_wait<0>();
            fence_proxy_async_smem();
            mbar_arrive(bar(kBarFull + 3));
        }
    } else {
        // ------------------------------------------------------------ softmax
        const int quad = warp & 3, half = warp >> 2;
        const int i = quad * 32 + lane;  // token lane of the tile
        const int hb = half * 32;        // this warp's first head
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        float lp[32];                    // running row-sum partials, heads hb .. hb+31
#pragma unroll
        for (int h = 0; h < 32; ++h) lp[h] = 0.f;
        bool ok = true;
        for (int jj = 0; jj < nt; ++jj) {
            ok = named_bar_all(1, kAtSoftThreads, mbar_wait(bar(kBarS), jj & 1, abort_flag, P.status));
            if (!ok) break;
            tc_fence_after();
            uint32_t r[32];
            tmem_ld_32x32b_x32(tmem + lane_base + kAtSCol + hb, r);
            tmem_ld_wait();
            const int n_valid = min(kAtTok, n_pool_tok - (tb + jj) * kAtTok);
            const bool valid = i < n_valid;
            float x[32];
#pragma unroll
            for (int h = 0; h < 32; ++h) {
                x[h] = valid ? __uint_as_float(r[h]) * P.scale_log2 : -INFINITY;
                const float m = warp_max_f32(x[h]);
                if (lane == h) red_s[quad * 64 + hb + h] = m;
            }
            named_bar(1, kAtSoftThreads);
            if (tid < kMlaHeads) {
                const float mt = fmaxf(fmaxf(red_s[tid], red_s[64 + tid]), fmaxf(red_s[128 + tid], red_s[192 + tid]));
                const float mo = mused_s[tid];
                if (mt > mo + kAtRescaleLog2) {
                    mused_s[tid] = mt;
                    fac_s[tid] = exp2f(mo - mt);  // 0 on the first tile (mo = -inf)
                } else {
                    fac_s[tid] = 1.f;
                }
            }
            named_bar(1, kAtSoftThreads);
            bool any = false;
#pragma unroll
            for (int h = 0; h < 32; h += 4) {
                const float4 f = *reinterpret_cast<const float4 *>(fac_s + hb + h);
                lp[h] *= f.x;
                lp[h + 1] *= f.y;
                lp[h + 2] *= f.z;
                lp[h + 3] *= f.w;
                any |= (f.x != 1.f) | (f.y != 1.f) | (f.z != 1.f) | (f.w != 1.f);
            }
            // p = 2^(x - m), row partial sums, bf16 P (token i, heads hb..hb+31), swizzled.
            uint8_t *prow = smem + kOffP + i * 128;
#pragma unroll
            for (int k = 0; k < 4; ++k) {
                uint32_t pk[4];
#pragma unroll
                for (int e = 0; e < 4; ++e) {
                    const int h = 8 * k + 2 * e;
                    const float2 m2 = *reinterpret_cast<const float2 *>(mused_s + hb + h);
                    const float p0 = exp2f(x[h] - m2.x);
                    const float p1 = exp2f(x[h + 1] - m2.y);
                    lp[h] += p0;
                    lp[h + 1] += p1;
                    pk[e] = pack_bf16x2(p0, p1);
                }
                const int chunk = 4 * half + k;
                *reinterpret_cast<uint4 *>(prow + ((chunk ^ (i & 7)) << 4)) = make_uint4(pk[0], pk[1], pk[2], pk[3]);
            }
            if (any && jj > 0) {
                // O^T is stable here: every P.V of the previous tile completed before S^T.
                // (Done after P so that the logits' registers are free.)
                for (int c = 0; c < kAtChunks; ++c) {
                    uint32_t o[32];
                    const uint32_t ta = tmem + lane_base + kAtOCol + 64 * c + hb;
                    tmem_ld_32x32b_x32(ta, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int h = 0; h < 32; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * fac_s[hb + h]);
                    tmem_st_32x32b_x32(ta, o);
                }
                tmem_st_wait();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(kBarP));
        }
        // ---- after the last tile: O^T -> shared memory as O[h][d] (fp32, unnormalised)
        if (ok) ok = named_bar_all(1, kAtSoftThreads, mbar_wait(bar(kBarO), 0, abort_flag, P.status));
        if (ok) {
            tc_fence_after();
            if (nt > 0) {
                float *odump = reinterpret_cast<float *>(smem + kOffTile);
                for (int c = 0; c < kAtChunks; ++c) {
                    uint32_t o[32];
                    tmem_ld_32x32b_x32(tmem + lane_base + kAtOCol + 64 * c + hb, o);
                    tmem_ld_wait();
                    const int d = c * 128 + i;
#pragma unroll
                    for (int h = 0; h < 32; ++h) odump[(hb + h) * kNopeDim + d] = __uint_as_float(o[h]);
                }
            }
            // Row sums: transpose-reduce the 32 per-thread partials over the warp
            // (lane l ends with head hb + l), then add the 4 quadrants.
#pragma unroll
            for (int j = 0; j < 16; ++j) {
                const bool hi = lane & 16;
                const float send = hi ? lp[j] : lp[j + 16];
                const float keep = hi ? lp[j + 16] : lp[j];
                lp[j] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
            }
#pragma unroll
            for (int j = 0; j < 8; ++j) {
                const bool hi = lane & 8;
                const float send = hi ? lp[j] : lp[j + 8];
                const float keep = hi ? lp[j + 8] : lp[j];
                lp[j] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
            }
#pragma unroll
            for (int j = 0; j < 4; ++j) {
                const bool hi = lane & 4;
                const float send = hi ? lp[j] : lp[j + 4];
                const float keep = hi ? lp[j + 4] : lp[j];
                lp[j] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
            }
#pragma unroll
            for (int j = 0; j < 2; ++j) {
                const bool hi = lane & 2;
                const float send = hi ? lp[j] : lp[j + 2];
                const float keep = hi ? lp[j + 2] : lp[j];
                lp[j] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
            }
            {
                const bool hi = lane & 1;
                const float send = hi ? lp[0] : lp[1];
                const float keep = hi ? lp[1] : lp[0];
                lp[0] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
            }
            atomicAdd(lsum_s + hb + lane, lp[0]);
        }
    }

    // ---- merge over the cluster, tail tokens, output
    tc_fence_before();
    __syncthreads();
    if (S > 1) cluster_barrier();

    const int h0 = kMlaHeads * split / S, h1 = kMlaHeads * (split + 1) / S, nh = h1 - h0;
    const bool aborted = *abort_flag != 0;
    if (qvalid && !aborted) {
        // tail rows -> shared memory
        for (int k = tid; k < n_tail * 64; k += kAtThreads) {
            const int j = k >> 6, piece = k & 63;
            const int64_t row = base_row + static_cast<int64_t>(nf) * kKpool + j;
            *reinterpret_cast<uint4 *>(tail_s + j * kNopeDim + piece * 8) =
                *reinterpret_cast<const uint4 *>(P.latent + row * kLatentDim + piece * 8);
        }
        // Q has landed (the tail logits read it; nothing may be in flight at exit).
        const bool have_q = mbar_wait(bar(kBarQ), 0, abort_flag, P.status);
        __syncthreads();
        // tail logits: one warp per (head, tail token)
        if (have_q) {
            for (int pr = warp; pr < nh * n_tail; pr += kAtThreads / 32) {
                const int h = h0 + pr / n_tail, j = pr % n_tail;
                float acc = 0.f;
#pragma unroll
                for (int e = 0; e < 16; e += 2) {
                    const int d = lane * 16 + e;
                    const uint32_t qv =
                        *reinterpret_cast<const uint32_t *>(smem + kOffQ + (d >> 6) * kAtQBlockBytes +
                                                            sw128_off(h, d & 63));
                    const uint32_t cv = *reinterpret_cast<const uint32_t *>(tail_s + j * kNopeDim + d);
                    acc = fmaf(bf16_lo(qv), bf16_lo(cv), acc);
                    acc = fmaf(bf16_hi(qv), bf16_hi(cv), acc);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
                if (lane == 0) ztail_s[h * 4 + j] = acc * P.scale_log2;
            }
        }
        __syncthreads();
        // per-head merge weights
        if (tid < nh) {
            const int h = h0 + tid;
            float M = -INFINITY;
            for (int s = 0; s < S; ++s) M = fmaxf(M, dsmem_ld_f32(dsmem_addr(smem_u32(mused_s + h), s)));
            for (int j = 0; j < n_tail; ++j) M = fmaxf(M, ztail_s[h * 4 + j]);
            float L = 0.f;
            float *w = wm_s + tid * 16;
            for (int s = 0; s < kAtMaxSplits; ++s) {
                float ws = 0.f;
                if (s < S) {
                    const float ms = dsmem_ld_f32(dsmem_addr(smem_u32(mused_s + h), s));
                    if (ms > -INFINITY) {
                        ws = exp2f(ms - M);
                        L += ws * dsmem_ld_f32(dsmem_addr(smem_u32(lsum_s + h), s));
                    }
                }
                w[s] = ws;
            }
            for (int j = 0; j < kAtMaxTail; ++j) {
                const float wt = j < n_tail ? exp2f(ztail_s[h * 4 + j] - M) : 0.f;
                w[8 + j] = wt;
                L += wt;
            }
            w[12] = L > 0.f ? 1.f / L : 0.f;
            if (P.lse) P.lse[static_cast<int64_t>(q) * kMlaHeads + h] = L > 0.f ? (M + log2f(L)) * 0.69314718055994530942f : -INFINITY;
        }
        __syncthreads();
        // out[q][h][d] = (sum_s w_s O_s[h][d] + sum_j w_j c_j[d]) / L
        const uint32_t odump_addr = sbase + kOffTile;
        for (int idx = tid; idx < nh * (kNopeDim / 2); idx += kAtThreads) {
            const int hl = idx / (kNopeDim / 2), d = 2 * (idx % (kNopeDim / 2));
            const int h = h0 + hl;
            const float *w = wm_s + hl * 16;
            float a0 = 0.f, a1 = 0.f;
            for (int s = 0; s < S; ++s) {
                if (w[s] > 0.f) {
                    const float2 v = dsmem_ld_f32x2(dsmem_addr(odump_addr + (h * kNopeDim + d) * 4, s));
                    a0 = fmaf(w[s], v.x, a0);
                    a1 = fmaf(w[s], v.y, a1);
                }
            }
            for (int j = 0; j < n_tail; ++j) {
                const uint32_t cv = *reinterpret_cast<const uint32_t *>(tail_s + j * kNopeDim + d);
                a0 = fmaf(w[8 + j], bf16_lo(cv), a0);
                a1 = fmaf(w[8 + j], bf16_hi(cv), a1);
            }
            *reinterpret_cast<uint32_t *>(P.out + (static_cast<int64_t>(q) * kMlaHeads + h) * kNopeDim + d) =
                pack_bf16x2(a0 * w[12], a1 * w[12]);
        }
    } else if (!qvalid && !aborted) {
        // Nothing to attend: out = 0, lse = -inf.
        for (int idx = tid; idx < nh * (kNopeDim / 2); idx += kAtThreads) {
            const int h = h0 + idx / (kNopeDim / 2), d = 2 * (idx % (kNopeDim / 2));
            *reinterpret_cast<uint32_t *>(P.out + (static_cast<int64_t>(q) * kMlaHeads + h) * kNopeDim + d) = 0u;
        }
        if (P.lse && tid < nh) P.lse[static_cast<int64_t>(q) * kMlaHeads + h0 + tid] = -INFINITY;
    }

    // Peers may still read this CTA's shared memory until everyone is done.
    if (S > 1) cluster_barrier();
    if (aborted && qvalid && tid == 0) mbar_wait(bar(kBarQ), 0, nullptr, P.status);  // no TMA left in flight
    tc_fence_before();
    __syncthreads();
    if (warp == kAtMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kAtTmemCols);
    }
}

// Largest cluster size whose clusters, one CTA per SM, all fit at once (cached per device).
int max_active_clusters(int cluster) {
    static int cache[64][kAtMaxSplits + 1] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    if (cache[dev][cluster] != 0) return cache[dev][cluster];
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cluster * 64);
    cfg.blockDim = dim3(kAtThreads);
    cfg.dynamicSmemBytes = kAtSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, sparse_mla_tc_kernel, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    cache[dev][cluster] = n > 0 ? n : -1;
    return n;
}

bool attend_smem_configured() {
    static int done[64] = {};
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    if (done[dev]) return true;
    cudaError_t e = cudaFuncSetAttribute(sparse_mla_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         kAtSmemBytes);
    if (e != cudaSuccess) {
        record_cuda_error("cudaFuncSetAttribute(sparse_mla_tc_kernel)", e);
        return false;
    }
    done[dev] = 1;
    return true;
}

}  // namespace

// Splits of one query's token list = CTAs of its cluster: as many as keep
// every cluster resident in one wave, at most 8, at most one per tile.
int attend_splits(const kp_config &cfg, int32_t num_queries, int sm_count) {
    if (num_queries <= 0) return 1;
    const int tiles = (cfg.topk_tokens + kAtTok - 1) / kAtTok;
    int s = sm_count / num_queries;
    if (s > kAtMaxSplits) s = kAtMaxSplits;
    if (s > tiles) s = tiles;
    if (s < 1) s = 1;
    return s;
}

size_t attend_ws_bytes(const kp_config &cfg, int32_t num_queries, int splits) {
    (void)cfg;
    (void)num_queries;
    (void)splits;
    return 256;  // the cluster merge needs no global scratch
}

kp_status launch_attend(const kp_attend_args &a, cudaStream_t s) {
    const int nq = a.q.num_queries;
    if (nq == 0) return KP_OK;
    const int sms = device_sm_count();
    if (sms <= 0) return KP_ERR_CUDA;
    if (!attend_smem_configured()) return KP_ERR_CUDA;
    int splits = attend_splits(a.cfg, nq, sms);
    while (splits > 1 && max_active_clusters(splits) < nq) --splits;

    CUtensorMap tm_q;
    if (!make_tmap_bf16_sw128(&tm_q, a.q_lat, kLatentDim, static_cast<uint64_t>(nq) * kMlaHeads,
                              kLatentDim * 2, 64, kMlaHeads))
        return KP_ERR_CUDA;
    AttendParams P;
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
    P.scale_log2 = a.cfg.sm_scale * 1.44269504088896340736f;
    P.out = a.out;
    P.lse = a.lse;
    P.splits = splits;
    P.status = a.d_status;

    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(static_cast<unsigned>(nq) * splits);
    cfg.blockDim = dim3(kAtThreads);
    cfg.dynamicSmemBytes = kAtSmemBytes;
    cfg.stream = s;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = splits;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    cudaError_t e = cudaLaunchKernelEx(&cfg, sparse_mla_tc_kernel, tm_q, P);
    if (e != cudaSuccess) {
        record_cuda_error("cudaLaunchKernelEx(sparse_mla_tc_kernel)", e);
        return KP_ERR_CUDA;
    }
    return check_launch("sparse_mla_tc_kernel");
}

}  // namespace kp
