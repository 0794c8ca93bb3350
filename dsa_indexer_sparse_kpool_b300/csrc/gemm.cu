// gemm.cu -- bf16 GEMM on tcgen05 tensor cores for the steps either side of
// the DSA step: the lightning indexer's projections from the hidden state
// and the MLA absorption of W_UK into the query and of W_UV / o_proj out of
// the latent output (MAX docs, max.pipelines.architectures.glm5_next:
// Glm5NextConfig q_lora_rank, kv_lora_rank, qk_nope_head_dim, v_head_dim,
// index_n_heads, index_head_dim; llm-atlas GLM-5.3-Flash card, raw config:
// hidden_size 4096, q_lora_rank 1536, qk_nope_head_dim 256).
//
//   C[b][m][n] = sum_k A[b][m][k] * B[b][n][k]      (bf16 in, fp32 accumulate)
//
// Batch b selects a column block of A (A's row holds every batch's K slice
// side by side, as a per-head query [T][heads * dim] does), a row block of B
// (B holds every batch's [N][K] weight one after another) and a column block
// of C.  Output bf16 (round to nearest even) or fp32.
//
// B300 design: persistent CTAs, one per SM, over (problem, batch, 128-row
// tile, BN-column tile) units; up to four independent problems share one
// launch, so small products run side by side instead of one after another.
// Warp 0 streams 64-wide K slices of A (128 x 64) and B (BN x 64) by TMA with
// 128-byte swizzle into a ring of 192 KB: four stages at BN 256, up to nine
// when every problem's tiles are narrow, so a CTA that streams weights alone
// keeps more bytes in flight.  Warp 1 issues tcgen05.mma (M 128, N = BN <=
// 256, K 16) into one of two TMEM accumulators, so the epilogue of one unit
// overlaps the MMAs of the next; warps 2-9 read the accumulator back with
// tcgen05.ld (two warps per TMEM lane quadrant, splitting the 32-column
// chunks) and store converted rows.
#include <cuda.h>

#include <cstring>

#include "kp_common.cuh"
#include "kp_internal.h"

namespace kp {

namespace {

constexpr int kGmM = 128;                       // rows per tile (MMA M)
constexpr int kGmMaxN = 256;                    // columns per tile (MMA N max)
constexpr int kGmK = 64;                        // K per stage: one 128-byte swizzle row of bf16
constexpr int kGmABytes = kGmM * 128;           // 16 KB
constexpr int kGmRingBytes = 4 * (kGmABytes + kGmMaxN * 128);   // 192 KB: four stages at BN 256
constexpr int kGmMaxStages = 24;
constexpr int kGmMaxProblems = 4;
constexpr int kGmEpiThreads = 256;
constexpr int kGmThreads = 64 + kGmEpiThreads;
constexpr int kGmNumBars = 2 * kGmMaxStages + 4 + 1;
// The MMA reads a 128-row A window from each stage; with fewer A rows loaded
// the window runs past the stage (rows >= m only feed output rows that are never
// stored), so the ring is followed by one A tile of slack.
// Per epilogue warp, a 32-row x 32-column bf16 block staged on its way out, so
// that the warp writes whole 64-byte row pieces (8 rows per store) instead of
// 16 bytes in each of 32 rows.
constexpr int kGmStageWarpBytes = 32 * 64;
constexpr int kGmOffStage = kGmRingBytes + kGmABytes + (kGmNumBars * 8 + 127) / 128 * 128;
constexpr int kGmSmemBytes = kGmOffStage + (kGmEpiThreads / 32) * kGmStageWarpBytes + 1024;
static_assert(kGmSmemBytes <= 232448, "GEMM shared memory over the per-CTA limit");

// One product of a launch.  Its units are unit0 .. unit0 + batch * m_tiles *
// n_tiles - 1, in the order batch, column tile, row tile (row tiles of one
// column tile run on neighbouring CTAs and share the B tile in L2).
struct GemmProblem {
    int m, n, k, batch;
    int bn;                      // columns per tile (multiple of 32, <= 256)
    int m_tiles, n_tiles, unit0;
    int64_t a_batch_off;         // A columns between batches
    int64_t b_batch_off;         // B rows between batches
    void *c;
    int64_t ldc, c_batch_off;    // C row pitch and columns between batches (elements)
    int c_f32;                   // 1: fp32 output, 0: bf16
};

struct GemmMaps {
    CUtensorMap a[kGmMaxProblems], b[kGmMaxProblems];
};

struct GemmParams {
    GemmProblem pr[kGmMaxProblems];
    int n_problems, units;
    int stages;                  // ring stages (<= kGmMaxStages)
    uint32_t a_bytes;            // A rows loaded per K block x 128 (rows a multiple of 8, <= 128)
    int kb;                      // 64-wide K blocks per stage (one TMA box each for A and B when > 1)
    uint32_t stage_bytes;        // kb x (a_bytes + the widest B tile), a multiple of 1024
    unsigned long long wait_ns;
    int32_t *status;
};

__device__ __forceinline__ bool gm_epi_bar_all(bool v) {
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

// Stores columns col0 .. col0 + 31 (clipped to n) of one row of batch b.
__device__ __forceinline__ void store_row_chunk(const GemmProblem &P, int b, int row, int col0,
                                                const uint32_t (&r)[32]) {
    const int64_t off = static_cast<int64_t>(row) * P.ldc + b * P.c_batch_off + col0;
    const int ncol = min(32, P.n - col0);
    if (P.c_f32) {
        float *c = static_cast<float *>(P.c) + off;
        if (ncol == 32 && (reinterpret_cast<uintptr_t>(c) & 15) == 0) {
#pragma unroll
            for (int j = 0; j < 32; j += 4)
                *reinterpret_cast<float4 *>(c + j) = make_float4(__uint_as_float(r[j]), __uint_as_float(r[j + 1]),
                                                                 __uint_as_float(r[j + 2]), __uint_as_float(r[j + 3]));
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (j < ncol) c[j] = __uint_as_float(r[j]);
        }
    } else {
        uint16_t *c = static_cast<uint16_t *>(P.c) + off;
        if (ncol == 32 && (reinterpret_cast<uintptr_t>(c) & 15) == 0) {
#pragma unroll
            for (int j = 0; j < 32; j += 8)
                *reinterpret_cast<uint4 *>(c + j) =
                    make_uint4(pack_bf16x2(__uint_as_float(r[j]), __uint_as_float(r[j + 1])),
                               pack_bf16x2(__uint_as_float(r[j + 2]), __uint_as_float(r[j + 3])),
                               pack_bf16x2(__uint_as_float(r[j + 4]), __uint_as_float(r[j + 5])),
                               pack_bf16x2(__uint_as_float(r[j + 6]), __uint_as_float(r[j + 7])));
        } else {
#pragma unroll
            for (int j = 0; j < 32; ++j)
                if (j < ncol) c[j] = static_cast<uint16_t>(pack_bf16x2(__uint_as_float(r[j]), 0.f) & 0xffffu);
        }
    }
}

__global__ void __launch_bounds__(kGmThreads, 1)
    gemm_bf16_kernel(const __grid_constant__ GemmMaps M, const __grid_constant__ GemmParams P) {
    extern __shared__ uint8_t smem_raw[];
    __shared__ uint32_t tmem_base_s;
    __shared__ int abort_s;
    uint8_t *smem = reinterpret_cast<uint8_t *>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                                ~static_cast<uintptr_t>(1023));
    const uint32_t s0 = smem_u32(smem);
    const uint32_t bar0 = s0 + kGmRingBytes + kGmABytes;
    auto full_bar = [&](int s) { return bar0 + 8u * s; };
    auto empty_bar = [&](int s) { return bar0 + 8u * (kGmMaxStages + s); };
    auto accf_bar = [&](int a) { return bar0 + 8u * (2 * kGmMaxStages + a); };
    auto acce_bar = [&](int a) { return bar0 + 8u * (2 * kGmMaxStages + 2 + a); };
    const uint32_t drain_bar = bar0 + 8u * (2 * kGmMaxStages + 4);
    const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
    const int stages = P.stages;

    if (threadIdx.x == 0) {
        for (int s = 0; s < kGmMaxStages; ++s) {
            mbar_init(full_bar(s), 1);
            mbar_init(empty_bar(s), 1);
        }
        for (int a = 0; a < 2; ++a) {
            mbar_init(accf_bar(a), 1);
            mbar_init(acce_bar(a), kGmEpiThreads);
        }
        mbar_init(drain_bar, 1);
        fence_mbar_init();
        abort_s = 0;
        for (int p = 0; p < P.n_problems; ++p) {
            tma_prefetch_desc(&M.a[p]);
            tma_prefetch_desc(&M.b[p]);
        }
    }
    if (warp == 1) {
        tmem_alloc(smem_u32(&tmem_base_s), 512);
        tmem_relinquish();
    }
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    pdl_wait_then_release();
    const uint32_t tmem = tmem_base_s;
    volatile int *abort_flag = &abort_s;
    // unit u -> problem p, batch b, row tile mt, column tile nt
    auto decode = [&](int u, int &p, int &b, int &mt, int &nt) {
        p = 0;
        while (p + 1 < P.n_problems && u >= P.pr[p + 1].unit0) ++p;
        const GemmProblem &g = P.pr[p];
        const int v = u - g.unit0;
        mt = v % g.m_tiles;
        const int r = v / g.m_tiles;
        nt = r % g.n_tiles;
        b = r / g.n_tiles;
    };

    if (warp == 0) {
        if (lane == 0) {
            int stage = 0, a_phase[kGmMaxStages];
            uint32_t phase = 0;
            for (int i = 0; i < kGmMaxStages; ++i) a_phase[i] = -1;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < P.units; u += gridDim.x) {
                int p, b, mt, nt;
                decode(u, p, b, mt, nt);
                const GemmProblem &g = P.pr[p];
                const uint32_t b_blk = static_cast<uint32_t>(g.bn) * 128u;
                const uint32_t bytes = static_cast<uint32_t>(P.kb) * (P.a_bytes + b_blk);
                const int ya = mt * kGmM;
                const int yb = static_cast<int>(b * g.b_batch_off) + nt * g.bn;
                const int a_blk0 = static_cast<int>(b * g.a_batch_off) / kGmK;   // A's first K block of batch b
                const int k_steps = g.k / (kGmK * P.kb);
                for (int ks = 0; ks < k_steps; ++ks) {
                    if (!mbar_wait(empty_bar(stage), phase ^ 1, abort_flag, P.status, P.wait_ns)) {
                        ok = false;
                        break;
                    }
                    const uint32_t dst = s0 + static_cast<uint32_t>(stage) * P.stage_bytes;
                    mbar_expect_tx(full_bar(stage), bytes);
                    if (P.kb == 1) {
                        tma_load_2d(dst, &M.a[p], full_bar(stage), static_cast<int>(b * g.a_batch_off) + ks * kGmK, ya);
                        tma_load_2d(dst + P.a_bytes, &M.b[p], full_bar(stage), ks * kGmK, yb);
                    } else {  // kb K blocks per box: [kb][rows][128 B] slabs, A's then B's
                        tma_load_3d(dst, &M.a[p], full_bar(stage), 0, ya, a_blk0 + ks * P.kb);
                        tma_load_3d(dst + P.kb * P.a_bytes, &M.b[p], full_bar(stage), 0, yb, ks * P.kb);
                    }
                    a_phase[stage] = static_cast<int>(phase);
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
            }
            if (!ok)  // gave up: every load issued lands before the CTA goes away
                for (int i = 0; i < kGmMaxStages; ++i)
                    if (a_phase[i] >= 0) mbar_wait(full_bar(i), static_cast<uint32_t>(a_phase[i]), nullptr, P.status);
        }
    } else if (warp == 1) {
        if (lane == 0) {
            int stage = 0, acc = 0;
            uint32_t phase = 0, acc_phase = 0;
            bool ok = true;
            for (int u = blockIdx.x; ok && u < P.units; u += gridDim.x) {
                int p, b, mt, nt;
                decode(u, p, b, mt, nt);
                const GemmProblem &g = P.pr[p];
                const uint32_t idesc = idesc_bf16_f32(kGmM, g.bn);
                const uint32_t b_blk = static_cast<uint32_t>(g.bn) * 128u;
                const int k_steps = g.k / (kGmK * P.kb);
                if (!(ok = mbar_wait(acce_bar(acc), acc_phase ^ 1, abort_flag, P.status, P.wait_ns))) break;
                const uint32_t d_tmem = tmem + acc * kGmMaxN;
                for (int ks = 0; ks < k_steps; ++ks) {
                    if (!(ok = mbar_wait(full_bar(stage), phase, abort_flag, P.status, P.wait_ns))) break;
                    tc_fence_after();
                    const uint32_t a_base = s0 + static_cast<uint32_t>(stage) * P.stage_bytes;
                    const uint32_t b_base = a_base + static_cast<uint32_t>(P.kb) * P.a_bytes;
                    for (int j = 0; j < P.kb; ++j) {
#pragma unroll
                        for (int kk = 0; kk < kGmK / 16; ++kk) {
                            const uint64_t ad = desc_kmajor_sw128(a_base + j * P.a_bytes + kk * 32);
                            const uint64_t bd = desc_kmajor_sw128(b_base + j * b_blk + kk * 32);
                            tc_mma_bf16(d_tmem, ad, bd, idesc, (ks | j | kk) ? 1u : 0u);
                        }
                    }
                    tc_commit(empty_bar(stage));
                    if (++stage == stages) {
                        stage = 0;
                        phase ^= 1;
                    }
                }
                if (!ok) break;
                tc_commit(accf_bar(acc));
                if (++acc == 2) {
                    acc = 0;
                    acc_phase ^= 1;
                }
            }
            if (!ok) {  // gave up: every MMA issued completes before the TMEM is freed
                tc_commit(drain_bar);
                mbar_wait(drain_bar, 0, nullptr, P.status);
            }
        }
    } else {
        // Epilogue: warp w reads TMEM lanes 32*(w%4) .. +31 (its tile rows);
        // the two warps of a lane quadrant take alternate 32-column chunks.
        const int quad = warp & 3, et = threadIdx.x - 64, half = et >> 7;
        int acc = 0;
        uint32_t acc_phase = 0;
        for (int u = blockIdx.x; u < P.units; u += gridDim.x) {
            int p, b, mt, nt;
            decode(u, p, b, mt, nt);
            const GemmProblem &g = P.pr[p];
            if (!gm_epi_bar_all(mbar_wait(accf_bar(acc), acc_phase, abort_flag, P.status, P.wait_ns))) break;
            tc_fence_after();
            const int row = mt * kGmM + quad * 32 + lane;
            const uint32_t tbase = tmem + acc * kGmMaxN + (static_cast<uint32_t>(quad * 32) << 16);
            const int row0 = mt * kGmM + quad * 32;   // the warp's first row
            for (int ch = half; ch < g.bn / 32; ch += 2) {
                uint32_t r[32];
                tmem_ld_32x32b_x32(tbase + ch * 32, r);
                tmem_ld_wait();
                const int col0 = nt * g.bn + ch * 32;  // column inside the batch
                uint16_t *c0 = static_cast<uint16_t *>(g.c) + static_cast<int64_t>(row0) * g.ldc +
                               b * g.c_batch_off + col0;
                if (!g.c_f32 && col0 + 32 <= g.n && (g.ldc & 7) == 0 &&
                    (reinterpret_cast<uintptr_t>(c0) & 15) == 0) {
                    // bf16 rows through the warp's staging block: lane l writes its
                    // row's four 16-byte pieces (piece slots swizzled by the row, so
                    // neither side conflicts), then 4 lanes per row store 8 rows at a time
                    uint32_t *st = reinterpret_cast<uint32_t *>(smem + kGmOffStage) + (warp - 2) * (kGmStageWarpBytes / 4);
#pragma unroll
                    for (int pc = 0; pc < 4; ++pc)
                        *reinterpret_cast<uint4 *>(st + lane * 16 + ((pc ^ ((lane >> 1) & 3)) << 2)) =
                            make_uint4(pack_bf16x2(__uint_as_float(r[8 * pc]), __uint_as_float(r[8 * pc + 1])),
                                       pack_bf16x2(__uint_as_float(r[8 * pc + 2]), __uint_as_float(r[8 * pc + 3])),
                                       pack_bf16x2(__uint_as_float(r[8 * pc + 4]), __uint_as_float(r[8 * pc + 5])),
                                       pack_bf16x2(__uint_as_float(r[8 * pc + 6]), __uint_as_float(r[8 * pc + 7])));
                    __syncwarp();
                    const int part = lane & 3;
#pragma unroll
                    for (int i = 0; i < 4; ++i) {
                        const int rr = 8 * i + (lane >> 2);
                        const uint4 v = *reinterpret_cast<const uint4 *>(st + rr * 16 + ((part ^ ((rr >> 1) & 3)) << 2));
                        if (row0 + rr < g.m) *reinterpret_cast<uint4 *>(c0 + static_cast<int64_t>(rr) * g.ldc + 8 * part) = v;
                    }
                    __syncwarp();   // the block is rewritten by the next chunk
                } else if (row < g.m && col0 < g.n) {
                    store_row_chunk(g, b, row, col0, r);
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
        tmem_dealloc(tmem, 512);
    }
}

}  // namespace

kp_status launch_gemm_group(const kp_gemm_args *gs, int count, cudaStream_t s) {
    if (count < 1 || count > kGmMaxProblems) return KP_ERR_INVALID_ARG;
    const int sms = device_sm_count();
    if (sms <= 0) return KP_ERR_CUDA;
    GemmMaps maps;
    GemmParams P;
    std::memset(&maps, 0, sizeof maps);
    std::memset(&P, 0, sizeof P);
    int64_t units = 0;
    uint32_t widest = 0;
    // A rows loaded per stage: a product of at most 128 rows loads only its rows
    // (rounded up to 8, one swizzle atom), which leaves ring room for more stages.
    int a_rows = 8;
    for (int i = 0; i < count; ++i) {
        const kp_gemm_args &g = gs[i];
        if (g.m == 0 || g.n == 0) continue;
        const int r = g.m > kGmM ? kGmM : (g.m + 7) / 8 * 8;
        if (r > a_rows) a_rows = r;
    }
    const uint32_t a_bytes = static_cast<uint32_t>(a_rows) * 128u;
    // K blocks per stage: with few rows the tiles are small, and the TMA box
    // count, not the bytes, sets the pace; a box then carries four 64-wide K
    // blocks (fewer where K or a batch offset does not divide).
    int kb = 1;
    if (a_rows < kGmM) {
        kb = 4;
        for (int i = 0; i < count; ++i) {
            const kp_gemm_args &g = gs[i];
            if (g.m == 0 || g.n == 0) continue;
            while (kb > 1 && ((g.k / kGmK) % kb != 0 || g.a_batch_off % kGmK != 0)) kb /= 2;
        }
    }
    for (int i = 0; i < count; ++i) {
        const kp_gemm_args &g = gs[i];
        if (g.m == 0 || g.n == 0) continue;
        // Columns per tile (a multiple of 32, <= 256): the width whose waves of
        // units cost least, a unit's cost taken as (64 + bn) -- its MMA and B
        // bytes grow with bn, its A tile and fixed costs do not.  Large products
        // keep 256; a product of few rows (decode) takes narrow tiles so that
        // every SM streams a share of the weights instead of a few SMs all of it.
        const int64_t m_tiles = (g.m + kGmM - 1) / kGmM;
        int bn = 32;
        int64_t best = -1;
        for (int cand = kGmMaxN; cand >= 32; cand /= 2) {
            const int64_t u = static_cast<int64_t>(g.batch) * m_tiles * ((g.n + cand - 1) / cand);
            const int64_t cost = (u + sms - 1) / sms * (64 + cand);
            if (best < 0 || cost < best) {
                best = cost;
                bn = cand;
            }
        }
        const int p = P.n_problems++;
        const uint64_t a_cols = static_cast<uint64_t>(g.a_batch_off) * (g.batch - 1) + g.k;
        const uint64_t b_rows = static_cast<uint64_t>(g.b_batch_off) * (g.batch - 1) + g.n;
        const bool ok =
            kb == 1 ? make_tmap_bf16_sw128(&maps.a[p], g.a, a_cols, static_cast<uint64_t>(g.m),
                                           static_cast<uint64_t>(g.lda) * 2, kGmK, static_cast<uint32_t>(a_rows)) &&
                          make_tmap_bf16_sw128(&maps.b[p], g.b, static_cast<uint64_t>(g.k), b_rows,
                                               static_cast<uint64_t>(g.ldb) * 2, kGmK, static_cast<uint32_t>(bn))
                    : make_tmap_bf16_sw128_kblocks(&maps.a[p], g.a, a_cols, static_cast<uint64_t>(g.m),
                                                   static_cast<uint64_t>(g.lda) * 2, static_cast<uint32_t>(a_rows),
                                                   static_cast<uint32_t>(kb)) &&
                          make_tmap_bf16_sw128_kblocks(&maps.b[p], g.b, static_cast<uint64_t>(g.k), b_rows,
                                                       static_cast<uint64_t>(g.ldb) * 2, static_cast<uint32_t>(bn),
                                                       static_cast<uint32_t>(kb));
        if (!ok) return KP_ERR_CUDA;
        GemmProblem &q = P.pr[p];
        q.m = g.m;
        q.n = g.n;
        q.k = g.k;
        q.batch = g.batch;
        q.bn = bn;
        q.m_tiles = static_cast<int>(m_tiles);
        q.n_tiles = (g.n + bn - 1) / bn;
        q.unit0 = static_cast<int>(units);
        q.a_batch_off = g.a_batch_off;
        q.b_batch_off = g.b_batch_off;
        q.c = g.c;
        q.ldc = g.ldc;
        q.c_batch_off = g.c_batch_off;
        q.c_f32 = g.c_dtype == KP_DTYPE_F32 ? 1 : 0;
        units += static_cast<int64_t>(g.batch) * q.m_tiles * q.n_tiles;
        const uint32_t stage = static_cast<uint32_t>(kb) * (a_bytes + static_cast<uint32_t>(bn) * 128u);
        if (stage > widest) widest = stage;
        // the first problem's limits stand for the launch (every problem of a
        // call carries the same wait limit and status word)
        if (p == 0) {
            P.wait_ns = wait_limit_ns(g.wait_limit_us);
            P.status = g.d_status;
        }
    }
    if (P.n_problems == 0) return KP_OK;
    if (units > INT32_MAX) return KP_ERR_UNSUPPORTED;
    P.units = static_cast<int>(units);
    P.a_bytes = a_bytes;
    P.kb = kb;
    P.stage_bytes = widest;   // multiples of 1024 (A: 8-row atoms; B: 32-row tiles): stages stay 1024-aligned
    P.stages = static_cast<int>(kGmRingBytes / widest);
    if (P.stages > kGmMaxStages) P.stages = kGmMaxStages;
    cudaError_t e = cudaFuncSetAttribute(gemm_bf16_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kGmSmemBytes);
    if (e != cudaSuccess) {
        record_cuda_error("cudaFuncSetAttribute(gemm_bf16_kernel)", e);
        return KP_ERR_CUDA;
    }
    const int grid = static_cast<int>(units < sms ? units : sms);
    return launch_kernel("gemm_bf16_kernel", gemm_bf16_kernel, LaunchCfg(dim3(grid), dim3(kGmThreads), kGmSmemBytes, s),
                         maps, P);
}

kp_status launch_gemm(const kp_gemm_args &g, cudaStream_t s) { return launch_gemm_group(&g, 1, s); }

}  // namespace kp
