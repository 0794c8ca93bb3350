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
// tokens their M.  64-token tiles of latent rows (64 KB) are gathered into two
// shared-memory slots in the 128-byte-swizzle layout, so the next tile streams
// in while this one is computed; Q takes the other 64 KB, so two slots is all
// that fits.  Measured on B300, an M = 64 or 128, N = 64 product costs about
// 50 cycles per instruction at best (about 75 in this kernel), whatever M is,
// while M = 128 with N = 128 or more runs at the full 4,096 FMA/clk.  So the
// logits come from one M = 128, N = 128 product per K step that stacks the
// two halves of the latent columns (L = columns 0-255, H = 256-511):
//   [C_L; C_H] . [Q_L; Q_H]^T   (A: the tile's 64 rows twice, K-halves L and H;
//                               B: Q's 64 heads twice; K = 256 in 16 steps)
//   S^T[tok, h] = D[tok, h] + D[64 + tok, 64 + h]
// (the off-diagonal blocks are computed and ignored): 16 instructions per tile
// instead of 32 at N = 64.  The tile and Q keep each 64-column block j at
// block position 2(j % 4) + j / 4, so blocks j and j + 4 sit next to each other
// and every such pair is one K-major 128-row operand (8-row groups 1 KB apart).
//   O^T[d, h] += C[tok, d]^T . P[tok, h]   M = 128 latent columns (x4), N = 64, K = 64 tokens
// reads the same pairs M-major: chunk c of O^T holds columns 64c + i (lane i <
// 64) and 256 + 64c + i (lane 64 + i).  Each latent row crosses HBM once.  A
// selected pool is kpool = 4 consecutive latent rows, so the gather is a plain
// tiled TMA load per (pool, 64-column block): a 4-row box of 512 bytes that
// lands at a 512-byte offset of its 1 KB swizzle atom (the swizzle follows the
// shared-memory address, so a half atom gets the rows 4-7 pattern).  Pools
// missing from a partial tile load rows at a negative coordinate, which the
// TMA fills with zeros, so P.V never multiplies stale bytes.  D (two buffers
// of 128 columns) and O^T (4 x 64 columns) live in TMEM.  A token's two
// partial logits sit in lane quadrants q and q + 2, read by different warps:
// each warp pair swaps half of its 32 heads through shared memory, so each
// thread ends with 1 token x 16 heads.  The running max is raised only when a
// tile's max exceeds it by 2^8 (then O^T and the row sums are rescaled), so
// the correction pass almost never runs.
//
// A query's token list is split over the S CTAs of a thread-block cluster
// (up to 8; any count but 7).  After its tiles, each CTA dumps its
// unnormalised O^T to its own shared memory and sends each head's running max
// and row sum to the CTA that merges the head; after a cluster barrier, CTA r
// merges heads [64r/S, 64(r+1)/S) (rounded down) across the cluster through
// distributed shared memory, adds the <= kpool - 1 tail tokens (computed on
// CUDA cores, so the tail never costs a tensor-core tile), normalises and
// writes bf16 out and fp32 lse.  No global scratch, no second launch.
//
// Warp roles (416 threads, one CTA per SM):
//   warps 0-7  softmax: warp w reads TMEM lane quadrant w % 4 (tokens
//              32 (w % 2) .. +31; column half (w % 4) / 2) and ends with heads
//              32 (w / 4) + 16 ((w % 4) / 2) .. +15 of its token; then the O^T dump
//   warp 8     TMEM allocation, Q TMA, MMA issue (one lane)
//   warps 9-12 gather: all four load each 128-column chunk of a tile in turn,
//              8 TMA boxes per warp per chunk (TMA issue is serial within a
//              warp, so four warps issue at four times the rate of one)
//   all        cluster merge and output
#include <atomic>

#include "kp_common.cuh"
#include "kp_internal.h"

namespace kp {

namespace {

constexpr int kAtTok = 64;                                // tokens per tile (16 pools)
constexpr int kAtSlots = 2;                               // tiles resident in shared memory
constexpr int kAtChunks = 4;                              // 128-column chunks of a latent row
constexpr int kAtBlockBytes = kAtTok * 128;               // [64 rows][64 bf16] swizzle block, 8 KB
constexpr int kAtChunkBytes = 2 * kAtBlockBytes;          // 16 KB
constexpr int kAtTileBytes = kAtChunks * kAtChunkBytes;   // 64 KB
constexpr int kAtQBlockBytes = kMlaHeads * 128;           // [64 heads][64 bf16] = 8 KB
constexpr int kAtQBytes = 8 * kAtQBlockBytes;             // 64 KB
constexpr int kAtPBytes = kAtTok * kMlaHeads * 2;         // 8 KB per buffer (two buffers)
constexpr int kAtMaxSplits = 8;
constexpr int kAtSoftWarps = 8;
constexpr int kAtSoftThreads = 32 * kAtSoftWarps;
constexpr int kAtMmaWarp = 8;
constexpr int kAtProdWarp0 = 9;
constexpr int kAtProdWarps = 4;                           // TMA gather warps
constexpr int kAtThreads = 416;
static_assert(kAtThreads == 32 * (kAtSoftWarps + 1 + kAtProdWarps), "softmax, MMA and gather warps");
static_assert(kAtTok % 16 == 0 && kAtTok <= 64, "a tile is whole K-steps of P.V and fits the M = 64 product");
static_assert(kAtBlockBytes % 1024 == 0, "blocks start on a swizzle atom");
constexpr int kAtTmemCols = 512;
constexpr uint32_t kAtOCol = 0;                           // O^T: chunk c at columns 64c .. 64c+63
constexpr uint32_t kAtSCol = 256;                         // D (stacked logits): two buffers of 128 columns
constexpr float kAtRescaleLog2 = 8.f;                     // raise the running max only past 2^8
// Softmax exchange during the tile loop, in the merge buffers' place: per warp
// pair (token half, head half) and direction, [16 heads][32 tokens] f32.
constexpr int kAtXBytes = 4 * 2 * 16 * 32 * 4;
static_assert(kAtTok == 64, "the stacked S product and the softmax assume 64-token tiles");

// Shared-memory position of 64-column block j of a tile or of Q: blocks j and
// j + 4 (the two K-halves of one S step) are adjacent.
__host__ __device__ constexpr int at_block_pos(int j) { return 2 * (j & 3) + (j >> 2); }

// Shared memory (offsets from a 1024-aligned base).  During the tile loop:
// Q, the tile slots, the two P buffers and a small block of per-head state and
// barriers.  After the loop the slots hold this CTA's O^T dump, which the
// cluster's CTAs read; the merge's small buffers (tail rows and logits, merge
// weights, row-sum partials) follow it in the slots when they fit there, else
// they sit after the barriers.
constexpr int kOffQ = 0;
constexpr int kOffTile = kOffQ + kAtQBytes;               // slots; then this CTA's O^T dump
constexpr int kOffP = kOffTile + kAtSlots * kAtTileBytes;
constexpr int kOffMisc = kOffP + 2 * kAtPBytes;
constexpr int kMiscRed = 0;                               // [2][64] f32 per-token-half tile maxima
constexpr int kMiscMUsed = kMiscRed + 2 * 64 * 4;         // [64] f32 running max (log2 units)
constexpr int kMiscFac = kMiscMUsed + 64 * 4;             // [64] f32 rescale factors of this tile
constexpr int kMiscLSum = kMiscFac + 64 * 4;              // [64] f32 row sums
constexpr int kAtRecvSlots = 66;                          // max over splits S != 7 of S x ceil(64 / S)
constexpr int kMiscRecv = kMiscLSum + 64 * 4;             // [2][kAtRecvSlots] f32 running maxima, row
                                                          // sums of the heads this CTA merges,
                                                          // [head][split], from every CTA of the cluster
constexpr int kMiscBars = kMiscRecv + 2 * kAtRecvSlots * 4;   // mbarriers
constexpr int kNumBars = 4 * kAtSlots * 2 + 9;
constexpr int kMiscTmem = kMiscBars + kNumBars * 8;
constexpr int kMiscAbort = kMiscTmem + 4;
constexpr int kMiscCore = (kMiscAbort + 12 + 15) / 16 * 16;
constexpr int kMrgOBytes = kMlaHeads * kNopeDim * 4;      // [64 heads][512] f32 dump of this CTA's O^T
static_assert(kMrgOBytes <= kAtSlots * kAtTileBytes, "the O^T dump must fit in the tile slots");

// What depends on the pool size KP (tokens per pool, 4 or 16): a pool is KP
// consecutive latent rows, gathered as one TMA box of KP rows per 64-column
// block; the tail holds up to KP - 1 rows.  After the tile loop the tail rows
// sit in the P buffers' place, and the merge's small buffers after the
// barriers: tail logits [64][KP], merge weights [64][kWStride] (splits 0..7,
// tail tokens 8.., 1/L at kWInv) and row-sum partials [4][64].
template <int KP>
struct AtPool {
    static constexpr int kMaxTail = KP - 1;
    static constexpr int kPoolsPerTile = kAtTok / KP;     // 16 pools of 4 rows, or 4 of 16
    static constexpr int kBoxBytes = KP * 128;           // one pool's rows of one 64-column block
    static constexpr int kWInv = 8 + kMaxTail;
    static constexpr int kWStride = (kWInv + 1 + 15) / 16 * 16;
    static constexpr int kWF4 = (kWInv + 1 + 3) / 4;     // float4 loads that cover a weight row
    static constexpr int kZTail = 0;
    static constexpr int kW = kZTail + kMlaHeads * KP * 4;
    static constexpr int kLPart = kW + kMlaHeads * kWStride * 4;
    static constexpr int kAuxBytes = kLPart + 4 * kMlaHeads * 4;
    static constexpr int kOffAux = kOffMisc + kMiscCore;
    static constexpr int kSmemBytes = kOffMisc + kMiscCore + (kAuxBytes > kAtXBytes ? kAuxBytes : kAtXBytes) +
                                      1024;  // + alignment slack
    static_assert(kPoolsPerTile * 2 <= 32, "a gather lane per (pool, block) of a 128-column chunk");
    static_assert(kMaxTail * kNopeDim * 2 <= 2 * kAtPBytes, "the tail rows fit in the P buffers");
    static_assert(kSmemBytes <= 232448, "attention shared memory over the per-CTA limit");
};

// mbarrier indices
constexpr int kBarFull = 0;                        // [slot][4] chunk gathered (one arrival + TMA bytes)
constexpr int kBarFree = kBarFull + 4 * kAtSlots;  // [slot][4] chunk consumed by P.V (tcgen05.commit)
constexpr int kBarQ = kBarFree + 4 * kAtSlots;     // Q landed (TMA)
constexpr int kBarS = kBarQ + 1;                   // [2] S^T buffer ready (commit)
constexpr int kBarP = kBarS + 2;                   // [2] P buffer written, O^T rescaled (256 softmax arrivals)
constexpr int kBarO = kBarP + 2;                   // every MMA of the CTA done (commit)
constexpr int kBarDrain = kBarO + 1;               // teardown after an abort
constexpr int kBarPV = kBarDrain + 1;              // P.V of a tile done (commit): O^T is stable
constexpr int kBarNever = kBarPV + 1;              // nothing arrives (failure-path tests)
static_assert(kBarNever + 1 == kNumBars, "barrier count");

struct AttendParams {
    const uint16_t *latent;
    CacheMap cmap;               // where each sequence's latent rows live
    const int32_t *q_seq;
    const int32_t *q_pos;
    const int32_t *seq_len;
    int num_seqs;
    const int32_t *pool_idx;
    const int32_t *n_sel;
    const int32_t *share_src;    // [nq] shared selection (nullptr: none)
    int nq;
    int K;
    int tail;
    float scale_log2;
    uint16_t *out;
    float *lse;
    int splits;
    int32_t *status;
    unsigned long long wait_ns;  // limit of one pipeline wait
    int stall;                   // KP_DEBUG_STALL_FIRST_WAIT: the MMA warp's first wait never completes
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

// Named barrier that ORs a flag over the participating threads.
__device__ __forceinline__ bool named_bar_any(int id, int count, bool v) {
    uint32_t r;
    asm volatile(
        "{\n\t.reg .pred p, q;\n\t"
        "setp.ne.u32 q, %1, 0;\n\t"
        "bar.red.or.pred p, %2, %3, q;\n\t"
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

template <int KP>
__global__ void __launch_bounds__(kAtThreads, 1)
    sparse_mla_tc_kernel(const __grid_constant__ CUtensorMap tm_q, const __grid_constant__ CUtensorMap tm_lat,
                         AttendParams P) {
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
    float *recv_m = reinterpret_cast<float *>(misc + kMiscRecv);
    float *recv_l = recv_m + kAtRecvSlots;
    using Pool = AtPool<KP>;
    constexpr int kAtMaxTail = Pool::kMaxTail;
    constexpr int kAtPoolsPerTile = Pool::kPoolsPerTile;
    constexpr int kWS = Pool::kWStride, kWInv = Pool::kWInv;
    uint8_t *aux = smem + Pool::kOffAux;  // merge buffers: valid only after the tile loop
    float *lpart_s = reinterpret_cast<float *>(aux + Pool::kLPart);
    uint16_t *tail_s = reinterpret_cast<uint16_t *>(smem + kOffP);   // the P buffers' place
    float *ztail_s = reinterpret_cast<float *>(aux + Pool::kZTail);
    float *wm_s = reinterpret_cast<float *>(aux + Pool::kW);
    const uint32_t bar0 = sbase + kOffMisc + kMiscBars;
    auto bar = [&](int i) { return bar0 + 8u * static_cast<uint32_t>(i); };
    uint32_t *tmem_s = reinterpret_cast<uint32_t *>(misc + kMiscTmem);
    int *abort_s = reinterpret_cast<int *>(misc + kMiscAbort);
    volatile int *abort_flag = abort_s;

    const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
    const int S = P.splits;
    const int q = blockIdx.x / S, split = blockIdx.x % S;
    // Heads this CTA merges: [64 split / S, 64 (split + 1) / S), 64 / S rounded
    // either way when S does not divide 64.
    const int h0 = kMlaHeads * split / S;
    const int nh = kMlaHeads * (split + 1) / S - h0;

    // ---- set-up, and what this query is: inputs no earlier kernel of the step
    // writes, so they are read before the grid dependency resolves.
    if (tid == 0) {
        for (int c = 0; c < kAtSlots * kAtChunks; ++c) {
            mbar_init(bar(kBarFull + c), 1);
            mbar_init(bar(kBarFree + c), 1);
        }
        mbar_init(bar(kBarQ), 1);
        mbar_init(bar(kBarS), 1);
        mbar_init(bar(kBarS + 1), 1);
        mbar_init(bar(kBarPV), 1);
        mbar_init(bar(kBarP), kAtSoftThreads);
        mbar_init(bar(kBarP + 1), kAtSoftThreads);
        mbar_init(bar(kBarO), 1);
        mbar_init(bar(kBarDrain), 1);
        mbar_init(bar(kBarNever), 1);
        fence_mbar_init();
        *abort_s = 0;
        tma_prefetch_desc(&tm_q);
        tma_prefetch_desc(&tm_lat);
    }
    if (tid < kMlaHeads) {
        mused_s[tid] = -INFINITY;
        lsum_s[tid] = 0.f;
    }
    if (warp == kAtMmaWarp) {
        tmem_alloc(smem_u32(tmem_s), kAtTmemCols);
        tmem_relinquish();
    }
    const int b = P.q_seq[q];
    const int t = P.q_pos[q];
    bool qvalid = b >= 0 && b < P.num_seqs && t >= 0;
    const bool paged = P.cmap.paged();
    int64_t base_row = (qvalid && !paged) ? P.cmap.latent_row_off[b] : 0;
    if (qvalid && t >= P.seq_len[b]) qvalid = false;   // a query sits inside its sequence
    if (qvalid && !paged && (base_row < 0 || base_row + t >= P.cmap.latent_rows)) qvalid = false;
    if (qvalid && paged && (t >> P.cmap.page_shift) >= P.cmap.blocks_per_seq) qvalid = false;
    if (!qvalid && tid == 0) set_status(P.status, KP_ERR_DEVICE_BOUNDS);
    // The selection row this query attends: its own, or a shared source's (a
    // query of the same sequence that selects for itself); a bad source leaves
    // the query its tail alone.
    int sel_row = q;
    bool sel_ok = true;
    if (qvalid && P.share_src) {
        const int src = P.share_src[q];
        if (src >= 0) {
            if (src < P.nq && P.q_seq[src] == b && P.share_src[src] < 0) {
                sel_row = src;
            } else {
                sel_ok = false;
                if (tid == 0) set_status(P.status, KP_ERR_DEVICE_BOUNDS);
            }
        }
    }
    const int nf = qvalid ? (t + 1) / KP : 0;
    const int n_tail = (qvalid && P.tail) ? (t + 1) - nf * KP : 0;
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    const uint32_t tmem = *tmem_s;
    if (tid == 32 * kAtMmaWarp && qvalid) {  // Q: 64 heads x 512 columns, 8 swizzled blocks
        mbar_expect_tx(bar(kBarQ), kAtQBytes);
        for (int blk = 0; blk < 8; ++blk)
            tma_load_2d(sQ + at_block_pos(blk) * kAtQBlockBytes, &tm_q, bar(kBarQ), blk * 64, q * kMlaHeads);
    }

    // ---- the selection comes from the previous kernel
    pdl_wait_then_release();
    int ns = 0;
    if (qvalid && sel_ok) {
        ns = P.n_sel[sel_row];
        const int ns_max = min(P.K, nf);
        if (ns < 0 || ns > ns_max) {
            if (tid == 0) set_status(P.status, KP_ERR_DEVICE_BOUNDS);
            ns = max(0, min(ns, ns_max));
        }
    }
    const int n_pool_tok = ns * KP;
    const int n_tiles = (n_pool_tok + kAtTok - 1) / kAtTok;
    const int tb = n_tiles * split / S, te = n_tiles * (split + 1) / S;
    const int nt = te - tb;

    if (warp == kAtMmaWarp) {
        // ------------------------------------------------------------ MMA issuer
        // S(t) chunk by chunk as the gather lands it; P.V(t - 1) as soon as its P
        // is written, even between S(t)'s chunks, so tile t - 1's slot goes back
        // to the gather without waiting for tile t's data.  S(t) reuses the S^T
        // buffer of tile t - 2, so P.V(t - 2) (after its P) is issued before it.
        // The thread polls with test_wait: a suspended thread would wake late
        // with the pipe idle.
        if (lane == 0) {
            bool ok = !P.stall || mbar_wait(bar(kBarNever), 0, abort_flag, P.status, P.wait_ns);
            ok = ok && (nt == 0 || mbar_wait(bar(kBarQ), 0, abort_flag, P.status, P.wait_ns));
            const uint32_t idesc_s = idesc_bf16_f32(128, 2 * kMlaHeads);            // stacked K-halves
            const uint32_t idesc_pv = idesc_bf16_f32(128, kMlaHeads, true, true);   // M = 128 columns
            // Descriptors are built once; a step along K or to another block adds
            // (bytes >> 4) to the start-address field (addresses stay < 256 KB).
            const uint64_t dq0 = desc_sw128(sQ, 16, 1024);
            const uint64_t dt0 = desc_sw128(sTile, 16, 1024);
            // A of P.V = C^T, M-major: 64-column groups 8 KB apart, 8-token groups 1 KB apart.
            const uint64_t dv0 = desc_sw128(sTile, kAtBlockBytes, 1024);
            // B of P.V = P (tokens x heads), N-major, one 64-head group wide.
            const uint64_t dp0 = desc_sw128(sP, 4096, 1024);
            int pv_next = 0;  // oldest tile whose P.V is not issued yet
            auto issue_pv = [&]() {
                const int tp = pv_next, slot = tp % kAtSlots, pbuf = tp & 1;
                tc_fence_after();
#pragma unroll
                for (int c = 0; c < kAtChunks; ++c) {
#pragma unroll
                    for (int kk = 0; kk < kAtTok / 16; ++kk) {
                        const uint64_t ad = dv0 + ((slot * kAtTileBytes + 2 * c * kAtBlockBytes + kk * 2048) >> 4);
                        const uint64_t bd = dp0 + ((pbuf * kAtPBytes + kk * 2048) >> 4);
                        tc_mma_bf16(tmem + kAtOCol + 64 * c, ad, bd, idesc_pv, (tp | kk) ? 1u : 0u);
                    }
                    tc_commit(bar(kBarFree + slot * kAtChunks + c));
                }
                tc_commit(bar(kBarPV));
                ++pv_next;
            };
            for (int t = 0; ok && t < nt; ++t) {
                if (pv_next < t - 1) {  // P.V(t - 2): frees the S^T buffer S(t) writes
                    ok = mbar_spin(bar(kBarP + (pv_next & 1)), (pv_next >> 1) & 1, abort_flag, P.status, P.wait_ns);
                    if (!ok) break;
                    issue_pv();
                }
                const int slot = t % kAtSlots, sbuf = t & 1;
                for (int c = 0; ok && c < kAtChunks; ++c) {
                    const uint32_t fb = bar(kBarFull + slot * kAtChunks + c);
                    const uint32_t fpar = (t / kAtSlots) & 1;
                    if (!mbar_test(fb, fpar)) {
                        const unsigned long long t0 = globaltimer_ns();
                        for (uint32_t it = 1;; ++it) {
                            if (pv_next < t && mbar_test(bar(kBarP + (pv_next & 1)), (pv_next >> 1) & 1)) issue_pv();
                            if (mbar_test(fb, fpar)) break;
                            if ((it & 255u) == 0 &&
                                (*abort_flag || globaltimer_ns() - t0 > P.wait_ns)) {
                                set_status(P.status, KP_ERR_DEVICE_TIMEOUT);
                                *abort_flag = 1;
                                ok = false;
                                break;
                            }
                        }
                        if (!ok) break;
                    }
                    tc_fence_after();
                    // Chunk c holds blocks c and c + 4 (positions 2c, 2c + 1): the
                    // tile's rows over both K-halves as A, Q's heads over both as B.
#pragma unroll
                    for (int kk = 0; kk < 4; ++kk) {
                        const uint64_t ad = dt0 + ((slot * kAtTileBytes + c * kAtChunkBytes + kk * 32) >> 4);
                        const uint64_t bd = dq0 + ((2 * c * kAtQBlockBytes + kk * 32) >> 4);
                        tc_mma_bf16(tmem + kAtSCol + 128 * sbuf, ad, bd, idesc_s, (c | kk) ? 1u : 0u);
                    }
                }
                if (!ok) break;
                tc_commit(bar(kBarS + sbuf));
            }
            while (ok && pv_next < nt) {  // the last tiles' P.V
                ok = mbar_spin(bar(kBarP + (pv_next & 1)), (pv_next >> 1) & 1, abort_flag, P.status, P.wait_ns);
                if (ok) issue_pv();
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
        // A tile is 4 chunks of 32 TMA boxes (16 pools x 2 64-column blocks).
        // The four warps load every chunk together, chunk by chunk: lanes 8c ..
        // 8c + 7 of warp w issue boxes j = 4 (l % 8) + w of chunk c (pool j % 16,
        // latent column block c + 4 (j / 16)), so chunk 0 of a tile lands first and the S product
        // starts on it while chunks 1-3 are still in flight.  Warp 0 posts each
        // chunk's byte count (boxes of other warps may land before it: the
        // transaction count may go negative, the phase cannot complete without
        // this arrival).  Each lane reads its pool index two tiles ahead and,
        // with paged caches, the page of that pool one tile ahead, so no
        // global read sits between a freed slot and its refill.
        const int w = warp - kAtProdWarp0;
        const int my_chunk = lane >> 3, j = 4 * (lane & 7) + w;
        // chunk c = latent column blocks c and c + 4, at block positions 2c and 2c + 1
        const int my_pool = j % kAtPoolsPerTile, khalf = j / kAtPoolsPerTile;
        const int blk = my_chunk + 4 * khalf, spos = 2 * my_chunk + khalf;
        const bool active = j < 2 * kAtPoolsPerTile;
        const int pool0 = tb * kAtPoolsPerTile;
        const int npools = min(nt * kAtPoolsPerTile, ns - pool0);
        const int32_t *plist = P.pool_idx + static_cast<int64_t>(sel_row) * P.K + pool0 + my_pool;
        auto want = [&](int t) -> bool { return active && t * kAtPoolsPerTile + my_pool < npools; };
        auto fetch_p = [&](int t) -> int { return want(t) ? plist[t * kAtPoolsPerTile] : -1; };
        // Raw block-table entry of pool p's page (checked where it is used), -2
        // when p itself is out of range; 0 for contiguous caches.
        auto fetch_pg = [&](int p) -> int {
            if (!paged) return 0;
            if (p < 0 || p >= nf) return -2;
            const int blk = (p * KP) >> P.cmap.page_shift;
            if (blk >= P.cmap.blocks_per_seq) return -2;
            return P.cmap.block_table[static_cast<int64_t>(b) * P.cmap.blocks_per_seq + blk];
        };
        // First row of this lane's pool in tile t, or a coordinate wholly above
        // row 0 (zero fill) for a pool past the end of the list or out of range.
        auto row_at = [&](int t, int p, int pg) -> int {
            if (!want(t)) return -KP;
            bool good = p >= 0 && p < nf;
            int64_t r = 0;
            if (good && !paged) r = base_row + static_cast<int64_t>(p) * KP;
            if (good && paged) {
                good = pg >= 0 && pg < P.cmap.num_pages;
                r = (static_cast<int64_t>(pg) << P.cmap.page_shift) +
                    ((p * KP) & ((1 << P.cmap.page_shift) - 1));
            }
            if (!good) {
                set_status(P.status, KP_ERR_DEVICE_BOUNDS);
                return -KP;
            }
            return static_cast<int>(r);
        };
        int pf_p[kAtSlots], pf_pg[kAtSlots];
        pf_p[0] = fetch_p(0);
        pf_p[1] = fetch_p(1);
        pf_pg[0] = fetch_pg(pf_p[0]);
        pf_pg[1] = 0;
        bool ok = true;
        int issued[kAtSlots][kAtChunks];   // latest tile whose chunk this warp loaded, per slot
#pragma unroll
        for (int u = 0; u < kAtSlots; ++u)
#pragma unroll
            for (int cc = 0; cc < kAtChunks; ++cc) issued[u][cc] = -1;
        for (int j0 = 0; ok && j0 < nt; j0 += kAtSlots) {
#pragma unroll
            for (int u = 0; u < kAtSlots; ++u) {  // tile jj = j0 + u lives in slot u
                const int jj = j0 + u;
                if (!ok || jj >= nt) break;
                const int y = row_at(jj, pf_p[u], pf_pg[u]);
                pf_pg[u ^ 1] = fetch_pg(pf_p[u ^ 1]);   // page of tile jj + 1's pool
                pf_p[u] = fetch_p(jj + kAtSlots);       // pool of tile jj + 2
                const uint32_t dst = sTile + u * kAtTileBytes + spos * kAtBlockBytes + my_pool * Pool::kBoxBytes;
#pragma unroll
                for (int cc = 0; cc < kAtChunks; ++cc) {
                    if (jj >= kAtSlots) {  // P.V of the slot's previous tile has read this chunk
                        ok = __all_sync(0xffffffffu, mbar_wait(bar(kBarFree + u * kAtChunks + cc),
                                                              ((jj / kAtSlots) - 1) & 1, abort_flag, P.status,
                                                              P.wait_ns));
                        if (!ok) break;
                    }
                    const uint32_t fb = bar(kBarFull + u * kAtChunks + cc);
                    if (w == 0 && lane == 0) mbar_expect_tx(fb, kAtChunkBytes);
                    if (my_chunk == cc && active) tma_load_2d(dst, &tm_lat, fb, blk * 64, y);
                    issued[u][cc] = jj;
                }
            }
        }
        if (!ok) {
            // Every load this warp issued lands before the shared memory is reused
            // (bounded: a chunk whose other boxes were never issued times out).
#pragma unroll
            for (int u = 0; u < kAtSlots; ++u)
#pragma unroll
                for (int cc = 0; cc < kAtChunks; ++cc)
                    if (issued[u][cc] >= 0)
                        mbar_wait(bar(kBarFull + u * kAtChunks + cc), (issued[u][cc] / kAtSlots) & 1, nullptr,
                                  P.status);
        }
    } else {
        // ------------------------------------------------------------ softmax
        // D lane i < 64 holds token i's logits over the first column half
        // (heads in columns 0-63), lane 64 + i the same token's over the second
        // (heads in columns 64-127).  Warp w reads lane quadrant w % 4, columns
        // of head half w / 4: quadrants 0-1 (tokens 0-31, 32-63) the first
        // column half, 2-3 the second.  Warps w and w ^ 2 hold the same tokens:
        // each sends the other 16 of its 32 heads' partial sums through shared
        // memory, so each thread ends with its token's logits for 16 heads.
        const int quad = warp & 3, half = warp >> 2;
        const int second = quad >> 1;                      // reads the second column half
        const int tk = 32 * (quad & 1) + lane;             // this thread's token in the tile
        const int hb = 32 * half + 16 * second;            // this thread's first head
        const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
        const uint32_t scol = kAtSCol + 64 * second + 32 * half;
        float *xbuf = reinterpret_cast<float *>(smem + Pool::kOffAux);   // the merge buffers' place
        float *xsend = xbuf + (((quad & 1) * 2 + half) * 2 + second) * 512;        // [16][32] f32
        const float *xrecv = xbuf + (((quad & 1) * 2 + half) * 2 + (second ^ 1)) * 512;
        const int pair_bar = 3 + (quad & 1) * 2 + half;    // named barrier of warps w, w ^ 2
        // Per head k (head hb + k): row-sum partial and running max (log2 units,
        // a copy of mused_s).
        float lp[16], mr[16];
#pragma unroll
        for (int k = 0; k < 16; ++k) {
            lp[k] = 0.f;
            mr[k] = -INFINITY;
        }
        bool ok = true;
        for (int jj = 0; jj < nt; ++jj) {
            ok = named_bar_all(1, kAtSoftThreads,
                               mbar_wait(bar(kBarS + (jj & 1)), (jj >> 1) & 1, abort_flag, P.status, P.wait_ns));
            if (!ok) break;
            tc_fence_after();
            uint32_t r[32];   // heads 32 half + 0..31, this column half's partial sums
            tmem_ld_32x32b_x32(tmem + lane_base + scol + 128 * (jj & 1), r);
            tmem_ld_wait();
            // The partner's heads go out (the first-half warp keeps heads 0-15 of
            // the half, the second-half warp heads 16-31).
#pragma unroll
            for (int k = 0; k < 16; ++k) xsend[k * 32 + lane] = __uint_as_float(second ? r[k] : r[16 + k]);
            named_bar(pair_bar, 64);
            const int n_valid = min(kAtTok, n_pool_tok - (tb + jj) * kAtTok);
            const bool valid = tk < n_valid;
            float x[16];
            bool high = false;  // a logit more than 2^8 above the running max
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                const float mine = __uint_as_float(second ? r[16 + k] : r[k]);
                const float other = xrecv[k * 32 + lane];
                const float z = second ? other + mine : mine + other;   // first half + second half
                x[k] = valid ? z * P.scale_log2 : -INFINITY;
                high |= x[k] > mr[k] + kAtRescaleLog2;
            }
            bool rescale = false;
            if (named_bar_any(1, kAtSoftThreads, high)) {
                // Slow path (the first tile, and whenever a head's max jumps): exact
                // per-head tile max, raise the running max, rescale O^T and row sums.
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    float m = x[k];
#pragma unroll
                    for (int o = 16; o > 0; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
                    if (lane == 0) red_s[(quad & 1) * 64 + hb + k] = m;
                }
                named_bar(1, kAtSoftThreads);
                if (tid < kMlaHeads) {
                    const float mt = fmaxf(red_s[tid], red_s[64 + tid]);
                    const float mo = mused_s[tid];
                    if (mt > mo + kAtRescaleLog2) {
                        mused_s[tid] = mt;
                        fac_s[tid] = fast_exp2(mo - mt);  // 0 when mo = -inf
                    } else {
                        fac_s[tid] = 1.f;
                    }
                }
                named_bar(1, kAtSoftThreads);
#pragma unroll
                for (int k = 0; k < 16; ++k) {
                    lp[k] *= fac_s[hb + k];
                    mr[k] = mused_s[hb + k];
                }
                rescale = jj > 0;
            }
            // p = 2^(x - m), row partial sums, and this token's 16 heads of P as
            // two 16-byte pieces of its 128-byte row (128-byte swizzle).
            {
                uint8_t *pt = smem + kOffP + (jj & 1) * kAtPBytes;
                uint32_t pk[8];
#pragma unroll
                for (int g = 0; g < 8; ++g) {
                    const float p0 = fast_exp2(x[2 * g] - mr[2 * g]);
                    const float p1 = fast_exp2(x[2 * g + 1] - mr[2 * g + 1]);
                    lp[2 * g] += p0;
                    lp[2 * g + 1] += p1;
                    pk[g] = pack_bf16x2(p0, p1);
                }
                const int c0 = hb >> 3;
                *reinterpret_cast<uint4 *>(pt + tk * 128 + ((c0 ^ (tk & 7)) << 4)) =
                    make_uint4(pk[0], pk[1], pk[2], pk[3]);
                *reinterpret_cast<uint4 *>(pt + tk * 128 + (((c0 + 1) ^ (tk & 7)) << 4)) =
                    make_uint4(pk[4], pk[5], pk[6], pk[7]);
            }
            if (rescale) {
                // O^T must hold P.V of the previous tile before it is rescaled; P.V of
                // this tile waits for our arrival below.  Warp w rescales O^T lanes of
                // quadrant w % 4, heads 32 (w / 4) .. +31, in every chunk.
                mbar_wait(bar(kBarPV), (jj - 1) & 1, abort_flag, P.status, P.wait_ns);
                tc_fence_after();
                for (int c = 0; c < 2 * kAtChunks; ++c) {  // 16 heads at a time
                    uint32_t o[16];
                    const int h0c = 32 * half + 16 * (c & 1);
                    const uint32_t ta = tmem + lane_base + kAtOCol + 64 * (c >> 1) + h0c;
                    tmem_ld_32x32b_x16(ta, o);
                    tmem_ld_wait();
#pragma unroll
                    for (int h = 0; h < 16; ++h) o[h] = __float_as_uint(__uint_as_float(o[h]) * fac_s[h0c + h]);
                    tmem_st_32x32b_x16(ta, o);
                }
                tmem_st_wait();
            }
            fence_proxy_async_smem();
            tc_fence_before();
            mbar_arrive(bar(kBarP + (jj & 1)));
        }
        if (ok) ok = named_bar_all(1, kAtSoftThreads, mbar_wait(bar(kBarO), 0, abort_flag, P.status, P.wait_ns));
        if (ok) {
            tc_fence_after();
            // Row sums over the warp's 32 tokens (fixed order); the two token
            // halves are added in order below.  (Every exchange read is done:
            // the barrier above follows the last tile.)
#pragma unroll
            for (int k = 0; k < 16; ++k) {
                float v = lp[k];
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
                if (lane == 0) lpart_s[(quad & 1) * 64 + hb + k] = v;
            }
        }
    }

    // ---- merge over the cluster (pull).  Every CTA dumps its unnormalised O^T
    // into its own tile slots as [head][512] f32 while warps 8-12 stage the
    // tail rows and compute the tail logits of this CTA's heads; after one
    // cluster barrier, CTA r reads heads [64r/S, 64(r+1)/S) of every CTA's dump,
    // running max and row sums through distributed shared memory (16-byte
    // loads), merges them in split order with the tail and writes out and lse;
    // a second barrier keeps every dump alive until its readers are done.
    // (Measured on B300: pushing with 4- or 16-byte remote stores into a
    // receive buffer, or keeping more remote loads in flight, was slower.)
    tc_fence_before();
    __syncthreads();
    const bool aborted = *abort_flag != 0;
    float *dump = reinterpret_cast<float *>(smem + kOffTile);   // [64 heads][512] f32
    if (warp < kAtSoftWarps) {
        if (tid < kMlaHeads && nt > 0)  // row sums in a fixed order: repeated calls give the same bits
            lsum_s[tid] = lpart_s[tid] + lpart_s[64 + tid];
        if (S > 1 && tid < kMlaHeads) {
            // Head tid's running max and row sum go to the CTA that merges it, so
            // the merge weights read local memory after the cluster barrier.
            const int r = (tid * S + S - 1) / kMlaHeads;          // the CTA whose head range holds tid
            const int hl = tid - kMlaHeads * r / S;
            dsmem_st_f32(dsmem_addr(smem_u32(recv_m + hl * S + split), r), mused_s[tid]);
            dsmem_st_f32(dsmem_addr(smem_u32(recv_l + hl * S + split), r), lsum_s[tid]);
        }
        if (!aborted && nt > 0) {
            tc_fence_after();
            const int quad = warp & 3, hb = (warp >> 2) * 32;
            const uint32_t lane_base = static_cast<uint32_t>(quad * 32) << 16;
            for (int c = 0; c < 2 * kAtChunks; ++c) {  // 16 heads at a time
                uint32_t o[16];
                const int h0c = hb + 16 * (c & 1);
                tmem_ld_32x32b_x16(tmem + lane_base + kAtOCol + 64 * (c >> 1) + h0c, o);
                tmem_ld_wait();
                // O^T lane i of chunk cc is latent column 64 cc + i (i < 64), else 256 + 64 cc + i - 64
                const int d = 64 * (c >> 1) + 256 * (quad >> 1) + 32 * (quad & 1) + lane;
#pragma unroll
                for (int h = 0; h < 16; ++h) dump[(h0c + h) * kNopeDim + d] = __uint_as_float(o[h]);
            }
        }
    } else if (qvalid && !aborted) {
        constexpr int kTailThreads = kAtThreads - kAtSoftThreads;
        const int t2 = tid - kAtSoftThreads;
        for (int k = t2; k < n_tail * 64; k += kTailThreads) {
            const int j = k >> 6, piece = k & 63;
            const int64_t row = paged ? P.cmap.latent_row(b, nf * KP + j)
                                      : base_row + static_cast<int64_t>(nf) * KP + j;
            uint4 v = make_uint4(0u, 0u, 0u, 0u);
            if (row >= 0) v = *reinterpret_cast<const uint4 *>(P.latent + row * kLatentDim + piece * 8);
            else if (piece == 0) set_status(P.status, KP_ERR_DEVICE_BOUNDS);
            *reinterpret_cast<uint4 *>(tail_s + j * kNopeDim + piece * 8) = v;
        }
        // Q has landed (the tail logits read it; nothing may be in flight at exit).
        const bool have_q = mbar_wait(bar(kBarQ), 0, abort_flag, P.status, P.wait_ns);
        named_bar(2, kTailThreads);
        if (have_q) {  // tail logits of this CTA's heads: one warp per (head, tail token)
            for (int pr = warp - kAtSoftWarps; pr < nh * n_tail; pr += kTailThreads / 32) {
                const int h = h0 + pr / n_tail, j = pr % n_tail;
                float acc = 0.f;
#pragma unroll
                for (int e = 0; e < 16; e += 2) {
                    const int d = lane * 16 + e;
                    const uint32_t qv =
                        *reinterpret_cast<const uint32_t *>(smem + kOffQ + at_block_pos(d >> 6) * kAtQBlockBytes +
                                                            sw128_off(h, d & 63));
                    const uint32_t cv = *reinterpret_cast<const uint32_t *>(tail_s + j * kNopeDim + d);
                    acc = fmaf(bf16_lo(qv), bf16_lo(cv), acc);
                    acc = fmaf(bf16_hi(qv), bf16_hi(cv), acc);
                }
#pragma unroll
                for (int o = 16; o > 0; o >>= 1) acc += __shfl_xor_sync(0xffffffffu, acc, o);
                if (lane == 0) ztail_s[h * KP + j] = acc * P.scale_log2;
            }
        }
    }
    if (S > 1) cluster_barrier();  // every dump, running max and row sum is written
    else __syncthreads();
    const bool merge_ok = !aborted && *abort_flag == 0;  // the Q wait above may have timed out

    if (qvalid && merge_ok) {
        // per-head merge weights from every split's running max and row sums
        if (tid < nh) {
            const int h = h0 + tid;
            float ms[kAtMaxSplits], ls[kAtMaxSplits];
#pragma unroll
            for (int s2 = 0; s2 < kAtMaxSplits; ++s2) {
                ms[s2] = -INFINITY;
                ls[s2] = 0.f;
                if (s2 < S) {   // pushed by every CTA before the cluster barrier
                    ms[s2] = S > 1 ? recv_m[tid * S + s2] : mused_s[h];
                    ls[s2] = S > 1 ? recv_l[tid * S + s2] : lsum_s[h];
                }
            }
            float M = -INFINITY;
#pragma unroll
            for (int s2 = 0; s2 < kAtMaxSplits; ++s2) M = fmaxf(M, ms[s2]);
            for (int j = 0; j < n_tail; ++j) M = fmaxf(M, ztail_s[h * KP + j]);
            float L = 0.f;
            float *w = wm_s + tid * kWS;
#pragma unroll
            for (int s2 = 0; s2 < kAtMaxSplits; ++s2) {
                const float ws = ms[s2] > -INFINITY ? fast_exp2(ms[s2] - M) : 0.f;
                w[s2] = ws;
                if (ws > 0.f) L += ws * ls[s2];
            }
            for (int j = 0; j < kAtMaxTail; ++j) {
                const float wt = j < n_tail ? fast_exp2(ztail_s[h * KP + j] - M) : 0.f;
                w[8 + j] = wt;
                L += wt;
            }
            w[kWInv] = L > 0.f ? 1.f / L : 0.f;
            if (P.lse)
                P.lse[static_cast<int64_t>(q) * kMlaHeads + h] =
                    L > 0.f ? (M + fast_log2(L)) * 0.69314718055994530942f : -INFINITY;
        }
        __syncthreads();
        // out[q][h][d] = (sum_s w_s O_s[h][d] + sum_j w_j c_j[d]) / L, 4 columns per item;
        // a split with no tokens (w_s = 0) wrote no dump and is skipped.  A thread
        // takes kMrgItems items at a time and issues all their remote loads before
        // using any, so the distributed-shared-memory latency is paid once per group.
        const uint32_t dump_u32 = smem_u32(dump);
        constexpr int kMrgItems = 2;
        const int n_items = nh * (kNopeDim / 4);
        for (int idx0 = tid; idx0 < n_items; idx0 += kMrgItems * kAtThreads) {
            // weights of the items' heads into registers first (local reads), then
            // every remote load of the group, then the arithmetic
            float4 wv[kMrgItems][Pool::kWF4];
#pragma unroll
            for (int it = 0; it < kMrgItems; ++it) {
                const int idx = min(idx0 + it * kAtThreads, n_items - 1);
                const float4 *w4 = reinterpret_cast<const float4 *>(wm_s + (idx / (kNopeDim / 4)) * kWS);
#pragma unroll
                for (int k = 0; k < Pool::kWF4; ++k) wv[it][k] = w4[k];
            }
            float4 v[kMrgItems][kAtMaxSplits];
#pragma unroll
            for (int it = 0; it < kMrgItems; ++it) {
                const int idx = idx0 + it * kAtThreads;
                const float ws[8] = {wv[it][0].x, wv[it][0].y, wv[it][0].z, wv[it][0].w,
                                     wv[it][1].x, wv[it][1].y, wv[it][1].z, wv[it][1].w};
                if (idx < n_items) {
                    const int hl = idx / (kNopeDim / 4), d = 4 * (idx % (kNopeDim / 4));
                    const uint32_t off = static_cast<uint32_t>(((h0 + hl) * kNopeDim + d) * 4);
#pragma unroll
                    for (int s2 = 0; s2 < kAtMaxSplits; ++s2)
                        if (s2 < S && ws[s2] > 0.f) v[it][s2] = dsmem_ld_f32x4(dsmem_addr(dump_u32 + off, s2));
                }
            }
#pragma unroll
            for (int it = 0; it < kMrgItems; ++it) {
                const int idx = idx0 + it * kAtThreads;
                if (idx >= n_items) break;
                const int hl = idx / (kNopeDim / 4), d = 4 * (idx % (kNopeDim / 4));
                float ws[4 * Pool::kWF4];
#pragma unroll
                for (int k = 0; k < Pool::kWF4; ++k) {
                    ws[4 * k] = wv[it][k].x;
                    ws[4 * k + 1] = wv[it][k].y;
                    ws[4 * k + 2] = wv[it][k].z;
                    ws[4 * k + 3] = wv[it][k].w;
                }
                float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
                for (int s2 = 0; s2 < kAtMaxSplits; ++s2) {
                    const float w_s = s2 < S ? ws[s2] : 0.f;
                    if (w_s > 0.f) {
                        a.x = fmaf(w_s, v[it][s2].x, a.x);
                        a.y = fmaf(w_s, v[it][s2].y, a.y);
                        a.z = fmaf(w_s, v[it][s2].z, a.z);
                        a.w = fmaf(w_s, v[it][s2].w, a.w);
                    }
                }
#pragma unroll
                for (int j = 0; j < kAtMaxTail; ++j) {
                    if (j >= n_tail) break;
                    const uint2 cv = *reinterpret_cast<const uint2 *>(tail_s + j * kNopeDim + d);
                    const float wt = ws[8 + j];
                    a.x = fmaf(wt, bf16_lo(cv.x), a.x);
                    a.y = fmaf(wt, bf16_hi(cv.x), a.y);
                    a.z = fmaf(wt, bf16_lo(cv.y), a.z);
                    a.w = fmaf(wt, bf16_hi(cv.y), a.w);
                }
                const float il = ws[kWInv];
                *reinterpret_cast<uint2 *>(P.out + (static_cast<int64_t>(q) * kMlaHeads + h0 + hl) * kNopeDim + d) =
                    make_uint2(pack_bf16x2(a.x * il, a.y * il), pack_bf16x2(a.z * il, a.w * il));
            }
        }
    } else if (!qvalid && merge_ok) {
        // Nothing to attend: out = 0, lse = -inf.
        for (int idx = tid; idx < nh * (kNopeDim / 2); idx += kAtThreads) {
            const int h = h0 + idx / (kNopeDim / 2), d = 2 * (idx % (kNopeDim / 2));
            *reinterpret_cast<uint32_t *>(P.out + (static_cast<int64_t>(q) * kMlaHeads + h) * kNopeDim + d) = 0u;
        }
        if (P.lse && tid < nh) P.lse[static_cast<int64_t>(q) * kMlaHeads + h0 + tid] = -INFINITY;
    }
    if (S > 1) cluster_barrier();  // every peer is done reading this CTA's dump

    if (qvalid && aborted && tid == 0) mbar_wait(bar(kBarQ), 0, nullptr, P.status);  // no TMA left in flight
    tc_fence_before();
    __syncthreads();
    if (warp == kAtMmaWarp) {
        tc_fence_after();
        tmem_dealloc(tmem, kAtTmemCols);
    }
}

// Largest cluster size whose clusters, one CTA per SM, all fit at once
// (cached per device and pool size; host threads that race here compute the
// same value, and the cache entries are atomics, so the race is benign).
std::atomic<int> g_active_clusters[2][64][kAtMaxSplits + 1];
std::atomic<int> g_smem_configured[2][64];

template <int KP>
constexpr int pool_slot() { return KP == 4 ? 0 : 1; }

template <int KP>
bool attend_smem_configured() {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return false;
    if (g_smem_configured[pool_slot<KP>()][dev].load(std::memory_order_relaxed)) return true;
    cudaError_t e = cudaFuncSetAttribute(sparse_mla_tc_kernel<KP>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         AtPool<KP>::kSmemBytes);
    if (e != cudaSuccess) {
        record_cuda_error("cudaFuncSetAttribute(sparse_mla_tc_kernel)", e);
        return false;
    }
    g_smem_configured[pool_slot<KP>()][dev].store(1, std::memory_order_relaxed);
    return true;
}

template <int KP>
int max_active_clusters(int cluster) {
    if (!attend_smem_configured<KP>()) return 0;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
    std::atomic<int> &slot = g_active_clusters[pool_slot<KP>()][dev][cluster];
    const int cached = slot.load(std::memory_order_relaxed);
    if (cached != 0) return cached;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(cluster * 64);
    cfg.blockDim = dim3(kAtThreads);
    cfg.dynamicSmemBytes = AtPool<KP>::kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = cluster;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, sparse_mla_tc_kernel<KP>, &cfg) != cudaSuccess) {
        cudaGetLastError();
        n = 0;
    }
    slot.store(n > 0 ? n : -1, std::memory_order_relaxed);
    return n;
}

template <int KP>
kp_status launch_attend_kp(const kp_attend_args &a, cudaStream_t s) {
    const int nq = a.q.num_queries;
    const int sms = device_sm_count();
    if (sms <= 0) return KP_ERR_CUDA;
    if (!attend_smem_configured<KP>()) return KP_ERR_CUDA;
    int splits = attend_splits(a.cfg, nq, sms);
    while (splits > 1 && max_active_clusters<KP>(splits) < nq) splits = attend_splits_lower(splits);

    // The gather addresses latent rows by a signed 32-bit TMA coordinate
    // (validated: latent_rows <= INT32_MAX).
    CUtensorMap tm_q, tm_lat;
    if (!make_tmap_bf16_sw128(&tm_q, a.q_lat, kLatentDim, static_cast<uint64_t>(nq) * kMlaHeads,
                              kLatentDim * 2, 64, kMlaHeads))
        return KP_ERR_CUDA;
    if (!make_tmap_bf16_sw128(&tm_lat, a.latent, kLatentDim, static_cast<uint64_t>(a.seqs.latent_rows),
                              kLatentDim * 2, 64, KP))
        return KP_ERR_CUDA;
    AttendParams P;
    P.latent = a.latent;
    P.cmap = cache_map(a.seqs, a.cfg.kpool);
    P.q_seq = a.q.q_seq;
    P.q_pos = a.q.q_pos;
    P.seq_len = a.seqs.seq_len;
    P.num_seqs = a.seqs.num_seqs;
    P.pool_idx = a.pool_idx;
    P.n_sel = a.n_sel;
    P.share_src = a.q.share_src;
    P.nq = nq;
    P.K = a.cfg.topk_tokens / a.cfg.kpool;
    P.tail = a.cfg.always_select_tail ? 1 : 0;
    P.scale_log2 = a.cfg.sm_scale * 1.44269504088896340736f;
    P.out = a.out;
    P.lse = a.lse;
    P.splits = splits;
    P.status = a.d_status;
    P.wait_ns = wait_limit_ns(a.cfg.wait_limit_us);
    P.stall = (a.cfg.debug_flags & KP_DEBUG_STALL_FIRST_WAIT) ? 1 : 0;

    return launch_kernel("sparse_mla_tc_kernel", sparse_mla_tc_kernel<KP>,
                         LaunchCfg(dim3(static_cast<unsigned>(nq) * splits), dim3(kAtThreads), AtPool<KP>::kSmemBytes,
                                   s, splits),
                         tm_q, tm_lat, P);
}

}  // namespace

// Splits of one query's token list = CTAs of its cluster: at most 8, at most
// one per tile, and no more than keep the grid within the SMs; never 7, whose
// one 10-head CTA would need 70 merge slots (kAtRecvSlots holds 66).  The
// launch lowers the count further while the clusters do not all fit at once.
int attend_splits(const kp_config &cfg, int32_t num_queries, int sm_count) {
    if (num_queries <= 0) return 1;
    const int tiles = (cfg.topk_tokens + kAtTok - 1) / kAtTok;
    int s = kAtMaxSplits;
    while (s > 1 && (s > tiles || static_cast<int64_t>(num_queries) * s > sm_count || s == 7)) --s;
    return s;
}
// The next smaller split count the launch tries when the clusters of `s` do
// not all fit at once.
int attend_splits_lower(int s) { return s == 8 ? 6 : s - 1; }

size_t attend_ws_bytes(const kp_config &cfg, int32_t num_queries, int splits) {
    (void)cfg;
    (void)num_queries;
    (void)splits;
    return 256;  // the cluster merge needs no global scratch
}

kp_status launch_attend(const kp_attend_args &a, cudaStream_t s) {
    if (a.q.num_queries == 0) return KP_OK;
    return a.cfg.kpool == 16 ? launch_attend_kp<16>(a, s) : launch_attend_kp<4>(a, s);
}

}  // namespace kp
