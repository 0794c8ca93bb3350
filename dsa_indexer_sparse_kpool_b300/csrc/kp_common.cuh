// kp_common.cuh -- device helpers shared by the KPool DSA kernels (sm_103a).
//
// Thin inline-PTX wrappers for the Blackwell data movers and tensor cores
// (mbarrier, TMA tensor copies, tcgen05 MMA / TMEM, distributed shared
// memory), a block-wide scan, and the status word.  Every wait on an mbarrier is bounded in time:
// after KP_WAIT_NS it records KP_ERR_DEVICE_TIMEOUT and returns false so the
// caller can unwind instead of spinning forever.
#pragma once

#include <cuda_runtime.h>
#include <cuda_bf16.h>
#include <climits>
#include <stdint.h>

#include "kpool_dsa.h"

namespace kp {

constexpr int kIndexHeads = KP_INDEX_HEADS;
constexpr int kIndexDim = KP_INDEX_DIM;
constexpr int kMlaHeads = KP_MLA_HEADS;
constexpr int kLatentDim = KP_LATENT_DIM;
constexpr int kNopeDim = KP_NOPE_DIM;

// A single wait longer than this (1 s) means something is broken.  Callers
// can set a shorter limit per call (kp_config.wait_limit_us); the waits that
// drain in-flight copies and MMAs before teardown always use this one.
constexpr unsigned long long KP_WAIT_NS = 1000000000ull;

// Limit of one wait for a call: wait_limit_us, or KP_WAIT_NS when it is 0.
__host__ __device__ inline unsigned long long wait_limit_ns(int32_t wait_limit_us) {
    return wait_limit_us > 0 ? static_cast<unsigned long long>(wait_limit_us) * 1000ull : KP_WAIT_NS;
}

__device__ __forceinline__ uint32_t smem_u32(const void *p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ unsigned long long globaltimer_ns() {
    unsigned long long t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}

// Programmatic dependent launch: wait until the preceding kernel of the
// stream has completed and its writes are visible (a no-op when the launch has
// no programmatic dependency), then let the next kernel start launching.
// Every kernel calls this before its first global-memory access.
__device__ __forceinline__ void pdl_wait_then_release() {
    asm volatile("griddepcontrol.wait;" ::: "memory");
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// Where a sequence's latent rows and pooled keys live: per-sequence row
// offsets (contiguous mode) or a block table of pages (paged mode; a page of
// 2^page_shift token positions holds as many latent rows and 2^page_shift /
// kpool pooled rows, at the same physical page id in both caches).
struct CacheMap {
    const int64_t *latent_row_off;
    const int64_t *pool_row_off;
    const int32_t *block_table;  // nullptr: contiguous mode
    int page_shift;              // log2(tokens per page)
    int pool_shift;              // log2(tokens per pool)
    int blocks_per_seq;
    int num_pages;               // valid page ids: 0 .. num_pages - 1
    int64_t latent_rows;
    int64_t pool_rows;

    __device__ __forceinline__ bool paged() const { return block_table != nullptr; }
    // Physical page of logical page `blk` of sequence b, or -1 when out of range.
    __device__ __forceinline__ int page(int b, int blk) const {
        if (blk < 0 || blk >= blocks_per_seq) return -1;
        const int pg = block_table[static_cast<int64_t>(b) * blocks_per_seq + blk];
        return (pg >= 0 && pg < num_pages) ? pg : -1;
    }
    // Latent-cache row of position `pos` of sequence b, or -1 when out of range.
    __device__ __forceinline__ int64_t latent_row(int b, int pos) const {
        if (!paged()) {
            const int64_t r = latent_row_off[b] + pos;
            return (pos >= 0 && r >= 0 && r < latent_rows) ? r : -1;
        }
        if (pos < 0) return -1;
        const int pg = page(b, pos >> page_shift);
        return pg < 0 ? -1 : (static_cast<int64_t>(pg) << page_shift) + (pos & ((1 << page_shift) - 1));
    }
    // Pooled-cache row of pool p of sequence b, or -1 when out of range.
    __device__ __forceinline__ int64_t pool_row(int b, int p) const {
        if (!paged()) {
            const int64_t r = pool_row_off[b] + p;
            return (p >= 0 && r >= 0 && r < pool_rows) ? r : -1;
        }
        if (p < 0) return -1;
        const int ps = page_shift - pool_shift;  // log2(pools per page)
        const int pg = page(b, p >> ps);
        return pg < 0 ? -1 : (static_cast<int64_t>(pg) << ps) + (p & ((1 << ps) - 1));
    }
};

// log2 of a supported pool size (4 or 16).
__host__ __device__ constexpr int kpool_shift(int kpool) { return kpool == 16 ? 4 : 2; }

// First error wins; later ones are dropped.
__device__ __forceinline__ void set_status(int32_t *st, int code) {
    if (st) atomicCAS(st, 0, code);
}

// ------------------------------------------------------------------ mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
    asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
    asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_expect_tx(uint32_t bar, uint32_t bytes) {
    asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
                 : "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
    asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Non-blocking test of the same condition (try_wait may suspend the thread for
// a while when the phase is not complete; polling several barriers needs this).
__device__ __forceinline__ bool mbar_test(uint32_t bar, uint32_t parity) {
    uint32_t ok;
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "mbarrier.test_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
        "selp.u32 %0, 1, 0, p;\n\t}\n"
        : "=r"(ok)
        : "r"(bar), "r"(parity)
        : "memory");
    return ok != 0;
}
// Waits for the phase of parity `parity` to complete.  Returns false (and
// records a timeout in *status) after limit_ns, or early when *abort is set
// by another thread of the CTA.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int *abort,
                                          int32_t *status, unsigned long long limit_ns = KP_WAIT_NS) {
    if (mbar_try_wait(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_try_wait(bar, parity)) return true;
        if ((it & 63u) == 0) {
            if (abort && *abort) return false;
            if (globaltimer_ns() - t0 > limit_ns) {
                set_status(status, KP_ERR_DEVICE_TIMEOUT);
                if (abort) *abort = 1;
                return false;
            }
        }
    }
}
// Same contract as mbar_wait, but polls with test_wait and never suspends:
// for the one thread that feeds the tensor pipe, where a late wake-up leaves
// the pipe idle.
__device__ __forceinline__ bool mbar_spin(uint32_t bar, uint32_t parity, volatile int *abort, int32_t *status,
                                          unsigned long long limit_ns = KP_WAIT_NS) {
    if (mbar_test(bar, parity)) return true;
    const unsigned long long t0 = globaltimer_ns();
    for (uint32_t it = 1;; ++it) {
        if (mbar_test(bar, parity)) return true;
        if ((it & 255u) == 0) {
            if (abort && *abort) return false;
            if (globaltimer_ns() - t0 > limit_ns) {
                set_status(status, KP_ERR_DEVICE_TIMEOUT);
                if (abort) *abort = 1;
                return false;
            }
        }
    }
}

// ------------------------------------------------------------------ TMA
__device__ __forceinline__ void tma_prefetch_desc(const void *tmap) {
    asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(tmap)) : "memory");
}
// 2-D tiled load of one box into shared memory, completing on `bar`.
// x = innermost coordinate (elements; x * elem_size must be a multiple of 16).
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void *tmap, uint32_t bar, int x,
                                            int y) {
    asm volatile(
        "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3}], [%4];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(bar)
        : "memory");
}

__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void *tmap, uint32_t bar, int x, int y,
                                            int z) {
    asm volatile(
        "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
        " [%0], [%1, {%2, %3, %4}], [%5];" ::"r"(dst),
        "l"(reinterpret_cast<uint64_t>(tmap)), "r"(x), "r"(y), "r"(z), "r"(bar)
        : "memory");
}

// ------------------------------------------------------------------ tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem),
                 "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
                 : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
    asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
    asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem desc] * B[smem desc]^T, bf16 inputs, fp32 accumulate.
__device__ __forceinline__ void tc_mma_bf16(uint32_t d_tmem, uint64_t a_desc, uint64_t b_desc,
                                            uint32_t idesc, uint32_t accumulate) {
    asm volatile(
        "{\n\t.reg .pred p;\n\t"
        "setp.ne.b32 p, %4, 0;\n\t"
        "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}\n" ::"r"(d_tmem),
        "l"(a_desc), "l"(b_desc), "r"(idesc), "r"(accumulate)
        : "memory");
}
// Arrive once on `bar` when every tcgen05 op issued so far by this thread completes.
__device__ __forceinline__ void tc_commit(uint32_t bar) {
    asm volatile(
        "tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
        : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() {
    asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
}
// 32 TMEM lanes (one per thread of the warp) x 32 consecutive 32-bit columns.
__device__ __forceinline__ void tmem_ld_32x32b_x32(uint32_t taddr, uint32_t (&r)[32]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
        "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]),
          "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]),
          "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
        : "r"(taddr));
}

// 32 TMEM lanes x 16 consecutive columns (load and store).
__device__ __forceinline__ void tmem_ld_32x32b_x16(uint32_t taddr, uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.ld.sync.aligned.32x32b.x16.b32 "
        "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15}, [%16];"
        : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
          "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
          "=r"(r[14]), "=r"(r[15])
        : "r"(taddr));
}
__device__ __forceinline__ void tmem_st_32x32b_x16(uint32_t taddr, const uint32_t (&r)[16]) {
    asm volatile(
        "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], "
        "{%1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, %16};" ::"r"(taddr),
        "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
        "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
        : "memory");
}
__device__ __forceinline__ void tmem_st_wait() {
    asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
}
// Makes this thread's generic-proxy shared-memory writes visible to the async
// proxy (TMA, tcgen05.mma operand reads) once the thread synchronises.
__device__ __forceinline__ void fence_proxy_async_smem() {
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// 2^x and log2(x) as single approximate hardware instructions (relative error
// about 2^-22; denormal results flush to zero, 2^-inf = 0).
__device__ __forceinline__ float fast_exp2(float x) {
    float r;
    asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
__device__ __forceinline__ float fast_log2(float x) {
    float r;
    asm("lg2.approx.ftz.f32 %0, %1;" : "=f"(r) : "f"(x));
    return r;
}
// Shared-memory matrix descriptor, 128-byte swizzle, with explicit leading
// and stride byte offsets.  K-major operands: LBO unused (16), SBO = bytes
// between 8-row groups along M/N.  MN-major operands (64 contiguous M/N
// elements per 128-byte row, rows along K): LBO = bytes between 64-element
// groups along M/N, SBO = bytes between 8-row groups along K.
__device__ __forceinline__ uint64_t desc_sw128(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
    d |= static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16;
    d |= static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32;
    d |= static_cast<uint64_t>(1) << 46;
    d |= static_cast<uint64_t>(2) << 61;
    return d;
}

// ------------------------------------------------------------------ clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
    uint32_t r;
    asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
    return r;
}
__device__ __forceinline__ void cluster_barrier() {
    asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::
                     : "memory");
}
// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t dsmem_addr(uint32_t saddr, uint32_t rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
    return r;
}
// Loads from a peer's shared memory.  No memory clobber: callers order them
// after the peer's writes with a cluster barrier (itself a volatile asm with a
// memory clobber, which these volatile loads are not moved across), and
// leaving ordinary shared-memory reads free to move lets the compiler issue a
// group of remote loads back to back instead of interleaving local reads that
// wait behind them.
__device__ __forceinline__ float dsmem_ld_f32(uint32_t addr) {
    float v;
    asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr));
    return v;
}
// Store to a peer's shared memory (made visible to the peer by a cluster barrier).
__device__ __forceinline__ void dsmem_st_f32(uint32_t addr, float v) {
    asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}
__device__ __forceinline__ float4 dsmem_ld_f32x4(uint32_t addr) {
    float4 v;
    asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
                 : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w)
                 : "r"(addr));
    return v;
}

// Shared-memory matrix descriptor for a K-major operand stored in the
// 128-byte-swizzle canonical layout: rows of 64 bf16 (128 B), 8-row swizzle
// atoms of 1024 B stacked along M/N (stride 1024 B).  `saddr` is the byte
// address of the first element of the K slice to read (atoms 1024-aligned;
// advancing along K inside the 128 B row adds 32 B per 16 elements).
__device__ __forceinline__ uint64_t desc_kmajor_sw128(uint32_t saddr) {
    uint64_t d = 0;
    d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);  // start address
    d |= static_cast<uint64_t>(1) << 16;                  // leading byte offset (unused here)
    d |= static_cast<uint64_t>(1024 >> 4) << 32;          // stride byte offset: 8 rows
    d |= static_cast<uint64_t>(1) << 46;                  // descriptor version
    d |= static_cast<uint64_t>(2) << 61;                  // 128-byte swizzle
    return d;
}
// Instruction descriptor of kind::f16: bf16 A and B, fp32 D; A / B K-major
// unless a_mn / b_mn (then M- / N-major).
__host__ __device__ constexpr uint32_t idesc_bf16_f32(int m, int n, bool a_mn = false, bool b_mn = false) {
    return (1u << 4)                                  // D format f32
           | (1u << 7)                                // A format bf16
           | (1u << 10)                               // B format bf16
           | (a_mn ? (1u << 15) : 0u)                 // A major-ness
           | (b_mn ? (1u << 16) : 0u)                 // B major-ness
           | (static_cast<uint32_t>(n >> 3) << 17)    // N / 8
           | (static_cast<uint32_t>(m >> 4) << 24);   // M / 16
}

// Packed fp32 pairs: d = a * b + c on both halves (IEEE fp32 fma, round to
// nearest each), the sm_100-family paired FP32 pipe.
__device__ __forceinline__ uint64_t pack_f32x2(float lo, float hi) {
    uint64_t r;
    asm("mov.b64 %0, {%1, %2};" : "=l"(r) : "f"(lo), "f"(hi));
    return r;
}
__device__ __forceinline__ float2 unpack_f32x2(uint64_t v) {
    float2 r;
    asm("mov.b64 {%0, %1}, %2;" : "=f"(r.x), "=f"(r.y) : "l"(v));
    return r;
}
__device__ __forceinline__ uint64_t fma_f32x2(uint64_t a, uint64_t b, uint64_t c) {
    uint64_t d;
    asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
    return d;
}

// bf16 pair (round to nearest even), lo in the low half.
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
    __nv_bfloat162 v = __floats2bfloat162_rn(lo, hi);
    return *reinterpret_cast<uint32_t *>(&v);
}

// ------------------------------------------------------------------ block scan
// Inclusive scan over the threads of a block (blockDim.x a multiple of 32,
// <= 1024).  `scratch` holds >= 33 ints of shared memory.  Op: 0 = sum,
// 1 = max.  Returns the thread's inclusive value; *total = block aggregate.
template <int OP>
__device__ __forceinline__ int block_inclusive_scan(int v, int *scratch, int *total) {
    const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5, nwarps = blockDim.x >> 5;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        int n = __shfl_up_sync(0xffffffffu, v, o);
        if (lane >= o) v = OP == 0 ? v + n : max(v, n);
    }
    if (lane == 31) scratch[warp] = v;
    __syncthreads();
    if (warp == 0) {
        int w = lane < nwarps ? scratch[lane] : (OP == 0 ? 0 : INT_MIN);
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            int n = __shfl_up_sync(0xffffffffu, w, o);
            if (lane >= o) w = OP == 0 ? w + n : max(w, n);
        }
        scratch[lane] = w;
    }
    __syncthreads();
    if (warp > 0) {
        int prev = scratch[warp - 1];
        v = OP == 0 ? v + prev : max(v, prev);
    }
    *total = scratch[nwarps - 1];
    __syncthreads();
    return v;
}

}  // namespace kp
