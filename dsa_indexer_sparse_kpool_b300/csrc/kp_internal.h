// kp_internal.h -- host-side declarations shared by the library's .cu files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include <utility>

#include "kpool_dsa.h"
#include "kp_common.cuh"

namespace kp {

// Device-side view of a kp_seqs layout (validated) for pools of `kpool` tokens.
CacheMap cache_map(const kp_seqs &s, int kpool);

// Records the text of a failed CUDA call for kp_last_error() (per host thread).
void record_cuda_error(const char *where, cudaError_t err);
void record_error_text(const char *text);

// Status of the launch just enqueued: KP_OK or KP_ERR_CUDA.
kp_status check_launch(const char *where);

// Number of SMs of the current device (0 on failure).
int device_sm_count();

// 2-D bf16 tensor map with 128-byte swizzle: `rows` rows of `inner` elements
// (row pitch `row_bytes`, a multiple of 16), box of box_rows x box_inner
// elements (box_inner * 2 <= 128).  False (error recorded) on failure.
bool make_tmap_bf16_sw128(CUtensorMap *m, const void *base, uint64_t inner, uint64_t rows,
                          uint64_t row_bytes, uint32_t box_inner, uint32_t box_rows);
// The same matrix seen as (64 columns, rows, cols / 64 column blocks), boxes of
// box_rows rows x kblocks blocks (cols a multiple of 64).
bool make_tmap_bf16_sw128_kblocks(CUtensorMap *m, const void *base, uint64_t cols, uint64_t rows,
                                  uint64_t row_bytes, uint32_t box_rows, uint32_t kblocks);

// Launch configuration with programmatic stream serialisation (the kernel
// may start while the previous kernel of the stream drains; it waits in
// pdl_wait_then_release before touching memory) and, when cluster_x > 1, a
// 1-D thread-block cluster.  `attrs` must outlive the launch call.
struct LaunchCfg {
    cudaLaunchConfig_t cfg;
    cudaLaunchAttribute attrs[2];
    LaunchCfg(dim3 grid, dim3 block, size_t smem, cudaStream_t s, int cluster_x = 1) {
        cfg = cudaLaunchConfig_t{};
        cfg.gridDim = grid;
        cfg.blockDim = block;
        cfg.dynamicSmemBytes = smem;
        cfg.stream = s;
        int n = 0;
        attrs[n].id = cudaLaunchAttributeProgrammaticStreamSerialization;
        attrs[n].val.programmaticStreamSerializationAllowed = 1;
        ++n;
        if (cluster_x > 1) {
            attrs[n].id = cudaLaunchAttributeClusterDimension;
            attrs[n].val.clusterDim.x = static_cast<unsigned>(cluster_x);
            attrs[n].val.clusterDim.y = 1;
            attrs[n].val.clusterDim.z = 1;
            ++n;
        }
        cfg.attrs = attrs;
        cfg.numAttrs = n;
    }
};

// Launches a kernel with LaunchCfg; KP_ERR_CUDA (error recorded) on failure.
template <typename... KArgs, typename... Args>
kp_status launch_kernel(const char *name, void (*kernel)(KArgs...), const LaunchCfg &lc, Args &&...args) {
    const cudaError_t e = cudaLaunchKernelEx(&lc.cfg, kernel, std::forward<Args>(args)...);
    if (e != cudaSuccess) {
        record_cuda_error(name, e);
        return KP_ERR_CUDA;
    }
    return check_launch(name);
}

// Byte sizes of the step workspaces.
size_t score_plan_bytes(int32_t num_queries);
int attend_splits(const kp_config &cfg, int32_t num_queries, int sm_count);
int attend_splits_lower(int splits);
size_t attend_ws_bytes(const kp_config &cfg, int32_t num_queries, int splits);

// Inputs of the scorer's work plan, for building it inside another launch.
struct ScorePlanArgs {
    int nq;
    int num_seqs;
    const int32_t *q_seq;
    const int32_t *q_pos;
    const int32_t *seq_len;
    int kshift;        // log2(tokens per pool)
    int max_q;         // queries per group (8 for the scorer, 4 for the fused score-and-select)
    int max_tiles;
    int32_t *plan;     // nullptr: no plan to build
    int32_t *status;
};
ScorePlanArgs score_plan_args(const kp_score_args &a);

// Launchers (arguments already validated).  launch_compress with a plan also
// builds the scorer's plan (one extra CTA); launch_score with plan_ready then
// skips its own plan kernel.  Up to score_plan_is_local(nq) queries the scorer
// builds its plan in shared memory (no plan kernel, no plan read) unless
// allow_local_plan is false; with prev_len (the compression's prev_len) it
// also loads pooled-key tiles that the compression cannot have written before
// waiting for it.
kp_status launch_compress(const kp_compress_args &a, cudaStream_t s, const ScorePlanArgs *plan = nullptr);
bool score_plan_is_local(int32_t num_queries);
// The scorer's plan kernel on its own (one CTA).
kp_status launch_score_plan(const ScorePlanArgs &p, cudaStream_t s);
kp_status launch_score(const kp_score_args &a, cudaStream_t s, bool plan_ready = false,
                       const int32_t *prev_len = nullptr, bool allow_local_plan = true);
kp_status launch_topk(const kp_topk_args &a, cudaStream_t s);
// Fused scoring and top-k (no score matrix in global memory): when
// score_select_fits(...) holds.  plan_ready: the plan (groups of <= 4 queries)
// was built by the compression launch (score_select_plan_args); prev_len as
// for launch_score.
bool score_select_fits(const kp_config &cfg, const kp_queries &q);
ScorePlanArgs score_select_plan_args(const kp_score_args &a);
bool score_select_plan_is_local(int32_t num_queries);
kp_status launch_score_select(const kp_score_args &sc, const kp_topk_args &tk, cudaStream_t s, bool plan_ready,
                              const int32_t *prev_len);
// kp_indexer_score with its plan always in the caller's workspace (validated).
kp_status score_with_workspace_plan(const kp_score_args *a, cudaStream_t stream);
kp_status launch_attend(const kp_attend_args &a, cudaStream_t s);
kp_status launch_gemm(const kp_gemm_args &g, cudaStream_t s);
// Up to four independent products (validated, none reading another's output)
// in one launch.
kp_status launch_gemm_group(const kp_gemm_args *gs, int count, cudaStream_t s);

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace kp
