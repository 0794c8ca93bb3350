// kp_internal.h -- host-side declarations shared by the library's .cu files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "kpool_dsa.h"

namespace kp {

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

// Byte sizes of the step workspaces.
size_t score_plan_bytes(int32_t num_queries);
int attend_splits(const kp_config &cfg, int32_t num_queries, int sm_count);
size_t attend_ws_bytes(const kp_config &cfg, int32_t num_queries, int splits);

// Launchers (arguments already validated).
kp_status launch_compress(const kp_compress_args &a, cudaStream_t s);
kp_status launch_score(const kp_score_args &a, cudaStream_t s);
kp_status launch_topk(const kp_topk_args &a, cudaStream_t s);
kp_status launch_attend(const kp_attend_args &a, cudaStream_t s);

inline size_t align_up(size_t x, size_t a) { return (x + a - 1) / a * a; }

}  // namespace kp
