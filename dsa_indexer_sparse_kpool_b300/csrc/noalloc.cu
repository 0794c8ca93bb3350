// noalloc.cu -- kp_indexer_score_noalloc: indexer scoring for callers that
// cannot allocate device memory.
//
// kp_indexer_score needs a small caller-provided workspace for its work plan
// (the query groups and the 128-pool tiles each one covers).  Some callers
// cannot call cudaMalloc at the point where they score: code running inside
// a framework's own caching allocator that forbids raw allocations, plugins
// handed only input and output buffers, or hosts whose memory budget is
// fixed before the first step.  For them this entry point keeps the plan in a
// file-scope device array instead, so the call itself allocates nothing.
//
// The array is loaded with the library and held by every GPU that loads it
// until the process exits.  In host code its name is only a host-side
// stand-in, so its device address is looked up with the device current
// (cudaGetSymbolAddress) and passed to the kernels.  The lookup is repeated on
// every call made outside stream capture, so a device reset (which reloads the
// module at another address) is picked up; a call made while its stream is
// being captured uses the address cached by the last call outside capture.
#include <mutex>

#include "kp_common.cuh"
#include "kp_internal.h"

namespace kp {
namespace {

// Plan words for KP_NOALLOC_MAX_QUERIES queries: header (4) + four arrays of
// one word per query + the closing unit offset (1); rounded up to 256 bytes.
constexpr size_t kNoallocPlanWords =
    (4 + 4 * static_cast<size_t>(KP_NOALLOC_MAX_QUERIES) + 1 + 63) / 64 * 64;

static __device__ __align__(256) int32_t g_noalloc_plan[kNoallocPlanWords];

constexpr int kMaxDevices = 64;
std::mutex g_noalloc_mutex;
void *g_noalloc_addr[kMaxDevices] = {};

// Device address of g_noalloc_plan on the current device (nullptr on error,
// with the error recorded for kp_last_error).  Looked up afresh unless the
// stream is capturing, then taken from the per-device cache.
void *noalloc_plan_address(cudaStream_t stream) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) {
        record_cuda_error("cudaGetDevice", e);
        return nullptr;
    }
    if (dev < 0 || dev >= kMaxDevices) {
        record_error_text("kp_indexer_score_noalloc: device ordinal out of range");
        return nullptr;
    }
    cudaStreamCaptureStatus cs = cudaStreamCaptureStatusNone;
    e = cudaStreamIsCapturing(stream, &cs);
    if (e != cudaSuccess) {
        record_cuda_error("cudaStreamIsCapturing", e);
        return nullptr;
    }
    std::lock_guard<std::mutex> lock(g_noalloc_mutex);
    if (cs == cudaStreamCaptureStatusNone) {
        void *p = nullptr;
        e = cudaGetSymbolAddress(&p, g_noalloc_plan);
        if (e != cudaSuccess) {
            record_cuda_error("cudaGetSymbolAddress(g_noalloc_plan)", e);
            return nullptr;
        }
        g_noalloc_addr[dev] = p;
    } else if (!g_noalloc_addr[dev]) {
        record_error_text(
            "kp_indexer_score_noalloc: first call on this device made during stream capture; "
            "call it once outside capture first");
        return nullptr;
    }
    return g_noalloc_addr[dev];
}

}  // namespace
}  // namespace kp

extern "C" kp_status kp_indexer_score_noalloc(const kp_score_args *a, kp_stream_t stream) {
    if (!a) return KP_ERR_INVALID_ARG;
    if (a->q.num_queries > KP_NOALLOC_MAX_QUERIES) {
        kp::record_error_text(
            "kp_indexer_score_noalloc: num_queries exceeds KP_NOALLOC_MAX_QUERIES");
        return KP_ERR_UNSUPPORTED;
    }
    if (a->q.num_queries <= 0) return kp_indexer_score(a, stream);
    void *plan = kp::noalloc_plan_address(reinterpret_cast<cudaStream_t>(stream));
    if (!plan) return KP_ERR_CUDA;
    // Every word of the plan that the scorer reads is rewritten by the plan
    // kernel of this call, so nothing has to be cleared between calls.
    kp_score_args b = *a;
    b.workspace = plan;
    b.workspace_bytes = sizeof(int32_t) * kp::kNoallocPlanWords;
    return kp::score_with_workspace_plan(&b, reinterpret_cast<cudaStream_t>(stream));
}
