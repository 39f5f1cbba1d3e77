// moe_route_static: the routing step without a caller-provided workspace.
//
// Some callers cannot allocate device memory at the point where they route:
// an inference-engine plugin whose enqueue step must not allocate, or a
// runtime that owns all device memory in a fixed pool and forbids any other
// allocation.  For them this entry point keeps the
// routing scratch (per-chunk expert counts and bases) in a fixed-size array
// of device memory that belongs to the library itself.
//
// The array is file-scope `static __device__`, so every GPU that loads the
// library holds it until the process exits.  In host code its name is only a
// host-side stand-in, not a device address: the address a kernel may use is
// fetched once per device with cudaGetSymbolAddress, with that device
// current, by the first call on that device; make that first call before
// any stream capture.  Every call shares the one array, and calls whose
// kernels overlap on the GPU race on it: serialize them.
#include "../../include/moe.h"
#include "kernels.h"

#include <mutex>

namespace {

constexpr size_t kScratchBytes = MOE_ROUTE_STATIC_MAX_SCRATCH_BYTES;
static_assert(kScratchBytes % 256 == 0, "scratch size must keep 256-byte alignment");

static __device__ __align__(256) int32_t g_route_scratch[kScratchBytes / sizeof(int32_t)];

constexpr int kMaxDevices = 64;
int32_t *g_scratch_ptr[kMaxDevices] = {};
std::mutex g_scratch_mu;

// Device address of g_route_scratch on the current device (set up on first use).
moe_status_t scratch_address(int32_t **out) {
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return MOE_ERR_CUDA;
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_ptr[dev] == nullptr) {
        void *p = nullptr;
        if (cudaGetSymbolAddress(&p, g_route_scratch) != cudaSuccess || p == nullptr) return MOE_ERR_CUDA;
        g_scratch_ptr[dev] = static_cast<int32_t *>(p);
    }
    *out = g_scratch_ptr[dev];
    return MOE_OK;
}

inline bool aligned4(const void *p) { return (reinterpret_cast<uintptr_t>(p) & 3u) == 0; }

}  // namespace

extern "C" moe_status_t moe_route_static(const float *logits, int T, int E, int K, int32_t *topk_idx,
                                         float *topk_w, int32_t *counts, int32_t *offsets, int32_t *row_of,
                                         int32_t *src_tok, cudaStream_t stream) {
    if (!logits || !topk_idx || !topk_w || !counts || !offsets || !row_of || !src_tok) return MOE_ERR_INVALID_ARG;
    if (!aligned4(logits) || !aligned4(topk_idx) || !aligned4(topk_w) || !aligned4(counts) || !aligned4(offsets) ||
        !aligned4(row_of) || !aligned4(src_tok))
        return MOE_ERR_INVALID_ARG;
    if (T < 1 || E < 1 || K < 1 || K > E) return MOE_ERR_INVALID_ARG;
    if (E > 256 || K > 16 || static_cast<int64_t>(T) * K >= (int64_t(1) << 31)) return MOE_ERR_UNSUPPORTED;
    // too many tokens x experts for the fixed scratch: use moe_route instead
    if (moe::route_workspace_bytes(T, E) > kScratchBytes) return MOE_ERR_UNSUPPORTED;
    int32_t *scratch = nullptr;
    moe_status_t st = scratch_address(&scratch);
    if (st != MOE_OK) return st;
    // Nothing in the scratch needs to start at zero: the first kernel writes
    // every per-chunk count before the second one reads it, and the second
    // writes every per-chunk base before the third one reads it.
    const cudaError_t err = moe::launch_route(logits, T, E, K, topk_idx, topk_w, counts, offsets, row_of, src_tok,
                                              scratch, stream);
    return err == cudaSuccess ? MOE_OK : MOE_ERR_CUDA;
}
