// ep_layout_static.cu -- ep_layout_static_ws(): the routing layout for
// callers that cannot allocate device memory.  The layout's scratch lives in
// one fixed-size array in the library's own device memory instead of a
// caller-provided workspace.
#include <mutex>

#include "ep_internal.cuh"

namespace {

// Scratch for the layout's per-chunk counts (int32 [(E+R) x chunks]).  It is
// part of the loaded module, so every GPU that loads the library holds these
// EP_STATIC_WS_BYTES until the process exits.  Every call shares it and
// nothing clears it between calls; the layout writes every scratch entry it
// later reads within the same call, so no zeroing is needed.
static __device__ __align__(256) int32_t g_layout_scratch[EP_STATIC_WS_BYTES / sizeof(int32_t)];

constexpr int kMaxDevices = 64;
std::mutex g_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Device address of g_layout_scratch on the current device.  In host code
// the array's name is only a host-side stand-in, so the address is looked up
// once per device (with that device current) and cached.
int scratch_address(void** out) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return (int)e;
    if (dev < 0 || dev >= kMaxDevices) return (int)cudaErrorInvalidDevice;
    std::lock_guard<std::mutex> lock(g_mutex);
    if (g_scratch_ptr[dev] == nullptr) {
        void* p = nullptr;
        e = cudaGetSymbolAddress(&p, g_layout_scratch);
        if (e != cudaSuccess) return (int)e;
        g_scratch_ptr[dev] = p;
    }
    *out = g_scratch_ptr[dev];
    return 0;
}

}  // namespace

extern "C" int ep_layout_static_ws(const int32_t* topk_idx, int64_t T, int k, int E, int R,
                                   int kind, int capacity, int32_t* expert_counts,
                                   int32_t* expert_offsets, int32_t* dst_row,
                                   int32_t* rank_token_counts, uint32_t* status, void* stream) {
    // the checks of ep_layout first, against the fixed array's size, so that
    // both calls report a bad argument the same way; a size beyond the array
    // gives EP_ERR_WORKSPACE.  The placeholder pointer stands for the array
    // (aligned, never dereferenced on the host).
    void* const placeholder = reinterpret_cast<void*>(static_cast<uintptr_t>(256));
    const int rc = ep::check_layout_args(topk_idx, T, k, E, R, kind, capacity, 1, expert_counts,
                                         expert_offsets, dst_row, rank_token_counts, status,
                                         placeholder, (size_t)EP_STATIC_WS_BYTES);
    if (rc != EP_OK) return rc;
    const size_t need = ep_layout_workspace_bytes(T, k, E, R, rank_token_counts != nullptr);
    void* scratch = nullptr;
    if (need > 0) {
        const int err = scratch_address(&scratch);
        if (err != 0) {
            ep::record_cuda_error(err);
            return EP_ERR_CUDA;
        }
    }
    return ep_layout(topk_idx, T, k, E, R, kind, capacity, expert_counts, expert_offsets, dst_row,
                     rank_token_counts, status, scratch, (size_t)EP_STATIC_WS_BYTES, stream);
}
