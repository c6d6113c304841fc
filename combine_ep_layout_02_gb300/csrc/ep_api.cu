// ep_api.cu -- the C ABI: argument validation on the host, then the launches.
// Every check that can fail happens before anything is enqueued.
#include <stdint.h>

#include "ep_internal.cuh"

namespace {

thread_local int g_last_cuda_error = 0;

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) % a) == 0; }

inline int cuda_status(cudaError_t e) {
    if (e == cudaSuccess) return EP_OK;
    g_last_cuda_error = (int)e;
    return EP_ERR_CUDA;
}

inline cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }

// Common checks of (T, H, k, rows) for dispatch and combine.
int check_rows_args(int64_t T, int64_t H, int k, int64_t rows) {
    if (T < 0 || H <= 0 || k < 1 || k > EP_MAX_TOPK || rows < 0) return EP_ERR_INVALID_ARG;
    if (T > 0 && T > (int64_t)INT32_MAX / k) return EP_ERR_INVALID_ARG;
    if (rows > (int64_t)INT32_MAX + 1) return EP_ERR_INVALID_ARG;
    if (H % 8 != 0) return EP_ERR_ALIGNMENT;
    return EP_OK;
}

}  // namespace

namespace ep {
void record_cuda_error(int err) { g_last_cuda_error = err; }

int cached_device_attribute(cudaDeviceAttr attr, std::atomic<int> (&cache)[64]) {
    int dev = 0, v = 0;
    if (cudaGetDevice(&dev) != cudaSuccess) return 0;
    v = cache[dev & 63].load(std::memory_order_relaxed);
    if (v == 0 && cudaDeviceGetAttribute(&v, attr, dev) == cudaSuccess && v > 0)
        cache[dev & 63].store(v, std::memory_order_relaxed);
    return v > 0 ? v : 0;
}

RowSlices row_slices(int64_t T, int64_t nvec, int warps_per_sm, int64_t min_slice) {
    // SM count per device, read once (it only shapes grids)
    static std::atomic<int> sm_cache[64];
    int sms = cached_device_attribute(cudaDevAttrMultiProcessorCount, sm_cache);
    if (sms <= 0) sms = 1;
    const int64_t target = (int64_t)sms * warps_per_sm;
    int64_t S = 1;
    while (T * S < target && (nvec + 2 * S - 1) / (2 * S) >= min_slice) S *= 2;
    if (S == 1) return RowSlices{1, nvec};
    const int64_t slice = ((nvec + S - 1) / S + 31) / 32 * 32;
    return RowSlices{(int)((nvec + slice - 1) / slice), slice};
}
}  // namespace ep

extern "C" {

int ep_version(void) { return (1 << 16) | 0; }

const char* ep_status_string(int status) {
    switch (status) {
        case EP_OK: return "EP_OK";
        case EP_ERR_INVALID_ARG: return "EP_ERR_INVALID_ARG";
        case EP_ERR_ALIGNMENT: return "EP_ERR_ALIGNMENT";
        case EP_ERR_WORKSPACE: return "EP_ERR_WORKSPACE";
        case EP_ERR_CUDA: return "EP_ERR_CUDA";
        default: return "EP_ERR_UNKNOWN";
    }
}

int ep_last_cuda_error(void) { return g_last_cuda_error; }

size_t ep_layout_workspace_bytes(int64_t T, int k, int E, int R, int with_rank_counts) {
    if (T <= 0 || k < 1 || E < 1 || R < 1) return 0;
    const int64_t nchunk = ep::layout_num_chunks(T);
    const int64_t cols = E + (with_rank_counts ? R : 0);
    const size_t bytes = (size_t)(nchunk * cols) * sizeof(int32_t);
    return (bytes + 255) & ~(size_t)255;
}

}  // extern "C"

namespace ep {

// The host-side checks of ep_layout (EP_OK when the call may proceed).
int check_layout_args(const int32_t* topk_idx, int64_t T, int k, int E, int R, int kind,
                      int capacity, int align, int32_t* expert_counts, int32_t* expert_offsets,
                      int32_t* dst_row, int32_t* rank_token_counts, uint32_t* status,
                      void* workspace, size_t workspace_bytes) {
    if (T < 0 || k < 1 || k > EP_MAX_TOPK || E < 1 || E > EP_MAX_EXPERTS || R < 1 || E % R != 0)
        return EP_ERR_INVALID_ARG;
    if (T > (int64_t)INT32_MAX / k) return EP_ERR_INVALID_ARG;
    if (kind != EP_LAYOUT_CONTIGUOUS && kind != EP_LAYOUT_MASKED) return EP_ERR_INVALID_ARG;
    if (kind == EP_LAYOUT_MASKED && (capacity < 0 || (int64_t)E * capacity > (int64_t)INT32_MAX))
        return EP_ERR_INVALID_ARG;
    if (align < 1 || T * k + (int64_t)E * (align - 1) > (int64_t)INT32_MAX) return EP_ERR_INVALID_ARG;
    if (!expert_counts || !expert_offsets) return EP_ERR_INVALID_ARG;
    if (T > 0 && (!topk_idx || !dst_row)) return EP_ERR_INVALID_ARG;
    if (!aligned(topk_idx, 4) || !aligned(dst_row, 4) || !aligned(expert_counts, 4) ||
        !aligned(expert_offsets, 4) || !aligned(rank_token_counts, 4) || !aligned(status, 4))
        return EP_ERR_ALIGNMENT;
    const size_t need = ep_layout_workspace_bytes(T, k, E, R, rank_token_counts != nullptr);
    if (need > 0) {
        if (!workspace || workspace_bytes < need) return EP_ERR_WORKSPACE;
        if (!aligned(workspace, 16)) return EP_ERR_ALIGNMENT;
    }
    return EP_OK;
}

}  // namespace ep

namespace {

using ep::check_layout_args;

int layout_checked(const int32_t* topk_idx, int64_t T, int k, int E, int R, int kind, int capacity,
                   int align, int32_t* expert_counts, int32_t* expert_offsets, int32_t* dst_row,
                   int32_t* rank_token_counts, uint32_t* status, void* workspace,
                   size_t workspace_bytes, void* stream) {
    const int rc = check_layout_args(topk_idx, T, k, E, R, kind, capacity, align, expert_counts,
                                     expert_offsets, dst_row, rank_token_counts, status, workspace,
                                     workspace_bytes);
    if (rc != EP_OK) return rc;
    return cuda_status(ep::launch_layout(topk_idx, T, k, E, R, kind, capacity, align,
                                         expert_counts, expert_offsets, dst_row, rank_token_counts,
                                         status, static_cast<int32_t*>(workspace),
                                         as_stream(stream)));
}

}  // namespace

extern "C" {

int ep_layout(const int32_t* topk_idx, int64_t T, int k, int E, int R, int kind, int capacity,
              int32_t* expert_counts, int32_t* expert_offsets, int32_t* dst_row,
              int32_t* rank_token_counts, uint32_t* status, void* workspace,
              size_t workspace_bytes, void* stream) {
    return layout_checked(topk_idx, T, k, E, R, kind, capacity, 1, expert_counts, expert_offsets,
                          dst_row, rank_token_counts, status, workspace, workspace_bytes, stream);
}

int ep_layout_aligned(const int32_t* topk_idx, int64_t T, int k, int E, int R, int alignment,
                      int32_t* expert_counts, int32_t* expert_offsets, int32_t* dst_row,
                      int32_t* rank_token_counts, uint32_t* status, void* workspace,
                      size_t workspace_bytes, void* stream) {
    return layout_checked(topk_idx, T, k, E, R, EP_LAYOUT_CONTIGUOUS, 0, alignment, expert_counts,
                          expert_offsets, dst_row, rank_token_counts, status, workspace,
                          workspace_bytes, stream);
}

int ep_dispatch(const void* x, int64_t T, int64_t H, int k, const int32_t* dst_row, void* recv,
                int64_t rows, uint32_t* status, void* stream) {
    int rc = check_rows_args(T, H, k, rows);
    if (rc != EP_OK) return rc;
    if (T == 0) return EP_OK;
    if (!x || !dst_row || (!recv && rows > 0)) return EP_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(recv, 16) || !aligned(dst_row, 4) || !aligned(status, 4))
        return EP_ERR_ALIGNMENT;
    return cuda_status(
        ep::launch_dispatch_bf16(x, T, H, k, dst_row, recv, rows, status, as_stream(stream)));
}

int ep_dispatch_fp8(const void* x, int64_t T, int64_t H, int k, const int32_t* dst_row,
                    uint8_t* recv_q, float* recv_scale, int64_t rows, uint32_t* status,
                    void* stream) {
    int rc = check_rows_args(T, H, k, rows);
    if (rc != EP_OK) return rc;
    if (H % 128 != 0) return EP_ERR_ALIGNMENT;
    if (T == 0) return EP_OK;
    if (!x || !dst_row || ((!recv_q || !recv_scale) && rows > 0)) return EP_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(recv_q, 16) || !aligned(recv_scale, 4) ||
        !aligned(dst_row, 4) || !aligned(status, 4))
        return EP_ERR_ALIGNMENT;
    return cuda_status(ep::launch_dispatch_fp8(x, T, H, k, dst_row, recv_q, recv_scale, rows,
                                               status, as_stream(stream)));
}

}  // extern "C"

namespace {

// ep_layout then ep_dispatch (fp8: ep_dispatch_fp8) on one status word, as a
// single launch when the fused kernel covers the shape.
int layout_dispatch_checked(bool fp8, const int32_t* topk_idx, int64_t T, int k, int E, int R,
                            int kind, int capacity, const void* x, int64_t H, int32_t* expert_counts,
                            int32_t* expert_offsets, int32_t* dst_row, int32_t* rank_token_counts,
                            void* recv, uint8_t* recv_q, float* recv_scale, int64_t rows,
                            uint32_t* status, void* workspace, size_t workspace_bytes,
                            void* stream) {
    int rc = check_layout_args(topk_idx, T, k, E, R, kind, capacity, 1, expert_counts,
                               expert_offsets, dst_row, rank_token_counts, status, workspace,
                               workspace_bytes);
    if (rc != EP_OK) return rc;
    rc = check_rows_args(T, H, k, rows);
    if (rc != EP_OK) return rc;
    if (fp8 && H % 128 != 0) return EP_ERR_ALIGNMENT;
    if (T > 0 && (!x || (fp8 ? ((!recv_q || !recv_scale) && rows > 0) : (!recv && rows > 0))))
        return EP_ERR_INVALID_ARG;
    if (!aligned(x, 16) || !aligned(recv, 16) || !aligned(recv_q, 16) || !aligned(recv_scale, 4))
        return EP_ERR_ALIGNMENT;
    const cudaError_t e = ep::launch_layout_dispatch(
        topk_idx, T, k, E, R, kind, capacity, x, H, fp8, expert_counts, expert_offsets, dst_row,
        rank_token_counts, fp8 ? static_cast<void*>(recv_q) : recv, recv_scale, rows, status,
        as_stream(stream));
    if (e != cudaErrorNotSupported) return cuda_status(e);
    // outside the fused kernel's range: the layout, then the dispatch, which
    // reads its first rows of x before waiting for the layout to finish (the
    // layout kernel writes no x and lets it start only once all earlier work
    // in the stream is complete); same results as the two calls
    rc = cuda_status(ep::launch_layout(topk_idx, T, k, E, R, kind, capacity, 1, expert_counts,
                                       expert_offsets, dst_row, rank_token_counts, status,
                                       static_cast<int32_t*>(workspace), as_stream(stream)));
    if (rc != EP_OK || T == 0) return rc;
    return cuda_status(fp8 ? ep::launch_dispatch_fp8(x, T, H, k, dst_row, recv_q, recv_scale,
                                                     rows, status, as_stream(stream), true)
                           : ep::launch_dispatch_bf16(x, T, H, k, dst_row, recv, rows, status,
                                                      as_stream(stream), true));
}

}  // namespace

extern "C" {

int ep_layout_dispatch(const int32_t* topk_idx, int64_t T, int k, int E, int R, int kind,
                       int capacity, const void* x, int64_t H, int32_t* expert_counts,
                       int32_t* expert_offsets, int32_t* dst_row, int32_t* rank_token_counts,
                       void* recv, int64_t rows, uint32_t* status, void* workspace,
                       size_t workspace_bytes, void* stream) {
    return layout_dispatch_checked(false, topk_idx, T, k, E, R, kind, capacity, x, H, expert_counts,
                                   expert_offsets, dst_row, rank_token_counts, recv, nullptr,
                                   nullptr, rows, status, workspace, workspace_bytes, stream);
}

int ep_layout_dispatch_fp8(const int32_t* topk_idx, int64_t T, int k, int E, int R, int kind,
                           int capacity, const void* x, int64_t H, int32_t* expert_counts,
                           int32_t* expert_offsets, int32_t* dst_row, int32_t* rank_token_counts,
                           uint8_t* recv_q, float* recv_scale, int64_t rows, uint32_t* status,
                           void* workspace, size_t workspace_bytes, void* stream) {
    return layout_dispatch_checked(true, topk_idx, T, k, E, R, kind, capacity, x, H, expert_counts,
                                   expert_offsets, dst_row, rank_token_counts, nullptr, recv_q,
                                   recv_scale, rows, status, workspace, workspace_bytes, stream);
}

int ep_combine(const void* y, const float* topk_w, const int32_t* dst_row, int64_t T, int64_t H,
               int k, int64_t rows, void* out, uint32_t* status, void* stream) {
    int rc = check_rows_args(T, H, k, rows);
    if (rc != EP_OK) return rc;
    if (T == 0) return EP_OK;
    if (!topk_w || !dst_row || !out || (!y && rows > 0)) return EP_ERR_INVALID_ARG;
    if (!aligned(y, 16) || !aligned(out, 16) || !aligned(topk_w, 4) || !aligned(dst_row, 4) ||
        !aligned(status, 4))
        return EP_ERR_ALIGNMENT;
    return cuda_status(ep::launch_combine(y, topk_w, dst_row, T, H, k, rows, out, status,
                                          as_stream(stream)));
}

int ep_combine_fp8(const uint8_t* y_q, const float* y_scale, const float* topk_w,
                   const int32_t* dst_row, int64_t T, int64_t H, int k, int64_t rows, void* out,
                   uint32_t* status, void* stream) {
    int rc = check_rows_args(T, H, k, rows);
    if (rc != EP_OK) return rc;
    if (H % 128 != 0) return EP_ERR_ALIGNMENT;
    if (T == 0) return EP_OK;
    if (!topk_w || !dst_row || !out || ((!y_q || !y_scale) && rows > 0)) return EP_ERR_INVALID_ARG;
    if (!aligned(y_q, 16) || !aligned(y_scale, 4) || !aligned(out, 16) || !aligned(topk_w, 4) ||
        !aligned(dst_row, 4) || !aligned(status, 4))
        return EP_ERR_ALIGNMENT;
    return cuda_status(ep::launch_combine_fp8(y_q, y_scale, topk_w, dst_row, T, H, k, rows, out,
                                              status, as_stream(stream)));
}

size_t ep_rank_layout_workspace_bytes(int64_t T, int k, int E, int R) {
    if (T <= 0 || k < 1 || E < 1 || R < 1) return 0;
    return ep::rank_keys_bytes(T, k) + ep_layout_workspace_bytes(T, k, R, 1, 0);
}

int ep_rank_layout(const int32_t* topk_idx, int64_t T, int k, int E, int R,
                   int32_t* rank_counts, int32_t* rank_offsets, int32_t* rank_dst_row,
                   int32_t* pair_rank_row, int32_t* rank_row_token, int64_t rank_rows,
                   uint32_t* status, void* workspace, size_t workspace_bytes, void* stream) {
    if (T < 0 || k < 1 || k > EP_MAX_TOPK || E < 1 || E > EP_MAX_EXPERTS || R < 1 || E % R != 0)
        return EP_ERR_INVALID_ARG;
    if (T > (int64_t)INT32_MAX / k) return EP_ERR_INVALID_ARG;
    if (!rank_counts || !rank_offsets || rank_rows < 0) return EP_ERR_INVALID_ARG;
    if (T > 0 && (!topk_idx || !rank_dst_row || !pair_rank_row || !rank_row_token))
        return EP_ERR_INVALID_ARG;
    if (!aligned(topk_idx, 4) || !aligned(rank_counts, 4) || !aligned(rank_offsets, 4) ||
        !aligned(rank_dst_row, 4) || !aligned(pair_rank_row, 4) || !aligned(rank_row_token, 4) ||
        !aligned(status, 4))
        return EP_ERR_ALIGNMENT;
    const size_t need = ep_rank_layout_workspace_bytes(T, k, E, R);
    if (need > 0) {
        if (!workspace || workspace_bytes < need) return EP_ERR_WORKSPACE;
        if (!aligned(workspace, 16)) return EP_ERR_ALIGNMENT;
    }
    return cuda_status(ep::launch_rank_layout(topk_idx, T, k, E, R, rank_counts, rank_offsets,
                                              rank_dst_row, pair_rank_row, rank_row_token,
                                              rank_rows, status, workspace, as_stream(stream)));
}

int ep_expand(const void* rank_buf, const int32_t* rank_offsets, int R, int64_t rank_rows,
              const int32_t* rank_row_token, const int32_t* pair_rank_row,
              const int32_t* dst_row, int64_t T, int64_t H, int k, void* recv, int64_t rows,
              uint32_t* status, void* stream) {
    int rc = check_rows_args(T, H, k, rows);
    if (rc != EP_OK) return rc;
    if (R < 1 || rank_rows < 0 || rank_rows > (int64_t)INT32_MAX) return EP_ERR_INVALID_ARG;
    if (T == 0 || rank_rows == 0) return EP_OK;
    if (!rank_buf || !rank_offsets || !rank_row_token || !pair_rank_row || !dst_row ||
        (!recv && rows > 0))
        return EP_ERR_INVALID_ARG;
    if (!aligned(rank_buf, 16) || !aligned(recv, 16) || !aligned(rank_offsets, 4) ||
        !aligned(rank_row_token, 4) || !aligned(pair_rank_row, 4) || !aligned(dst_row, 4) ||
        !aligned(status, 4))
        return EP_ERR_ALIGNMENT;
    return cuda_status(ep::launch_expand(rank_buf, rank_offsets, R, rank_rows, rank_row_token,
                                         pair_rank_row, dst_row, T, H, k, recv, rows, status,
                                         as_stream(stream)));
}

int ep_expand_fp8(const uint8_t* rank_q, const float* rank_scale, const int32_t* rank_offsets,
                  int R, int64_t rank_rows, const int32_t* rank_row_token,
                  const int32_t* pair_rank_row, const int32_t* dst_row, int64_t T, int64_t H,
                  int k, uint8_t* recv_q, float* recv_scale, int64_t rows, uint32_t* status,
                  void* stream) {
    int rc = check_rows_args(T, H, k, rows);
    if (rc != EP_OK) return rc;
    if (H % 128 != 0) return EP_ERR_ALIGNMENT;
    if (R < 1 || rank_rows < 0 || rank_rows > (int64_t)INT32_MAX) return EP_ERR_INVALID_ARG;
    if (T == 0 || rank_rows == 0) return EP_OK;
    if (!rank_q || !rank_scale || !rank_offsets || !rank_row_token || !pair_rank_row ||
        !dst_row || ((!recv_q || !recv_scale) && rows > 0))
        return EP_ERR_INVALID_ARG;
    if (!aligned(rank_q, 16) || !aligned(recv_q, 16) || !aligned(rank_scale, 4) ||
        !aligned(recv_scale, 4) || !aligned(rank_offsets, 4) || !aligned(rank_row_token, 4) ||
        !aligned(pair_rank_row, 4) || !aligned(dst_row, 4) || !aligned(status, 4))
        return EP_ERR_ALIGNMENT;
    return cuda_status(ep::launch_expand_fp8(rank_q, rank_scale, rank_offsets, R, rank_rows,
                                             rank_row_token, pair_rank_row, dst_row, T, H, k,
                                             recv_q, recv_scale, rows, status, as_stream(stream)));
}

int ep_combine_partial(const void* y, int64_t rows, const float* topk_w, const int32_t* dst_row,
                       const int32_t* pair_rank_row, const int32_t* rank_row_token,
                       const int32_t* rank_offsets, int R, int64_t rank_rows, int64_t T,
                       int64_t H, int k, void* partial, uint32_t* status, void* stream) {
    int rc = check_rows_args(T, H, k, rows);
    if (rc != EP_OK) return rc;
    if (R < 1 || rank_rows < 0 || rank_rows > (int64_t)INT32_MAX) return EP_ERR_INVALID_ARG;
    if (T == 0 || rank_rows == 0) return EP_OK;
    if (!topk_w || !dst_row || !pair_rank_row || !rank_row_token || !rank_offsets || !partial ||
        (!y && rows > 0))
        return EP_ERR_INVALID_ARG;
    if (!aligned(y, 16) || !aligned(partial, 16) || !aligned(topk_w, 4) || !aligned(dst_row, 4) ||
        !aligned(pair_rank_row, 4) || !aligned(rank_row_token, 4) || !aligned(rank_offsets, 4) ||
        !aligned(status, 4))
        return EP_ERR_ALIGNMENT;
    return cuda_status(ep::launch_combine_partial(y, rows, topk_w, dst_row, pair_rank_row,
                                                  rank_row_token, rank_offsets, R, rank_rows, T,
                                                  H, k, partial, status, as_stream(stream)));
}

int ep_combine_reduce(const void* partial, int64_t rank_rows, const int32_t* rank_dst_row,
                      int64_t T, int64_t H, int k, void* out, uint32_t* status, void* stream) {
    int rc = check_rows_args(T, H, k, rank_rows);
    if (rc != EP_OK) return rc;
    if (T == 0) return EP_OK;
    if (!rank_dst_row || !out || (!partial && rank_rows > 0)) return EP_ERR_INVALID_ARG;
    if (!aligned(partial, 16) || !aligned(out, 16) || !aligned(rank_dst_row, 4) ||
        !aligned(status, 4))
        return EP_ERR_ALIGNMENT;
    return cuda_status(ep::launch_combine_reduce(partial, rank_rows, rank_dst_row, T, H, k, out,
                                                 status, as_stream(stream)));
}

int ep_status_read(const uint32_t* status, void* stream, uint32_t* host_flags) {
    if (!status || !host_flags) return EP_ERR_INVALID_ARG;
    cudaError_t e = cudaMemcpyAsync(host_flags, status, sizeof(uint32_t), cudaMemcpyDeviceToHost,
                                    as_stream(stream));
    if (e == cudaSuccess) e = cudaStreamSynchronize(as_stream(stream));
    return cuda_status(e);
}

}  // extern "C"
