// ep_pipeline.cu -- host-side executor: one layout + dispatch + combine step
// whose inputs and output live in pinned host memory.  The route goes to the
// device first (the layout needs all of it); the hidden states then stream to
// the device in token chunks on a copy stream while earlier chunks are
// dispatched and combined on the caller's stream, and each combined chunk
// streams back to the host on a third stream.  Dispatch and combine of a
// token chunk touch only that chunk's rows when combine reads the dispatched
// rows (identity experts) or a caller-provided device tensor, so chunks are
// independent once the layout is done.
#include <stdlib.h>

#include <new>
#include <vector>

#include "ep_internal.cuh"

struct ep_pipeline {
    int device = 0;
    int max_chunks = 0;
    cudaStream_t h2d = nullptr;
    cudaStream_t d2h = nullptr;
    cudaEvent_t start = nullptr;     // caller's stream reached the call
    cudaEvent_t route = nullptr;     // route on the device
    cudaEvent_t done = nullptr;      // last output chunk back on the host
    std::vector<cudaEvent_t> x_ready;
    std::vector<cudaEvent_t> out_ready;
};

namespace {

void destroy_events(ep_pipeline* p) {
    cudaEvent_t* singles[] = {&p->start, &p->route, &p->done};
    for (cudaEvent_t* e : singles)
        if (*e) cudaEventDestroy(*e), *e = nullptr;
    for (auto& e : p->x_ready)
        if (e) cudaEventDestroy(e);
    for (auto& e : p->out_ready)
        if (e) cudaEventDestroy(e);
    p->x_ready.clear();
    p->out_ready.clear();
    if (p->h2d) cudaStreamDestroy(p->h2d), p->h2d = nullptr;
    if (p->d2h) cudaStreamDestroy(p->d2h), p->d2h = nullptr;
}

inline bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15) == 0; }

}  // namespace

extern "C" {

int ep_pipeline_create(int max_chunks, void** handle) {
    if (!handle || max_chunks < 1 || max_chunks > 4096) return EP_ERR_INVALID_ARG;
    *handle = nullptr;
    ep_pipeline* p = new (std::nothrow) ep_pipeline();
    if (!p) return EP_ERR_INVALID_ARG;
    cudaError_t e = cudaGetDevice(&p->device);
    const unsigned ev_flags = cudaEventDisableTiming;
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->h2d, cudaStreamNonBlocking);
    if (e == cudaSuccess) e = cudaStreamCreateWithFlags(&p->d2h, cudaStreamNonBlocking);
    cudaEvent_t* singles[] = {&p->start, &p->route, &p->done};
    for (cudaEvent_t* ev : singles)
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(ev, ev_flags);
    p->x_ready.assign(max_chunks, nullptr);
    p->out_ready.assign(max_chunks, nullptr);
    for (int i = 0; i < max_chunks && e == cudaSuccess; ++i) {
        e = cudaEventCreateWithFlags(&p->x_ready[i], ev_flags);
        if (e == cudaSuccess) e = cudaEventCreateWithFlags(&p->out_ready[i], ev_flags);
    }
    if (e != cudaSuccess) {
        destroy_events(p);
        delete p;
        ep::record_cuda_error((int)e);
        return EP_ERR_CUDA;
    }
    p->max_chunks = max_chunks;
    *handle = p;
    return EP_OK;
}

int ep_pipeline_destroy(void* handle) {
    if (!handle) return EP_ERR_INVALID_ARG;
    ep_pipeline* p = static_cast<ep_pipeline*>(handle);
    if (p->h2d) cudaStreamSynchronize(p->h2d);
    if (p->d2h) cudaStreamSynchronize(p->d2h);
    destroy_events(p);
    delete p;
    return EP_OK;
}

int ep_roundtrip_host(void* handle, void* stream, const void* x_host, const int32_t* idx_host,
                      const float* w_host, void* out_host, int64_t T, int64_t H, int k, int E,
                      int R, int kind, int capacity, int64_t chunk_tokens, void* x_dev,
                      int32_t* idx_dev, float* w_dev, void* recv, uint8_t* recv_q,
                      float* recv_scale, int64_t rows, const void* y,
                      void* out_dev, int32_t* expert_counts, int32_t* expert_offsets,
                      int32_t* dst_row, int32_t* rank_token_counts, uint32_t* status,
                      void* workspace, size_t workspace_bytes) {
    if (!handle) return EP_ERR_INVALID_ARG;
    ep_pipeline* p = static_cast<ep_pipeline*>(handle);
    if (T < 0 || H <= 0 || k < 1 || k > EP_MAX_TOPK || chunk_tokens < 1 || rows < 0)
        return EP_ERR_INVALID_ARG;
    if (H % 8 != 0) return EP_ERR_ALIGNMENT;
    const int64_t nchunks = T > 0 ? (T + chunk_tokens - 1) / chunk_tokens : 0;
    if (nchunks > p->max_chunks) return EP_ERR_INVALID_ARG;
    const bool fp8 = recv_q != nullptr;
    if (T > 0 && (!x_host || !idx_host || !w_host || !out_host || !x_dev || !idx_dev || !w_dev ||
                  !out_dev))
        return EP_ERR_INVALID_ARG;
    // FP8 dispatch needs its scale buffer and expert outputs to combine;
    // BF16 dispatch needs its buffer (combined directly when y is NULL)
    if (fp8 ? (!recv_scale || !y) : (!recv && rows > 0)) return EP_ERR_INVALID_ARG;
    if (!aligned16(x_dev) || !aligned16(out_dev) || !aligned16(recv) || !aligned16(y) ||
        !aligned16(recv_q))
        return EP_ERR_ALIGNMENT;
    int dev = 0;
    if (cudaGetDevice(&dev) != cudaSuccess || dev != p->device) return EP_ERR_INVALID_ARG;
    cudaStream_t cs = static_cast<cudaStream_t>(stream);
    const size_t xrow = (size_t)H * 2;
    const size_t pair_bytes = (size_t)T * k * 4;

    auto fail = [](cudaError_t e) {
        ep::record_cuda_error((int)e);
        return EP_ERR_CUDA;
    };
    cudaError_t e;
    // nothing of this call may touch the device buffers before the caller's
    // stream has reached it (earlier steps may still be using them)
    if ((e = cudaEventRecord(p->start, cs)) != cudaSuccess) return fail(e);
    if ((e = cudaStreamWaitEvent(p->h2d, p->start, 0)) != cudaSuccess) return fail(e);
    if ((e = cudaStreamWaitEvent(p->d2h, p->start, 0)) != cudaSuccess) return fail(e);

    // 1. route to the device, layout on the caller's stream
    if (T > 0) {
        if ((e = cudaMemcpyAsync(idx_dev, idx_host, pair_bytes, cudaMemcpyHostToDevice, p->h2d)) !=
            cudaSuccess)
            return fail(e);
        if ((e = cudaMemcpyAsync(w_dev, w_host, pair_bytes, cudaMemcpyHostToDevice, p->h2d)) !=
            cudaSuccess)
            return fail(e);
    }
    if ((e = cudaEventRecord(p->route, p->h2d)) != cudaSuccess) return fail(e);
    if ((e = cudaStreamWaitEvent(cs, p->route, 0)) != cudaSuccess) return fail(e);
    int rc = ep_layout(idx_dev, T, k, E, R, kind, capacity, expert_counts, expert_offsets, dst_row,
                       rank_token_counts, status, workspace, workspace_bytes, stream);
    if (rc != EP_OK) return rc;

    // 2. hidden states in chunks on the copy stream
    for (int64_t c = 0; c < nchunks; ++c) {
        const int64_t t0 = c * chunk_tokens;
        const int64_t tn = (T - t0 < chunk_tokens) ? T - t0 : chunk_tokens;
        e = cudaMemcpyAsync(static_cast<char*>(x_dev) + t0 * xrow,
                            static_cast<const char*>(x_host) + t0 * xrow, tn * xrow,
                            cudaMemcpyHostToDevice, p->h2d);
        if (e == cudaSuccess) e = cudaEventRecord(p->x_ready[c], p->h2d);
        if (e != cudaSuccess) return fail(e);
    }
    // 3. dispatch + combine per chunk on the caller's stream, 4. results back
    const void* ysrc = y ? y : recv;
    for (int64_t c = 0; c < nchunks; ++c) {
        const int64_t t0 = c * chunk_tokens;
        const int64_t tn = (T - t0 < chunk_tokens) ? T - t0 : chunk_tokens;
        if ((e = cudaStreamWaitEvent(cs, p->x_ready[c], 0)) != cudaSuccess) return fail(e);
        rc = fp8 ? ep_dispatch_fp8(static_cast<const char*>(x_dev) + t0 * xrow, tn, H, k,
                                   dst_row + t0 * k, recv_q, recv_scale, rows, status, stream)
                 : ep_dispatch(static_cast<const char*>(x_dev) + t0 * xrow, tn, H, k,
                               dst_row + t0 * k, recv, rows, status, stream);
        if (rc != EP_OK) return rc;
        rc = ep_combine(ysrc, w_dev + t0 * k, dst_row + t0 * k, tn, H, k, rows,
                        static_cast<char*>(out_dev) + t0 * xrow, status, stream);
        if (rc != EP_OK) return rc;
        if ((e = cudaEventRecord(p->out_ready[c], cs)) != cudaSuccess) return fail(e);
        if ((e = cudaStreamWaitEvent(p->d2h, p->out_ready[c], 0)) != cudaSuccess) return fail(e);
        e = cudaMemcpyAsync(static_cast<char*>(out_host) + t0 * xrow,
                            static_cast<const char*>(out_dev) + t0 * xrow, tn * xrow,
                            cudaMemcpyDeviceToHost, p->d2h);
        if (e != cudaSuccess) return fail(e);
    }
    // the caller's stream completes only after the last output chunk landed
    if ((e = cudaEventRecord(p->done, p->d2h)) != cudaSuccess) return fail(e);
    if ((e = cudaStreamWaitEvent(cs, p->done, 0)) != cudaSuccess) return fail(e);
    return EP_OK;
}

}  // extern "C"
