// ep_internal.cuh -- device helpers and launcher declarations shared by the
// translation units of the CUDA library (layout, dispatch, combine, C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include "ep.h"

namespace ep {

constexpr unsigned kFullMask = 0xffffffffu;

__device__ __forceinline__ unsigned lanemask_lt() {
    unsigned m;
    asm("mov.u32 %0, %%lanemask_lt;" : "=r"(m));
    return m;
}

// 16-byte streaming load through the non-coherent path without allocating
// in L1 (each input byte is read once by the kernels that use this).
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
    uint4 v;
    asm volatile("ld.global.nc.L1::no_allocate.v4.u32 {%0, %1, %2, %3}, [%4];"
                 : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
                 : "l"(p));
    return v;
}

// 16-byte store.
__device__ __forceinline__ void st_v4(void* p, const uint4& v) {
    asm volatile("st.global.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z),
                 "r"(v.w)
                 : "memory");
}

// 16-byte store with the evict-first ("streaming") cache hint.
__device__ __forceinline__ void st_cs_v4(void* p, const uint4& v) {
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(v.x), "r"(v.y),
                 "r"(v.z), "r"(v.w)
                 : "memory");
}

// bf16 bit patterns (low / high half of a 32-bit word) to fp32: by
// definition the bf16 bits are the upper half of the binary32 encoding.
__device__ __forceinline__ float bf16lo_to_f32(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16hi_to_f32(uint32_t w) { return __uint_as_float(w & 0xffff0000u); }

// Round two fp32 values to bf16 (nearest even) and pack them, `lo` at the
// lower address.
__device__ __forceinline__ uint32_t pack_bf16x2_rn(float lo, float hi) {
    uint32_t r;
    asm("cvt.rn.bf16x2.f32 %0, %1, %2;" : "=r"(r) : "f"(hi), "f"(lo));
    return r;
}

// Convert two fp32 values to OCP E4M3 with round-to-nearest-even and
// saturation to the largest finite value; `lo` lands in the low byte.
__device__ __forceinline__ uint32_t cvt_e4m3x2_rn_sat(float lo, float hi) {
    uint16_t r;
    asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(r) : "f"(hi), "f"(lo));
    return r;
}

// OR device-side condition bits into the optional status word: one atomic
// per warp at most.
__device__ __forceinline__ void warp_flag(uint32_t* status, bool cond, uint32_t bit) {
    const unsigned any = __ballot_sync(kFullMask, cond);
    if (any && status && (threadIdx.x & 31) == 0) atomicOr(status, bit);
}

// ---- launchers (host) ------------------------------------------------------

// Record a CUDA error for ep_last_cuda_error() (host, per thread).
void record_cuda_error(int err);

// Tokens per layout chunk (one per thread of a 512-thread block).
constexpr int kLayoutThreads = 512;
constexpr int kLayoutWarps = kLayoutThreads / 32;
constexpr int kLayoutTokensPerChunk = kLayoutThreads;

inline int64_t layout_num_chunks(int64_t T) {
    return (T + kLayoutTokensPerChunk - 1) / kLayoutTokensPerChunk;
}

cudaError_t launch_layout(const int32_t* topk_idx, int64_t T, int k, int E, int R, int kind,
                          int capacity, int32_t* expert_counts, int32_t* expert_offsets,
                          int32_t* dst_row, int32_t* rank_token_counts, uint32_t* status,
                          int32_t* workspace, cudaStream_t stream);

cudaError_t launch_dispatch_bf16(const void* x, int64_t T, int64_t H, int k,
                                 const int32_t* dst_row, void* recv, int64_t rows,
                                 uint32_t* status, cudaStream_t stream);

cudaError_t launch_dispatch_fp8(const void* x, int64_t T, int64_t H, int k,
                                const int32_t* dst_row, uint8_t* recv_q, float* recv_scale,
                                int64_t rows, uint32_t* status, cudaStream_t stream);

cudaError_t launch_combine(const void* y, const float* topk_w, const int32_t* dst_row, int64_t T,
                           int64_t H, int k, int64_t rows, void* out, uint32_t* status,
                           cudaStream_t stream);

}  // namespace ep
