// ep_internal.cuh -- device helpers and launcher declarations shared by the
// translation units of the CUDA library (layout, dispatch, combine, C ABI).
#pragma once

#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <utility>

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

// 32-byte streaming load (sm_100+ 256-bit vector access); `p` 32-byte aligned.
struct Vec32 {
    uint4 lo, hi;
};
__device__ __forceinline__ Vec32 ld_stream_v8(const void* p) {
    Vec32 v;
    asm volatile("ld.global.nc.L1::no_allocate.v8.b32 {%0, %1, %2, %3, %4, %5, %6, %7}, [%8];"
                 : "=r"(v.lo.x), "=r"(v.lo.y), "=r"(v.lo.z), "=r"(v.lo.w), "=r"(v.hi.x),
                   "=r"(v.hi.y), "=r"(v.hi.z), "=r"(v.hi.w)
                 : "l"(p));
    return v;
}

// 32-byte store; `p` 32-byte aligned.
__device__ __forceinline__ void st_v8(void* p, const Vec32& v) {
    asm volatile("st.global.v8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};" ::"l"(p), "r"(v.lo.x),
                 "r"(v.lo.y), "r"(v.lo.z), "r"(v.lo.w), "r"(v.hi.x), "r"(v.hi.y), "r"(v.hi.z),
                 "r"(v.hi.w)
                 : "memory");
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

// Programmatic dependent launch: wait until the preceding kernel in the
// stream has completed and its writes are visible (a no-op when this kernel
// was launched without the attribute), and allow the next kernel in the
// stream to be launched (its blocks then sit in their own wait).
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void pdl_trigger() {
    asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// OR device-side condition bits into the optional status word: one atomic
// per warp at most.
__device__ __forceinline__ void warp_flag(uint32_t* status, bool cond, uint32_t bit) {
    const unsigned any = __ballot_sync(kFullMask, cond);
    if (any && status && (threadIdx.x & 31) == 0) atomicOr(status, bit);
}

// Row of pair (t, lane) for lane < k, validated against [-1, rows): a row
// outside raises EP_FLAG_BAD_ROW and the pair is skipped (-1).
__device__ __forceinline__ int load_dst_row(const int32_t* __restrict__ dst_row, int64_t t, int k,
                                            int64_t rows, uint32_t* status) {
    const int lane = threadIdx.x & 31;
    int r = -1;
    bool bad = false;
    if (lane < k) {
        r = __ldg(dst_row + t * k + lane);
        if (r < -1 || (int64_t)r >= rows) {
            bad = true;
            r = -1;
        }
    }
    warp_flag(status, bad, EP_FLAG_BAD_ROW);
    return r;
}

// ---- per-token FP8 e4m3 cast of one lane's 16 channels --------------------
// 8 consecutive lanes hold one 128-channel block: its amax comes from three
// xor-shuffles, the scale is max(amax, 1e-4) / 448 and the codes are
// e4m3_rn_satfinite(x * (448 / max(amax, 1e-4))), both divisions IEEE.
struct Fp8Group {
    uint4 q;   // 16 e4m3 codes of this lane
    float sf;  // scale of this lane's 128-channel block
};

__device__ __forceinline__ Fp8Group quantize16(const uint4& a, const uint4& b) {
    const uint32_t wv[8] = {a.x, a.y, a.z, a.w, b.x, b.y, b.z, b.w};
    float f[16];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        f[2 * i] = bf16lo_to_f32(wv[i]);
        f[2 * i + 1] = bf16hi_to_f32(wv[i]);
    }
    float amax = 0.0f;
#pragma unroll
    for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(f[i]));
    amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 2));
    amax = fmaxf(amax, __shfl_xor_sync(kFullMask, amax, 4));
    const float ap = fmaxf(amax, 1e-4f);
    Fp8Group g;
    g.sf = __fdiv_rn(ap, 448.0f);
    const float inv = __fdiv_rn(448.0f, ap);
    uint32_t qw[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        const uint32_t lo =
            cvt_e4m3x2_rn_sat(__fmul_rn(f[4 * i], inv), __fmul_rn(f[4 * i + 1], inv));
        const uint32_t hi =
            cvt_e4m3x2_rn_sat(__fmul_rn(f[4 * i + 2], inv), __fmul_rn(f[4 * i + 3], inv));
        qw[i] = lo | (hi << 16);
    }
    g.q = make_uint4(qw[0], qw[1], qw[2], qw[3]);
    return g;
}

// Row index of warp g when each row has S column slices.  S > 1 only when
// the grid holds fewer than 2 * EP_SLICE_WARPS_PER_SM warps per SM, so g then
// fits 32 bits and a 32-bit division suffices; S == 1 needs none.
__device__ __forceinline__ int64_t slice_row(int64_t g, int S) {
    return S == 1 ? g : (int64_t)((uint32_t)g / (uint32_t)S);
}

// ---- weighted reduction of up to k rows into one (combine and the two-stage
// partial / final reductions) -------------------------------------------------

constexpr int kRowBatch = 8;  // rows whose loads are issued together

// Accumulate one batch of up to kRowBatch rows into acc for the U column
// groups starting at v0 (vectors below vend only): all loads first, then the
// FMAs in j order.
template <int U>
__device__ __forceinline__ void accumulate_batch(const uint4* const (&src)[kRowBatch],
                                                 const float (&wj)[kRowBatch], int64_t v0,
                                                 int64_t vend, int lane, float (&acc)[U][8]) {
    uint4 buf[kRowBatch][U];
#pragma unroll
    for (int jj = 0; jj < kRowBatch; ++jj) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t v = v0 + u * 32 + lane;
            buf[jj][u] = make_uint4(0, 0, 0, 0);
            if (src[jj] != nullptr && v < vend) buf[jj][u] = ld_stream_v4(src[jj] + v);
        }
    }
#pragma unroll
    for (int jj = 0; jj < kRowBatch; ++jj) {
        if (src[jj] == nullptr) continue;  // warp-uniform: skipped pairs add nothing
        const float w = wj[jj];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const uint32_t wv[4] = {buf[jj][u].x, buf[jj][u].y, buf[jj][u].z, buf[jj][u].w};
#pragma unroll
            for (int i = 0; i < 4; ++i) {
                acc[u][2 * i] = __fmaf_rn(w, bf16lo_to_f32(wv[i]), acc[u][2 * i]);
                acc[u][2 * i + 1] = __fmaf_rn(w, bf16hi_to_f32(wv[i]), acc[u][2 * i + 1]);
            }
        }
    }
}

template <int U>
__device__ __forceinline__ void store_bf16(uint4* out_row, int64_t v0, int64_t vend, int lane,
                                           const float (&acc)[U][8]) {
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t v = v0 + u * 32 + lane;
        if (v < vend) {
            uint4 o;
            o.x = pack_bf16x2_rn(acc[u][0], acc[u][1]);
            o.y = pack_bf16x2_rn(acc[u][2], acc[u][3]);
            o.z = pack_bf16x2_rn(acc[u][4], acc[u][5]);
            o.w = pack_bf16x2_rn(acc[u][6], acc[u][7]);
            st_v4(out_row + v, o);
        }
    }
}

// out_row[vb, ve) = bf16(fp32 sum over j = 0..k-1 in increasing order of
// w_j * rows[r_j][vb, ve)), one fused multiply-add per term, where lane j
// (< k) of the warp holds r_j (-1: skipped) and w_j.  Each lane owns one
// 16-byte vector of each of U column groups per iteration; the loads of all
// rows of a batch are issued before the FMAs.  With w_j = 1 the chain is a
// plain fp32 sum (fma(1, x, a) rounds x + a once).
template <int U>
__device__ __forceinline__ void reduce_rows(const uint4* __restrict__ rows, int64_t nvec, int k,
                                            int my_row, float my_w, int64_t vb, int64_t ve,
                                            uint4* __restrict__ out_row, int lane) {
    if (k <= kRowBatch) {
        // one batch: row pointers and weights stay in registers for the row
        const uint4* src[kRowBatch];
        float wj[kRowBatch];
#pragma unroll
        for (int jj = 0; jj < kRowBatch; ++jj) {
            const int r = __shfl_sync(kFullMask, my_row, jj);
            wj[jj] = __shfl_sync(kFullMask, my_w, jj);
            src[jj] = (jj < k && r >= 0) ? rows + (int64_t)r * nvec : nullptr;
        }
        for (int64_t v0 = vb; v0 < ve; v0 += 32 * U) {
            float acc[U][8];
#pragma unroll
            for (int u = 0; u < U; ++u)
#pragma unroll
                for (int i = 0; i < 8; ++i) acc[u][i] = 0.0f;
            accumulate_batch<U>(src, wj, v0, ve, lane, acc);
            store_bf16<U>(out_row, v0, ve, lane, acc);
        }
        return;
    }
    // k > kRowBatch: batches of kRowBatch rows inside each column group
    for (int64_t v0 = vb; v0 < ve; v0 += 32 * U) {
        float acc[U][8];
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int i = 0; i < 8; ++i) acc[u][i] = 0.0f;
        for (int j0 = 0; j0 < k; j0 += kRowBatch) {
            const uint4* src[kRowBatch];
            float wj[kRowBatch];
#pragma unroll
            for (int jj = 0; jj < kRowBatch; ++jj) {
                const int j = j0 + jj;
                const int r = __shfl_sync(kFullMask, my_row, j & 31);
                wj[jj] = __shfl_sync(kFullMask, my_w, j & 31);
                src[jj] = (j < k && r >= 0) ? rows + (int64_t)r * nvec : nullptr;
            }
            accumulate_batch<U>(src, wj, v0, ve, lane, acc);
        }
        store_bf16<U>(out_row, v0, ve, lane, acc);
    }
}

// ---- launchers (host) ------------------------------------------------------

// Record a CUDA error for ep_last_cuda_error() (host, per thread).
void record_cuda_error(int err);

// Raise `kernel`'s dynamic shared-memory limit to `bytes`, once per device;
// `configured` is that kernel's flag word (one bit per device ordinal).
template <typename K>
cudaError_t raise_smem_limit(K kernel, size_t bytes, std::atomic<uint64_t>& configured) {
    int dev = 0;
    cudaError_t err = cudaGetDevice(&dev);
    if (err != cudaSuccess) return err;
    const uint64_t bit = 1ull << (dev & 63);
    if (!(configured.load(std::memory_order_acquire) & bit)) {
        err = cudaFuncSetAttribute(kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, (int)bytes);
        if (err != cudaSuccess) return err;
        configured.fetch_or(bit, std::memory_order_acq_rel);
    }
    return cudaSuccess;
}

// An attribute of the current device, read once per device into the
// caller's `cache` (0 = not read yet); 0 if it cannot be read.
int cached_device_attribute(cudaDeviceAttr attr, std::atomic<int> (&cache)[64]);

// Launch `kernel` with programmatic stream serialisation allowed, so that its
// launch overlaps the tail of the previous kernel in the stream.  Every kernel
// of this library starts with pdl_wait() before touching global memory.
template <typename... KArgs, typename... Args>
cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                       cudaStream_t stream, Args&&... args) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = grid;
    cfg.blockDim = block;
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[0].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    return cudaLaunchKernelEx(&cfg, kernel, std::forward<Args>(args)...);
}

// Column slices of the token-row kernels (BF16 dispatch, combine).  One warp
// per token leaves most SMs idle when there are few tokens, so each row is
// then split into S slices of `slice` 16-byte vectors (a multiple of 32: one
// vector per lane), one warp per (token, slice).  S doubles while the grid is
// below `warps_per_sm` warps per SM and the slices stay >= `min_slice`
// vectors (a multiple of 32); S = 1 (slice = nvec) otherwise.  The choice
// only shapes the grid: every output element is still computed by exactly
// one lane, in the same order.
#ifndef EP_SLICE_WARPS_PER_SM
#define EP_SLICE_WARPS_PER_SM 8
#endif
struct RowSlices {
    int S;          // slices (warps) per token
    int64_t slice;  // 16-byte vectors per slice
};
RowSlices row_slices(int64_t T, int64_t nvec, int warps_per_sm = EP_SLICE_WARPS_PER_SM,
                     int64_t min_slice = 32);

// The host-side argument checks of ep_layout (EP_OK when the call may
// proceed); `workspace` / `workspace_bytes` are what the layout would use.
int check_layout_args(const int32_t* topk_idx, int64_t T, int k, int E, int R, int kind,
                      int capacity, int align, int32_t* expert_counts, int32_t* expert_offsets,
                      int32_t* dst_row, int32_t* rank_token_counts, uint32_t* status,
                      void* workspace, size_t workspace_bytes);

// Tokens per layout chunk (one per thread of a 128-thread block).
constexpr int kLayoutThreads = 128;
constexpr int kLayoutWarps = kLayoutThreads / 32;
constexpr int kLayoutTokensPerChunk = kLayoutThreads;

inline int64_t layout_num_chunks(int64_t T) {
    return (T + kLayoutTokensPerChunk - 1) / kLayoutTokensPerChunk;
}

cudaError_t launch_layout(const int32_t* topk_idx, int64_t T, int k, int E, int R, int kind,
                          int capacity, int align, int32_t* expert_counts, int32_t* expert_offsets,
                          int32_t* dst_row, int32_t* rank_token_counts, uint32_t* status,
                          int32_t* workspace, cudaStream_t stream);

// Layout and dispatch in one launch for few tokens; cudaErrorNotSupported
// (nothing enqueued) when the shape is outside the fused kernel's range.
cudaError_t launch_layout_dispatch(const int32_t* topk_idx, int64_t T, int k, int E, int R,
                                   int kind, int capacity, const void* x, int64_t H, bool fp8,
                                   int32_t* expert_counts, int32_t* expert_offsets,
                                   int32_t* dst_row, int32_t* rank_token_counts, void* recv,
                                   float* recv_scale, int64_t rows, uint32_t* status,
                                   cudaStream_t stream);

// `early`: the kernel may read x before waiting on the preceding kernel in
// the stream (only when that kernel cannot write x; see ep_dispatch.cu).
cudaError_t launch_dispatch_bf16(const void* x, int64_t T, int64_t H, int k,
                                 const int32_t* dst_row, void* recv, int64_t rows,
                                 uint32_t* status, cudaStream_t stream, bool early = false);

cudaError_t launch_dispatch_fp8(const void* x, int64_t T, int64_t H, int k,
                                const int32_t* dst_row, uint8_t* recv_q, float* recv_scale,
                                int64_t rows, uint32_t* status, cudaStream_t stream,
                                bool early = false);

cudaError_t launch_combine(const void* y, const float* topk_w, const int32_t* dst_row, int64_t T,
                           int64_t H, int k, int64_t rows, void* out, uint32_t* status,
                           cudaStream_t stream);

cudaError_t launch_combine_fp8(const uint8_t* y_q, const float* y_scale, const float* topk_w,
                               const int32_t* dst_row, int64_t T, int64_t H, int k, int64_t rows,
                               void* out, uint32_t* status, cudaStream_t stream);

// two-stage (rank, then expert) path
size_t rank_keys_bytes(int64_t T, int k);
cudaError_t launch_rank_layout(const int32_t* topk_idx, int64_t T, int k, int E, int R,
                               int32_t* rank_counts, int32_t* rank_offsets,
                               int32_t* rank_dst_row, int32_t* pair_rank_row,
                               int32_t* rank_row_token, int64_t cap, uint32_t* status,
                               void* workspace, cudaStream_t stream);
cudaError_t launch_expand(const void* rank_buf, const int32_t* rank_offsets, int R, int64_t cap,
                          const int32_t* rank_row_token, const int32_t* pair_rank_row,
                          const int32_t* dst_row, int64_t T, int64_t H, int k, void* recv,
                          int64_t rows, uint32_t* status, cudaStream_t stream);
cudaError_t launch_expand_fp8(const uint8_t* rank_q, const float* rank_scale,
                              const int32_t* rank_offsets, int R, int64_t cap,
                              const int32_t* rank_row_token, const int32_t* pair_rank_row,
                              const int32_t* dst_row, int64_t T, int64_t H, int k,
                              uint8_t* recv_q, float* recv_scale, int64_t rows, uint32_t* status,
                              cudaStream_t stream);
cudaError_t launch_combine_partial(const void* y, int64_t rows, const float* topk_w,
                                   const int32_t* dst_row, const int32_t* pair_rank_row,
                                   const int32_t* rank_row_token, const int32_t* rank_offsets,
                                   int R, int64_t cap, int64_t T, int64_t H, int k, void* partial,
                                   uint32_t* status, cudaStream_t stream);
cudaError_t launch_combine_reduce(const void* partial, int64_t cap, const int32_t* rank_dst_row,
                                  int64_t T, int64_t H, int k, void* out, uint32_t* status,
                                  cudaStream_t stream);

}  // namespace ep
