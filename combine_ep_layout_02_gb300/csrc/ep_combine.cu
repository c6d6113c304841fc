// ep_combine.cu -- weighted top-k combine: out[t] = bf16(sum_j w[t,j] *
// y[dst_row[t,j]]), accumulated in fp32 fused multiply-adds in increasing j.
//
// One warp per token (per column slice of the token when there are few
// tokens).  Per iteration each lane owns 8 channels (one 16-byte vector) of U
// column groups; the loads of all k rows for those groups are
// issued before any arithmetic so that k*U 16-byte loads per lane are in
// flight, then the FMAs run in j order (the order fixes the fp32 result
// bit-for-bit).  Every expert-output byte is read once and every output byte
// written once: T*k*H*2 read + T*H*2 written is the HBM floor.  Large batches
// use the same kernel with 32-byte (256-bit) loads and stores.
#include "ep_internal.cuh"

namespace ep {
namespace {

#ifndef EP_COMBINE_U
#define EP_COMBINE_U 2  // column groups (16-byte vectors per lane) per pass
#endif
#ifndef EP_COMBINE_V8_MIN_TOKENS
// 32-byte loads/stores pay off once enough warps are in flight (measured at
// 65,536 tokens: -3.3 %; at 2,048 tokens: +13 %), so they are used from this
// many tokens up, when H % 16 == 0 and y, out are 32-byte aligned
#define EP_COMBINE_V8_MIN_TOKENS 16384
#endif
#ifndef EP_COMBINE_WARPS
#define EP_COMBINE_WARPS 4
#endif

constexpr int kCombineWarps = EP_COMBINE_WARPS;
template <int U>
__global__ void __launch_bounds__(kCombineWarps * 32)
combine_kernel(const uint4* __restrict__ y, const float* __restrict__ topk_w,
               const int32_t* __restrict__ dst_row, int64_t T, int64_t nvec, int k, int S,
               int64_t slice, int64_t rows, uint4* __restrict__ out,
               uint32_t* __restrict__ status) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t g = (int64_t)blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
    const int64_t t = slice_row(g, S);
    if (t >= T) return;  // warp-uniform
    const int64_t vb = (g - t * S) * slice;          // this warp's column slice [vb, ve)
    const int64_t ve = vb + slice < nvec ? vb + slice : nvec;

    int my_row = -1;
    float my_w = 0.0f;
    bool bad = false;
    if (lane < k) {
        my_row = __ldg(dst_row + t * k + lane);
        my_w = __ldg(topk_w + t * k + lane);
        if (my_row < -1 || (int64_t)my_row >= rows) {
            bad = true;
            my_row = -1;
        }
    }
    warp_flag(status, bad, EP_FLAG_BAD_ROW);
    reduce_rows<U>(y, nvec, k, my_row, my_w, vb, ve, out + t * nvec, lane);
}

// The same reduction with 32-byte accesses: each lane owns 16 channels (one
// 32-byte vector) per row, a warp 512 channels per iteration; as above, the
// row pointers and weights of a token stay in registers (k <= kRowBatch) and
// the k rows' loads of an iteration are issued before the FMA chain.  Needs
// H % 16 == 0 and 32-byte-aligned y and out.
__device__ __forceinline__ void fma16(float (&acc)[16], float w, const Vec32& b) {
    const uint32_t wv[8] = {b.lo.x, b.lo.y, b.lo.z, b.lo.w, b.hi.x, b.hi.y, b.hi.z, b.hi.w};
#pragma unroll
    for (int i = 0; i < 8; ++i) {
        acc[2 * i] = __fmaf_rn(w, bf16lo_to_f32(wv[i]), acc[2 * i]);
        acc[2 * i + 1] = __fmaf_rn(w, bf16hi_to_f32(wv[i]), acc[2 * i + 1]);
    }
}

__device__ __forceinline__ void store16(Vec32* p, const float (&acc)[16]) {
    Vec32 o;
    o.lo.x = pack_bf16x2_rn(acc[0], acc[1]);
    o.lo.y = pack_bf16x2_rn(acc[2], acc[3]);
    o.lo.z = pack_bf16x2_rn(acc[4], acc[5]);
    o.lo.w = pack_bf16x2_rn(acc[6], acc[7]);
    o.hi.x = pack_bf16x2_rn(acc[8], acc[9]);
    o.hi.y = pack_bf16x2_rn(acc[10], acc[11]);
    o.hi.z = pack_bf16x2_rn(acc[12], acc[13]);
    o.hi.w = pack_bf16x2_rn(acc[14], acc[15]);
    st_v8(p, o);
}

__global__ void __launch_bounds__(kCombineWarps * 32)
combine_v8_kernel(const Vec32* __restrict__ y, const float* __restrict__ topk_w,
                  const int32_t* __restrict__ dst_row, int64_t T, int64_t nvec, int k,
                  int64_t rows, Vec32* __restrict__ out, uint32_t* __restrict__ status) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * kCombineWarps + (threadIdx.x >> 5);
    if (t >= T) return;  // warp-uniform
    int my_row = -1;
    float my_w = 0.0f;
    bool bad = false;
    if (lane < k) {
        my_row = __ldg(dst_row + t * k + lane);
        my_w = __ldg(topk_w + t * k + lane);
        if (my_row < -1 || (int64_t)my_row >= rows) {
            bad = true;
            my_row = -1;
        }
    }
    warp_flag(status, bad, EP_FLAG_BAD_ROW);
    Vec32* out_row = out + t * nvec;
    if (k <= kRowBatch) {
        const Vec32* src[kRowBatch];
        float wj[kRowBatch];
#pragma unroll
        for (int jj = 0; jj < kRowBatch; ++jj) {
            const int r = __shfl_sync(kFullMask, my_row, jj);
            wj[jj] = __shfl_sync(kFullMask, my_w, jj);
            src[jj] = (jj < k && r >= 0) ? y + (int64_t)r * nvec : nullptr;
        }
        for (int64_t v0 = 0; v0 < nvec; v0 += 32) {
            const int64_t v = v0 + lane;
            Vec32 buf[kRowBatch];
#pragma unroll
            for (int jj = 0; jj < kRowBatch; ++jj) {
                buf[jj].lo = make_uint4(0, 0, 0, 0);
                buf[jj].hi = make_uint4(0, 0, 0, 0);
                if (src[jj] != nullptr && v < nvec) buf[jj] = ld_stream_v8(src[jj] + v);
            }
            float acc[16];
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
#pragma unroll
            for (int jj = 0; jj < kRowBatch; ++jj)
                if (src[jj] != nullptr) fma16(acc, wj[jj], buf[jj]);  // warp-uniform
            if (v < nvec) store16(out_row + v, acc);
        }
        return;
    }
    for (int64_t v0 = 0; v0 < nvec; v0 += 32) {
        const int64_t v = v0 + lane;
        float acc[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) acc[i] = 0.0f;
        for (int j0 = 0; j0 < k; j0 += kRowBatch) {
            Vec32 buf[kRowBatch];
            int rr[kRowBatch];
            float ww[kRowBatch];
#pragma unroll
            for (int jj = 0; jj < kRowBatch; ++jj) {
                const int j = j0 + jj;
                rr[jj] = __shfl_sync(kFullMask, my_row, j & 31);
                ww[jj] = __shfl_sync(kFullMask, my_w, j & 31);
                if (j >= k) rr[jj] = -1;
                buf[jj].lo = make_uint4(0, 0, 0, 0);
                buf[jj].hi = make_uint4(0, 0, 0, 0);
                if (rr[jj] >= 0 && v < nvec) buf[jj] = ld_stream_v8(y + (int64_t)rr[jj] * nvec + v);
            }
#pragma unroll
            for (int jj = 0; jj < kRowBatch; ++jj)
                if (rr[jj] >= 0) fma16(acc, ww[jj], buf[jj]);  // warp-uniform
        }
        if (v < nvec) store16(out_row + v, acc);
    }
}

}  // namespace

cudaError_t launch_combine(const void* y, const float* topk_w, const int32_t* dst_row, int64_t T,
                           int64_t H, int k, int64_t rows, void* out, uint32_t* status,
                           cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    if (T >= EP_COMBINE_V8_MIN_TOKENS && H % 16 == 0 &&
        (reinterpret_cast<uintptr_t>(y) & 31) == 0 && (reinterpret_cast<uintptr_t>(out) & 31) == 0) {
        const unsigned grid8 = (unsigned)((T + kCombineWarps - 1) / kCombineWarps);
        return launch_pdl(combine_v8_kernel, dim3(grid8), dim3(kCombineWarps * 32), 0, stream,
                          static_cast<const Vec32*>(y), topk_w, dst_row, T, H / 16, k, rows,
                          static_cast<Vec32*>(out), status);
    }
    const int64_t nvec = H / 8;
    const RowSlices sl = row_slices(T, nvec);
    const unsigned grid = (unsigned)((T * sl.S + kCombineWarps - 1) / kCombineWarps);
    return launch_pdl(combine_kernel<EP_COMBINE_U>, dim3(grid), dim3(kCombineWarps * 32), 0, stream,
                      static_cast<const uint4*>(y), topk_w, dst_row, T, nvec, k, sl.S, sl.slice,
                      rows, static_cast<uint4*>(out), status);
}

}  // namespace ep
