// ep_dispatch_fp8.cu -- dispatch with the per-token FP8 e4m3 cast fused into
// the copy.  One warp per token (per 512-channel-aligned slice of the token
// when there are few tokens): each lane owns 16 consecutive channels, 8
// lanes form one 128-channel block whose amax comes from three xor-shuffles,
// so the cast costs no extra pass over memory (PR #1238 measures the unfused
// cast as a separate launch-bound step).  Every input byte is read once and
// every code and scale written once: T*H*2 read + T*k*(H + H/32) written.
#include "ep_internal.cuh"

#ifndef EP_FP8_WARPS
#define EP_FP8_WARPS 8  // warps per block
#endif
#ifndef EP_FP8_MIN_BLOCKS
#define EP_FP8_MIN_BLOCKS 0  // >0: resident blocks per SM the FP8 kernel is compiled for
#endif
#if EP_FP8_MIN_BLOCKS > 0
#define EP_FP8_BOUNDS __launch_bounds__(EP_FP8_WARPS * 32, EP_FP8_MIN_BLOCKS)
#else
#define EP_FP8_BOUNDS __launch_bounds__(EP_FP8_WARPS * 32)
#endif
#ifndef EP_FP8_U
#define EP_FP8_U 2  // 512-channel groups per FP8 iteration (loads issued together)
#endif
#ifndef EP_FP8_LOAD32
#define EP_FP8_LOAD32 0  // 1: one 32-byte load per lane and group instead of two 16-byte loads
#endif

namespace ep {
namespace {

constexpr int kDispatchWarps = EP_FP8_WARPS;  // warps per block
constexpr int kRowRegs = 8;        // destination rows held in registers per pass

// FP8: each lane owns 16 consecutive channels (two 16-byte loads, one
// 16-byte store of codes per destination row; quantize16 in ep_internal.cuh);
// 8 lanes form one 128-channel block; a warp covers 512 channels per group
// and EP_FP8_U groups per iteration (their loads are issued together).
//
// EARLY: the first iteration's loads are issued before the wait on the
// preceding kernel in the stream -- correct only when that kernel cannot
// write x (ep_layout_dispatch: its own layout kernel, which lets this kernel
// start only after having waited for all earlier work itself).
template <bool EARLY>
__global__ void EP_FP8_BOUNDS
dispatch_fp8_kernel(const uint16_t* __restrict__ x, int64_t T, int64_t H, int k, int S,
                    int64_t slice_ch, const int32_t* __restrict__ dst_row,
                    uint8_t* __restrict__ recv_q, float* __restrict__ recv_scale, int64_t rows,
                    uint32_t* __restrict__ status) {
    constexpr int U = EP_FP8_U;
    const int lane = threadIdx.x & 31;
    const int64_t g = (int64_t)blockIdx.x * kDispatchWarps + (threadIdx.x >> 5);
    const int64_t t = slice_row(g, S);
    // this warp's channels [cb, ce): multiples of 512 (S > 1) or the whole row,
    // so that all 8 lanes of a 128-channel block agree on every bound below
    const int64_t cb = (g - t * S) * slice_ch;
    const int64_t ce = cb + slice_ch < H ? cb + slice_ch : H;
    const uint16_t* src = x + t * H;
    uint4 ea[U], eb[U];  // EARLY: the first iteration's loads
    if (EARLY && t < T) {
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t c = cb + u * 512 + lane * 16;
            ea[u] = make_uint4(0, 0, 0, 0);
            eb[u] = make_uint4(0, 0, 0, 0);
            if (c < ce) {
                ea[u] = ld_stream_v4(src + c);
                eb[u] = ld_stream_v4(src + c + 8);
            }
        }
    }
    pdl_wait();
    pdl_trigger();
    if (t >= T) return;
    const int my_row = load_dst_row(dst_row, t, k, rows, status);
    const int64_t nblk = H / 128;
    for (int j0 = 0; j0 < k; j0 += kRowRegs) {
        int rr[kRowRegs];
#pragma unroll
        for (int jj = 0; jj < kRowRegs; ++jj) {
            const int r = __shfl_sync(kFullMask, my_row, (j0 + jj) & 31);
            rr[jj] = (j0 + jj < k) ? r : -1;
        }
        for (int64_t c0 = cb; c0 < ce; c0 += 512 * U) {
            uint4 a[U], b[U];
            const bool pre = EARLY && j0 == 0 && c0 == cb;  // warp-uniform
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c = c0 + u * 512 + lane * 16;
                a[u] = make_uint4(0, 0, 0, 0);
                b[u] = make_uint4(0, 0, 0, 0);
                if (pre) {
                    a[u] = ea[u];
                    b[u] = eb[u];
                } else if (c < ce) {  // H % 128 == 0: all 8 lanes of a block agree
#if EP_FP8_LOAD32
                    const Vec32 v = ld_stream_v8(src + c);  // 32-byte aligned: H % 128 == 0
                    a[u] = v.lo;
                    b[u] = v.hi;
#else
                    a[u] = ld_stream_v4(src + c);
                    b[u] = ld_stream_v4(src + c + 8);
#endif
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c = c0 + u * 512 + lane * 16;
                const bool act = c < ce;
                const Fp8Group g = quantize16(a[u], b[u]);
                const bool scale_writer = act && (lane & 7) == 0;
#pragma unroll
                for (int jj = 0; jj < kRowRegs; ++jj) {
                    const int r = rr[jj];
                    if (r < 0) continue;  // warp-uniform
                    if (act) st_v4(recv_q + (int64_t)r * H + c, g.q);
                    if (scale_writer) recv_scale[(int64_t)r * nblk + (c >> 7)] = g.sf;
                }
            }
        }
    }
}

}  // namespace

cudaError_t launch_dispatch_fp8(const void* x, int64_t T, int64_t H, int k,
                                const int32_t* dst_row, uint8_t* recv_q, float* recv_scale,
                                int64_t rows, uint32_t* status, cudaStream_t stream,
                                bool early) {
    if (T == 0) return cudaSuccess;
    // slices in units of one lane's 16 channels (32 units = one 512-channel group)
    const RowSlices sl = row_slices(T, H / 16);
    const unsigned grid = (unsigned)((T * sl.S + kDispatchWarps - 1) / kDispatchWarps);
    return launch_pdl(early ? dispatch_fp8_kernel<true> : dispatch_fp8_kernel<false>, dim3(grid), dim3(kDispatchWarps * 32), 0, stream,
                      static_cast<const uint16_t*>(x), T, H, k, sl.S, sl.slice * 16, dst_row,
                      recv_q, recv_scale, rows, status);
}

}  // namespace ep
