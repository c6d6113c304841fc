// ep_dispatch.cu -- dispatch (scatter of token rows into the per-expert
// buffer), BF16 bit copy and the fused per-token FP8 e4m3 cast.
//
// One warp per token.  The warp reads the token row once in 16-byte vectors
// (streaming, no L1 allocation) and writes it to each of its k destination
// rows, so every input byte is read once and every output byte written once:
// the HBM floor is T*H*2 read + T*k*H*2 (BF16) or T*k*(H + H/32) (FP8) written.
// The FP8 variant computes the block amax with three xor-shuffles over the 8
// lanes that share a 128-channel block, so the cast costs no extra pass over
// memory (PR #1238 measures the unfused cast as a separate launch-bound step).
#include "ep_internal.cuh"

namespace ep {
namespace {

constexpr int kDispatchWarps = 8;  // warps (= tokens) per block

// Row of pair (t, lane) for lane < k, validated against [-1, rows).
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

template <int U>
__global__ void __launch_bounds__(kDispatchWarps * 32)
dispatch_bf16_kernel(const uint4* __restrict__ x, int64_t T, int64_t nvec, int k,
                     const int32_t* __restrict__ dst_row, uint4* __restrict__ recv, int64_t rows,
                     uint32_t* __restrict__ status) {
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * kDispatchWarps + (threadIdx.x >> 5);
    if (t >= T) return;  // warp-uniform
    const int my_row = load_dst_row(dst_row, t, k, rows, status);
    const uint4* src = x + t * nvec;
    for (int64_t v0 = 0; v0 < nvec; v0 += 32 * U) {
        uint4 buf[U];
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t v = v0 + u * 32 + lane;
            if (v < nvec) buf[u] = ld_stream_v4(src + v);
        }
        for (int j = 0; j < k; ++j) {
            const int r = __shfl_sync(kFullMask, my_row, j);
            if (r < 0) continue;
            uint4* dst = recv + (int64_t)r * nvec;
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t v = v0 + u * 32 + lane;
                if (v < nvec) st_v4(dst + v, buf[u]);
            }
        }
    }
}

// FP8: each lane owns 16 consecutive channels (two 16-byte loads, one
// 16-byte store of codes per destination row); 8 lanes form one 128-channel
// block; a warp covers 512 channels per iteration.
__global__ void __launch_bounds__(kDispatchWarps * 32)
dispatch_fp8_kernel(const uint16_t* __restrict__ x, int64_t T, int64_t H, int k,
                    const int32_t* __restrict__ dst_row, uint8_t* __restrict__ recv_q,
                    float* __restrict__ recv_scale, int64_t rows, uint32_t* __restrict__ status) {
    const int lane = threadIdx.x & 31;
    const int64_t t = (int64_t)blockIdx.x * kDispatchWarps + (threadIdx.x >> 5);
    if (t >= T) return;
    const int my_row = load_dst_row(dst_row, t, k, rows, status);
    const int64_t nblk = H / 128;
    const uint16_t* src = x + t * H;
    for (int64_t c0 = 0; c0 < H; c0 += 512) {
        const int64_t c = c0 + lane * 16;
        const bool act = c < H;  // H % 128 == 0: all 8 lanes of a block agree
        uint4 a = make_uint4(0, 0, 0, 0), b = make_uint4(0, 0, 0, 0);
        if (act) {
            a = ld_stream_v4(src + c);
            b = ld_stream_v4(src + c + 8);
        }
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
        const float sf = __fdiv_rn(ap, 448.0f);
        const float inv = __fdiv_rn(448.0f, ap);
        uint4 q;
        uint32_t qw[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
            const uint32_t lo = cvt_e4m3x2_rn_sat(__fmul_rn(f[4 * i], inv), __fmul_rn(f[4 * i + 1], inv));
            const uint32_t hi =
                cvt_e4m3x2_rn_sat(__fmul_rn(f[4 * i + 2], inv), __fmul_rn(f[4 * i + 3], inv));
            qw[i] = lo | (hi << 16);
        }
        q = make_uint4(qw[0], qw[1], qw[2], qw[3]);
        const bool scale_writer = act && (lane & 7) == 0;
        for (int j = 0; j < k; ++j) {
            const int r = __shfl_sync(kFullMask, my_row, j);
            if (r < 0) continue;
            if (act) st_v4(recv_q + (int64_t)r * H + c, q);
            if (scale_writer) recv_scale[(int64_t)r * nblk + (c >> 7)] = sf;
        }
    }
}

}  // namespace

cudaError_t launch_dispatch_bf16(const void* x, int64_t T, int64_t H, int k,
                                 const int32_t* dst_row, void* recv, int64_t rows,
                                 uint32_t* status, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const int64_t nvec = H / 8;
    const unsigned grid = (unsigned)((T + kDispatchWarps - 1) / kDispatchWarps);
    dispatch_bf16_kernel<4><<<grid, kDispatchWarps * 32, 0, stream>>>(
        static_cast<const uint4*>(x), T, nvec, k, dst_row, static_cast<uint4*>(recv), rows, status);
    return cudaGetLastError();
}

cudaError_t launch_dispatch_fp8(const void* x, int64_t T, int64_t H, int k,
                                const int32_t* dst_row, uint8_t* recv_q, float* recv_scale,
                                int64_t rows, uint32_t* status, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const unsigned grid = (unsigned)((T + kDispatchWarps - 1) / kDispatchWarps);
    dispatch_fp8_kernel<<<grid, kDispatchWarps * 32, 0, stream>>>(
        static_cast<const uint16_t*>(x), T, H, k, dst_row, recv_q, recv_scale, rows, status);
    return cudaGetLastError();
}

}  // namespace ep
