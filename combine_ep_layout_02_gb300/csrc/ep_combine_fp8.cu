// ep_combine_fp8.cu -- weighted top-k combine of expert outputs held in the
// FP8 payload encoding: e4m3 codes y_q[rows, H] and one float32 scale
// y_scale[rows, H/128] per 128 channels, the value of a code being
// decode(q) * scale.  For each token t, channel h and 128-channel block b:
//     c_j    = fl32(w[t,j] * y_scale[r_j, b])            (one rounding)
//     acc    = fmaf(c_j, decode(y_q[r_j, h]), acc)        in increasing j, from +0
//     out    = bf16_rne(acc)
// over the pairs j with r_j = dst_row[t,j] != -1.  decode() is exact in fp32
// (e4m3 values have at most 4 significant bits), so each step rounds once.
//
// The pages (PR #1238, review section 9 "Smaller notes") name a compressed
// combine path without defining it; this one carries the expert outputs in
// the dispatch payload's own encoding, so it reads T*k*(H + H/32) bytes where
// the BF16 combine reads T*k*H*2.
//
// One warp per token (per column slice of the token when there are few
// tokens); each lane owns 16 consecutive channels (one 16-byte vector of
// codes per row) of U groups of 512 channels per iteration.  The loads of
// all rows of a batch (codes and scales) are issued before the FMAs.  U = 1
// and 4-warp blocks measured fastest: 131,072 x 7168 (Zipf 1.2) 1466 us
// against 1478 us with U = 2 and 1580 us with 8-warp blocks; 2,048 tokens
// (masked, L2 flushed) 36.4 us against 41.8 us with U = 2.
#include "ep_internal.cuh"

namespace ep {
namespace {

#ifndef EP_COMBINE_FP8_U
#define EP_COMBINE_FP8_U 1  // 512-channel groups per lane iteration (loads issued together)
#endif
#ifndef EP_COMBINE_FP8_WARPS
#define EP_COMBINE_FP8_WARPS 4
#endif
constexpr int kWarps = EP_COMBINE_FP8_WARPS;
#ifndef EP_COMBINE_FP8_SLICE_WARPS_PER_SM
// Column slices (whole 512-channel groups) while the grid has fewer than this
// many warps per SM: each warp then walks fewer groups one after the other.
// 2,048 x 7168 (L2 flushed): 36.8 -> 33.1 us (8 slices); 4,096 tokens
// 66.2 -> 59.2 us (4 slices); 1,024 tokens and below within 1 %.
#define EP_COMBINE_FP8_SLICE_WARPS_PER_SM 100
#endif

// Four e4m3 codes (bytes of w, lowest first) to fp32, exactly: the hardware
// conversion to an f16 pair (every e4m3 value, NaN included, is an f16
// value), then f16 to fp32.
__device__ __forceinline__ void e4m3x4_to_f32(uint32_t w, float& f0, float& f1, float& f2,
                                              float& f3) {
    uint32_t h01, h23;
    asm("{\n\t.reg .b16 lo, hi;\n\t"
        "mov.b32 {lo, hi}, %2;\n\t"
        "cvt.rn.f16x2.e4m3x2 %0, lo;\n\t"
        "cvt.rn.f16x2.e4m3x2 %1, hi;\n\t}"
        : "=r"(h01), "=r"(h23)
        : "r"(w));
    asm("{\n\t.reg .f16 a, b;\n\t"
        "mov.b32 {a, b}, %2;\n\t"
        "cvt.f32.f16 %0, a;\n\t"
        "cvt.f32.f16 %1, b;\n\t}"
        : "=f"(f0), "=f"(f1)
        : "r"(h01));
    asm("{\n\t.reg .f16 a, b;\n\t"
        "mov.b32 {a, b}, %2;\n\t"
        "cvt.f32.f16 %0, a;\n\t"
        "cvt.f32.f16 %1, b;\n\t}"
        : "=f"(f2), "=f"(f3)
        : "r"(h23));
}

// acc[0..16) += c * decode(16 codes of q), one FMA per channel.
__device__ __forceinline__ void fma16_e4m3(float (&acc)[16], float c, const uint4& q) {
    const uint32_t wv[4] = {q.x, q.y, q.z, q.w};
#pragma unroll
    for (int i = 0; i < 4; ++i) {
        float f0, f1, f2, f3;
        e4m3x4_to_f32(wv[i], f0, f1, f2, f3);
        acc[4 * i + 0] = __fmaf_rn(c, f0, acc[4 * i + 0]);
        acc[4 * i + 1] = __fmaf_rn(c, f1, acc[4 * i + 1]);
        acc[4 * i + 2] = __fmaf_rn(c, f2, acc[4 * i + 2]);
        acc[4 * i + 3] = __fmaf_rn(c, f3, acc[4 * i + 3]);
    }
}

template <int U>
__global__ void __launch_bounds__(kWarps * 32)
combine_fp8_kernel(const uint8_t* __restrict__ y_q, const float* __restrict__ y_scale,
                   const float* __restrict__ topk_w, const int32_t* __restrict__ dst_row,
                   int64_t T, int64_t H, int k, int S, int64_t slice_ch, int64_t rows,
                   uint16_t* __restrict__ out, uint32_t* __restrict__ status) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t g = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int64_t t = slice_row(g, S);
    if (t >= T) return;  // warp-uniform
    // this warp's channels [cb, ce): multiples of 512 (S > 1) or the whole row
    const int64_t cb = (g - t * S) * slice_ch;
    const int64_t ce = cb + slice_ch < H ? cb + slice_ch : H;
    const int64_t nblk = H / 128;

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
    uint16_t* out_row = out + t * H;

    for (int64_t c0 = cb; c0 < ce; c0 += 512 * U) {
        float acc[U][16];
#pragma unroll
        for (int u = 0; u < U; ++u)
#pragma unroll
            for (int i = 0; i < 16; ++i) acc[u][i] = 0.0f;
        for (int j0 = 0; j0 < k; j0 += kRowBatch) {  // one batch for k <= 8
            int rr[kRowBatch];
            float ww[kRowBatch];
#pragma unroll
            for (int jj = 0; jj < kRowBatch; ++jj) {
                const int j = j0 + jj;
                rr[jj] = __shfl_sync(kFullMask, my_row, j & 31);
                ww[jj] = __shfl_sync(kFullMask, my_w, j & 31);
                if (j >= k) rr[jj] = -1;
            }
            uint4 q[kRowBatch][U];
            float sc[kRowBatch][U];
#pragma unroll
            for (int jj = 0; jj < kRowBatch; ++jj) {
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t c = c0 + u * 512 + lane * 16;
                    q[jj][u] = make_uint4(0, 0, 0, 0);
                    sc[jj][u] = 0.0f;
                    if (rr[jj] >= 0 && c < ce) {
                        q[jj][u] = ld_stream_v4(y_q + (int64_t)rr[jj] * H + c);
                        sc[jj][u] = __ldg(y_scale + (int64_t)rr[jj] * nblk + (c >> 7));
                    }
                }
            }
#pragma unroll
            for (int jj = 0; jj < kRowBatch; ++jj) {
                if (rr[jj] < 0) continue;  // warp-uniform: skipped pairs add nothing
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const float cj = __fmul_rn(ww[jj], sc[jj][u]);
                    fma16_e4m3(acc[u], cj, q[jj][u]);
                }
            }
        }
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t c = c0 + u * 512 + lane * 16;
            if (c < ce) {
                uint4 lo, hi;
                lo.x = pack_bf16x2_rn(acc[u][0], acc[u][1]);
                lo.y = pack_bf16x2_rn(acc[u][2], acc[u][3]);
                lo.z = pack_bf16x2_rn(acc[u][4], acc[u][5]);
                lo.w = pack_bf16x2_rn(acc[u][6], acc[u][7]);
                hi.x = pack_bf16x2_rn(acc[u][8], acc[u][9]);
                hi.y = pack_bf16x2_rn(acc[u][10], acc[u][11]);
                hi.z = pack_bf16x2_rn(acc[u][12], acc[u][13]);
                hi.w = pack_bf16x2_rn(acc[u][14], acc[u][15]);
                st_v4(out_row + c, lo);
                st_v4(out_row + c + 8, hi);
            }
        }
    }
}

}  // namespace

cudaError_t launch_combine_fp8(const uint8_t* y_q, const float* y_scale, const float* topk_w,
                               const int32_t* dst_row, int64_t T, int64_t H, int k, int64_t rows,
                               void* out, uint32_t* status, cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    // slices in units of one lane's 16 channels (32 units = one 512-channel group)
    const RowSlices sl = row_slices(T, H / 16, EP_COMBINE_FP8_SLICE_WARPS_PER_SM);
    const unsigned grid = (unsigned)((T * sl.S + kWarps - 1) / kWarps);
    return launch_pdl(combine_fp8_kernel<EP_COMBINE_FP8_U>, dim3(grid), dim3(kWarps * 32), 0,
                      stream, y_q, y_scale, topk_w, dst_row, T, H, k, sl.S, sl.slice * 16, rows,
                      static_cast<uint16_t*>(out), status);
}

}  // namespace ep
