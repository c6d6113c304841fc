// ep_two_stage.cu -- the two-stage (rank, then expert) form of dispatch and
// combine that the pages' transport uses: one copy of a token per virtual
// rank it reaches, expanded on arrival into that rank's experts
// (dispatch_copy_epilogue in the afdEP kernel traces), and on the way back a
// rank-local partial reduction followed by the final reduction over the
// token's ranks (combine_reduce_epilogue).  Here the "ranks" are regions of
// one GPU's memory, so the copy to ranks is ep_dispatch with rank_dst_row.
//
//   rank layout : keys kernel (one key per (token, rank): the rank for the
//                 token's first pair in that rank, -1 for its other pairs)
//                 -> the ordinary layout over keys with E' = R experts
//                 -> finish kernel (pair_rank_row for every pair, the token
//                 of every rank row).
//   expand      : one warp per rank row, copying it to the expert rows of its
//                 token's pairs in that rank (BF16 rows, or FP8 code rows plus
//                 their fp32 scale rows).
//   partial     : one warp per rank row, fp32 FMA chain over those pairs in
//                 increasing j, rounded to bf16.
//   reduce      : one warp per token, fp32 sum of its rank rows' partials in
//                 increasing j of their first pair, rounded to bf16 (the same
//                 reducer with unit weights).
// With few rows each row is split into column slices, one warp each, as in
// the single-stage row kernels.
#include "ep_internal.cuh"

namespace ep {
namespace {

constexpr int kWarps = 8;

// Keys for the rank layout: the rank for the first pair of each (token,
// rank), -1 for the token's other pairs in that rank and for id -1, and R
// (out of range for the inner layout, which flags it) for any other bad id.
__global__ void rank_keys_kernel(const int32_t* __restrict__ idx, int64_t T, int k, int E, int R,
                                 int32_t* __restrict__ keys) {
    pdl_wait();
    pdl_trigger();
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T) return;
    const int per_rank = E / R;
    const int32_t* row = idx + t * k;
    int32_t* out = keys + t * k;
    uint64_t seen = 0;  // ranks < 64 already keyed for this token
    for (int j = 0; j < k; ++j) {
        const int e = row[j];
        int key;
        if (e == -1) {
            key = -1;
        } else if (e < -1 || e >= E) {
            key = R;
        } else {
            const int r = e / per_rank;
            bool first;
            if (r < 64) {
                first = !((seen >> r) & 1);
                seen |= 1ull << r;
            } else {
                first = true;
                for (int jj = 0; jj < j; ++jj) {
                    const int e2 = row[jj];
                    if (e2 >= 0 && e2 < E && e2 / per_rank == r) { first = false; break; }
                }
            }
            key = first ? r : -1;
        }
        out[j] = key;
    }
}

// pair_rank_row for every pair and the token of every rank row.
__global__ void rank_finish_kernel(const int32_t* __restrict__ idx, int64_t T, int k, int E, int R,
                                   const int32_t* __restrict__ rank_dst_row,
                                   int32_t* __restrict__ pair_rank_row,
                                   int32_t* __restrict__ rank_row_token, int64_t cap,
                                   uint32_t* __restrict__ status) {
    pdl_wait();
    pdl_trigger();
    const int64_t t = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
    if (t >= T) return;
    const int per_rank = E / R;
    const int32_t* row = idx + t * k;
    const int32_t* rdst = rank_dst_row + t * k;
    for (int j = 0; j < k; ++j) {
        const int e = row[j];
        int out = -1;
        const int first_row = rdst[j];
        if (first_row >= 0) {
            out = first_row;
            if (first_row < cap) rank_row_token[first_row] = (int32_t)t;
            else if (status) atomicOr(status, EP_FLAG_BAD_ROW);  // caller's buffer too small
        } else if (e >= 0 && e < E) {
            const int r = e / per_rank;
            for (int jj = 0; jj < j; ++jj) {
                const int e2 = row[jj];
                if (rdst[jj] >= 0 && e2 / per_rank == r) { out = rdst[jj]; break; }
            }
        }
        pair_rank_row[t * k + j] = out;
    }
}

// The pairs of rank row i's token that belong to row i: lane j (< k) returns
// its destination row (validated against [0, rows)) or -1.
__device__ __forceinline__ int rank_row_pair(int64_t i, int64_t t, int k,
                                             const int32_t* __restrict__ pair_rank_row,
                                             const int32_t* __restrict__ dst_row, int64_t rows,
                                             uint32_t* status) {
    const int lane = threadIdx.x & 31;
    int d = -1;
    bool bad = false;
    if (lane < k) {
        const int pr = __ldg(pair_rank_row + t * k + lane);
        const int dd = __ldg(dst_row + t * k + lane);
        if (dd < -1 || (int64_t)dd >= rows) bad = true;
        else if (pr == i) d = dd;
    }
    warp_flag(status, bad, EP_FLAG_BAD_ROW);
    return d;
}

// Number of rank rows (rank_offsets[R]); rows beyond `cap` are not touched
// and raise EP_FLAG_BAD_ROW.
__device__ __forceinline__ int64_t live_rank_rows(const int32_t* rank_offsets, int R, int64_t cap,
                                                  uint32_t* status) {
    int64_t n = __ldg(rank_offsets + R);
    if (n > cap) {
        if (threadIdx.x == 0 && blockIdx.x == 0 && status) atomicOr(status, EP_FLAG_BAD_ROW);
        n = cap;
    }
    return n;
}

// Copy of a rank row to the expert rows of its token's pairs in that rank.
// Rows are `nvec` vectors of type V (16-byte uint4 for bf16 rows and e4m3
// codes, 4-byte words for fp32 scale rows).
template <typename V>
__device__ __forceinline__ V ld_row_vec(const V* p);
template <>
__device__ __forceinline__ uint4 ld_row_vec<uint4>(const uint4* p) { return ld_stream_v4(p); }
template <>
__device__ __forceinline__ uint32_t ld_row_vec<uint32_t>(const uint32_t* p) { return __ldg(p); }

template <typename V>
__device__ __forceinline__ void expand_row(const V* __restrict__ src, V* __restrict__ dst_base,
                                           int64_t nvec, int64_t vb, int64_t ve, int k,
                                           int my_row, int lane) {
    constexpr int U = 4;
    for (int j0 = 0; j0 < k; j0 += 8) {
        V* dst[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
            const int r = __shfl_sync(kFullMask, my_row, (j0 + jj) & 31);
            dst[jj] = (j0 + jj < k && r >= 0) ? dst_base + (int64_t)r * nvec : nullptr;
        }
        for (int64_t v0 = vb; v0 < ve; v0 += 32 * U) {
            V buf[U];
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t v = v0 + u * 32 + lane;
                if (v < ve) buf[u] = ld_row_vec<V>(src + v);
            }
#pragma unroll
            for (int jj = 0; jj < 8; ++jj) {
                if (dst[jj] == nullptr) continue;  // warp-uniform
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t v = v0 + u * 32 + lane;
                    if (v < ve) dst[jj][v] = buf[u];
                }
            }
        }
    }
}

// One warp per rank row (per column slice of it when there are few rows, as
// for the single-stage row kernels): copies rank row i of up to two arrays
// (the payload rows a, sliced, and optionally the scale rows b, copied whole
// by the first slice's warp) to the expert rows of its pairs.
template <typename VA, typename VB>
__global__ void __launch_bounds__(kWarps * 32)
expand_kernel(const VA* __restrict__ a_src, VA* __restrict__ a_dst, int64_t a_nvec, int S,
              int64_t slice, const VB* __restrict__ b_src, VB* __restrict__ b_dst,
              int64_t b_nvec, const int32_t* __restrict__ rank_offsets, int R, int64_t cap,
              const int32_t* __restrict__ rank_row_token,
              const int32_t* __restrict__ pair_rank_row, const int32_t* __restrict__ dst_row,
              int64_t T, int k, int64_t rows, uint32_t* __restrict__ status) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t g = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int64_t i = slice_row(g, S);
    if (i >= live_rank_rows(rank_offsets, R, cap, status)) return;  // warp-uniform
    const int64_t sl = g - i * S;
    const int64_t vb = sl * slice;
    const int64_t ve = vb + slice < a_nvec ? vb + slice : a_nvec;
    const int64_t t = __ldg(rank_row_token + i);
    if (t < 0 || t >= T) {
        if (lane == 0 && status) atomicOr(status, EP_FLAG_BAD_ROW);
        return;
    }
    const int my_row = rank_row_pair(i, t, k, pair_rank_row, dst_row, rows, status);
    expand_row<VA>(a_src + i * a_nvec, a_dst, a_nvec, vb, ve, k, my_row, lane);
    if (b_src != nullptr && sl == 0)
        expand_row<VB>(b_src + i * b_nvec, b_dst, b_nvec, 0, b_nvec, k, my_row, lane);
}

// SLICED: rows split into column slices (few rows).  The unsliced instance
// keeps the loop bounds plain: with the slice bounds live, ptxas spilled in
// the unrolled pair loop and the kernel lost 2.7 % at prefill.
template <bool SLICED>
__global__ void __launch_bounds__(kWarps * 32)
combine_partial_kernel(const uint4* __restrict__ y, int64_t rows, const float* __restrict__ topk_w,
                       const int32_t* __restrict__ dst_row,
                       const int32_t* __restrict__ pair_rank_row,
                       const int32_t* __restrict__ rank_row_token,
                       const int32_t* __restrict__ rank_offsets, int R, int64_t cap, int64_t T,
                       int64_t nvec, int k, int S, int64_t slice, uint4* __restrict__ partial,
                       uint32_t* __restrict__ status) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t g = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int64_t i = SLICED ? slice_row(g, S) : g;
    if (i >= live_rank_rows(rank_offsets, R, cap, status)) return;
    const int64_t vb = SLICED ? (g - i * S) * slice : 0;  // this warp's column slice [vb, ve)
    const int64_t ve = SLICED ? (vb + slice < nvec ? vb + slice : nvec) : nvec;
    const int64_t t = __ldg(rank_row_token + i);
    if (t < 0 || t >= T) {
        if (lane == 0 && status) atomicOr(status, EP_FLAG_BAD_ROW);
        return;
    }
    const int my_row = rank_row_pair(i, t, k, pair_rank_row, dst_row, rows, status);
    const float my_w = lane < k ? __ldg(topk_w + t * k + lane) : 0.0f;
    // a rank row holds few of the token's pairs (1.8 on average at 8 of 256
    // experts over 16 ranks), so this walks the pairs one at a time: at 40
    // registers it keeps 48 warps per SM in flight, which beats batching the
    // loads of all k slots (121 registers, 29 % slower at prefill)
    uint4* out_row = partial + i * nvec;
    for (int64_t v0 = vb; v0 < ve; v0 += 64) {  // two 16-byte vectors per lane
        float acc[2][8];
#pragma unroll
        for (int u = 0; u < 2; ++u)
#pragma unroll
            for (int q = 0; q < 8; ++q) acc[u][q] = 0.0f;
        for (int j = 0; j < k; ++j) {
            const int r = __shfl_sync(kFullMask, my_row, j);
            const float w = __shfl_sync(kFullMask, my_w, j);
            if (r < 0) continue;  // warp-uniform
            const uint4* src = y + (int64_t)r * nvec;
#pragma unroll
            for (int u = 0; u < 2; ++u) {
                const int64_t v = v0 + u * 32 + lane;
                if (v >= ve) continue;
                const uint4 b = ld_stream_v4(src + v);
                const uint32_t wv[4] = {b.x, b.y, b.z, b.w};
#pragma unroll
                for (int q = 0; q < 4; ++q) {
                    acc[u][2 * q] = __fmaf_rn(w, bf16lo_to_f32(wv[q]), acc[u][2 * q]);
                    acc[u][2 * q + 1] = __fmaf_rn(w, bf16hi_to_f32(wv[q]), acc[u][2 * q + 1]);
                }
            }
        }
        store_bf16<2>(out_row, v0, ve, lane, acc);
    }
}

__global__ void __launch_bounds__(kWarps * 32)
combine_reduce_kernel(const uint4* __restrict__ partial, int64_t cap,
                      const int32_t* __restrict__ rank_dst_row, int64_t T, int64_t nvec, int k,
                      int S, int64_t slice, uint4* __restrict__ out,
                      uint32_t* __restrict__ status) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int64_t g = (int64_t)blockIdx.x * kWarps + (threadIdx.x >> 5);
    const int64_t t = slice_row(g, S);
    if (t >= T) return;
    const int64_t vb = (g - t * S) * slice;  // this warp's column slice [vb, ve)
    const int64_t ve = vb + slice < nvec ? vb + slice : nvec;
    int my_row = -1;
    bool bad = false;
    if (lane < k) {
        my_row = __ldg(rank_dst_row + t * k + lane);
        if (my_row < -1 || (int64_t)my_row >= cap) {
            bad = true;
            my_row = -1;
        }
    }
    warp_flag(status, bad, EP_FLAG_BAD_ROW);
    reduce_rows<2>(partial, nvec, k, my_row, 1.0f, vb, ve, out + t * nvec, lane);
}

inline unsigned blocks_for(int64_t n, int per_block) {
    return (unsigned)((n + per_block - 1) / per_block);
}

}  // namespace

size_t rank_keys_bytes(int64_t T, int k) {
    return ((size_t)T * k * sizeof(int32_t) + 255) & ~(size_t)255;
}

cudaError_t launch_rank_layout(const int32_t* topk_idx, int64_t T, int k, int E, int R,
                               int32_t* rank_counts, int32_t* rank_offsets,
                               int32_t* rank_dst_row, int32_t* pair_rank_row,
                               int32_t* rank_row_token, int64_t cap, uint32_t* status,
                               void* workspace, cudaStream_t stream) {
    int32_t* keys = static_cast<int32_t*>(workspace);
    int32_t* inner_ws =
        reinterpret_cast<int32_t*>(static_cast<char*>(workspace) + rank_keys_bytes(T, k));
    cudaError_t e;
    if (T > 0) {
        e = launch_pdl(rank_keys_kernel, dim3(blocks_for(T, 256)), dim3(256), 0, stream, topk_idx,
                       T, k, E, R, keys);
        if (e != cudaSuccess) return e;
    }
    // the ordinary layout over the keys: R "experts", one virtual rank
    e = launch_layout(keys, T, k, R, 1, EP_LAYOUT_CONTIGUOUS, 0, 1, rank_counts, rank_offsets,
                      rank_dst_row, nullptr, status, inner_ws, stream);
    if (e != cudaSuccess || T == 0) return e;
    return launch_pdl(rank_finish_kernel, dim3(blocks_for(T, 256)), dim3(256), 0, stream,
                      topk_idx, T, k, E, R, (const int32_t*)rank_dst_row, pair_rank_row,
                      rank_row_token, cap, status);
}

cudaError_t launch_expand(const void* rank_buf, const int32_t* rank_offsets, int R, int64_t cap,
                          const int32_t* rank_row_token, const int32_t* pair_rank_row,
                          const int32_t* dst_row, int64_t T, int64_t H, int k, void* recv,
                          int64_t rows, uint32_t* status, cudaStream_t stream) {
    if (cap == 0 || T == 0) return cudaSuccess;
    const RowSlices sl = row_slices(cap, H / 8);
    return launch_pdl(expand_kernel<uint4, uint4>, dim3(blocks_for(cap * sl.S, kWarps)),
                      dim3(kWarps * 32), 0, stream, static_cast<const uint4*>(rank_buf),
                      static_cast<uint4*>(recv), H / 8, sl.S, sl.slice, (const uint4*)nullptr,
                      (uint4*)nullptr, (int64_t)0, rank_offsets, R, cap, rank_row_token,
                      pair_rank_row, dst_row, T, k, rows, status);
}

cudaError_t launch_expand_fp8(const uint8_t* rank_q, const float* rank_scale,
                              const int32_t* rank_offsets, int R, int64_t cap,
                              const int32_t* rank_row_token, const int32_t* pair_rank_row,
                              const int32_t* dst_row, int64_t T, int64_t H, int k,
                              uint8_t* recv_q, float* recv_scale, int64_t rows, uint32_t* status,
                              cudaStream_t stream) {
    if (cap == 0 || T == 0) return cudaSuccess;
    const RowSlices sl = row_slices(cap, H / 16);
    return launch_pdl(expand_kernel<uint4, uint32_t>, dim3(blocks_for(cap * sl.S, kWarps)),
                      dim3(kWarps * 32), 0, stream, reinterpret_cast<const uint4*>(rank_q),
                      reinterpret_cast<uint4*>(recv_q), H / 16, sl.S, sl.slice,
                      reinterpret_cast<const uint32_t*>(rank_scale),
                      reinterpret_cast<uint32_t*>(recv_scale), H / 128, rank_offsets, R, cap,
                      rank_row_token, pair_rank_row, dst_row, T, k, rows, status);
}

cudaError_t launch_combine_partial(const void* y, int64_t rows, const float* topk_w,
                                   const int32_t* dst_row, const int32_t* pair_rank_row,
                                   const int32_t* rank_row_token, const int32_t* rank_offsets,
                                   int R, int64_t cap, int64_t T, int64_t H, int k, void* partial,
                                   uint32_t* status, cudaStream_t stream) {
    if (cap == 0 || T == 0) return cudaSuccess;
    const RowSlices sl = row_slices(cap, H / 8);
    return launch_pdl(sl.S > 1 ? combine_partial_kernel<true> : combine_partial_kernel<false>,
                      dim3(blocks_for(cap * sl.S, kWarps)), dim3(kWarps * 32), 0, stream,
                      static_cast<const uint4*>(y), rows, topk_w, dst_row, pair_rank_row,
                      rank_row_token, rank_offsets, R, cap, T, H / 8, k, sl.S, sl.slice,
                      static_cast<uint4*>(partial), status);
}

cudaError_t launch_combine_reduce(const void* partial, int64_t cap, const int32_t* rank_dst_row,
                                  int64_t T, int64_t H, int k, void* out, uint32_t* status,
                                  cudaStream_t stream) {
    if (T == 0) return cudaSuccess;
    const RowSlices sl = row_slices(T, H / 8);
    return launch_pdl(combine_reduce_kernel, dim3(blocks_for(T * sl.S, kWarps)),
                      dim3(kWarps * 32), 0, stream, static_cast<const uint4*>(partial), cap,
                      rank_dst_row, T, H / 8, k, sl.S, sl.slice, static_cast<uint4*>(out),
                      status);
}

}  // namespace ep
