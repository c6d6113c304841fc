// ep_layout.cu -- routing layout on the GPU: per-expert counts, exclusive
// scan and stable slot assignment (the "dispatch layout" that the Prefill-like
// profile of awsome-distributed-ai PR #1238 times inside its boundary).
//
// Three small kernels, no inter-block waiting:
//   1. count  : one block per chunk of 512 tokens; a warp-aggregated
//               (match.any) shared-memory histogram of the chunk's experts and
//               of the tokens per virtual rank.  Written transposed,
//               ws[column][chunk], so that phase 2 reads rows.
//   2. scan   : one warp per column (expert or rank): exclusive scan over the
//               chunks in place; the column total is the expert count.
//   3. assign : one block per chunk; every block re-derives the exclusive
//               scan over experts (E <= 1024 values), splits its chunk into 16
//               warp sub-chunks with a shared histogram + scan, and each warp
//               walks its pairs 32 at a time in flattened order, ranking equal
//               experts with match.any + popc(lanemask_lt).  The slot of a
//               pair is therefore the number of earlier pairs with the same
//               expert: a stable, deterministic assignment.
// Masked layouts use the same slots with row = e * capacity + slot.
#include "ep_internal.cuh"

namespace ep {
namespace {

__global__ void __launch_bounds__(kLayoutThreads)
layout_count_kernel(const int32_t* __restrict__ idx, int64_t T, int k, int E, int R_cols,
                    int64_t nchunk, int32_t* __restrict__ ws, uint32_t* __restrict__ status) {
    extern __shared__ int32_t s_hist[];  // [E + R_cols]
    const int ncol = E + R_cols;
    for (int i = threadIdx.x; i < ncol; i += blockDim.x) s_hist[i] = 0;
    if (blockIdx.x == 0 && threadIdx.x == 0 && status) *status = 0u;
    __syncthreads();

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int64_t c = blockIdx.x;
    const int64_t tok0 = c * kLayoutTokensPerChunk + warp * 32;
    const int64_t npairs = T * k;
    const int64_t p0 = tok0 * k;

    // experts: k pieces of 32 consecutive pairs per warp
    for (int piece = 0; piece < k; ++piece) {
        const int64_t p = p0 + piece * 32 + lane;
        int e = -1;
        if (p < npairs) e = __ldg(idx + p);
        const bool valid = (e >= 0) && (e < E);
        const unsigned peers = __match_any_sync(kFullMask, valid ? e : -1 - lane);
        if (valid && (__ffs(peers) - 1) == lane) atomicAdd(&s_hist[e], __popc(peers));
    }

    // tokens per virtual rank: one token per lane, count each rank once
    if (R_cols > 0) {
        const int per_rank = E / R_cols;
        const int64_t t = tok0 + lane;
        const int32_t* row = idx + t * k;
        for (int j = 0; j < k; ++j) {
            int r = -1;
            if (t < T) {
                const int e = __ldg(row + j);
                if (e >= 0 && e < E) {
                    r = e / per_rank;
                    for (int jj = 0; jj < j; ++jj) {
                        const int e2 = __ldg(row + jj);
                        if (e2 >= 0 && e2 < E && e2 / per_rank == r) { r = -1; break; }
                    }
                }
            }
            const unsigned peers = __match_any_sync(kFullMask, r >= 0 ? r : -1 - lane);
            if (r >= 0 && (__ffs(peers) - 1) == lane) atomicAdd(&s_hist[E + r], __popc(peers));
        }
    }
    __syncthreads();
    for (int i = threadIdx.x; i < ncol; i += blockDim.x) ws[(int64_t)i * nchunk + c] = s_hist[i];
}

constexpr int kScanWarps = 8;

__global__ void __launch_bounds__(kScanWarps * 32)
layout_scan_kernel(int32_t* __restrict__ ws, int64_t nchunk, int E, int R_cols,
                   int32_t* __restrict__ expert_counts, int32_t* __restrict__ rank_token_counts) {
    const int lane = threadIdx.x & 31;
    const int col = blockIdx.x * kScanWarps + (threadIdx.x >> 5);
    if (col >= E + R_cols) return;
    int32_t* row = ws + (int64_t)col * nchunk;
    int carry = 0;
    for (int64_t c0 = 0; c0 < nchunk; c0 += 32) {
        const int64_t c = c0 + lane;
        const int v = c < nchunk ? row[c] : 0;
        int incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(kFullMask, incl, o);
            if (lane >= o) incl += n;
        }
        if (c < nchunk) row[c] = carry + incl - v;
        carry += __shfl_sync(kFullMask, incl, 31);
    }
    if (lane == 0) {
        if (col < E) expert_counts[col] = carry;
        else rank_token_counts[col - E] = carry;
    }
}

// Exclusive scan of counts[0..E) into s_off[0..E] by one 512-thread block.
__device__ void block_exclusive_scan(const int32_t* __restrict__ counts, int E, int32_t* s_off,
                                     int32_t* s_warp) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    // each thread owns two consecutive experts (E <= 1024 = 2 * 512)
    const int e0 = 2 * threadIdx.x;
    const int a = e0 < E ? counts[e0] : 0;
    const int b = e0 + 1 < E ? counts[e0 + 1] : 0;
    int incl = a + b;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int n = __shfl_up_sync(kFullMask, incl, o);
        if (lane >= o) incl += n;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    if (warp == 0) {
        int v = lane < kLayoutWarps ? s_warp[lane] : 0;
        int w_incl = v;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int n = __shfl_up_sync(kFullMask, w_incl, o);
            if (lane >= o) w_incl += n;
        }
        if (lane < kLayoutWarps) s_warp[lane] = w_incl - v;  // exclusive warp prefix
    }
    __syncthreads();
    const int excl = s_warp[warp] + incl - (a + b);
    if (e0 < E) s_off[e0] = excl;
    if (e0 + 1 < E) s_off[e0 + 1] = excl + a;
    if (e0 + 1 == E || e0 + 2 == E) s_off[E] = excl + a + b;  // thread holding the last expert
}

__global__ void __launch_bounds__(kLayoutThreads)
layout_assign_kernel(const int32_t* __restrict__ idx, int64_t T, int k, int E, int kind,
                     int capacity, int64_t nchunk, const int32_t* __restrict__ ws,
                     const int32_t* __restrict__ expert_counts, int32_t* __restrict__ expert_offsets,
                     int32_t* __restrict__ dst_row, uint32_t* __restrict__ status) {
    extern __shared__ __align__(16) unsigned char smem[];
    int32_t* s_off = reinterpret_cast<int32_t*>(smem);                  // [E + 1]
    int32_t* s_base = s_off + (E + 1);                                  // [E]
    int32_t* s_warp = s_base + E;                                       // [kLayoutWarps]
    uint16_t* s_w = reinterpret_cast<uint16_t*>(s_warp + kLayoutWarps);  // [kLayoutWarps][E]

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int64_t c = blockIdx.x;

    block_exclusive_scan(expert_counts, E, s_off, s_warp);
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_base[e] = ws[(int64_t)e * nchunk + c];
    for (int i = threadIdx.x; i < kLayoutWarps * E; i += blockDim.x) s_w[i] = 0;
    __syncthreads();
    if (c == 0)
        for (int e = threadIdx.x; e <= E; e += blockDim.x) expert_offsets[e] = s_off[e];

    const int64_t npairs = T * k;
    const int64_t p0 = (c * kLayoutTokensPerChunk + warp * 32) * k;
    uint16_t* my_w = s_w + warp * E;

    // per-warp histogram of the warp's sub-chunk (each warp owns its row of
    // s_w; within one piece distinct experts have distinct leaders)
    for (int piece = 0; piece < k; ++piece) {
        const int64_t p = p0 + piece * 32 + lane;
        int e = -1;
        if (p < npairs) e = __ldg(idx + p);
        const bool valid = (e >= 0) && (e < E);
        const unsigned peers = __match_any_sync(kFullMask, valid ? e : -1 - lane);
        if (valid && (__ffs(peers) - 1) == lane) my_w[e] = (uint16_t)(my_w[e] + __popc(peers));
        __syncwarp();
    }
    __syncthreads();
    // exclusive scan over the warps, per expert
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = 0;
#pragma unroll
        for (int w = 0; w < kLayoutWarps; ++w) {
            const int v = s_w[w * E + e];
            s_w[w * E + e] = (uint16_t)run;
            run += v;
        }
    }
    __syncthreads();

    const unsigned lt = lanemask_lt();
    for (int piece = 0; piece < k; ++piece) {
        const int64_t p = p0 + piece * 32 + lane;
        int e = -1;
        const bool in_range = p < npairs;
        if (in_range) e = __ldg(idx + p);
        const bool valid = (e >= 0) && (e < E);
        const bool bad = in_range && !valid && e != -1;
        const unsigned peers = __match_any_sync(kFullMask, valid ? e : -1 - lane);
        bool overflow = false;
        int dst = -1;
        if (valid) {
            const int slot = s_base[e] + (int)my_w[e] + __popc(peers & lt);
            if (kind == EP_LAYOUT_CONTIGUOUS) {
                dst = s_off[e] + slot;
            } else if (slot < capacity) {
                dst = e * capacity + slot;
            } else {
                overflow = true;
            }
        }
        if (in_range) dst_row[p] = dst;
        __syncwarp();
        if (valid && (__ffs(peers) - 1) == lane) my_w[e] = (uint16_t)(my_w[e] + __popc(peers));
        __syncwarp();
        warp_flag(status, bad, EP_FLAG_BAD_EXPERT);
        warp_flag(status, overflow, EP_FLAG_OVERFLOW);
    }
}

// T == 0: write the (all-zero) outputs so that callers always get defined data.
__global__ void layout_empty_kernel(int E, int R, int32_t* expert_counts,
                                    int32_t* expert_offsets, int32_t* rank_token_counts,
                                    uint32_t* status) {
    for (int i = threadIdx.x; i <= E; i += blockDim.x) {
        if (i < E) expert_counts[i] = 0;
        expert_offsets[i] = 0;
    }
    if (rank_token_counts)
        for (int i = threadIdx.x; i < R; i += blockDim.x) rank_token_counts[i] = 0;
    if (threadIdx.x == 0 && status) *status = 0u;
}

}  // namespace

size_t layout_assign_smem_bytes(int E) {
    return (size_t)(2 * E + 1 + kLayoutWarps) * sizeof(int32_t) +
           (size_t)kLayoutWarps * E * sizeof(uint16_t);
}

cudaError_t launch_layout(const int32_t* topk_idx, int64_t T, int k, int E, int R, int kind,
                          int capacity, int32_t* expert_counts, int32_t* expert_offsets,
                          int32_t* dst_row, int32_t* rank_token_counts, uint32_t* status,
                          int32_t* workspace, cudaStream_t stream) {
    if (T == 0) {
        layout_empty_kernel<<<1, 256, 0, stream>>>(E, R, expert_counts, expert_offsets,
                                                   rank_token_counts, status);
        return cudaGetLastError();
    }
    const int64_t nchunk = layout_num_chunks(T);
    const int R_cols = rank_token_counts ? R : 0;
    const size_t count_smem = (size_t)(E + R_cols) * sizeof(int32_t);
    layout_count_kernel<<<(unsigned)nchunk, kLayoutThreads, count_smem, stream>>>(
        topk_idx, T, k, E, R_cols, nchunk, workspace, status);
    const int ncol = E + R_cols;
    layout_scan_kernel<<<(ncol + kScanWarps - 1) / kScanWarps, kScanWarps * 32, 0, stream>>>(
        workspace, nchunk, E, R_cols, expert_counts, rank_token_counts);
    layout_assign_kernel<<<(unsigned)nchunk, kLayoutThreads, layout_assign_smem_bytes(E),
                           stream>>>(topk_idx, T, k, E, kind, capacity, nchunk, workspace,
                                     expert_counts, expert_offsets, dst_row, status);
    return cudaGetLastError();
}

}  // namespace ep
