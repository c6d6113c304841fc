// ep_layout.cu -- routing layout on the GPU: per-expert counts, exclusive
// scan and stable slot assignment (the "dispatch layout" that the Prefill-like
// profile of awsome-distributed-ai PR #1238 times inside its boundary).
//
// Batches of up to 2048 tokens take one launch (a single block or one cluster
// of 8 or 16 blocks, in ep_layout_onelaunch.cu); larger batches use three small
// kernels chained with programmatic dependent launch, where no block ever
// waits on another block:
//   1. count  : one 128-thread block per chunk of 128 tokens.  The chunk's
//               ids are staged in shared memory with one coalesced pass, then
//               shared-memory atomic histograms of experts and of tokens per
//               virtual rank.  Written transposed, ws[column][chunk], so that
//               phase 2 reads contiguous rows.
//   2. scan   : one warp per column (expert or rank): each lane owns 16
//               consecutive chunks of a 512-chunk segment (coalesced int4
//               loads), lane sums are warp-scanned, and the exclusive prefix
//               over chunks is written back in place.  The column total is the
//               expert count (or the rank's token count).
//   3. assign : one block per chunk; every block re-derives the exclusive
//               scan over the E expert counts, splits its chunk into four
//               32-token warp sub-chunks with a shared histogram + scan, and
//               each warp walks its pairs 32 at a time in flattened order,
//               ranking equal experts with popc(peers & lanemask_lt), where the
//               peers of a lane (lanes holding the same expert) come from one
//               ballot per bit of the expert id (8 or 10 independent votes)
//               instead of match.any, whose per-SM throughput made it the
//               bottleneck of this kernel.  The
//               slot of a pair is the number of earlier pairs with the same
//               expert: a stable, deterministic assignment.
// Masked layouts use the same slots with row = e * capacity + slot.  With an
// expert alignment m > 1 (contiguous only) each expert's segment is padded to
// a multiple of m rows: the offsets scan ceil(count / m) * m instead.
#include "ep_internal.cuh"
#include "ep_layout_onelaunch.cuh"

namespace ep {
namespace {

// Stage the chunk's pairs [p0, p0 + n) into s_idx[0 .. kLayoutTokensPerChunk*k),
// padding the tail with kPad.
constexpr int kPad = -2147483647 - 1;

__device__ __forceinline__ void stage_ids(const int32_t* __restrict__ idx, int64_t p0, int n,
                                          int npad, int32_t* s_idx) {
    const bool vec = ((reinterpret_cast<uintptr_t>(idx + p0) & 15) == 0);
    int done = 0;
    if (vec) {
        const int n4 = n >> 2;
        const int4* src = reinterpret_cast<const int4*>(idx + p0);
        int4* dst = reinterpret_cast<int4*>(s_idx);
#pragma unroll 4
        for (int i = threadIdx.x; i < n4; i += blockDim.x) dst[i] = __ldg(src + i);
        done = n4 << 2;
    }
    for (int i = done + threadIdx.x; i < n; i += blockDim.x) s_idx[i] = __ldg(idx + p0 + i);
    for (int i = n + threadIdx.x; i < npad; i += blockDim.x) s_idx[i] = kPad;
}

// rank_of[e] = e / (E / R) for the block (one division per expert, once).
__device__ __forceinline__ void fill_rank_table(int E, int R, int32_t* s_rank_of) {
    const int per_rank = E / R;
    for (int e = threadIdx.x; e < E; e += blockDim.x) s_rank_of[e] = e / per_rank;
}

// Add one to s_rank_hist[r] for every virtual rank r that the token's k
// experts (row[0..k)) reach, each rank once.  The row is read in a skewed
// order so that the 32 lanes of a warp (32 consecutive tokens) hit distinct
// shared-memory banks.
__device__ __forceinline__ void count_token_ranks(const int32_t* row, int k, int E, int R,
                                                  const int32_t* s_rank_of, int32_t* s_rank_hist) {
    const int skew = ((threadIdx.x & 31) >> 2) % k;
    if (R <= 64) {
        uint64_t mask = 0;
        for (int j = 0; j < k; ++j) {
            int jj = j + skew;
            if (jj >= k) jj -= k;
            const int e = row[jj];
            if (e >= 0 && e < E) mask |= 1ull << s_rank_of[e];
        }
        while (mask) {
            const int r = __ffsll((long long)mask) - 1;
            atomicAdd(&s_rank_hist[r], 1);
            mask &= mask - 1;
        }
        return;
    }
    for (int j = 0; j < k; ++j) {
        const int e = row[j];
        if (e < 0 || e >= E) continue;
        const int r = s_rank_of[e];
        bool first = true;
        for (int jj = 0; jj < j; ++jj) {
            const int e2 = row[jj];
            if (e2 >= 0 && e2 < E && s_rank_of[e2] == r) { first = false; break; }
        }
        if (first) atomicAdd(&s_rank_hist[r], 1);
    }
}

__global__ void __launch_bounds__(kLayoutThreads)
layout_count_kernel(const int32_t* __restrict__ idx, int64_t T, int k, int E, int R_cols,
                    int64_t nchunk, int32_t* __restrict__ ws, uint32_t* __restrict__ status) {
    extern __shared__ __align__(16) int32_t smem_i[];
    const int npad = kLayoutTokensPerChunk * k;
    int32_t* s_idx = smem_i;            // [npad]
    int32_t* s_hist = smem_i + npad;    // [E + R_cols]
    int32_t* s_rank_of = s_hist + E + R_cols;  // [E] when R_cols > 0
    const int ncol = E + R_cols;
    const int64_t c = blockIdx.x;
    const int64_t t0 = c * kLayoutTokensPerChunk;
    const int64_t left = T - t0;
    const int ntok = left < kLayoutTokensPerChunk ? (int)left : kLayoutTokensPerChunk;

    // shared memory only: before waiting for the previous grid
    for (int i = threadIdx.x; i < ncol; i += blockDim.x) s_hist[i] = 0;
    if (R_cols > 0) fill_rank_table(E, R_cols, s_rank_of);
    pdl_wait();
    pdl_trigger();
    if (c == 0 && threadIdx.x == 0 && status) *status = 0u;
    stage_ids(idx, t0 * k, ntok * k, npad, s_idx);
    __syncthreads();

    // experts: k strided passes over the chunk's pairs
    for (int m = 0; m < k; ++m) {
        const int e = s_idx[m * kLayoutThreads + threadIdx.x];
        if (e >= 0 && e < E) atomicAdd(&s_hist[e], 1);
    }
    // tokens per virtual rank: one token per thread, each rank counted once
    if (R_cols > 0 && threadIdx.x < ntok)
        count_token_ranks(s_idx + threadIdx.x * k, k, E, R_cols, s_rank_of, s_hist + E);
    __syncthreads();
    for (int i = threadIdx.x; i < ncol; i += blockDim.x) ws[(int64_t)i * nchunk + c] = s_hist[i];
}

constexpr int kScanWarps = 4;
constexpr int kScanPerLane = 16;              // chunks per lane per segment
constexpr int kScanSegment = 32 * kScanPerLane;

__global__ void __launch_bounds__(kScanWarps * 32)
layout_scan_kernel(int32_t* __restrict__ ws, int64_t nchunk, int E, int R_cols,
                   int32_t* __restrict__ expert_counts, int32_t* __restrict__ rank_token_counts) {
    pdl_wait();
    pdl_trigger();
    const int lane = threadIdx.x & 31;
    const int col = blockIdx.x * kScanWarps + (threadIdx.x >> 5);
    if (col >= E + R_cols) return;
    int32_t* row = ws + (int64_t)col * nchunk;
    // rows start 16-byte aligned only when nchunk % 4 == 0
    const bool vec = (nchunk & 3) == 0;
    int carry = 0;
    for (int64_t s0 = 0; s0 < nchunk; s0 += kScanSegment) {
        const int64_t c0 = s0 + lane * kScanPerLane;
        int v[kScanPerLane];
        if (vec && c0 + kScanPerLane <= nchunk) {
#pragma unroll
            for (int q = 0; q < kScanPerLane / 4; ++q) {
                const int4 a = *reinterpret_cast<const int4*>(row + c0 + 4 * q);
                v[4 * q] = a.x; v[4 * q + 1] = a.y; v[4 * q + 2] = a.z; v[4 * q + 3] = a.w;
            }
        } else {
#pragma unroll
            for (int q = 0; q < kScanPerLane; ++q) v[q] = (c0 + q < nchunk) ? row[c0 + q] : 0;
        }
        int local = 0;
#pragma unroll
        for (int q = 0; q < kScanPerLane; ++q) local += v[q];
        int incl = local;
#pragma unroll
        for (int o = 1; o < 32; o <<= 1) {
            const int nb = __shfl_up_sync(kFullMask, incl, o);
            if (lane >= o) incl += nb;
        }
        int run = carry + incl - local;
        if (vec && c0 + kScanPerLane <= nchunk) {
#pragma unroll
            for (int q = 0; q < kScanPerLane / 4; ++q) {
                int4 a;
                a.x = run; run += v[4 * q];
                a.y = run; run += v[4 * q + 1];
                a.z = run; run += v[4 * q + 2];
                a.w = run; run += v[4 * q + 3];
                *reinterpret_cast<int4*>(row + c0 + 4 * q) = a;
            }
        } else {
#pragma unroll
            for (int q = 0; q < kScanPerLane; ++q) {
                if (c0 + q < nchunk) row[c0 + q] = run;
                run += v[q];
            }
        }
        carry += __shfl_sync(kFullMask, incl, 31);
    }
    if (lane == 0) {
        if (col < E) expert_counts[col] = carry;
        else rank_token_counts[col - E] = carry;
    }
}

// Exclusive scan of in[0..E) (shared) into s_off[0..E] by one block of NT
// threads (NT <= 1024); s_warp holds NT/32 ints.  Two barriers: each warp
// adds up the totals of the warps before it itself.  Ends with the block
// synchronised.
template <int NT>
__device__ void block_exclusive_scan(const int32_t* in, int E, int32_t* s_off, int32_t* s_warp) {
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int per = (E + NT - 1) / NT;
    const int e0 = threadIdx.x * per;
    int local = 0;
    for (int i = 0; i < per; ++i)
        if (e0 + i < E) local += in[e0 + i];
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int nb = __shfl_up_sync(kFullMask, incl, o);
        if (lane >= o) incl += nb;
    }
    if (lane == 31) s_warp[warp] = incl;
    __syncthreads();
    int base = lane < warp ? s_warp[lane] : 0;  // warps before this one
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) base += __shfl_xor_sync(kFullMask, base, o);
    int run = base + incl - local;
    if (threadIdx.x == NT - 1) s_off[E] = base + incl;  // grand total
    for (int i = 0; i < per; ++i) {
        if (e0 + i < E) {
            s_off[e0 + i] = run;
            run += in[e0 + i];
        }
    }
    __syncthreads();
}

// Peers of this lane: the lanes with valid set whose id equals this lane's,
// from B independent ballots, one per id bit (valid ids are below 2^B).
template <int B>
__device__ __forceinline__ unsigned peers_of_id(bool valid, int e) {
    unsigned p = __ballot_sync(kFullMask, valid);
#pragma unroll
    for (int b = 0; b < B; ++b) {
        const unsigned m = __ballot_sync(kFullMask, (e >> b) & 1);
        p &= ((e >> b) & 1) ? m : ~m;
    }
    return valid ? p : 0u;
}
static_assert(EP_MAX_EXPERTS <= 1024, "ten id bits");

__global__ void __launch_bounds__(kLayoutThreads)
layout_assign_kernel(const int32_t* __restrict__ idx, int64_t T, int k, int E, int kind,
                     int capacity, int align, int64_t nchunk, const int32_t* __restrict__ ws,
                     const int32_t* __restrict__ expert_counts, int32_t* __restrict__ expert_offsets,
                     int32_t* __restrict__ dst_row, uint32_t* __restrict__ status) {
    extern __shared__ __align__(16) int32_t smem_i[];
    const int npad = kLayoutTokensPerChunk * k;
    int32_t* s_idx = smem_i;                                              // [npad]
    int32_t* s_off = s_idx + npad;                                        // [E + 1]
    int32_t* s_base = s_off + (E + 1);                                    // [E]
    int32_t* s_tot = s_base + E;                                          // [E]
    int32_t* s_warp = s_tot + E;                                          // [kLayoutWarps]
    int32_t* s_w = s_warp + kLayoutWarps;                                 // [kLayoutWarps][E]

    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const int64_t c = blockIdx.x;
    const int64_t t0 = c * kLayoutTokensPerChunk;
    const int64_t left = T - t0;
    const int ntok = left < kLayoutTokensPerChunk ? (int)left : kLayoutTokensPerChunk;

    for (int i = threadIdx.x; i < kLayoutWarps * E; i += blockDim.x) s_w[i] = 0;  // shared only
    pdl_wait();
    pdl_trigger();
    // issue every global load of the prologue before the first shared store
    constexpr int kPer = EP_MAX_EXPERTS / kLayoutThreads;
    int cnt_v[kPer], base_v[kPer];
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        const int e = threadIdx.x + q * kLayoutThreads;
        cnt_v[q] = e < E ? expert_counts[e] : 0;
        base_v[q] = e < E ? ws[(int64_t)e * nchunk + c] : 0;
    }
    stage_ids(idx, t0 * k, ntok * k, npad, s_idx);
#pragma unroll
    for (int q = 0; q < kPer; ++q) {
        const int e = threadIdx.x + q * kLayoutThreads;
        if (e < E) {
            s_tot[e] = align > 1 ? (cnt_v[q] + align - 1) / align * align : cnt_v[q];  // padded length
            s_base[e] = base_v[q];
        }
    }
    __syncthreads();
    block_exclusive_scan<kLayoutThreads>(s_tot, E, s_off, s_warp);
    if (c == 0)
        for (int e = threadIdx.x; e <= E; e += blockDim.x) expert_offsets[e] = s_off[e];

    const int wp0 = warp * 32 * k;  // this warp's first pair within the chunk
    int32_t* my_w = s_w + warp * E;

    // per-warp histogram of the warp's 32-token sub-chunk
    for (int m = 0; m < k; ++m) {
        const int e = s_idx[wp0 + m * 32 + lane];
        if (e >= 0 && e < E) atomicAdd(&my_w[e], 1);
    }
    __syncthreads();
    // exclusive scan over the warps, per expert
    for (int e = threadIdx.x; e < E; e += blockDim.x) {
        int run = 0;
#pragma unroll
        for (int w = 0; w < kLayoutWarps; ++w) {
            const int v = s_w[w * E + e];
            s_w[w * E + e] = run;
            run += v;
        }
    }
    __syncthreads();

    const unsigned lt = lanemask_lt();
    const int64_t npairs = (int64_t)ntok * k;
    int32_t* out = dst_row + t0 * k;
    uint32_t flags = 0;
    for (int m = 0; m < k; ++m) {
        const int lp = wp0 + m * 32 + lane;   // pair within the chunk
        const bool in_range = lp < npairs;
        const int e = s_idx[lp];
        const bool valid = (e >= 0) && (e < E);
        const bool bad = in_range && !valid && e != -1;
        // warp-uniform: eight ballots up to 256 experts, ten above
        const unsigned peers = E <= 256 ? peers_of_id<8>(valid, e) : peers_of_id<10>(valid, e);
        bool overflow = false;
        int dst = -1;
        if (valid) {
            const int slot = s_base[e] + my_w[e] + __popc(peers & lt);
            if (kind == EP_LAYOUT_CONTIGUOUS) {
                dst = s_off[e] + slot;
            } else if (slot < capacity) {
                dst = e * capacity + slot;
            } else {
                overflow = true;
            }
        }
        if (in_range) out[lp] = dst;
        __syncwarp();
        if (valid && (__ffs(peers) - 1) == lane) my_w[e] += __popc(peers);
        __syncwarp();
        if (bad) flags |= EP_FLAG_BAD_EXPERT;
        if (overflow) flags |= EP_FLAG_OVERFLOW;
    }
    const unsigned wf = __reduce_or_sync(kFullMask, flags);  // one atomic per warp at most
    if (wf && lane == 0 && status) atomicOr(status, wf);
}

// T == 0: write the (all-zero) outputs so that callers always get defined data.
__global__ void layout_empty_kernel(int E, int R, int32_t* expert_counts,
                                    int32_t* expert_offsets, int32_t* rank_token_counts,
                                    uint32_t* status) {
    pdl_wait();
    pdl_trigger();
    for (int i = threadIdx.x; i <= E; i += blockDim.x) {
        if (i < E) expert_counts[i] = 0;
        expert_offsets[i] = 0;
    }
    if (rank_token_counts)
        for (int i = threadIdx.x; i < R; i += blockDim.x) rank_token_counts[i] = 0;
    if (threadIdx.x == 0 && status) *status = 0u;
}

size_t count_smem_bytes(int k, int E, int R_cols) {
    return ((size_t)kLayoutTokensPerChunk * k + E + R_cols + (R_cols > 0 ? E : 0)) * sizeof(int32_t);
}

size_t assign_smem_bytes(int k, int E) {
    return ((size_t)kLayoutTokensPerChunk * k + 3 * E + 1 + kLayoutWarps + kLayoutWarps * E) *
           sizeof(int32_t);
}

}  // namespace

cudaError_t launch_layout(const int32_t* topk_idx, int64_t T, int k, int E, int R, int kind,
                          int capacity, int align, int32_t* expert_counts, int32_t* expert_offsets,
                          int32_t* dst_row, int32_t* rank_token_counts, uint32_t* status,
                          int32_t* workspace, cudaStream_t stream) {
    if (T == 0)
        return launch_pdl(layout_empty_kernel, dim3(1), dim3(256), 0, stream, E, R, expert_counts,
                          expert_offsets, rank_token_counts, status);
    const int R_cols = rank_token_counts ? R : 0;
    if (T <= EP_LAYOUT_BLOCK_MAX_TOKENS) {
        const cudaError_t err =
            launch_layout_block(topk_idx, T, k, E, R_cols, R, kind, capacity, align,
                                EP_LAYOUT_BLOCK_THREADS, expert_counts, expert_offsets, dst_row,
                                rank_token_counts, status, stream);
        if (err != cudaErrorNotSupported) return err;
    }
    if (T <= EP_LAYOUT_CLUSTER_MAX_TOKENS) {
        cudaError_t err = cudaErrorNotSupported;
        if (T >= EP_LAYOUT_CLUSTER16_MIN_TOKENS)
            err = launch_layout_cluster(topk_idx, T, k, E, R_cols, R, kind, capacity, align, 16,
                                        EP_LAYOUT_CLUSTER16_THREADS, expert_counts,
                                        expert_offsets, dst_row, rank_token_counts, status,
                                        stream);
        if (err != cudaErrorNotSupported) return err;
        err = launch_layout_cluster(topk_idx, T, k, E, R_cols, R, kind, capacity, align, 8,
                                    T <= EP_LAYOUT_CLUSTER_SMALL_MAX_TOKENS
                                        ? EP_LAYOUT_CLUSTER_THREADS_SMALL
                                        : EP_LAYOUT_CLUSTER_THREADS,
                                    expert_counts, expert_offsets, dst_row, rank_token_counts,
                                    status, stream);
        if (err != cudaErrorNotSupported) return err;
    }
    const int64_t nchunk = layout_num_chunks(T);
    const int ncol = E + R_cols;
    cudaError_t err = launch_pdl(layout_count_kernel, dim3((unsigned)nchunk), dim3(kLayoutThreads),
                                 count_smem_bytes(k, E, R_cols), stream, topk_idx, T, k, E, R_cols,
                                 nchunk, workspace, status);
    if (err != cudaSuccess) return err;
    err = launch_pdl(layout_scan_kernel, dim3((unsigned)((ncol + kScanWarps - 1) / kScanWarps)),
                     dim3(kScanWarps * 32), 0, stream, workspace, nchunk, E, R_cols, expert_counts,
                     rank_token_counts);
    if (err != cudaSuccess) return err;
    return launch_pdl(layout_assign_kernel, dim3((unsigned)nchunk), dim3(kLayoutThreads),
                      assign_smem_bytes(k, E), stream, topk_idx, T, k, E, kind, capacity, align, nchunk,
                      workspace, expert_counts, expert_offsets, dst_row, status);
}

}  // namespace ep
