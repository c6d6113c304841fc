// ep_layout.cu -- routing layout on the GPU: per-expert counts, exclusive
// scan and stable slot assignment (the "dispatch layout" that the Prefill-like
// profile of awsome-distributed-ai PR #1238 times inside its boundary).
//
// Batches of up to 384 tokens use one single-block kernel, up to 2048 tokens
// one 8-block cluster kernel (both further down); larger batches use three
// small kernels chained with programmatic dependent launch, where no block
// ever waits on another block:
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
//               ballot per bit of the expert id -- a handful of vote
//               instructions instead of match.any, whose per-SM throughput
//               made it the bottleneck of this kernel.  The
//               slot of a pair is the number of earlier pairs with the same
//               expert: a stable, deterministic assignment.
// Masked layouts use the same slots with row = e * capacity + slot.  With an
// expert alignment m > 1 (contiguous only) each expert's segment is padded to
// a multiple of m rows: the offsets scan ceil(count / m) * m instead.
#include <cooperative_groups.h>

#include "ep_internal.cuh"

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

    pdl_wait();
    pdl_trigger();
    if (c == 0 && threadIdx.x == 0 && status) *status = 0u;
    for (int i = threadIdx.x; i < ncol; i += blockDim.x) s_hist[i] = 0;
    if (R_cols > 0) fill_rank_table(E, R_cols, s_rank_of);
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

// Lanes of the warp whose (valid) key equals this lane's: one ballot per key
// bit.  Invalid lanes get an empty set and appear in no valid lane's set.
__device__ __forceinline__ unsigned warp_peers(bool valid, int key, int key_bits) {
    unsigned peers = __ballot_sync(kFullMask, valid);
    for (int b = 0; b < key_bits; ++b) {
        const bool bit = (key >> b) & 1;
        const unsigned ones = __ballot_sync(kFullMask, bit);
        peers &= bit ? ones : ~ones;
    }
    return valid ? peers : 0u;
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
    for (int i = threadIdx.x; i < kLayoutWarps * E; i += blockDim.x) s_w[i] = 0;
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
    const int key_bits = 32 - __clz(E - 1 > 0 ? E - 1 : 1);  // bits that distinguish ids in [0, E)
    const int64_t npairs = (int64_t)ntok * k;
    int32_t* out = dst_row + t0 * k;
    for (int m = 0; m < k; ++m) {
        const int lp = wp0 + m * 32 + lane;   // pair within the chunk
        const bool in_range = lp < npairs;
        const int e = s_idx[lp];
        const bool valid = (e >= 0) && (e < E);
        const bool bad = in_range && !valid && e != -1;
        const unsigned peers = warp_peers(valid, e, key_bits);
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
        warp_flag(status, bad, EP_FLAG_BAD_EXPERT);
        warp_flag(status, overflow, EP_FLAG_OVERFLOW);
    }
}

// ---- one-launch layouts for small and medium batches -----------------------
// Both split their tokens into warp-owned runs.  Each warp builds a shared
// histogram of its pairs; an exclusive prefix over the warps turns it into
// the warp's base slot per expert; then the warp walks its pairs 32 at a time
// in flattened order and ranks equal experts within the piece with
// popc(peers & lanemask_lt).  Short runs per warp (many warps per block) keep
// the serial part of the walk short.

// Tokens per launch of the single-block kernel, and its block sizes: blocks
// of up to 128 tokens and larger ones (up to kFusedMaxTokens).  Above 384
// tokens the 8-block cluster is faster (512 tokens: 6.9 vs 7.7 us; 384:
// 7.0 vs 6.7 us).
constexpr int kFusedMaxTokens = 384;
#ifndef EP_FUSED_NT_SMALL
#define EP_FUSED_NT_SMALL 1024
#endif
#ifndef EP_FUSED_NT_LARGE
#define EP_FUSED_NT_LARGE 1024
#endif

// Per-warp histograms s_w[w * ES + e] (NT/32 warps; row stride ES = E | 1 is
// odd, so the warps' entries of one expert sit in distinct banks) are
// replaced by their exclusive prefix over w, and s_sum[e] gets the total.
// Up to 8 warps: one thread per expert walks the warps.  More: one warp per
// expert, lane w holding warp w's count, scanned with shuffles.
template <int NT>
__device__ __forceinline__ void warp_hist_prefix(int32_t* s_w, int ES, int E, int32_t* s_sum) {
    constexpr int NW = NT / 32;
    if constexpr (NW <= 8) {
        for (int e = threadIdx.x; e < E; e += NT) {
            int run = 0;
#pragma unroll
            for (int w = 0; w < NW; ++w) {
                const int v = s_w[w * ES + e];
                s_w[w * ES + e] = run;
                run += v;
            }
            s_sum[e] = run;
        }
    } else {
        const int lane = threadIdx.x & 31;
        for (int e = threadIdx.x >> 5; e < E; e += NW) {
            const int v = lane < NW ? s_w[lane * ES + e] : 0;
            int incl = v;
#pragma unroll
            for (int o = 1; o < 32; o <<= 1) {
                const int nb = __shfl_up_sync(kFullMask, incl, o);
                if (lane >= o) incl += nb;
            }
            if (lane < NW) s_w[lane * ES + e] = incl - v;
            if (lane == 31) s_sum[e] = incl;
        }
    }
}

// Histogram of one warp's `wpairs` pairs (s_ids) into its row my_w.
__device__ __forceinline__ void warp_count_pairs(const int32_t* s_ids, int wpairs, int E,
                                                 int32_t* my_w) {
    for (int q = threadIdx.x & 31; q < wpairs; q += 32) {
        const int e = s_ids[q];
        if (e >= 0 && e < E) atomicAdd(&my_w[e], 1);
    }
}

// Slots of one warp's pairs: slot = s_base[e] (if given) + my_w[e] + the
// earlier lanes of the piece holding e; my_w[e] then advances by the piece's
// count of e.  Writes out[0 .. wpairs) and raises the status flags.
__device__ __forceinline__ void warp_assign_pairs(const int32_t* s_ids, int wpairs, int E, int kind,
                                                  int capacity, int32_t* my_w,
                                                  const int32_t* s_base, const int32_t* s_off,
                                                  int32_t* __restrict__ out, uint32_t* status) {
    const int lane = threadIdx.x & 31;
    const unsigned lt = lanemask_lt();
    const int key_bits = 32 - __clz(E - 1 > 0 ? E - 1 : 1);
    for (int q0 = 0; q0 < wpairs; q0 += 32) {  // warp-uniform
        const int q = q0 + lane;
        const bool in_range = q < wpairs;
        const int e = in_range ? s_ids[q] : -1;
        const bool valid = (e >= 0) && (e < E);
        const bool bad = in_range && !valid && e != -1;
        const unsigned peers = warp_peers(valid, e, key_bits);
        bool overflow = false;
        int dst = -1;
        if (valid) {
            const int slot = (s_base ? s_base[e] : 0) + my_w[e] + __popc(peers & lt);
            if (kind == EP_LAYOUT_CONTIGUOUS) {
                dst = s_off[e] + slot;
            } else if (slot < capacity) {
                dst = e * capacity + slot;
            } else {
                overflow = true;
            }
        }
        if (in_range) out[q] = dst;
        __syncwarp();
        if (valid && (__ffs(peers) - 1) == lane) my_w[e] += __popc(peers);
        __syncwarp();
        warp_flag(status, bad, EP_FLAG_BAD_EXPERT);
        warp_flag(status, overflow, EP_FLAG_OVERFLOW);
    }
}

// Shared-memory arrays of the single-block layout (carved by the caller).
struct BlockLayoutSmem {
    int32_t* idx;      // [npad] staged ids (npad = warps * tpw * k >= T * k)
    int32_t* w;        // [warps][E | 1] per-warp histograms, then base slots
    int32_t* tot;      // [E] (padded) segment lengths
    int32_t* off;      // [E + 1] their exclusive scan
    int32_t* rank;     // [R_cols] tokens per virtual rank
    int32_t* rank_of;  // [E]
    int32_t* warp;     // [warps] scan scratch
};

// The single-block layout up to the slot walk, for T tokens in one block of
// NT threads (warp w owns tokens [w*tpw, (w+1)*tpw)): ids staged, per-warp
// histograms and their exclusive prefix over the warps, expert totals
// (stored to expert_counts when given), segment lengths rounded up to
// `align` and scanned into sm.off (stored to expert_offsets when given), and
// the tokens per rank (stored to rank_token_counts when given).  Ends with
// the block synchronised.
template <int NT>
__device__ void block_layout_scan(const int32_t* __restrict__ idx, int T, int k, int E, int R_cols,
                                  int align, int tpw, const BlockLayoutSmem& sm,
                                  int32_t* __restrict__ expert_counts,
                                  int32_t* __restrict__ expert_offsets,
                                  int32_t* __restrict__ rank_token_counts) {
    constexpr int NW = NT / 32;
    const int ES = E | 1;
    const int npairs = T * k;
    const int npad = NW * tpw * k;
    const int warp = threadIdx.x >> 5;
    stage_ids(idx, 0, npairs, npad, sm.idx);
    for (int i = threadIdx.x; i < NW * ES; i += NT) sm.w[i] = 0;
    for (int i = threadIdx.x; i < R_cols; i += NT) sm.rank[i] = 0;
    if (R_cols > 0) fill_rank_table(E, R_cols, sm.rank_of);
    __syncthreads();
    const int wp0 = warp * tpw * k;
    const int wrem = npairs - wp0;
    const int wpairs = wrem <= 0 ? 0 : (wrem < tpw * k ? wrem : tpw * k);
    warp_count_pairs(sm.idx + wp0, wpairs, E, sm.w + warp * ES);
    if (R_cols > 0)
        for (int t = threadIdx.x; t < T; t += NT)
            count_token_ranks(sm.idx + t * k, k, E, R_cols, sm.rank_of, sm.rank);
    __syncthreads();
    warp_hist_prefix<NT>(sm.w, ES, E, sm.tot);
    __syncthreads();
    for (int e = threadIdx.x; e < E; e += NT) {
        const int c = sm.tot[e];
        if (expert_counts) expert_counts[e] = c;
        if (align > 1) sm.tot[e] = (c + align - 1) / align * align;  // padded segment length
    }
    __syncthreads();
    block_exclusive_scan<NT>(sm.tot, E, sm.off, sm.warp);
    if (expert_offsets)
        for (int e = threadIdx.x; e <= E; e += NT) expert_offsets[e] = sm.off[e];
    if (rank_token_counts)
        for (int r = threadIdx.x; r < R_cols; r += NT) rank_token_counts[r] = sm.rank[r];
}

// Small batches (T <= kFusedMaxTokens): the whole layout in one block of NT
// threads; warp w owns tokens [w*tpw, (w+1)*tpw).  The block scan over the
// expert totals gives the offsets -- the same stable slots as the chunked
// kernels, in one launch.  One SM does all the work, so larger batches use
// the cluster or chunked kernels, which spread it over more SMs.
template <int NT>
__global__ void __launch_bounds__(NT)
layout_fused_kernel(const int32_t* __restrict__ idx, int T, int k, int E, int R_cols, int kind,
                    int capacity, int align, int tpw, int32_t* __restrict__ expert_counts,
                    int32_t* __restrict__ expert_offsets, int32_t* __restrict__ dst_row,
                    int32_t* __restrict__ rank_token_counts, uint32_t* __restrict__ status) {
    constexpr int NW = NT / 32;
    extern __shared__ __align__(16) int32_t smem_i[];
    const int ES = E | 1;
    const int npairs = T * k;
    const int npad = NW * tpw * k;              // >= npairs
    BlockLayoutSmem sm;
    sm.idx = smem_i;                            // [npad]
    sm.w = sm.idx + npad;                       // [NW][ES]
    sm.tot = sm.w + NW * ES;                    // [E]
    sm.off = sm.tot + E;                        // [E + 1]
    sm.rank = sm.off + E + 1;                   // [R_cols]
    sm.rank_of = sm.rank + R_cols;              // [E]
    sm.warp = sm.rank_of + E;                   // [NW]
    const int warp = threadIdx.x >> 5;

    pdl_wait();
    pdl_trigger();
    if (threadIdx.x == 0 && status) *status = 0u;
    block_layout_scan<NT>(idx, T, k, E, R_cols, align, tpw, sm, expert_counts, expert_offsets,
                          rank_token_counts);
    const int wp0 = warp * tpw * k;
    const int wrem = npairs - wp0;
    const int wpairs = wrem <= 0 ? 0 : (wrem < tpw * k ? wrem : tpw * k);
    warp_assign_pairs(sm.idx + wp0, wpairs, E, kind, capacity, sm.w + warp * ES, nullptr, sm.off,
                      dst_row + wp0, status);
}

// Medium batches (T <= kClusterMaxTokens): the whole layout in ONE launch of
// one 8-block thread-block cluster.  Each block owns 256 tokens and builds
// per-warp expert histograms; after a cluster barrier every block reads the 8
// block totals through distributed shared memory (the blocks before it give
// its base slots, all of them the totals), and a second cluster barrier keeps
// every block resident until all remote reads are done.  The barriers are
// hardware cluster barriers: no block ever spins on memory.
namespace cg = cooperative_groups;
constexpr int kClusterBlocks = 8;
constexpr int kClusterTokens = 256;  // tokens per block
constexpr int kClusterMaxTokens = kClusterBlocks * kClusterTokens;
#ifndef EP_CLUSTER_NT
#define EP_CLUSTER_NT 1024
#endif

template <int NT>
__global__ void __launch_bounds__(NT)
layout_cluster_kernel(const int32_t* __restrict__ idx, int T, int k, int E, int R_cols, int kind,
                      int capacity, int align, int32_t* __restrict__ expert_counts,
                      int32_t* __restrict__ expert_offsets, int32_t* __restrict__ dst_row,
                      int32_t* __restrict__ rank_token_counts, uint32_t* __restrict__ status) {
    constexpr int NW = NT / 32;
    constexpr int TPW = kClusterTokens / NW;      // tokens per warp
    cg::cluster_group cluster = cg::this_cluster();
    const int b = (int)cluster.block_rank();
    extern __shared__ __align__(16) int32_t smem_i[];
    const int ES = E | 1;
    const int npad = kClusterTokens * k;
    int32_t* s_idx = smem_i;                      // [npad]
    int32_t* s_w = s_idx + npad;                  // [NW][ES]
    int32_t* s_hist = s_w + NW * ES;              // [E + R_cols]  block totals (read remotely)
    int32_t* s_tot = s_hist + E + R_cols;         // [E]
    int32_t* s_base = s_tot + E;                  // [E]
    int32_t* s_off = s_base + E;                  // [E + 1]
    int32_t* s_rank_of = s_off + E + 1;           // [E]
    int32_t* s_rank = s_rank_of + E;              // [R_cols]
    int32_t* s_warp = s_rank + R_cols;            // [NW]
    const int warp = threadIdx.x >> 5;
    const int t0 = b * kClusterTokens;
    const int ntok = T - t0 < 0 ? 0 : (T - t0 < kClusterTokens ? T - t0 : kClusterTokens);

    pdl_wait();
    pdl_trigger();
    if (b == 0 && threadIdx.x == 0 && status) *status = 0u;
    stage_ids(idx, (int64_t)t0 * k, ntok * k, npad, s_idx);
    for (int i = threadIdx.x; i < NW * ES; i += NT) s_w[i] = 0;
    for (int i = threadIdx.x; i < R_cols; i += NT) s_rank[i] = 0;
    if (R_cols > 0) fill_rank_table(E, R_cols, s_rank_of);
    __syncthreads();

    const int wp0 = warp * TPW * k;
    const int wrem = ntok * k - wp0;
    const int wpairs = wrem <= 0 ? 0 : (wrem < TPW * k ? wrem : TPW * k);
    int32_t* my_w = s_w + warp * ES;
    warp_count_pairs(s_idx + wp0, wpairs, E, my_w);
    if (R_cols > 0)
        for (int t = threadIdx.x; t < ntok; t += NT)
            count_token_ranks(s_idx + t * k, k, E, R_cols, s_rank_of, s_rank);
    __syncthreads();
    warp_hist_prefix<NT>(s_w, ES, E, s_hist);
    for (int r = threadIdx.x; r < R_cols; r += NT) s_hist[E + r] = s_rank[r];
    cluster.sync();  // every block's histogram is complete and visible

    for (int e = threadIdx.x; e < E; e += NT) {
        int before = 0, total = 0;
#pragma unroll
        for (int q = 0; q < kClusterBlocks; ++q) {
            const int v = cluster.map_shared_rank(s_hist, q)[e];
            before += q < b ? v : 0;
            total += v;
        }
        s_base[e] = before;
        s_tot[e] = align > 1 ? (total + align - 1) / align * align : total;  // padded length
        if (b == 0) expert_counts[e] = total;
    }
    if (b == 0 && rank_token_counts)
        for (int r = threadIdx.x; r < R_cols; r += NT) {
            int total = 0;
#pragma unroll
            for (int q = 0; q < kClusterBlocks; ++q) total += cluster.map_shared_rank(s_hist, q)[E + r];
            rank_token_counts[r] = total;
        }
    cluster.sync();  // no block leaves while another still reads its histogram

    block_exclusive_scan<NT>(s_tot, E, s_off, s_warp);
    if (b == 0)
        for (int e = threadIdx.x; e <= E; e += NT) expert_offsets[e] = s_off[e];

    warp_assign_pairs(s_idx + wp0, wpairs, E, kind, capacity, my_w, s_base, s_off,
                      dst_row + (int64_t)t0 * k + wp0, status);
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

size_t fused_smem_bytes(int warps, int tpw, int k, int E, int R_cols) {
    return ((size_t)warps * tpw * k + (size_t)warps * (E | 1) + 3 * (size_t)E + 1 + R_cols +
            warps) * sizeof(int32_t);
}

constexpr size_t kFusedSmemLimit = 160 * 1024;

template <int NT>
cudaError_t launch_fused(const int32_t* topk_idx, int64_t T, int k, int E, int R_cols, int kind,
                         int capacity, int align, int tpw, int32_t* expert_counts,
                         int32_t* expert_offsets, int32_t* dst_row, int32_t* rank_token_counts,
                         uint32_t* status, size_t smem, cudaStream_t stream) {
    static std::atomic<uint64_t> configured{0};
    cudaError_t err = raise_smem_limit(layout_fused_kernel<NT>, kFusedSmemLimit, configured);
    if (err != cudaSuccess) return err;
    return launch_pdl(layout_fused_kernel<NT>, dim3(1), dim3(NT), smem, stream, topk_idx, (int)T,
                      k, E, R_cols, kind, capacity, align, tpw, expert_counts, expert_offsets,
                      dst_row, rank_token_counts, status);
}

// The single-block layout with the largest block (down to 128 threads, from
// `nt`) whose shared memory fits; cudaErrorNotSupported if none does.
cudaError_t try_fused(int nt, const int32_t* topk_idx, int64_t T, int k, int E, int R_cols,
                      int kind, int capacity, int align, int32_t* expert_counts,
                      int32_t* expert_offsets, int32_t* dst_row, int32_t* rank_token_counts,
                      uint32_t* status, cudaStream_t stream) {
    for (; nt >= 128; nt /= 2) {
        if (nt != 1024 && nt != 512 && nt != 256 && nt != 128) continue;
        const int warps = nt / 32;
        const int tpw = (int)((T + warps - 1) / warps);
        const size_t smem = fused_smem_bytes(warps, tpw, k, E, R_cols);
        if (smem > kFusedSmemLimit) continue;
#define EP_FUSED_CASE(N)                                                                       \
    case N:                                                                                    \
        return launch_fused<N>(topk_idx, T, k, E, R_cols, kind, capacity, align, tpw,          \
                               expert_counts, expert_offsets, dst_row, rank_token_counts,      \
                               status, smem, stream);
        switch (nt) {
            EP_FUSED_CASE(1024)
            EP_FUSED_CASE(512)
            EP_FUSED_CASE(256)
            EP_FUSED_CASE(128)
        }
#undef EP_FUSED_CASE
    }
    return cudaErrorNotSupported;
}

size_t cluster_smem_bytes(int nt, int k, int E, int R_cols) {
    const size_t warps = nt / 32;
    return ((size_t)kClusterTokens * k + warps * (E | 1) + 5 * (size_t)E + 1 + 2 * (size_t)R_cols +
            warps) * sizeof(int32_t);
}

template <int NT>
cudaError_t launch_cluster(const int32_t* topk_idx, int64_t T, int k, int E, int R_cols, int kind,
                           int capacity, int align, int32_t* expert_counts,
                           int32_t* expert_offsets, int32_t* dst_row, int32_t* rank_token_counts,
                           uint32_t* status, size_t smem, cudaStream_t stream) {
    static std::atomic<uint64_t> configured{0};
    cudaError_t err = raise_smem_limit(layout_cluster_kernel<NT>, kFusedSmemLimit, configured);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(kClusterBlocks);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = kClusterBlocks;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    return cudaLaunchKernelEx(&cfg, layout_cluster_kernel<NT>, topk_idx, (int)T, k, E, R_cols,
                              kind, capacity, align, expert_counts, expert_offsets, dst_row,
                              rank_token_counts, status);
}

// The cluster layout with the largest block (down to 256 threads, from `nt`)
// whose shared memory fits; cudaErrorNotSupported if none does.
cudaError_t try_cluster(int nt, const int32_t* topk_idx, int64_t T, int k, int E, int R_cols,
                        int kind, int capacity, int align, int32_t* expert_counts,
                        int32_t* expert_offsets, int32_t* dst_row, int32_t* rank_token_counts,
                        uint32_t* status, cudaStream_t stream) {
    for (; nt >= 256; nt /= 2) {
        if (nt != 1024 && nt != 512 && nt != 256) continue;
        const size_t smem = cluster_smem_bytes(nt, k, E, R_cols);
        if (smem > kFusedSmemLimit) continue;
#define EP_CLUSTER_CASE(N)                                                                     \
    case N:                                                                                    \
        return launch_cluster<N>(topk_idx, T, k, E, R_cols, kind, capacity, align,             \
                                 expert_counts, expert_offsets, dst_row, rank_token_counts,    \
                                 status, smem, stream);
        switch (nt) {
            EP_CLUSTER_CASE(1024)
            EP_CLUSTER_CASE(512)
            EP_CLUSTER_CASE(256)
        }
#undef EP_CLUSTER_CASE
    }
    return cudaErrorNotSupported;
}

// ---- layout fused with dispatch (few tokens) --------------------------------
// One launch for ep_layout_dispatch: every block computes the whole layout in
// shared memory with the single-block algorithm above, then each of its warps
// dispatches one (token, column slice) unit from it.  Block 0 alone stores the
// layout outputs and the status word; every block derives the same flags
// (bad ids, masked overflow, rows outside the dispatch buffer), so no block
// races another on the status.  Each warp loads its slice of x before the
// layout, so those loads overlap the layout's latency.
constexpr int kLDThreads = 256;
constexpr int kLDWarps = kLDThreads / 32;
constexpr int kLDMaxTokens = 128;  // above, the two launches measured faster (256 tokens: 8.8 vs 11.3 us)

// warp_assign_pairs for the fused kernel: slots into s_out (and g_out if
// given), conditions OR-ed into the block's flag word.
__device__ __forceinline__ void warp_assign_pairs_shared(const int32_t* s_ids, int wpairs, int E,
                                                         int kind, int capacity, int32_t* my_w,
                                                         const int32_t* s_off, int32_t* s_out,
                                                         int32_t* __restrict__ g_out, int64_t rows,
                                                         uint32_t* s_flags) {
    const int lane = threadIdx.x & 31;
    const unsigned lt = lanemask_lt();
    const int key_bits = 32 - __clz(E - 1 > 0 ? E - 1 : 1);
    for (int q0 = 0; q0 < wpairs; q0 += 32) {  // warp-uniform
        const int q = q0 + lane;
        const bool in_range = q < wpairs;
        const int e = in_range ? s_ids[q] : -1;
        const bool valid = (e >= 0) && (e < E);
        const bool bad = in_range && !valid && e != -1;
        const unsigned peers = warp_peers(valid, e, key_bits);
        bool overflow = false;
        int dst = -1;
        if (valid) {
            const int slot = my_w[e] + __popc(peers & lt);
            if (kind == EP_LAYOUT_CONTIGUOUS) {
                dst = s_off[e] + slot;
            } else if (slot < capacity) {
                dst = e * capacity + slot;
            } else {
                overflow = true;
            }
        }
        if (in_range) {
            s_out[q] = dst;
            if (g_out) g_out[q] = dst;
        }
        __syncwarp();
        if (valid && (__ffs(peers) - 1) == lane) my_w[e] += __popc(peers);
        __syncwarp();
        const unsigned f = (__ballot_sync(kFullMask, bad) ? EP_FLAG_BAD_EXPERT : 0u) |
                           (__ballot_sync(kFullMask, overflow) ? EP_FLAG_OVERFLOW : 0u) |
                           (__ballot_sync(kFullMask, (int64_t)dst >= rows) ? EP_FLAG_BAD_ROW : 0u);
        if (f && lane == 0) atomicOr(s_flags, f);
    }
}

template <bool FP8>
__global__ void __launch_bounds__(kLDThreads)
layout_dispatch_kernel(const int32_t* __restrict__ idx, int T, int k, int E, int R_cols, int kind,
                       int capacity, int tpw, const uint16_t* __restrict__ x, int64_t H, int S,
                       int64_t slice, int32_t* __restrict__ expert_counts,
                       int32_t* __restrict__ expert_offsets, int32_t* __restrict__ dst_row,
                       int32_t* __restrict__ rank_token_counts, void* __restrict__ recv,
                       float* __restrict__ recv_scale, int64_t rows, uint32_t* __restrict__ status) {
    constexpr int NT = kLDThreads;
    constexpr int NW = kLDWarps;
    constexpr int U = FP8 ? 2 : 4;  // 512-channel groups (FP8) or 16-byte vectors per pass
    extern __shared__ __align__(16) int32_t smem_i[];
    __shared__ uint32_t s_flags;
    const int ES = E | 1;
    const int npairs = T * k;
    const int npad = NW * tpw * k;              // >= npairs
    int32_t* s_dst = smem_i;                    // [npad] slots of all pairs
    BlockLayoutSmem sm;
    sm.idx = s_dst + npad;                      // [npad]
    sm.w = sm.idx + npad;                       // [NW][ES]
    sm.tot = sm.w + NW * ES;                    // [E]
    sm.off = sm.tot + E;                        // [E + 1]
    sm.rank = sm.off + E + 1;                   // [R_cols]
    sm.rank_of = sm.rank + R_cols;              // [E]
    sm.warp = sm.rank_of + E;                   // [NW]
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const bool lead = blockIdx.x == 0;

    pdl_wait();
    pdl_trigger();

    // this warp's unit: token t, columns [cb, ce) in units of 8 channels
    // (BF16 vectors) or 16 channels (FP8 lane groups)
    const int64_t unit = (int64_t)blockIdx.x * NW + warp;
    const int64_t t = slice_row(unit, S);
    const bool has_unit = t < T;  // warp-uniform
    const int64_t nunits = FP8 ? H / 16 : H / 8;
    const int64_t cb = has_unit ? (unit - t * S) * slice : 0;
    const int64_t ce = has_unit ? (cb + slice < nunits ? cb + slice : nunits) : 0;
    const uint16_t* src = x + (has_unit ? t : 0) * H;
    uint4 pa[U], pb[U];  // the first pass of this unit, loaded before the layout
#pragma unroll
    for (int u = 0; u < U; ++u) {
        const int64_t c = cb + u * 32 + lane;  // unit index
        pa[u] = make_uint4(0, 0, 0, 0);
        pb[u] = make_uint4(0, 0, 0, 0);
        if (c < ce) {
            if (FP8) {
                pa[u] = ld_stream_v4(src + c * 16);
                pb[u] = ld_stream_v4(src + c * 16 + 8);
            } else {
                pa[u] = ld_stream_v4(src + c * 8);
            }
        }
    }

    // ---- the layout, as layout_fused_kernel, into shared memory
    if (threadIdx.x == 0) s_flags = 0u;
    block_layout_scan<NT>(idx, T, k, E, R_cols, 1, tpw, sm, lead ? expert_counts : nullptr,
                          lead ? expert_offsets : nullptr, lead ? rank_token_counts : nullptr);
    const int wp0 = warp * tpw * k;
    const int wrem = npairs - wp0;
    const int wpairs = wrem <= 0 ? 0 : (wrem < tpw * k ? wrem : tpw * k);
    warp_assign_pairs_shared(sm.idx + wp0, wpairs, E, kind, capacity, sm.w + warp * ES, sm.off,
                             s_dst + wp0, lead ? dst_row + wp0 : nullptr, rows, &s_flags);
    __syncthreads();  // s_dst and s_flags complete
    if (lead && threadIdx.x == 0 && status) *status = s_flags;
    if (!has_unit) return;

    // ---- dispatch of this warp's unit from the shared layout
    int my_row = -1;
    if (lane < k) {
        const int d = s_dst[t * k + lane];
        my_row = (d >= 0 && (int64_t)d < rows) ? d : -1;  // out-of-range rows were flagged
    }
    for (int j0 = 0; j0 < k; j0 += 8) {
        int rr[8];
#pragma unroll
        for (int jj = 0; jj < 8; ++jj) {
            const int r = __shfl_sync(kFullMask, my_row, (j0 + jj) & 31);
            rr[jj] = (j0 + jj < k) ? r : -1;
        }
        for (int64_t c0 = cb; c0 < ce; c0 += 32 * U) {
            uint4 a[U], b[U];
            if (j0 == 0 && c0 == cb) {  // warp-uniform: the loads issued before the layout
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    a[u] = pa[u];
                    b[u] = pb[u];
                }
            } else {
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t c = c0 + u * 32 + lane;
                    a[u] = make_uint4(0, 0, 0, 0);
                    b[u] = make_uint4(0, 0, 0, 0);
                    if (c < ce) {
                        if (FP8) {
                            a[u] = ld_stream_v4(src + c * 16);
                            b[u] = ld_stream_v4(src + c * 16 + 8);
                        } else {
                            a[u] = ld_stream_v4(src + c * 8);
                        }
                    }
                }
            }
#pragma unroll
            for (int u = 0; u < U; ++u) {
                const int64_t c = c0 + u * 32 + lane;
                const bool act = c < ce;  // FP8: all 8 lanes of a 128-channel block agree
                if (FP8) {
                    const Fp8Group g = quantize16(a[u], b[u]);
                    uint8_t* q = static_cast<uint8_t*>(recv);
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        if (rr[jj] < 0) continue;  // warp-uniform
                        if (act) st_v4(q + (int64_t)rr[jj] * H + c * 16, g.q);
                        if (act && (lane & 7) == 0)
                            recv_scale[(int64_t)rr[jj] * (H / 128) + (c >> 3)] = g.sf;
                    }
                } else {
                    uint4* v = static_cast<uint4*>(recv);
#pragma unroll
                    for (int jj = 0; jj < 8; ++jj) {
                        if (rr[jj] < 0) continue;  // warp-uniform
                        if (act) st_cs_v4(v + (int64_t)rr[jj] * (H / 8) + c, a[u]);
                    }
                }
            }
        }
    }
}

size_t layout_dispatch_smem_bytes(int tpw, int k, int E, int R_cols) {
    return ((size_t)2 * kLDWarps * tpw * k + (size_t)kLDWarps * (E | 1) + 3 * (size_t)E + 1 +
            R_cols + kLDWarps) * sizeof(int32_t);
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
    if (T <= kFusedMaxTokens) {
        const cudaError_t err =
            try_fused(T <= 128 ? EP_FUSED_NT_SMALL : EP_FUSED_NT_LARGE, topk_idx, T, k, E, R_cols,
                      kind, capacity, align, expert_counts, expert_offsets, dst_row,
                      rank_token_counts, status, stream);
        if (err != cudaErrorNotSupported) return err;
    }
    if (T <= kClusterMaxTokens) {
        const cudaError_t err =
            try_cluster(EP_CLUSTER_NT, topk_idx, T, k, E, R_cols, kind, capacity, align,
                        expert_counts, expert_offsets, dst_row, rank_token_counts, status, stream);
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

cudaError_t launch_layout_dispatch(const int32_t* topk_idx, int64_t T, int k, int E, int R,
                                   int kind, int capacity, const void* x, int64_t H, bool fp8,
                                   int32_t* expert_counts, int32_t* expert_offsets,
                                   int32_t* dst_row, int32_t* rank_token_counts, void* recv,
                                   float* recv_scale, int64_t rows, uint32_t* status,
                                   cudaStream_t stream) {
    if (T < 1 || T > kLDMaxTokens) return cudaErrorNotSupported;
    const int R_cols = rank_token_counts ? R : 0;
    const int tpw = (int)((T + kLDWarps - 1) / kLDWarps);
    const size_t smem = layout_dispatch_smem_bytes(tpw, k, E, R_cols);
    if (smem > kFusedSmemLimit) return cudaErrorNotSupported;
    const RowSlices sl = row_slices(T, fp8 ? H / 16 : H / 8);
    const unsigned grid = (unsigned)((T * sl.S + kLDWarps - 1) / kLDWarps);
    static std::atomic<uint64_t> configured_bf16{0}, configured_fp8{0};
    cudaError_t err =
        fp8 ? raise_smem_limit(layout_dispatch_kernel<true>, kFusedSmemLimit, configured_fp8)
            : raise_smem_limit(layout_dispatch_kernel<false>, kFusedSmemLimit, configured_bf16);
    if (err != cudaSuccess) return err;
    return launch_pdl(fp8 ? layout_dispatch_kernel<true> : layout_dispatch_kernel<false>,
                      dim3(grid), dim3(kLDThreads), smem, stream, topk_idx, (int)T, k, E, R_cols,
                      kind, capacity, tpw, static_cast<const uint16_t*>(x), H, sl.S, sl.slice,
                      expert_counts, expert_offsets, dst_row, rank_token_counts, recv, recv_scale,
                      rows, status);
}

}  // namespace ep
