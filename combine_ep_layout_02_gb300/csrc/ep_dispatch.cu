// ep_dispatch.cu -- BF16 dispatch: scatter of token rows into the
// per-expert buffer (bit copy).  The FP8 variant is in ep_dispatch_fp8.cu.
//
// One warp per token (per column slice of the token when there are few
// tokens).  The warp reads its part of the row once in 16-byte vectors
// (streaming, no L1 allocation) and writes it to each of the k destination
// rows, so every input byte is read once and every output byte written once:
// the HBM floor is T*H*2 read + T*k*H*2 written.  Large batches run at most
// one 8-warp block per SM, where this write-bound scatter is fastest.
#include "ep_internal.cuh"

#ifndef EP_DISPATCH_U
#define EP_DISPATCH_U 4  // 16-byte vectors per lane in flight per row pass
#endif
#ifndef EP_DISPATCH_PREFETCH_MIN_TOKENS
#define EP_DISPATCH_PREFETCH_MIN_TOKENS 16384  // batches this large use PREFETCH
#endif
#ifndef EP_DISPATCH_PERSISTENT
#define EP_DISPATCH_PERSISTENT 0  // 1: large batches on a grid of one block per SM (slower)
#endif
#ifndef EP_DISPATCH_SLICE_WARPS_PER_SM
// Column slices (see row_slices) down to 64 vectors (1 KB) while the grid has
// fewer than this many warps per SM, on top of the default rule (down to 32
// vectors below 8 warps per SM), whichever gives more slices.  Measured at
// H = 2048 (L2 flushed): 2,048 tokens 16.4 -> 14.5 us (4 slices), 4,096
// tokens 26.7 -> 24.7 us (2 slices), 2,048 x 7168 45.7 -> 44.1 us; 1,024
// tokens and below unchanged.  Slices of 32 vectors up to this grid size were
// slower at 1,024 tokens (11.3 us against 10.5), and 64-vector slices at 128
// tokens (6.6 us against 6.2).
#define EP_DISPATCH_SLICE_WARPS_PER_SM 48
#endif
#ifndef EP_DISPATCH_MIN_SLICE
#define EP_DISPATCH_MIN_SLICE 64  // 16-byte vectors
#endif
#ifndef EP_DISPATCH_STORE_CS
#define EP_DISPATCH_STORE_CS 1  // evict-first stores for the dispatched rows (0: default policy)
#endif

namespace ep {
namespace {

#ifndef EP_DISPATCH_WARPS
#define EP_DISPATCH_WARPS 8
#endif
constexpr int kDispatchWarps = EP_DISPATCH_WARPS;  // warps per block
constexpr int kRowRegs = 8;        // destination rows held in registers per pass

// Units are (token, column slice) pairs, unit g = t * S + slice; warp w of
// the grid takes units w, w + W, w + 2W, ... (W = warps in the grid), so the
// same kernel serves a grid that covers every unit once and a persistent grid
// of one block per SM.
//
// PREFETCH: a unit's first-pass loads are issued before its destination rows
// are read, so the two latencies overlap (88 registers instead of 58).  Used
// with the persistent launch for large batches (65,536 tokens x 7168: 1275 ->
// 1257 us at 2 blocks per SM, 1245 us at one); 1-2 % slower at 1,024 to 2,048
// tokens and no faster below, so smaller batches use the plain instance.  The
// same change in the FP8 dispatch measured 0.15 % slower.
//
// EARLY: the first unit's first-pass loads are also issued before the wait on
// the preceding kernel in the stream.  That is correct only when the
// preceding kernel does not write x: ep_layout_dispatch launches this kernel
// right behind its own layout kernel, which lets it start only after having
// waited for all earlier work itself, so x is final by then.  The loads then
// overlap the layout.
template <int U, bool PREFETCH, bool EARLY>
__global__ void __launch_bounds__(kDispatchWarps * 32)
dispatch_bf16_kernel(const uint4* __restrict__ x, int64_t T, int64_t nvec, int k, int S,
                     int64_t slice, const int32_t* __restrict__ dst_row, uint4* __restrict__ recv,
                     int64_t rows, uint32_t* __restrict__ status) {
    const int lane = threadIdx.x & 31;
    const int64_t nunits = T * S;
    const int64_t stride = (int64_t)gridDim.x * kDispatchWarps;
    const int64_t g0 = (int64_t)blockIdx.x * kDispatchWarps + (threadIdx.x >> 5);
    // the first pass's loads of unit g do not depend on the destination rows
    uint4 first[U];
    auto load_first = [&](int64_t g) {
        const int64_t t = slice_row(g, S);
        const int64_t vb = (g - t * S) * slice;
        const int64_t ve = vb + slice < nvec ? vb + slice : nvec;
#pragma unroll
        for (int u = 0; u < U; ++u) {
            const int64_t v = vb + u * 32 + lane;
            if (v < ve) first[u] = ld_stream_v4(x + t * nvec + v);
        }
    };
    if (EARLY && g0 < nunits) load_first(g0);
    pdl_wait();
    pdl_trigger();
    for (int64_t g = g0; g < nunits; g += stride) {  // warp-uniform
        const int64_t t = slice_row(g, S);
        const int64_t vb = (g - t * S) * slice;  // this warp's column slice [vb, ve)
        const int64_t ve = vb + slice < nvec ? vb + slice : nvec;
        const uint4* src = x + t * nvec;
        // issue the first pass's loads before the rows are read, so the two
        // latencies overlap
        const bool early = EARLY && g == g0;  // warp-uniform
        if (PREFETCH && !early) load_first(g);
        const bool have_first = PREFETCH || early;
        const int my_row = load_dst_row(dst_row, t, k, rows, status);
        // k <= 8 is one pass; larger k re-reads the slice once per 8 destinations
        for (int j0 = 0; j0 < k; j0 += kRowRegs) {
            uint4* dst[kRowRegs];
#pragma unroll
            for (int jj = 0; jj < kRowRegs; ++jj) {
                const int r = __shfl_sync(kFullMask, my_row, (j0 + jj) & 31);
                dst[jj] = (j0 + jj < k && r >= 0) ? recv + (int64_t)r * nvec : nullptr;
            }
            for (int64_t v0 = vb; v0 < ve; v0 += 32 * U) {
                uint4 buf[U];
                const bool pre = have_first && j0 == 0 && v0 == vb;  // warp-uniform
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t v = v0 + u * 32 + lane;
                    if (pre) buf[u] = first[u];
                    else if (v < ve) buf[u] = ld_stream_v4(src + v);
                }
#pragma unroll
                for (int jj = 0; jj < kRowRegs; ++jj) {
                    if (dst[jj] == nullptr) continue;  // warp-uniform
#pragma unroll
                    for (int u = 0; u < U; ++u) {
                        const int64_t v = v0 + u * 32 + lane;
                        if (v < ve) {
                            if (EP_DISPATCH_STORE_CS) st_cs_v4(dst[jj] + v, buf[u]);
                            else st_v4(dst[jj] + v, buf[u]);
                        }
                    }
                }
            }
        }
    }
}

// Dynamic shared memory that admits one block per SM: just over half of an
// SM's shared memory (0, no request, if the device reports too little).  The
// kernel does not use it; the request only limits residency.
size_t dispatch_occupancy_smem() {
    static std::atomic<int> per_sm_cache[64], per_block_cache[64];
    const int per_sm =
        cached_device_attribute(cudaDevAttrMaxSharedMemoryPerMultiprocessor, per_sm_cache);
    const int per_block =
        cached_device_attribute(cudaDevAttrMaxSharedMemoryPerBlockOptin, per_block_cache);
    const int v = per_sm / 2 + 1024;
    return (per_sm > 0 && v <= per_block) ? (size_t)v : 0;
}

}  // namespace

cudaError_t launch_dispatch_bf16(const void* x, int64_t T, int64_t H, int k,
                                 const int32_t* dst_row, void* recv, int64_t rows,
                                 uint32_t* status, cudaStream_t stream, bool early) {
    if (T == 0) return cudaSuccess;
    const int64_t nvec = H / 8;
    // few tokens: slices down to 32 vectors while the grid is small; more
    // tokens: slices down to EP_DISPATCH_MIN_SLICE vectors up to a larger grid
    RowSlices sl = row_slices(T, nvec);
    const RowSlices wide =
        row_slices(T, nvec, EP_DISPATCH_SLICE_WARPS_PER_SM, EP_DISPATCH_MIN_SLICE);
    if (wide.S > sl.S) sl = wide;
    const unsigned grid = (unsigned)((T * sl.S + kDispatchWarps - 1) / kDispatchWarps);
    if (T < EP_DISPATCH_PREFETCH_MIN_TOKENS)
        return launch_pdl(early ? dispatch_bf16_kernel<EP_DISPATCH_U, false, true>
                                : dispatch_bf16_kernel<EP_DISPATCH_U, false, false>,
                          dim3(grid),
                          dim3(kDispatchWarps * 32), 0, stream, static_cast<const uint4*>(x), T,
                          nvec, k, sl.S, sl.slice, dst_row, static_cast<uint4*>(recv), rows,
                          status);
    // Large batches: at most one 8-warp block resident per SM.  A write-bound
    // scatter into k rows per token measured fastest with 8 warps per SM
    // (65,536 x 7168: 1257 us at 16 warps, 1245 us at 8, 1403 us at 4).  The
    // residency limit is set by the block's dynamic shared-memory request
    // (more than half of an SM's shared memory, which the kernel does not
    // use).  A persistent grid of one block per SM looping over the tokens
    // (EP_DISPATCH_PERSISTENT=1) measured slower: 1408 us against 1263 us
    // with the same residency limit, 1422 us without it.
    auto kern = early ? dispatch_bf16_kernel<EP_DISPATCH_U, true, true>
                      : dispatch_bf16_kernel<EP_DISPATCH_U, true, false>;
    unsigned pgrid = grid;
#if EP_DISPATCH_PERSISTENT
    {
        static std::atomic<int> sm_cache[64];
        const int sms = cached_device_attribute(cudaDevAttrMultiProcessorCount, sm_cache);
        if (sms > 0 && (unsigned)sms < grid) pgrid = (unsigned)sms;
    }
#endif
    const size_t smem = dispatch_occupancy_smem();
    if (smem > 0) {
        static std::atomic<uint64_t> configured[2];
        const cudaError_t e = raise_smem_limit(kern, smem, configured[early ? 1 : 0]);
        if (e != cudaSuccess) return e;
    }
    return launch_pdl(kern, dim3(pgrid), dim3(kDispatchWarps * 32), smem, stream,
                      static_cast<const uint4*>(x), T, nvec, k, sl.S, sl.slice, dst_row,
                      static_cast<uint4*>(recv), rows, status);
}

}  // namespace ep
