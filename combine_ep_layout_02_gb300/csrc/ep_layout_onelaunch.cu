// ep_layout_onelaunch.cu -- the routing layout (per-expert counts, exclusive
// scan, stable slots) in ONE kernel launch for small and medium batches, and
// the layout fused with dispatch for the smallest ones.  The layout is the
// "dispatch layout" that the Prefill-like profile of awsome-distributed-ai
// PR #1238 times inside its boundary; the Decode-like profile runs 128 tokens
// per rank, where the layout's latency, not its bytes, is the cost.
//
// Both kernels split the pairs (t, j) into pieces of P = floor(32 / k) whole
// tokens, one pair per lane (lane l: token l / k of the piece, j = l % k), and
// give each warp a contiguous run of pieces.  Per piece a warp ranks equal
// experts with popc(peers & lanemask_lt), the peers coming from one ballot
// per bit of the expert id (independent ballots: eight up to 256 experts, ten
// up to 1,024; the peers of the expert's virtual rank are the same ballots
// above the rank's shift), and keeps a running per-warp count of each expert in its
// own shared-memory row -- no block barrier until every warp has counted.
// (match.any gives the peers in one instruction but runs on a shared per-SM
// unit: 2,048 tokens 6.9 -> 7.8 us.)  The ids and slots of a lane's pieces
// live in shared memory: the piece loop is not unrolled (one copy of its code
// in the instruction cache), and a register array indexed by the loop counter
// would sit in local memory, whose stores every later warp and cluster
// barrier waits for.  Then:
//   single block (layout_block_kernel): one thread per expert turns the warps'
//     counts into their exclusive prefix over warps and the expert's total;
//     each warp scans its 32 experts' (padded) totals; after the second
//     barrier every warp scans the <= 32 range sums with shuffles and each
//     lane forms its pairs' rows.  Two block barriers in all.
//   cluster (layout_cluster_kernel, 8 or 16 blocks): the same per block, with the
//     block totals pushed into every block's shared memory (st.async,
//     completed on the receiving block's mbarrier) instead of read remotely.
// The status word is written once, by one thread: bad ids are collected per
// warp and the masked overflow is read off the expert totals.  The slot of a
// pair is the number of earlier pairs (flattened t*k + j) with the same
// expert, as in the chunked kernels of ep_layout.cu.
#include <cooperative_groups.h>

#include "ep_internal.cuh"
#include "ep_layout_onelaunch.cuh"

namespace ep {
namespace {

namespace cg = cooperative_groups;

// Pieces per warp at most (ids and slots in shared memory, ppw * 32 * 8
// bytes per warp): 8 in 1024-thread blocks, 16 in smaller ones.
template <int NT>
__host__ __device__ constexpr int max_pieces() { return NT >= 1024 ? 8 : 16; }
constexpr int kClusterMaxTokens = 2048;
constexpr size_t kSmemLimit = 160 * 1024;
// Bits of an expert id: one ballot each.
constexpr int kKeyBits = 10;
static_assert((1 << kKeyBits) >= EP_MAX_EXPERTS, "one ballot per expert-id bit");

// The virtual rank of expert e: e / (E / R), a shift when E / R is a power of two.
struct RankOf {
    int shift;  // >= 0: e >> shift
    int div;
    __device__ __forceinline__ int operator()(int e) const {
        return shift >= 0 ? (e >> shift) : e / div;
    }
};

RankOf make_rank_of(int E, int R) {
    const int per = E / R;
    RankOf r{-1, per};
    if ((per & (per - 1)) == 0) {
        int s = 0;
        while ((1 << s) < per) ++s;
        r.shift = s;
    }
    return r;
}

// Peers of this lane: the lanes with valid set whose key has the same bits
// [lo, B) as this lane's (0 for a lane without valid).  m[b] is the ballot of
// key bit b; keys of valid lanes are below 2^B.
template <int B>
__device__ __forceinline__ unsigned peers_from_bits(unsigned vmask, const unsigned (&m)[B],
                                                    int key, int lo, bool valid) {
    unsigned p = vmask;
#pragma unroll
    for (int b = 0; b < B; ++b) {
        const unsigned sel = ((key >> b) & 1) ? m[b] : ~m[b];
        p &= b >= lo ? sel : kFullMask;
    }
    return valid ? p : 0u;
}

template <int B>
__device__ __forceinline__ void key_ballots(int key, unsigned (&m)[B]) {
#pragma unroll
    for (int b = 0; b < B; ++b) m[b] = __ballot_sync(kFullMask, (key >> b) & 1);
}

// Shared-memory arrays of the one-launch layouts (carved by the kernels).
struct OneLaunchSmem {
    int32_t* cnt;        // [NW][E]  per-warp expert counts, then their exclusive prefix over warps
    int32_t* rc;         // [NW][R_cols]  per-warp tokens per virtual rank
    int32_t* off_local;  // [E]  exclusive scan of the padded totals within each 32-expert range
    int32_t* range_sum;  // [32] sum of the padded totals of each 32-expert range
    uint32_t* wflags;    // [NW] condition flags each warp found among its ids
    int32_t* pe;         // [NW][ppw][32]  expert id of each lane's pair in each piece (-1: none)
    int32_t* plr;        // [NW][ppw][32]  that pair's slot among its warp's pairs of the expert
    int32_t* btot;       // [E + R_cols + 1]  block totals and the block's flags, read by
                         // the other blocks (cluster)
    int32_t* base;       // [E]  pairs of expert e in the cluster's earlier blocks (cluster)
    int32_t* ctot;       // [E + R_cols]  cluster totals, stored by block 0 (cluster)
};

// Zero this warp's rows of expert and rank counts.  Shared memory only, so
// the kernels do it before waiting for the previous grid.
__device__ __forceinline__ void zero_warp_rows(const OneLaunchSmem& sm, int E, int R_cols) {
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    for (int i = lane; i < E; i += 32) sm.cnt[warp * E + i] = 0;
    for (int i = lane; i < R_cols; i += 32) sm.rc[warp * R_cols + i] = 0;
    __syncwarp();
}

// The piece loop of phase 1 for ids below 2^B (B ballots per piece).
template <bool RANKS, int B>
__device__ __forceinline__ void count_pieces(const int32_t* my_e, int np, int E, RankOf rank_of,
                                             unsigned grp, unsigned lt, int32_t* my_cnt,
                                             int32_t* my_rc, int32_t* my_lr, uint32_t& flags) {
    const int lane = threadIdx.x & 31;
#pragma unroll 1
    for (int q = 0; q < np; ++q) {  // warp-uniform
        const int e = my_e[q * 32 + lane];
        const bool valid = e >= 0 && e < E;
        if (e < -1 || e >= E) flags |= EP_FLAG_BAD_EXPERT;
        unsigned m[B];
        key_ballots<B>(e, m);
        const unsigned vmask = __ballot_sync(kFullMask, valid);
        const unsigned peers = peers_from_bits<B>(vmask, m, e, 0, valid);
        int c = 0;
        if (valid) {
            c = my_cnt[e];
            my_lr[q * 32 + lane] = c + __popc(peers & lt);
        }
        int r = 0;
        unsigned rpeers = 0;
        if (RANKS) {
            r = valid ? rank_of(e) : 0;
            if (rank_of.shift >= 0) {  // warp-uniform: the rank is the id's upper bits
                rpeers = peers_from_bits<B>(vmask, m, e, rank_of.shift, valid);
            } else {
                unsigned mr[B];
                key_ballots<B>(r, mr);
                rpeers = peers_from_bits<B>(vmask, mr, r, 0, valid);
            }
            rpeers &= grp;  // same token, same rank
        }
        __syncwarp();
        if (valid && (__ffs(peers) - 1) == lane) my_cnt[e] = c + __popc(peers);
        if (RANKS && valid && (rpeers & lt) == 0) atomicAdd(&my_rc[r], 1);  // first of the token
        __syncwarp();
    }
}

// Phase 1 (per warp, no block barrier): load the warp's ids into my_e, count
// them into the warp's row `my_cnt` (and tokens per rank into `my_rc`) and
// store in my_lr each pair's slot among the warp's earlier pairs with the
// same expert.  my_e / my_lr hold piece q's lane l at [q * 32 + l]; the
// count rows start zeroed (zero_warp_rows).
template <bool RANKS, int MAXP>
__device__ __forceinline__ void warp_count_pieces(const int32_t* __restrict__ idx, int T, int k,
                                                  int E, int R_cols, int P, int p0, int np,
                                                  RankOf rank_of, int32_t* my_cnt,
                                                  int32_t* my_rc, int32_t* my_e, int32_t* my_lr,
                                                  uint32_t& flags) {
    const int lane = threadIdx.x & 31;
    const int tl = lane / k;
    const int jl = lane - tl * k;
    const bool used = lane < P * k;
    const unsigned lt = lanemask_lt();
    // the lanes of this lane's token (for counting each rank once per token)
    const unsigned grp = !used ? 0u : (k >= 32 ? kFullMask : ((1u << k) - 1u) << (tl * k));
    {
        int ids[MAXP];  // all loads issued before the first store
#pragma unroll
        for (int q = 0; q < MAXP; ++q) {
            const int t = (p0 + q) * P + tl;
            ids[q] = (q < np && used && t < T) ? __ldg(idx + (int64_t)t * k + jl) : -1;
        }
#pragma unroll
        for (int q = 0; q < MAXP; ++q)
            if (q < np) my_e[q * 32 + lane] = ids[q];
    }
    if (E <= 256)  // warp-uniform: ids of up to 8 bits need 8 ballots, not 10
        count_pieces<RANKS, 8>(my_e, np, E, rank_of, grp, lt, my_cnt, my_rc, my_lr, flags);
    else
        count_pieces<RANKS, kKeyBits>(my_e, np, E, rank_of, grp, lt, my_cnt, my_rc, my_lr, flags);
}

// Inclusive warp scan.
__device__ __forceinline__ int warp_incl_scan(int v) {
    const int lane = threadIdx.x & 31;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
        const int nb = __shfl_up_sync(kFullMask, v, o);
        if (lane >= o) v += nb;
    }
    return v;
}

// Padded segment length of an expert with `c` pairs.
__device__ __forceinline__ int padded(int c, int align) {
    return align > 1 ? (c + align - 1) / align * align : c;
}

// Phase 2, part of one thread per expert e (< E): the warps' counts of e
// become their exclusive prefix over the warps; returns the total.
template <int NW>
__device__ __forceinline__ int expert_prefix_over_warps(int32_t* cnt, int E, int e) {
    constexpr int G = NW < 16 ? NW : 16;  // loads issued together
    int run = 0;
#pragma unroll
    for (int w0 = 0; w0 < NW; w0 += G) {
        int v[G];
#pragma unroll
        for (int i = 0; i < G; ++i) v[i] = cnt[(w0 + i) * E + e];
#pragma unroll
        for (int i = 0; i < G; ++i) {
            cnt[(w0 + i) * E + e] = run;
            run += v[i];
        }
    }
    return run;
}

// Phase 2, the range scan: the (padded) totals tt of the 32 experts
// [e0w, e0w + 32) held by this warp's lanes are scanned into off_local, and
// the range's sum is stored.  Warp-uniform call.
__device__ __forceinline__ void range_scan(int tt, int e, int E, OneLaunchSmem& sm) {
    const int incl = warp_incl_scan(tt);
    if (e < E) sm.off_local[e] = incl - tt;
    if ((threadIdx.x & 31) == 31) sm.range_sum[e >> 5] = incl;
}

// Phase 3 helper: every warp scans the range sums; lane r gets the first row
// of range r, and the call returns the rows used in all.
__device__ __forceinline__ int range_bases(const OneLaunchSmem& sm, int E, int& rp) {
    const int lane = threadIdx.x & 31;
    const int nr = (E + 31) >> 5;
    const int rs = lane < nr ? sm.range_sum[lane] : 0;
    const int incl = warp_incl_scan(rs);
    rp = incl - rs;
    return __shfl_sync(kFullMask, incl, 31);
}

// Phase 3: the rows of this lane's pairs.  base_e(e) adds the pairs of e in
// earlier blocks (cluster) to the warp's prefix.  Rows go to g_dst (global,
// if given) and s_dst (shared, if given); a row at or past `rows` raises
// EP_FLAG_BAD_ROW in `flags`.
template <typename BaseFn>
__device__ __forceinline__ void assign_pieces(const int32_t* my_e, const int32_t* my_lr, int k,
                                              int E, int kind, int capacity, int P, int p0,
                                              int np, int t_end, const OneLaunchSmem& sm,
                                              const int32_t* my_cnt, int rp, int64_t rows,
                                              BaseFn base_e, int32_t* __restrict__ g_dst,
                                              int32_t* s_dst, uint32_t& flags) {
    const int lane = threadIdx.x & 31;
    const int tl = lane / k;
    const int jl = lane - tl * k;
    const bool used = lane < P * k;
#pragma unroll 1
    for (int q = 0; q < np; ++q) {  // warp-uniform
        const int e = my_e[q * 32 + lane];
        const bool valid = e >= 0 && e < E;
        const int rbase = __shfl_sync(kFullMask, rp, valid ? (e >> 5) : 0);
        const int t = (p0 + q) * P + tl;
        int dst = -1;
        if (valid) {
            const int slot = base_e(e) + my_cnt[e] + my_lr[q * 32 + lane];
            if (kind == EP_LAYOUT_CONTIGUOUS) dst = rbase + sm.off_local[e] + slot;
            else if (slot < capacity) dst = e * capacity + slot;  // else overflow: -1
            if ((int64_t)dst >= rows) flags |= EP_FLAG_BAD_ROW;
        }
        if (used && t < t_end) {
            const int p = t * k + jl;
            if (g_dst) g_dst[p] = dst;
            if (s_dst) s_dst[p] = dst;
        }
    }
}

struct NoBase {
    __device__ __forceinline__ int operator()(int) const { return 0; }
};

// The whole layout of T tokens by one block of NT threads; pieces of P
// tokens, `ppw` per warp.  Outputs that are null are not written.  Returns
// the layout's condition flags (bad ids, masked overflow: an expert's count
// above the capacity), the same in every thread; `row_flags` gets this
// lane's EP_FLAG_BAD_ROW (a row at or past `rows`).  Two block barriers.
// The warps' count rows must be zeroed first (zero_warp_rows).
template <int NT, bool RANKS>
__device__ __forceinline__ uint32_t block_layout(const int32_t* __restrict__ idx, int T, int k,
                                                 int E, int R_cols, int kind, int capacity,
                                                 int align, int P, int ppw, RankOf rank_of,
                                                 const OneLaunchSmem& sm_in,
                                                 int32_t* __restrict__ expert_counts,
                                                 int32_t* __restrict__ expert_offsets,
                                                 int32_t* __restrict__ rank_token_counts,
                                                 int32_t* __restrict__ g_dst, int32_t* s_dst,
                                                 int64_t rows, uint32_t& row_flags) {
    constexpr int NW = NT / 32;
    OneLaunchSmem sm = sm_in;
    const int warp = threadIdx.x >> 5;
    const int lane = threadIdx.x & 31;
    const int npieces = (T + P - 1) / P;
    const int p0 = warp * ppw;
    const int np = p0 >= npieces ? 0 : (npieces - p0 < ppw ? npieces - p0 : ppw);
    int32_t* my_cnt = sm.cnt + warp * E;
    int32_t* my_e = sm.pe + warp * ppw * 32;
    int32_t* my_lr = sm.plr + warp * ppw * 32;
    uint32_t flags = 0;
    warp_count_pieces<RANKS, max_pieces<NT>()>(idx, T, k, E, R_cols, P, p0, np, rank_of, my_cnt,
                                               sm.rc + warp * R_cols, my_e, my_lr, flags);
    {
        const unsigned wf = __reduce_or_sync(kFullMask, flags);
        if (lane == 0) sm.wflags[warp] = wf;
    }
    __syncthreads();
    // one thread per expert: prefix over warps, totals, 32-expert range scans
    int ovf = 0;
    for (int e0 = 0; e0 < E; e0 += NT) {  // block-uniform
        const int e = e0 + threadIdx.x;
        int tt = 0;
        if (e < E) {
            const int c = expert_prefix_over_warps<NW>(sm.cnt, E, e);
            if (expert_counts) expert_counts[e] = c;
            if (kind == EP_LAYOUT_MASKED && c > capacity) ovf = 1;
            tt = padded(c, align);
        }
        if (e0 + (threadIdx.x & ~31) < E) range_scan(tt, e, E, sm);  // warp-uniform
    }
    if (RANKS) {
        // tokens per rank: the threads after the experts' warps (or all, if none are left)
        const int first = ((E + 31) & ~31) + R_cols <= NT ? ((E + 31) & ~31) : 0;
        for (int r = (int)threadIdx.x - first; r >= 0 && r < R_cols; r += NT) {
            int s = 0;
#pragma unroll
            for (int w = 0; w < NW; ++w) s += sm.rc[w * R_cols + r];
            if (rank_token_counts) rank_token_counts[r] = s;
        }
    }
    uint32_t lflags = __syncthreads_or(ovf) ? EP_FLAG_OVERFLOW : 0u;
#pragma unroll
    for (int w = 0; w < NW; ++w) lflags |= sm.wflags[w];
    int rp;
    const int total = range_bases(sm, E, rp);
    if (expert_offsets) {
        for (int e0 = 0; e0 < E; e0 += NT) {  // block-uniform
            const int e = e0 + threadIdx.x;
            const int rb = __shfl_sync(kFullMask, rp, ((e0 + (threadIdx.x & ~31)) >> 5) & 31);
            if (e < E) expert_offsets[e] = rb + sm.off_local[e];
        }
        if (threadIdx.x == 0) expert_offsets[E] = total;
    }
    assign_pieces(my_e, my_lr, k, E, kind, capacity, P, p0, np, T, sm, my_cnt, rp, rows,
                  NoBase(), g_dst, s_dst, row_flags);
    return lflags;
}

// Ints of the single-block arrays before the piece state, rounded to 16 bytes.
__host__ __device__ __forceinline__ int block_head_ints(int NW, int E, int R_cols) {
    return (NW * (E + R_cols) + E + 32 + NW + 3) & ~3;
}

// Carve the single-block arrays out of dynamic shared memory.
__device__ __forceinline__ OneLaunchSmem carve_block(int32_t* p, int NW, int E, int R_cols,
                                                     int ppw) {
    OneLaunchSmem sm;
    sm.cnt = p;
    sm.rc = sm.cnt + NW * E;
    sm.off_local = sm.rc + NW * R_cols;
    sm.range_sum = sm.off_local + E;
    sm.wflags = reinterpret_cast<uint32_t*>(sm.range_sum + 32);
    sm.pe = p + block_head_ints(NW, E, R_cols);
    sm.plr = sm.pe + NW * ppw * 32;
    sm.btot = nullptr;
    sm.base = nullptr;
    sm.ctot = nullptr;
    return sm;
}

size_t block_smem_bytes(int NW, int E, int R_cols, int ppw) {
    return ((size_t)block_head_ints(NW, E, R_cols) + (size_t)2 * NW * ppw * 32) * sizeof(int32_t);
}

// Small batches: the whole layout in one block.
template <int NT, bool RANKS>
__global__ void __launch_bounds__(NT)
layout_block_kernel(const int32_t* __restrict__ idx, int T, int k, int E, int R_cols, int kind,
                    int capacity, int align, int P, int ppw, RankOf rank_of,
                    int32_t* __restrict__ expert_counts, int32_t* __restrict__ expert_offsets,
                    int32_t* __restrict__ dst_row, int32_t* __restrict__ rank_token_counts,
                    uint32_t* __restrict__ status) {
    extern __shared__ __align__(16) int32_t smem_i[];
    const OneLaunchSmem sm = carve_block(smem_i, NT / 32, E, R_cols, ppw);
    zero_warp_rows(sm, E, R_cols);
    pdl_wait();
    pdl_trigger();
    uint32_t row_flags = 0;  // no row limit here
    const uint32_t f = block_layout<NT, RANKS>(idx, T, k, E, R_cols, kind, capacity, align, P, ppw,
                                               rank_of, sm, expert_counts, expert_offsets,
                                               rank_token_counts, dst_row, nullptr,
                                               (int64_t)1 << 40, row_flags);
    if (threadIdx.x == 0 && status) *status = f;  // the one write of the status word
}

// Medium batches: ONE launch of one cluster of CB blocks (8, or 16 where the
// GPU can place a cluster that large); block b
// owns tokens [b * tpb, (b + 1) * tpb).  The blocks exchange their totals by
// pushing them: each block stores its E + R_cols + 1 totals and flags into
// slot b of every block's `recv` with st.async, whose bytes complete on the
// receiving block's mbarrier; a block reads its own recv once its mbarrier
// has seen all the bytes.  So there is one cluster barrier, arrived at right
// after the mbarriers are initialised and waited on just before the first
// push (by then every block has long arrived), and no block reads another's
// shared memory, so none has to wait for the others before exiting.
__device__ __forceinline__ uint32_t smem_addr(const void* p) {
    return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}
__device__ __forceinline__ uint32_t cluster_map(uint32_t addr, int rank) {
    uint32_t r;
    asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(addr), "r"(rank));
    return r;
}
__device__ __forceinline__ void push_v4(uint32_t remote, const int4& v, uint32_t remote_bar) {
    asm volatile(
        "st.async.shared::cluster.mbarrier::complete_tx::bytes.v4.b32 [%0], {%1, %2, %3, %4}, [%5];"
        ::"r"(remote), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w), "r"(remote_bar)
        : "memory");
}
__device__ __forceinline__ uint64_t global_ns() {
    uint64_t t;
    asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
    return t;
}
// Wait for phase 0 of the mbarrier at `bar` to complete; false if it has not
// after kPushWaitNs (and at least 2^16 polls, so a context switch alone
// cannot end the wait).
constexpr uint64_t kPushWaitNs = 1000000000ull;
__device__ __forceinline__ bool wait_phase0(uint32_t bar) {
    const uint64_t t0 = global_ns();
    for (uint32_t polls = 0;; ++polls) {
        uint32_t done;
        asm volatile(
            "{\n\t.reg .pred p;\n\t"
            "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], 0;\n\t"
            "selp.u32 %0, 1, 0, p;\n\t}"
            : "=r"(done)
            : "r"(bar)
            : "memory");
        if (done) return true;
        if (polls >= (1u << 16) && global_ns() - t0 > kPushWaitNs) return false;
    }
}

template <int NT, bool RANKS, int CB>
__global__ void __launch_bounds__(NT)
layout_cluster_kernel(const int32_t* __restrict__ idx, int T, int k, int E, int R_cols, int kind,
                      int capacity, int align, int P, int ppw, int tpb, RankOf rank_of,
                      int32_t* __restrict__ expert_counts, int32_t* __restrict__ expert_offsets,
                      int32_t* __restrict__ dst_row, int32_t* __restrict__ rank_token_counts,
                      uint32_t* __restrict__ status) {
    constexpr int NW = NT / 32;
    extern __shared__ __align__(16) int32_t smem_i[];
    __shared__ __align__(8) uint64_t s_bar;
    cg::cluster_group cluster = cg::this_cluster();
    const int b = (int)cluster.block_rank();
    const int nb = (E + R_cols + 1 + 3) & ~3;  // pushed ints per block (16-byte multiple)
    OneLaunchSmem sm = carve_block(smem_i, NW, E, R_cols, ppw);
    sm.btot = sm.plr + NW * ppw * 32;             // [nb]  this block's totals, then its flags
    int32_t* recv = sm.btot + nb;                 // [CB][nb]  every block's btot
    sm.base = recv + CB * nb;                     // [E]
    const int warp = threadIdx.x >> 5;
    const int t0 = b * tpb;
    const int tb = T - t0 < 0 ? 0 : (T - t0 < tpb ? T - t0 : tpb);  // this block's tokens
    const int npieces = (tb + P - 1) / P;
    const int p0 = warp * ppw;
    const int np = p0 >= npieces ? 0 : (npieces - p0 < ppw ? npieces - p0 : ppw);
    const int32_t* bidx = idx + (int64_t)t0 * k;
    const uint32_t bar = smem_addr(&s_bar);
    zero_warp_rows(sm, E, R_cols);
    if (threadIdx.x == 0) {
        asm volatile("mbarrier.init.shared::cta.b64 [%0], 1;" ::"r"(bar) : "memory");
        asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
    }
    asm volatile("barrier.cluster.arrive.relaxed.aligned;" ::: "memory");

    pdl_wait();
    pdl_trigger();
    int32_t* my_cnt = sm.cnt + warp * E;
    int32_t* my_e = sm.pe + warp * ppw * 32;
    int32_t* my_lr = sm.plr + warp * ppw * 32;
    uint32_t flags = 0;
    warp_count_pieces<RANKS, max_pieces<NT>()>(bidx, tb, k, E, R_cols, P, p0, np, rank_of,
                                               my_cnt, sm.rc + warp * R_cols, my_e, my_lr, flags);
    {
        const unsigned wf = __reduce_or_sync(kFullMask, flags);
        if ((threadIdx.x & 31) == 0) sm.wflags[warp] = wf;
    }
    __syncthreads();
    // block totals (prefix over this block's warps kept in cnt), rank totals, flags
    for (int e = threadIdx.x; e < E; e += NT) sm.btot[e] = expert_prefix_over_warps<NW>(sm.cnt, E, e);
    if (RANKS)
        for (int r = threadIdx.x; r < R_cols; r += NT) {
            int s = 0;
#pragma unroll
            for (int w = 0; w < NW; ++w) s += sm.rc[w * R_cols + r];
            sm.btot[E + r] = s;
        }
    if (threadIdx.x == 0) {
        uint32_t bf = 0;
        for (int w = 0; w < NW; ++w) bf |= sm.wflags[w];
        sm.btot[E + R_cols] = (int32_t)bf;
    }
    for (int i = E + R_cols + 1 + (int)threadIdx.x; i < nb; i += NT) sm.btot[i] = 0;
    __syncthreads();
    asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory");  // every mbarrier is initialised
    if (threadIdx.x == 0)
        asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar),
                     "r"((uint32_t)(CB * nb * 4))
                     : "memory");
    {
        const uint32_t slot = smem_addr(recv + b * nb);
        for (int i = threadIdx.x; i < nb / 4; i += NT) {
            const int4 v = reinterpret_cast<const int4*>(sm.btot)[i];
#pragma unroll
            for (int q = 0; q < CB; ++q)
                push_v4(cluster_map(slot + 16u * i, q), v, cluster_map(bar, q));
        }
    }
    uint32_t cflags = 0;
    if (!__syncthreads_and(wait_phase0(bar))) {  // a block's totals never arrived: give up
        if (threadIdx.x == 0 && status) atomicOr(status, EP_FLAG_TIMEOUT);
        return;
    }
    // one thread per expert: pairs in earlier blocks and the cluster total;
    // masked overflow is a total above the capacity
    int ovf = 0;
    for (int e0 = 0; e0 < E; e0 += NT) {  // block-uniform
        const int e = e0 + threadIdx.x;
        int tt = 0;
        if (e < E) {
            int before = 0, total = 0;
#pragma unroll
            for (int q = 0; q < CB; ++q) {
                const int v = recv[q * nb + e];
                before += q < b ? v : 0;
                total += v;
            }
            sm.base[e] = before;
            if (b == 0) expert_counts[e] = total;
            if (kind == EP_LAYOUT_MASKED && total > capacity) ovf = 1;
            tt = padded(total, align);
        }
        if (e0 + (threadIdx.x & ~31) < E) range_scan(tt, e, E, sm);  // warp-uniform
    }
    if (RANKS && b == 0 && rank_token_counts) {
        const int first = ((E + 31) & ~31) + R_cols <= NT ? ((E + 31) & ~31) : 0;
        for (int r = (int)threadIdx.x - first; r >= 0 && r < R_cols; r += NT) {
            int s = 0;
#pragma unroll
            for (int q = 0; q < CB; ++q) s += recv[q * nb + E + r];
            rank_token_counts[r] = s;
        }
    }
    if (b == 0 && threadIdx.x == 0)
        for (int q = 0; q < CB; ++q) cflags |= (uint32_t)recv[q * nb + E + R_cols];
    if (__syncthreads_or(ovf)) cflags |= EP_FLAG_OVERFLOW;
    int rp;
    const int total = range_bases(sm, E, rp);
    if (b == 0) {
        for (int e0 = 0; e0 < E; e0 += NT) {  // block-uniform
            const int e = e0 + threadIdx.x;
            const int rb = __shfl_sync(kFullMask, rp, ((e0 + (threadIdx.x & ~31)) >> 5) & 31);
            if (e < E) expert_offsets[e] = rb + sm.off_local[e];
        }
        if (threadIdx.x == 0) expert_offsets[E] = total;
    }
    const int32_t* base = sm.base;
    uint32_t row_flags = 0;  // no row limit here
    assign_pieces(my_e, my_lr, k, E, kind, capacity, P, p0, np, tb, sm, my_cnt, rp,
                  (int64_t)1 << 40, [base](int e) { return base[e]; }, dst_row + (int64_t)t0 * k,
                  nullptr, row_flags);
    if (b == 0 && threadIdx.x == 0 && status) *status = cflags;  // the one write of the status word
}

size_t cluster_smem_bytes(int NW, int E, int R_cols, int ppw, int CB) {
    const size_t nb = (size_t)((E + R_cols + 1 + 3) & ~3);
    return block_smem_bytes(NW, E, R_cols, ppw) + ((1 + CB) * nb + (size_t)E) * sizeof(int32_t);
}

// Pieces per warp for `tokens` tokens over NW warps (pieces of P = 32/k tokens).
int pieces_per_warp(int64_t tokens, int k, int NW) {
    const int P = 32 / k;
    const int64_t npieces = (tokens + P - 1) / P;
    return (int)((npieces + NW - 1) / NW);
}

template <typename K>
cudaError_t prepare(K kernel, size_t smem, std::atomic<uint64_t>& configured) {
    return raise_smem_limit(kernel, kSmemLimit, configured);
}

template <int NT, bool RANKS>
cudaError_t launch_block_nt(const int32_t* idx, int T, int k, int E, int R_cols, int kind,
                            int capacity, int align, int ppw, RankOf rof,
                            int32_t* counts, int32_t* offsets, int32_t* dst_row, int32_t* rtc,
                            uint32_t* status, size_t smem, cudaStream_t stream) {
    static std::atomic<uint64_t> configured{0};
    cudaError_t err = prepare(layout_block_kernel<NT, RANKS>, smem, configured);
    if (err != cudaSuccess) return err;
    return launch_pdl(layout_block_kernel<NT, RANKS>, dim3(1), dim3(NT), smem, stream, idx, T, k,
                      E, R_cols, kind, capacity, align, 32 / k, ppw, rof, counts, offsets,
                      dst_row, rtc, status);
}

template <int NT, bool RANKS, int CB>
cudaError_t launch_cluster_nt(const int32_t* idx, int T, int k, int E, int R_cols, int kind,
                              int capacity, int align, int ppw, int tpb, RankOf rof,
                              int32_t* counts, int32_t* offsets, int32_t* dst_row, int32_t* rtc,
                              uint32_t* status, size_t smem, cudaStream_t stream) {
    static std::atomic<uint64_t> configured{0};
    auto kern = layout_cluster_kernel<NT, RANKS, CB>;
    cudaError_t err = prepare(kern, smem, configured);
    if (err != cudaSuccess) return err;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(CB);
    cfg.blockDim = dim3(NT);
    cfg.dynamicSmemBytes = smem;
    cfg.stream = stream;
    cudaLaunchAttribute attr[2];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = CB;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;
    attr[1].val.programmaticStreamSerializationAllowed = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 2;
    if (CB > 8) {  // above the portable cluster size: allowed per kernel, and only if the
                   // device can place such a cluster (checked once per device)
        static std::atomic<uint64_t> allowed{0}, refused{0};
        int dev = 0;
        err = cudaGetDevice(&dev);
        if (err != cudaSuccess) return err;
        const uint64_t bit = 1ull << (dev & 63);
        if (refused.load(std::memory_order_acquire) & bit) return cudaErrorNotSupported;
        if (!(allowed.load(std::memory_order_acquire) & bit)) {
            err = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
            int n = 0;
            if (err == cudaSuccess) err = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
            if (err != cudaSuccess || n < 1) {
                (void)cudaGetLastError();  // a refused size is not this call's failure
                refused.fetch_or(bit, std::memory_order_acq_rel);
                return cudaErrorNotSupported;
            }
            allowed.fetch_or(bit, std::memory_order_acq_rel);
        }
    }
    return cudaLaunchKernelEx(&cfg, kern, idx, T, k, E, R_cols, kind, capacity, align, 32 / k, ppw,
                              tpb, rof, counts, offsets, dst_row, rtc, status);
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

template <bool FP8, bool RANKS>
__global__ void __launch_bounds__(kLDThreads)
layout_dispatch_kernel(const int32_t* __restrict__ idx, int T, int k, int E, int R_cols, int kind,
                       int capacity, int P, int ppw, RankOf rank_of,
                       const uint16_t* __restrict__ x, int64_t H, int S, int64_t slice,
                       int32_t* __restrict__ expert_counts, int32_t* __restrict__ expert_offsets,
                       int32_t* __restrict__ dst_row, int32_t* __restrict__ rank_token_counts,
                       void* __restrict__ recv, float* __restrict__ recv_scale, int64_t rows,
                       uint32_t* __restrict__ status) {
    constexpr int NT = kLDThreads;
    constexpr int NW = kLDWarps;
    constexpr int U = FP8 ? 2 : 4;  // 512-channel groups (FP8) or 16-byte vectors per pass
    extern __shared__ __align__(16) int32_t smem_i[];
    __shared__ uint32_t s_flags;
    int32_t* s_dst = smem_i;  // [T * k] rows of all pairs
    const OneLaunchSmem sm = carve_block(s_dst + ((T * k + 3) & ~3), NW, E, R_cols, ppw);
    const int lane = threadIdx.x & 31;
    const int warp = threadIdx.x >> 5;
    const bool lead = blockIdx.x == 0;
    zero_warp_rows(sm, E, R_cols);

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

    // ---- the layout, as layout_block_kernel, into shared memory
    if (threadIdx.x == 0) s_flags = 0u;  // ordered before the atomics by block_layout's barriers
    uint32_t row_flags = 0;
    const uint32_t f = block_layout<NT, RANKS>(
        idx, T, k, E, R_cols, kind, capacity, 1, P, ppw, rank_of, sm,
        lead ? expert_counts : nullptr, lead ? expert_offsets : nullptr,
        lead ? rank_token_counts : nullptr, lead ? dst_row : nullptr, s_dst, rows, row_flags);
    const unsigned any = __reduce_or_sync(kFullMask, row_flags);
    if (any && lane == 0) atomicOr(&s_flags, any);
    __syncthreads();  // s_dst and s_flags complete
    if (lead && threadIdx.x == 0 && status) *status = s_flags | f;
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
            uint4 a[U], bb[U];
            if (j0 == 0 && c0 == cb) {  // warp-uniform: the loads issued before the layout
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    a[u] = pa[u];
                    bb[u] = pb[u];
                }
            } else {
#pragma unroll
                for (int u = 0; u < U; ++u) {
                    const int64_t c = c0 + u * 32 + lane;
                    a[u] = make_uint4(0, 0, 0, 0);
                    bb[u] = make_uint4(0, 0, 0, 0);
                    if (c < ce) {
                        if (FP8) {
                            a[u] = ld_stream_v4(src + c * 16);
                            bb[u] = ld_stream_v4(src + c * 16 + 8);
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
                    const Fp8Group g = quantize16(a[u], bb[u]);
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

size_t layout_dispatch_smem_bytes(int T, int k, int E, int R_cols, int ppw) {
    return ((size_t)((T * k + 3) & ~3)) * sizeof(int32_t) +
           block_smem_bytes(kLDWarps, E, R_cols, ppw);
}

template <bool FP8, bool RANKS>
cudaError_t launch_ld(const int32_t* topk_idx, int T, int k, int E, int R_cols, int kind,
                      int capacity, int ppw, RankOf rof, const void* x, int64_t H,
                      RowSlices sl, unsigned grid, int32_t* counts, int32_t* offsets,
                      int32_t* dst_row, int32_t* rtc, void* recv, float* recv_scale,
                      int64_t rows, uint32_t* status, size_t smem, cudaStream_t stream) {
    static std::atomic<uint64_t> configured{0};
    auto kern = layout_dispatch_kernel<FP8, RANKS>;
    cudaError_t err = prepare(kern, smem, configured);
    if (err != cudaSuccess) return err;
    return launch_pdl(kern, dim3(grid), dim3(kLDThreads), smem, stream, topk_idx, T, k, E, R_cols,
                      kind, capacity, 32 / k, ppw, rof, static_cast<const uint16_t*>(x), H,
                      sl.S, sl.slice, counts, offsets, dst_row, rtc, recv, recv_scale, rows,
                      status);
}

}  // namespace

cudaError_t launch_layout_dispatch(const int32_t* topk_idx, int64_t T, int k, int E, int R,
                                   int kind, int capacity, const void* x, int64_t H, bool fp8,
                                   int32_t* expert_counts, int32_t* expert_offsets,
                                   int32_t* dst_row, int32_t* rank_token_counts, void* recv,
                                   float* recv_scale, int64_t rows, uint32_t* status,
                                   cudaStream_t stream) {
    if (T < 1 || T > kLDMaxTokens) return cudaErrorNotSupported;
    const int R_cols = rank_token_counts ? R : 0;
    const int ppw = pieces_per_warp(T, k, kLDWarps);
    const size_t smem = layout_dispatch_smem_bytes((int)T, k, E, R_cols, ppw);
    if (ppw > max_pieces<kLDThreads>() || smem > kSmemLimit) return cudaErrorNotSupported;
    const RankOf rof = make_rank_of(E, R);
    const RowSlices sl = row_slices(T, fp8 ? H / 16 : H / 8);
    const unsigned grid = (unsigned)((T * sl.S + kLDWarps - 1) / kLDWarps);
#define EP_LD_ARGS                                                                             \
    topk_idx, (int)T, k, E, R_cols, kind, capacity, ppw, rof, x, H, sl, grid,           \
        expert_counts, expert_offsets, dst_row, rank_token_counts, recv, recv_scale, rows, status, \
        smem, stream
    if (fp8)
        return R_cols > 0 ? launch_ld<true, true>(EP_LD_ARGS) : launch_ld<true, false>(EP_LD_ARGS);
    return R_cols > 0 ? launch_ld<false, true>(EP_LD_ARGS) : launch_ld<false, false>(EP_LD_ARGS);
#undef EP_LD_ARGS
}

cudaError_t launch_layout_block(const int32_t* topk_idx, int64_t T, int k, int E, int R_cols,
                                int R, int kind, int capacity, int align, int max_threads,
                                int32_t* expert_counts, int32_t* expert_offsets, int32_t* dst_row,
                                int32_t* rank_token_counts, uint32_t* status,
                                cudaStream_t stream) {
    if (T < 1 || T > kClusterMaxTokens) return cudaErrorNotSupported;
    const RankOf rof = make_rank_of(E, R);
    for (int nt = max_threads; nt >= 32; nt /= 2) {
        const int NW = nt / 32;
        const int ppw = pieces_per_warp(T, k, NW);
        const size_t smem = block_smem_bytes(NW, E, R_cols, ppw);
        if (ppw > (nt >= 1024 ? max_pieces<1024>() : max_pieces<512>()) || smem > kSmemLimit)
            continue;
#define EP_BLOCK_CASE(N)                                                                         \
    case N:                                                                                      \
        return R_cols > 0                                                                        \
                   ? launch_block_nt<N, true>(topk_idx, (int)T, k, E, R_cols, kind, capacity,    \
                                              align, ppw, rof, expert_counts,             \
                                              expert_offsets, dst_row, rank_token_counts,        \
                                              status, smem, stream)                              \
                   : launch_block_nt<N, false>(topk_idx, (int)T, k, E, R_cols, kind, capacity,   \
                                               align, ppw, rof, expert_counts,            \
                                               expert_offsets, dst_row, rank_token_counts,       \
                                               status, smem, stream);
        switch (nt) {
            EP_BLOCK_CASE(1024)
            EP_BLOCK_CASE(512)
            EP_BLOCK_CASE(256)
            EP_BLOCK_CASE(128)
            EP_BLOCK_CASE(64)
            EP_BLOCK_CASE(32)
            default: break;
        }
#undef EP_BLOCK_CASE
    }
    return cudaErrorNotSupported;
}

namespace {

template <int CB>
cudaError_t launch_cluster_cb(const int32_t* topk_idx, int64_t T, int k, int E, int R_cols, int R,
                              int kind, int capacity, int align, int max_threads,
                              int32_t* expert_counts, int32_t* expert_offsets, int32_t* dst_row,
                              int32_t* rank_token_counts, uint32_t* status, cudaStream_t stream) {
    const RankOf rof = make_rank_of(E, R);
    const int tpb = (int)((T + CB - 1) / CB);
    for (int nt = max_threads; nt >= 32; nt /= 2) {
        const int NW = nt / 32;
        const int ppw = pieces_per_warp(tpb, k, NW);
        const size_t smem = cluster_smem_bytes(NW, E, R_cols, ppw, CB);
        if (ppw > (nt >= 1024 ? max_pieces<1024>() : max_pieces<512>()) || smem > kSmemLimit)
            continue;
#define EP_CLUSTER_CASE(N)                                                                       \
    case N:                                                                                      \
        return R_cols > 0                                                                        \
                   ? launch_cluster_nt<N, true, CB>(topk_idx, (int)T, k, E, R_cols, kind,        \
                                                    capacity, align, ppw, tpb, rof,              \
                                                    expert_counts, expert_offsets, dst_row,      \
                                                    rank_token_counts, status, smem, stream)     \
                   : launch_cluster_nt<N, false, CB>(topk_idx, (int)T, k, E, R_cols, kind,       \
                                                     capacity, align, ppw, tpb, rof,             \
                                                     expert_counts, expert_offsets, dst_row,     \
                                                     rank_token_counts, status, smem, stream);
        switch (nt) {
            EP_CLUSTER_CASE(1024)
            EP_CLUSTER_CASE(512)
            EP_CLUSTER_CASE(256)
            EP_CLUSTER_CASE(128)
            EP_CLUSTER_CASE(64)
            EP_CLUSTER_CASE(32)
            default: break;
        }
#undef EP_CLUSTER_CASE
    }
    return cudaErrorNotSupported;
}

}  // namespace

cudaError_t launch_layout_cluster(const int32_t* topk_idx, int64_t T, int k, int E, int R_cols,
                                  int R, int kind, int capacity, int align, int cluster_blocks,
                                  int max_threads, int32_t* expert_counts,
                                  int32_t* expert_offsets, int32_t* dst_row,
                                  int32_t* rank_token_counts, uint32_t* status,
                                  cudaStream_t stream) {
    if (T < 1 || T > kClusterMaxTokens) return cudaErrorNotSupported;
    if (cluster_blocks == 16)
        return launch_cluster_cb<16>(topk_idx, T, k, E, R_cols, R, kind, capacity, align,
                                     max_threads, expert_counts, expert_offsets, dst_row,
                                     rank_token_counts, status, stream);
    if (cluster_blocks == 8)
        return launch_cluster_cb<8>(topk_idx, T, k, E, R_cols, R, kind, capacity, align,
                                    max_threads, expert_counts, expert_offsets, dst_row,
                                    rank_token_counts, status, stream);
    return cudaErrorNotSupported;
}

}  // namespace ep
