/*
 * ep.h -- C ABI of the GB300 (sm_103a) MoE expert-parallel hot path:
 * routing layout, dispatch (BF16 or FP8 e4m3 with per-128-channel scales)
 * and weighted top-k combine, all on one GPU.
 *
 * The operations are the local steps of DeepEP-style dispatch/combine as the
 * pages state the problem ("Replace EP backend comparison with Decode-like
 * and Prefill-like B200 benchmarks", awsome-distributed-ai PR #1238, section
 * "What changed": BF16 input with an exact top-k route and weights; FP8
 * conversion, the dispatch layout, dispatch and combine inside one timed
 * boundary; and the afdEP-comm validation record, "setup": masked
 * [experts, capacity, hidden] buffers with capacity 2048).  "Virtual ranks"
 * are only a grouping of experts here: rank r owns experts
 * [r*E/R, (r+1)*E/R).  There is no communication.
 *
 * Conventions for every call
 *  - Pointers are DEVICE pointers unless stated otherwise.  The caller owns
 *    (allocates and frees) every buffer; the library allocates no device
 *    memory (ep_layout_static_ws uses one fixed array of the library's own;
 *    ep_pipeline_create makes streams and events, no memory).
 *  - Work runs on the caller's current CUDA device; the pointers and
 *    `stream` must belong to it.
 *  - `stream` is a cudaStream_t passed as void*; NULL is the legacy default
 *    stream.  Every call only enqueues work on `stream` and returns; nothing
 *    synchronises except ep_status_read().
 *  - Return value: an ep_status_t.  A non-zero value detected on the host
 *    (bad sizes, NULL or misaligned pointers, small workspace) means that
 *    NOTHING was enqueued.  EP_ERR_CUDA means a launch failed (the CUDA error
 *    is available from ep_last_cuda_error()).
 *  - Conditions found on the device never trap: they are OR-ed as EP_FLAG_*
 *    bits into the optional `status` word (a device uint32), which the caller
 *    reads with ep_status_read().  ep_layout() zeroes the word first;
 *    ep_dispatch*() and ep_combine() only OR into it.
 *  - Kernels are launched with programmatic stream serialisation: each one
 *    waits for the preceding work in the stream before touching memory, and
 *    lets the next kernel launch early.  A caller's own kernel launched right
 *    after one of ours WITH that launch attribute must wait on the grid
 *    dependency (griddepcontrol.wait / cudaGridDependencySynchronize) before
 *    reading our outputs; ordinary launches, copies and events need nothing.
 *  - bf16 tensors are passed as raw 16-bit patterns, row-major.
 *  - dst_row[t*k + j] is the row of the dispatch buffer that receives token t
 *    for its j-th expert, or -1 when the pair is not routed (expert id -1, a
 *    bad id, or a masked-capacity overflow).  Pairs with dst_row == -1 are
 *    skipped by dispatch and contribute nothing to combine.
 *
 * Limits: 1 <= k <= EP_MAX_TOPK; 1 <= E <= EP_MAX_EXPERTS; R >= 1 divides E;
 * T*k < 2^31; E*capacity < 2^31 (masked); H % 8 == 0 (BF16 rows are whole
 * 16-byte vectors); H % 128 == 0 for FP8; 16-byte-aligned bf16/e4m3 buffers.
 */
#ifndef EP_GB300_H
#define EP_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#if defined(__GNUC__)
#define EP_API __attribute__((visibility("default")))
#else
#define EP_API
#endif

#define EP_MAX_TOPK 32
#define EP_MAX_EXPERTS 1024
#define EP_STATIC_WS_BYTES (2u << 20) /* scratch held by ep_layout_static_ws() */

typedef enum {
    EP_OK = 0,
    EP_ERR_INVALID_ARG = 1, /* NULL pointer, size out of range, E % R != 0 ... */
    EP_ERR_ALIGNMENT = 2,   /* H or a pointer violates the alignment rules     */
    EP_ERR_WORKSPACE = 3,   /* workspace smaller than ep_layout_workspace_bytes */
    EP_ERR_CUDA = 4         /* a kernel launch or copy failed                   */
} ep_status_t;

/* Device-side condition bits (OR-ed into *status). */
enum {
    EP_FLAG_BAD_EXPERT = 1u, /* an expert id outside [-1, E): the pair was skipped */
    EP_FLAG_OVERFLOW = 2u,   /* masked layout: slot >= capacity, the pair was dropped */
    EP_FLAG_BAD_ROW = 4u,    /* dispatch/combine: dst_row outside [-1, rows): skipped */
    EP_FLAG_TIMEOUT = 8u     /* layout: a block of the one-launch cluster layout waited
                                over a second for the others' totals and gave up; the
                                outputs are incomplete (not expected on a working GPU) */
};

typedef enum { EP_LAYOUT_CONTIGUOUS = 0, EP_LAYOUT_MASKED = 1 } ep_layout_kind_t;

/* Library version, (major << 16) | minor. */
EP_API int ep_version(void);

/* Human-readable name of an ep_status_t. Never NULL. */
EP_API const char* ep_status_string(int status);

/* The CUDA error (cudaError_t as int) of the last EP_ERR_CUDA on this host
 * thread, 0 if none. */
EP_API int ep_last_cuda_error(void);

/* Bytes of device workspace ep_layout() needs for these sizes (0 when T == 0).
 * with_rank_counts: non-zero if rank_token_counts will be requested. */
EP_API size_t ep_layout_workspace_bytes(int64_t T, int k, int E, int R, int with_rank_counts);

/*
 * ep_layout -- routing layout: per-expert counts, exclusive scan, stable slot.
 * (PR #1238 "What changed": the Prefill-like profile includes the dispatch
 * layout the normal API requires; masked buffers from the afdEP "setup".)
 *
 *  topk_idx          [T, k] int32 expert ids; -1 = no expert.
 *  kind, capacity    EP_LAYOUT_CONTIGUOUS (capacity ignored) or
 *                    EP_LAYOUT_MASKED with `capacity` rows per expert.
 *  expert_counts     [E] int32 out: pairs routed to each expert (the true
 *                    count, also when a masked expert overflows).
 *  expert_offsets    [E+1] int32 out: exclusive scan of expert_counts;
 *                    expert_offsets[E] = rows used by the contiguous layout.
 *  dst_row           [T, k] int32 out.  A pair's slot is the number of
 *                    earlier pairs (in flattened order t*k+j) with the same
 *                    expert.  Contiguous: expert_offsets[e] + slot.
 *                    Masked: e*capacity + slot, or -1 with EP_FLAG_OVERFLOW
 *                    when slot >= capacity.  Ids outside [-1, E) give -1 and
 *                    EP_FLAG_BAD_EXPERT.
 *  rank_token_counts [R] int32 out or NULL: tokens with at least one valid
 *                    expert in virtual rank r.
 *                    The layout may be computed once and reused by any number
 *                    of ep_dispatch / ep_combine calls for the same route
 *                    (the pages' "cached dispatch").
 *  status            [1] uint32 or NULL: zeroed, then device flags OR-ed in.
 *  workspace         device scratch of at least
 *                    ep_layout_workspace_bytes(T, k, E, R, rank_token_counts != NULL)
 *                    bytes, 16-byte aligned; contents need no initialisation
 *                    and are clobbered.  May be NULL when that size is 0.
 * T == 0 is valid: counts, offsets and rank counts are written as zeros.
 */
EP_API int ep_layout(const int32_t* topk_idx, int64_t T, int k, int E, int R,
              int kind, int capacity,
              int32_t* expert_counts, int32_t* expert_offsets, int32_t* dst_row,
              int32_t* rank_token_counts, uint32_t* status,
              void* workspace, size_t workspace_bytes, void* stream);

/*
 * ep_layout_aligned -- the contiguous layout for a grouped-GEMM consumer that
 * wants every expert's rows to start on a multiple of `alignment` rows (the
 * "expert_alignment" setting of the DeepEP dispatch mode that PR #1238's
 * kernel-level re-run pins to 1).  Expert e's segment is
 * ceil(expert_counts[e] / alignment) * alignment rows long, so
 * expert_offsets[e] is a multiple of `alignment`; slots are those of
 * ep_layout.  The padding rows receive no pair: dispatch leaves them untouched
 * and combine never reads them.  The buffer needs expert_offsets[E] rows, at
 * most T*k + E*(alignment-1).  alignment == 1 is ep_layout(..contiguous..).
 * Requires alignment >= 1 and T*k + E*(alignment-1) < 2^31.
 */
EP_API int ep_layout_aligned(const int32_t* topk_idx, int64_t T, int k, int E, int R,
                             int alignment, int32_t* expert_counts, int32_t* expert_offsets,
                             int32_t* dst_row, int32_t* rank_token_counts, uint32_t* status,
                             void* workspace, size_t workspace_bytes, void* stream);

/*
 * ep_layout_static_ws -- ep_layout() for callers that cannot allocate device
 * memory: for example a plug-in whose host application owns all device
 * memory through its own pool and gives the plug-in no way to allocate, or a
 * real-time loop that must not allocate once it is running.  The pages have
 * no counterpart; this call exists only for such callers.
 *
 * Arguments, outputs and status are those of ep_layout(), minus the
 * workspace: the layout's scratch is one fixed array of EP_STATIC_WS_BYTES
 * (2 MiB) in the library's own device memory, which every GPU that loads the
 * library holds until the process exits.
 *  - Returns EP_ERR_WORKSPACE, enqueueing nothing, when
 *    ep_layout_workspace_bytes(T, k, E, R, rank_token_counts != NULL) exceeds
 *    EP_STATIC_WS_BYTES.  (Example: T = 131072, E = 256, R = 32 needs 1.18 MB;
 *    the limit is 512k int32 counters of (E+R) x ceil(T/128).)
 *  - The first call on a device looks up the array's device address, with
 *    the caller's current device; that device must be the one `stream`
 *    belongs to.  Make the first call on each device before any stream
 *    capture begins.  The address is kept for the life of the process:
 *    cudaDeviceReset() (or anything else that destroys the device's primary
 *    context) between calls is not supported.
 *  - Argument errors are reported as ep_layout() reports them; a size beyond
 *    the array's limit then gives EP_ERR_WORKSPACE.
 *  - Every call on a device shares the one array, and it keeps the last
 *    call's contents (the layout fully rewrites what it reads, so nothing
 *    needs clearing).  Calls whose kernels overlap on the GPU (for example
 *    on two streams without an event between them) race on it and produce
 *    wrong layouts: serialise them.
 *  - Allocates nothing: no cudaMalloc, cudaFree or allocating library call.
 */
EP_API int ep_layout_static_ws(const int32_t* topk_idx, int64_t T, int k, int E, int R,
                               int kind, int capacity,
                               int32_t* expert_counts, int32_t* expert_offsets,
                               int32_t* dst_row, int32_t* rank_token_counts,
                               uint32_t* status, void* stream);

/*
 * ep_dispatch -- BF16 dispatch (scatter): recv[dst_row[t,j], :] = x[t, :],
 * a bit copy (PR #1238 "What changed": each token is sent to its top-k
 * experts; the BF16 payload is T*k*H*2 bytes).
 *
 *  x        [T, H] bf16, 16-byte aligned.
 *  dst_row  [T, k] int32 from ep_layout.
 *  recv     [rows, H] bf16, 16-byte aligned.  Rows no pair maps to (masked
 *           padding, rows past expert_offsets[E]) are not touched.
 *  rows     number of rows of recv; a dst_row outside [-1, rows) is skipped
 *           and raises EP_FLAG_BAD_ROW.
 */
EP_API int ep_dispatch(const void* x, int64_t T, int64_t H, int k, const int32_t* dst_row,
                void* recv, int64_t rows, uint32_t* status, void* stream);

/*
 * ep_dispatch_fp8 -- dispatch with the per-token FP8 cast fused into the copy
 * (PR #1238: the standalone cast is a separate launch-bound step in the
 * timed boundary; the low-latency API quantises inside the dispatch kernel;
 * the payload carries one float32 scale per 128 channels).  For each token t
 * and block b of 128 channels:
 *     a   = max |x[t, 128b .. 128b+127]|         (fp32)
 *     a'  = max(a, 1e-4f)
 *     sf  = a' / 448.0f                          (IEEE fp32 division, RNE)
 *     inv = 448.0f / a'                          (IEEE fp32 division, RNE)
 *     q   = e4m3(x * inv)   fp32 product rounded to nearest even, then
 *                           e4m3 "fn" with round-to-nearest-even and
 *                           saturation to +-448
 * q and sf are written to every dst_row of the token; x ~= e4m3_value(q) * sf.
 *
 *  recv_q      [rows, H] uint8 e4m3 codes, 16-byte aligned.
 *  recv_scale  [rows, H/128] float32, row-major, 4-byte aligned.
 *  H % 128 == 0 is required.
 */
EP_API int ep_dispatch_fp8(const void* x, int64_t T, int64_t H, int k, const int32_t* dst_row,
                    uint8_t* recv_q, float* recv_scale, int64_t rows,
                    uint32_t* status, void* stream);

/*
 * ep_layout_dispatch -- ep_layout followed by ep_dispatch on the same status
 * word, in one call (PR #1238, "What changed": the dispatch layout is part
 * of the timed dispatch boundary, and the Decode-like profile measures 128
 * tokens per rank, where separate launches dominate).  Arguments are those
 * of the two calls; the layout kind, capacity and rank counts are as for
 * ep_layout (no alignment), recv and rows as for ep_dispatch.  The outputs
 * (counts, offsets, dst_row, rank_token_counts, recv, status) are identical
 * to the two calls made in sequence.  Up to 128 tokens this is one kernel
 * launch: every block computes the whole layout in shared memory and
 * dispatches its share of the rows.  Larger batches run the two launches,
 * the dispatch issuing its first loads of x while the layout still runs
 * (x must therefore not be written by earlier work that is still running on
 * another stream without an event between them -- as for any input).  The
 * workspace rules of ep_layout apply.
 */
EP_API int ep_layout_dispatch(const int32_t* topk_idx, int64_t T, int k, int E, int R, int kind,
                              int capacity, const void* x, int64_t H, int32_t* expert_counts,
                              int32_t* expert_offsets, int32_t* dst_row,
                              int32_t* rank_token_counts, void* recv, int64_t rows,
                              uint32_t* status, void* workspace, size_t workspace_bytes,
                              void* stream);

/* ep_layout_dispatch_fp8 -- the same with ep_dispatch_fp8 (H % 128 == 0). */
EP_API int ep_layout_dispatch_fp8(const int32_t* topk_idx, int64_t T, int k, int E, int R,
                                  int kind, int capacity, const void* x, int64_t H,
                                  int32_t* expert_counts, int32_t* expert_offsets,
                                  int32_t* dst_row, int32_t* rank_token_counts, uint8_t* recv_q,
                                  float* recv_scale, int64_t rows, uint32_t* status,
                                  void* workspace, size_t workspace_bytes, void* stream);

/*
 * ep_combine -- weighted top-k reduction back into token order (the combine
 * step of the PR's timed boundary; BF16 in either payload mode):
 *     out[t, h] = bf16_rne( sum over j with dst_row[t,j] != -1 of
 *                           topk_w[t,j] * y[dst_row[t,j], h] )
 * accumulated in fp32 as fused multiply-adds in increasing j, starting from
 * +0, then rounded to bf16 (nearest even).  A token with no valid pair
 * gives +0.
 *
 *  y        [rows, H] bf16 expert outputs in the dispatch layout, 16-byte aligned.
 *  topk_w   [T, k] float32 top-k weights.
 *  out      [T, H] bf16, 16-byte aligned; must not overlap y.
 */
EP_API int ep_combine(const void* y, const float* topk_w, const int32_t* dst_row,
               int64_t T, int64_t H, int k, int64_t rows, void* out,
               uint32_t* status, void* stream);

/*
 * ep_combine_fp8 -- the combine for expert outputs carried in the FP8
 * payload's own encoding (PR #1238, review section 9 "Smaller notes", names a
 * compressed combine path but fixes no format; this is the reading taken):
 * e4m3 codes and one float32 scale per 128 channels, the value of a code
 * being decode(code) * scale, as for the output of ep_dispatch_fp8.
 *     out[t, h] = bf16_rne( sum over j with dst_row[t,j] != -1 of
 *                           topk_w[t,j] * decode(y_q[r, h]) * y_scale[r, h/128] )
 * computed in fp32 as: c = fl32(topk_w[t,j] * y_scale[r, h/128]), then
 * acc = fmaf(c, decode(y_q[r, h]), acc) in increasing j from +0, then one
 * rounding to bf16 (decode is exact in fp32).  A token with no valid pair
 * gives +0; a NaN code (0x7F, 0xFF) gives NaN.
 *
 *  y_q      [rows, H] uint8 e4m3 codes, 16-byte aligned.
 *  y_scale  [rows, H/128] float32, row-major, 4-byte aligned.
 *  topk_w   [T, k] float32;  dst_row [T, k] int32 as for ep_combine.
 *  out      [T, H] bf16, 16-byte aligned.  H % 128 == 0.
 */
EP_API int ep_combine_fp8(const uint8_t* y_q, const float* y_scale, const float* topk_w,
                          const int32_t* dst_row, int64_t T, int64_t H, int k, int64_t rows,
                          void* out, uint32_t* status, void* stream);

/*
 * Two-stage (rank, then expert) form of dispatch and combine -- the shape of
 * the pages' transport: one copy of a token per virtual rank it reaches,
 * expanded on arrival into that rank's experts (dispatch_copy_epilogue in the
 * afdEP kernel traces; PR #1238's review: one copy per destination node, then
 * forwarding to the local experts), and on the way back a rank-local partial
 * reduction followed by the final reduction over the token's ranks
 * (combine_reduce_epilogue).  With ranks being regions of one GPU, the copy to
 * ranks is ep_dispatch(x, .., rank_dst_row, rank_buf, rank_rows, ..).
 *
 * ep_rank_layout: every (token t, rank r) that t reaches gets one row of a
 * rank buffer; rank r owns rows [rank_offsets[r], rank_offsets[r+1]), in
 * token order.
 *  rank_counts      [R] out: tokens reaching rank r.
 *  rank_offsets     [R+1] out: exclusive scan; rank_offsets[R] = rows used
 *                   (at most T * min(k, R): size rank buffers for that).
 *  rank_dst_row     [T,k] out: the rank row for the FIRST pair of each
 *                   (token, rank), -1 for the token's other pairs in that rank
 *                   and for pairs without a valid expert.
 *  pair_rank_row    [T,k] out: the rank row of every pair with a valid expert.
 *  rank_row_token   [rank_rows] out: the token of each rank row; rank_rows
 *                   should be T * min(k, R) (rows beyond it are not written
 *                   and raise EP_FLAG_BAD_ROW).
 *  workspace        ep_rank_layout_workspace_bytes(T, k, E, R) bytes,
 *                   16-byte aligned, no initialisation needed.
 *  status           zeroed, then EP_FLAG_BAD_EXPERT for ids outside [-1, E).
 */
EP_API size_t ep_rank_layout_workspace_bytes(int64_t T, int k, int E, int R);
EP_API int ep_rank_layout(const int32_t* topk_idx, int64_t T, int k, int E, int R,
                          int32_t* rank_counts, int32_t* rank_offsets, int32_t* rank_dst_row,
                          int32_t* pair_rank_row, int32_t* rank_row_token, int64_t rank_rows,
                          uint32_t* status, void* workspace, size_t workspace_bytes,
                          void* stream);

/*
 * ep_expand: recv[dst_row[t,j]] = rank_buf[pair_rank_row[t,j]] for every pair
 * (bit copy), one pass over each rank row.  rank_buf is [rank_rows, H] bf16
 * (rank_rows = its allocated rows, >= rank_offsets[R]); the kernels read the
 * live row count from rank_offsets[R] on the device.
 */
EP_API int ep_expand(const void* rank_buf, const int32_t* rank_offsets, int R, int64_t rank_rows,
                     const int32_t* rank_row_token, const int32_t* pair_rank_row,
                     const int32_t* dst_row, int64_t T, int64_t H, int k, void* recv,
                     int64_t rows, uint32_t* status, void* stream);

/*
 * ep_expand_fp8: the same for an FP8 rank buffer (the copy to ranks being
 * ep_dispatch_fp8(x, .., rank_dst_row, rank_q, rank_scale, rank_rows, ..)):
 * codes [rank_rows, H] and scales [rank_rows, H/128] of each rank row are
 * copied to recv_q / recv_scale rows dst_row[t,j].  H % 128 == 0.
 */
EP_API int ep_expand_fp8(const uint8_t* rank_q, const float* rank_scale,
                         const int32_t* rank_offsets, int R, int64_t rank_rows,
                         const int32_t* rank_row_token, const int32_t* pair_rank_row,
                         const int32_t* dst_row, int64_t T, int64_t H, int k, uint8_t* recv_q,
                         float* recv_scale, int64_t rows, uint32_t* status, void* stream);

/*
 * ep_combine_partial: for each rank row i of token t,
 *   partial[i] = bf16_rne( fp32 FMA chain, increasing j, over the pairs of t
 *                with pair_rank_row == i and dst_row != -1, of
 *                topk_w[t,j] * y[dst_row[t,j]] ).
 * ep_combine_reduce: out[t] = bf16_rne( fp32 sum, increasing j, of
 *   partial[rank_dst_row[t,j]] over the pairs with rank_dst_row != -1 ).
 * The two together equal ep_combine up to the extra bf16 rounding of each
 * partial (|difference| <= 2^-9 * sum_r |partial_r| + one final rounding).
 */
EP_API int ep_combine_partial(const void* y, int64_t rows, const float* topk_w,
                              const int32_t* dst_row, const int32_t* pair_rank_row,
                              const int32_t* rank_row_token, const int32_t* rank_offsets, int R,
                              int64_t rank_rows, int64_t T, int64_t H, int k, void* partial,
                              uint32_t* status, void* stream);
EP_API int ep_combine_reduce(const void* partial, int64_t rank_rows, const int32_t* rank_dst_row,
                             int64_t T, int64_t H, int k, void* out, uint32_t* status,
                             void* stream);

/*
 * Host-buffer executor.  ep_roundtrip_host() runs one whole step -- route to
 * the device, ep_layout, ep_dispatch, ep_combine, result back -- for inputs and
 * output in pinned HOST memory, overlapping the copies with the kernels in
 * token chunks: the route is copied first (the layout needs all of it), then
 * the hidden states stream in chunk by chunk on a copy stream while earlier
 * chunks are dispatched and combined on `stream`, and each combined chunk is
 * copied back on a second copy stream.  (The pages time one boundary from
 * "BF16 input and route ready" to combine completion; this call is that step
 * seen from host memory.)
 *
 * A pipeline handle owns the two copy streams and the events the overlap
 * needs; it is created once for the current device and reused.  It holds no
 * device memory.
 */
EP_API int ep_pipeline_create(int max_chunks, void** handle);
EP_API int ep_pipeline_destroy(void* handle); /* synchronises its copy streams first */

/*
 *  handle        from ep_pipeline_create on the current device;
 *                ceil(T / chunk_tokens) <= its max_chunks.
 *  stream        the caller's stream: when it has run past this call the
 *                whole step, including the copy of `out_host`, is complete.
 *  x_host        [T, H] bf16, idx_host [T, k] int32, w_host [T, k] float32,
 *  out_host      [T, H] bf16: HOST pointers, pinned (page-locked).
 *  x_dev, idx_dev, w_dev, out_dev   device staging buffers of the same shapes
 *                (x_dev, out_dev 16-byte aligned).
 *  recv, rows    the BF16 dispatch buffer, as for ep_dispatch; or, when
 *  recv_q        is not NULL, FP8 dispatch into recv_q / recv_scale as for
 *                ep_dispatch_fp8 (recv may then be NULL).
 *  y             expert outputs [rows, H] bf16 on the device, or NULL (BF16
 *                dispatch only) to combine the dispatched rows themselves
 *                (identity experts).
 *  the rest      as for ep_layout.
 * Returns as the underlying calls do; on a non-zero return some work may
 * already be enqueued.
 */
EP_API int ep_roundtrip_host(void* handle, void* stream, const void* x_host,
                             const int32_t* idx_host, const float* w_host, void* out_host,
                             int64_t T, int64_t H, int k, int E, int R, int kind, int capacity,
                             int64_t chunk_tokens, void* x_dev, int32_t* idx_dev, float* w_dev,
                             void* recv, uint8_t* recv_q, float* recv_scale, int64_t rows,
                             const void* y, void* out_dev,
                             int32_t* expert_counts, int32_t* expert_offsets, int32_t* dst_row,
                             int32_t* rank_token_counts, uint32_t* status, void* workspace,
                             size_t workspace_bytes);

/* Copy the device status word to *host_flags (a HOST pointer) after
 * synchronising `stream`. */
EP_API int ep_status_read(const uint32_t* status, void* stream, uint32_t* host_flags);

#ifdef __cplusplus
}
#endif
#endif /* EP_GB300_H */
