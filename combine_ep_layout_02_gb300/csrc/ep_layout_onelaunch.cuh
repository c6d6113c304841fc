// ep_layout_onelaunch.cuh -- launchers of the one-launch layouts
// (ep_layout_onelaunch.cu) and the batch sizes at which ep_layout uses them
// (ep_layout.cu).
#pragma once

#include "ep_internal.cuh"

namespace ep {

// One-launch layouts (ep_layout_onelaunch.cu): a single block up to
// EP_LAYOUT_BLOCK_MAX_TOKENS tokens, one cluster up to
// EP_LAYOUT_CLUSTER_MAX_TOKENS (at most 2048): 8 blocks up to
// EP_LAYOUT_CLUSTER16_MIN_TOKENS - 1 tokens, 16 above (8 where the device
// cannot place 16); cudaErrorNotSupported (nothing enqueued) when the shape
// does not fit their registers or shared memory.  Sizes measured fastest
// (graph-replayed, E = 128 and 256): one 256-thread block up to 64 tokens
// (2.7-3.0 us), 8 blocks of 256 threads up to 256 tokens (128: 2.9-3.3 us;
// 16 blocks 3.1-3.5 us; 8 blocks of 128 threads the same or slower), 16
// blocks of 256 threads above (2048: 4.4-5.1 us; 16 x 512 threads 4.8-5.2 us;
// 8 x 512 threads 5.8-5.9 us).  The 8-block
// fallback keeps 256-thread blocks up to EP_LAYOUT_CLUSTER_SMALL_MAX_TOKENS
// tokens and 512-thread blocks above.
#ifndef EP_LAYOUT_BLOCK_MAX_TOKENS
#define EP_LAYOUT_BLOCK_MAX_TOKENS 64
#endif
#ifndef EP_LAYOUT_CLUSTER_MAX_TOKENS
#define EP_LAYOUT_CLUSTER_MAX_TOKENS 2048
#endif
#ifndef EP_LAYOUT_BLOCK_THREADS
#define EP_LAYOUT_BLOCK_THREADS 256
#endif
#ifndef EP_LAYOUT_CLUSTER16_MIN_TOKENS
#define EP_LAYOUT_CLUSTER16_MIN_TOKENS 257
#endif
#ifndef EP_LAYOUT_CLUSTER16_THREADS
#define EP_LAYOUT_CLUSTER16_THREADS 256
#endif
#ifndef EP_LAYOUT_CLUSTER_SMALL_MAX_TOKENS
#define EP_LAYOUT_CLUSTER_SMALL_MAX_TOKENS 768
#endif
#ifndef EP_LAYOUT_CLUSTER_THREADS_SMALL
#define EP_LAYOUT_CLUSTER_THREADS_SMALL 256
#endif
#ifndef EP_LAYOUT_CLUSTER_THREADS
#define EP_LAYOUT_CLUSTER_THREADS 512
#endif
cudaError_t launch_layout_block(const int32_t* topk_idx, int64_t T, int k, int E, int R_cols,
                                int R, int kind, int capacity, int align, int max_threads,
                                int32_t* expert_counts, int32_t* expert_offsets, int32_t* dst_row,
                                int32_t* rank_token_counts, uint32_t* status, cudaStream_t stream);
// cluster_blocks: 8 or 16.
cudaError_t launch_layout_cluster(const int32_t* topk_idx, int64_t T, int k, int E, int R_cols,
                                  int R, int kind, int capacity, int align, int cluster_blocks,
                                  int max_threads, int32_t* expert_counts,
                                  int32_t* expert_offsets, int32_t* dst_row,
                                  int32_t* rank_token_counts, uint32_t* status,
                                  cudaStream_t stream);

}  // namespace ep
