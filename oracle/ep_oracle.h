/*
 * ep_oracle.h -- plain, single-threaded CPU oracle for MoE expert-parallel
 * routing layout, dispatch (BF16 and FP8 e4m3 with per-128-channel scales)
 * and weighted top-k combine.
 *
 * TEST INFRASTRUCTURE ONLY.  Nothing in the product path may link, load or
 * call this library: only the test-suite, the smoke check and the CPU-baseline
 * leg of the benchmark use it.  It shares no code, header, table or constant
 * with the CUDA library and includes no CUDA header.
 *
 * Every function computes the plain definition of its step; see the comments
 * in ep_oracle.c for the passage each one follows and the reading taken where
 * the pages leave a step open.
 */
#ifndef EP_ORACLE_H
#define EP_ORACLE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

enum { ORACLE_LAYOUT_CONTIGUOUS = 0, ORACLE_LAYOUT_MASKED = 1 };
enum { ORACLE_FLAG_BAD_EXPERT = 1u, ORACLE_FLAG_OVERFLOW = 2u };

/* Scalar format helpers (definitions of the number formats). */
float    oracle_bf16_to_float(uint16_t b);
uint16_t oracle_bf16_from_double(double v);
float    oracle_e4m3_decode(uint8_t code);
uint8_t  oracle_e4m3_encode(float v);

/* Routing layout.  topk_idx is [T,k] row-major.  Writes counts[E],
 * offsets[E+1], dst_row[T*k] and, if rank_token_counts is not NULL,
 * rank_token_counts[R].  Returns the OR of ORACLE_FLAG_* conditions.
 * Returns 0xFFFFFFFF (and writes nothing) on invalid sizes. */
uint32_t oracle_layout(const int32_t* topk_idx, int64_t T, int k, int E, int R,
                       int kind, int capacity, int32_t* counts,
                       int32_t* offsets, int32_t* dst_row,
                       int32_t* rank_token_counts);

/* Routing layout with each expert's contiguous segment padded to a multiple
 * of `alignment` rows: offsets are the exclusive scan of
 * ceil(count / alignment) * alignment.  Contiguous kind only; alignment 1 is
 * oracle_layout(). */
uint32_t oracle_layout_aligned(const int32_t* topk_idx, int64_t T, int k, int E, int R,
                               int alignment, int32_t* counts, int32_t* offsets,
                               int32_t* dst_row, int32_t* rank_token_counts);

/* BF16 dispatch: recv[dst_row[t,j], :] = x[t, :] for every pair with
 * dst_row >= 0.  x is [T,H], recv is [rows,H], both bf16 bit patterns. */
void oracle_dispatch_bf16(const uint16_t* x, int64_t T, int64_t H, int k,
                          const int32_t* dst_row, uint16_t* recv);

/* Per-token, per-128-channel FP8 e4m3 quantisation of one token row:
 * q[H] codes and scale[H/128] float32.  H must be a multiple of 128. */
void oracle_quantize_row_fp8(const uint16_t* x_row, int64_t H, uint8_t* q,
                             float* scale);

/* FP8 dispatch: the quantised row and its scales copied to every dst_row of
 * the token.  recv_q is [rows,H] e4m3 codes, recv_scale is [rows,H/128]. */
void oracle_dispatch_fp8(const uint16_t* x, int64_t T, int64_t H, int k,
                         const int32_t* dst_row, uint8_t* recv_q,
                         float* recv_scale);

/* Combine with fp64 accumulation.  out[t,h] = bf16(sum_j w[t,j]*y[row,h])
 * rounded once from the fp64 sum.  ref (may be NULL) receives the fp64 sum,
 * absum (may be NULL) the fp64 sum of |w*y| over the valid pairs. */
void oracle_combine_f64(const uint16_t* y, const float* topk_w,
                        const int32_t* dst_row, int64_t T, int64_t H, int k,
                        uint16_t* out, double* ref, double* absum);

/* Combine as a sequence of fp32 fused multiply-adds in increasing j, each
 * rounded to nearest even, then rounded once to bf16. */
void oracle_combine_fp32_seq(const uint16_t* y, const float* topk_w,
                             const int32_t* dst_row, int64_t T, int64_t H,
                             int k, uint16_t* out);

/* Combine of FP8 expert outputs: codes y_q [rows,H], scales y_scale
 * [rows,H/128] (value = decode(q) * scale).  out[t,h] = bf16 of the fp64 sum
 * of w[t,j] * value over the valid pairs (every product exact in double);
 * ref / absum as for oracle_combine_f64 (may be NULL). */
void oracle_combine_fp8_f64(const uint8_t* y_q, const float* y_scale,
                            const float* topk_w, const int32_t* dst_row,
                            int64_t T, int64_t H, int k, uint16_t* out,
                            double* ref, double* absum);

/* The same in fp32: c = fl32(w * scale) per pair and block, then fmaf(c,
 * decode(q), acc) in increasing j, then one rounding to bf16. */
void oracle_combine_fp8_fp32_seq(const uint8_t* y_q, const float* y_scale,
                                 const float* topk_w, const int32_t* dst_row,
                                 int64_t T, int64_t H, int k, uint16_t* out);

/* ---- two-stage (rank, then expert) path ---------------------------------
 * Rank layout: every (token t, virtual rank r) that t reaches gets one row of
 * a rank buffer, rank r's rows in token order.  rank_dst_row[t,j] is that row
 * for the FIRST pair of t in rank r and -1 for its other pairs (and for
 * pairs with no valid expert); pair_rank_row[t,j] is the row for every pair
 * with a valid expert.  rank_row_token[row] is the row's token. */
uint32_t oracle_rank_layout(const int32_t* topk_idx, int64_t T, int k, int E, int R,
                            int32_t* rank_counts, int32_t* rank_offsets,
                            int32_t* rank_dst_row, int32_t* pair_rank_row,
                            int32_t* rank_row_token);

/* Expansion: recv[dst_row[t,j]] = rank_buf[pair_rank_row[t,j]] for every
 * pair with both rows valid. */
void oracle_expand(const uint16_t* rank_buf, const int32_t* pair_rank_row,
                   const int32_t* dst_row, int64_t T, int64_t H, int k, uint16_t* recv);

/* Rank-local partial reduction: partial[i] = bf16(fp32 fma chain over the
 * pairs j (increasing) of token rank_row_token[i] with pair_rank_row == i and
 * dst_row >= 0 of w[t,j] * y[dst_row[t,j]]), for i < n_rows. */
void oracle_combine_partial(const uint16_t* y, const float* topk_w,
                            const int32_t* dst_row, const int32_t* pair_rank_row,
                            const int32_t* rank_row_token, int64_t n_rows, int64_t H,
                            int k, uint16_t* partial);

/* Final reduction: out[t] = bf16(fp32 sum, in increasing j, of
 * partial[rank_dst_row[t,j]] over the pairs with rank_dst_row >= 0). */
void oracle_combine_reduce(const uint16_t* partial, const int32_t* rank_dst_row,
                           int64_t T, int64_t H, int k, uint16_t* out);

#ifdef __cplusplus
}
#endif
#endif
