/*
 * Plain fp64 CPU oracle for the Kimi-K3 shared-expert SwiGLU MLP.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * bench's CPU-baseline leg may load this library.  It shares no code, header,
 * table or helper with the CUDA library, and it does not include that
 * library's header.
 *
 * All tensors are row-major.  bf16 tensors are passed as their uint16 bit
 * patterns and decoded exactly to double.  Every sum runs in double over the
 * reduction index in ascending order.
 */
#ifndef MSE_ORACLE_H
#define MSE_ORACLE_H
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

double   oracle_bf16_to_f64(uint16_t b);
uint16_t oracle_f64_to_bf16_rne(double d);
double   oracle_silu(double z);

/* h[r, j - j_begin] = bf16_rne(silu(g) * u) for j in [j_begin, j_end);
 * g_out/u_out (nullable) receive the fp64 pre-activation sums. */
void oracle_swiglu_hidden(const uint16_t *x, int64_t T, int64_t H, int64_t I,
                          const uint16_t *w_gate_up, int64_t j_begin, int64_t j_end,
                          const int64_t *rows, int64_t n_rows,
                          uint16_t *h, double *g_out, double *u_out, int nthreads);

/* Replicated layer.  y (bf16) and y_f64 (pre-rounding sums) are [n_rows x H];
 * h_out (nullable) is [n_rows x I]. */
void oracle_mlp_forward(const uint16_t *x, int64_t T, int64_t H, int64_t I,
                        const uint16_t *w_gate_up, const uint16_t *w_down,
                        const int64_t *rows, int64_t n_rows,
                        uint16_t *y, double *y_f64, uint16_t *h_out, int nthreads);

/* Partial output of shard `rank` of `tp` over its intermediate slice.
 * p_f64 is [n_rows x H] (nullable); p_round receives bf16 (dtype 0, uint16)
 * or fp32 (dtype 1, float) roundings of p_f64. */
int oracle_shard_partial(const uint16_t *x, int64_t T, int64_t H, int64_t I,
                         const uint16_t *w_gate_up, const uint16_t *w_down,
                         int tp, int rank, const int64_t *rows, int64_t n_rows,
                         double *p_f64, void *p_round, int dtype, int nthreads);

/* out[t, n] = bf16_rne(sum_r partial_r[t, n]), r ascending, in double. */
void oracle_shard_sum(const void *partials, int dtype, int n_parts, int64_t T, int64_t H,
                      uint16_t *out);

/* out = round(sum_{r = rank_first .. rank_first + rank_count - 1} P_r), the fp64
 * partials summed r ascending before any rounding; out_f64 (nullable) is the sum,
 * out_round (nullable) its bf16 (dtype 0) or fp32 (dtype 1) rounding. */
int oracle_shard_group_sum(const uint16_t *x, int64_t T, int64_t H, int64_t I,
                           const uint16_t *w_gate_up, const uint16_t *w_down,
                           int tp, int rank_first, int rank_count,
                           const int64_t *rows, int64_t n_rows,
                           double *out_f64, void *out_round, int dtype, int nthreads);

/* Gathered (rank-major) column g  ->  logical column of [q_a | kv_a]. */
int oracle_rank_major_to_logical(int64_t q_dim, int64_t kv_dim, int tp, int64_t *logical_of_gathered);

/* Merged q_a/kv_a projection.  out_logical / out_rank_major are [n_rows x (q+kv)],
 * both nullable; out_f64 (nullable) holds the logical pre-rounding sums. */
int oracle_merged_proj(const uint16_t *x, int64_t T, int64_t H, const uint16_t *w,
                       int64_t q_dim, int64_t kv_dim, int tp,
                       const int64_t *rows, int64_t n_rows,
                       uint16_t *out_logical, uint16_t *out_rank_major, double *out_f64,
                       int nthreads);

/* Pure permutation of 16-bit words: logical[t, c(g)] = rank_major[t, g]. */
int oracle_reorder(const uint16_t *rank_major, uint16_t *logical, int64_t T,
                   int64_t q_dim, int64_t kv_dim, int tp);

#ifdef __cplusplus
}
#endif
#endif
