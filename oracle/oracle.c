/*
 * Plain fp64 CPU oracle for the Kimi-K3 shared-expert SwiGLU MLP.
 *
 * TEST INFRASTRUCTURE ONLY: the test suite, the smoke check and the bench's
 * CPU-baseline leg are the only callers.  Nothing here is shared with the CUDA
 * library (no header, helper, table or constant generator).
 *
 * What is computed, and where the pages define it:
 *   - the SwiGLU MLP  y = W_down (SiLU(W_gate x) * (W_up x)), hidden 7168 and
 *     shared intermediate 6144, gate_up a merged 12288-row weight
 *     ("[Kimi-K3] Add option to shard the shared expert instead of replicating",
 *     sections "Problem" and "Change"; prhub analysis of vllm PR #50656,
 *     section "关键源码片段": the replicated output is the activation of
 *     x @ cat([gate, up]).T, times down.T);
 *   - the shard partial of rank r over intermediate slice [r*s, (r+1)*s), s = I/tp,
 *     and the sum of partials (same prhub section: per-rank slices of gate, up
 *     and of the down columns, then stack(partials).sum(0)), either of partials
 *     already rounded to their storage dtype or of a group of shards' fp64
 *     partials rounded once;
 *   - the merged q_a/kv_a projection stored as column shards whose gathered
 *     output is rank-major and is reordered to logical [q_a | kv_a]
 *     ("[II] TP-shard Kimi MLA latent projections", sections "Behavior" and
 *     "Technical reason").
 *
 * Readings where the pages are silent (each one is listed in the design notes):
 *   - SiLU(z) = z / (1 + exp(-z)), no clamp; SiluAndMul = silu(first half) * second half.
 *   - g and u are not rounded before the activation; h is rounded to bf16 once,
 *     after the multiply.  Outputs are rounded fp64 -> bf16 directly with
 *     round-to-nearest-even.
 *   - Every reduction is a plain fp64 sum over its index in ascending order.
 *
 * Built with -ffp-contract=off so that x86 and Arm hosts give identical bits.
 */
#include "oracle.h"

#include <math.h>
#include <pthread.h>
#include <stdlib.h>
#include <string.h>

/* ------------------------------------------------------------------------- */
/* bf16 <-> double, from the IEEE-754 binary16-brain layout: 1 sign bit,     */
/* 8 exponent bits (bias 127), 7 fraction bits; i.e. the top half of fp32.   */
/* ------------------------------------------------------------------------- */

double oracle_bf16_to_f64(uint16_t b) {
    uint32_t u = (uint32_t)b << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f; /* exact: every bf16 value is an fp32 value */
}

/* Round a double to the nearest bf16 value, ties to even, directly (no
 * intermediate fp32 rounding).  The grid spacing is 2^(e-7) inside the binade
 * [2^e, 2^(e+1)) for e >= -126, and 2^-133 below (subnormals). */
uint16_t oracle_f64_to_bf16_rne(double d) {
    if (isnan(d)) return 0x7FC0;
    uint16_t sign = signbit(d) ? 0x8000 : 0;
    double a = fabs(d);
    if (isinf(a)) return sign | 0x7F80;
    if (a == 0.0) return sign;
    int e2;
    (void)frexp(a, &e2);      /* a = m * 2^e2, m in [0.5, 1) */
    int e = e2 - 1;           /* a in [2^e, 2^(e+1)) */
    if (e < -126) e = -126;   /* subnormal range shares the smallest spacing */
    double q = ldexp(1.0, e - 7);
    double n = a / q;         /* exact: q is a power of two */
    double fl = floor(n);
    double frac = n - fl;
    double r;
    if (frac > 0.5) r = fl + 1.0;
    else if (frac < 0.5) r = fl;
    else r = (fmod(fl, 2.0) == 0.0) ? fl : fl + 1.0;
    double v = r * q;         /* exactly representable in bf16, or 2^128 */
    if (v >= 0x1p128) return sign | 0x7F80;
    float f = (float)v;       /* exact */
    uint32_t u;
    memcpy(&u, &f, sizeof u);
    return sign | (uint16_t)(u >> 16);
}

double oracle_silu(double z) { return z / (1.0 + exp(-z)); }

/* ------------------------------------------------------------------------- */
/* a tiny parallel-for over [0, n) with static contiguous blocks             */
/* ------------------------------------------------------------------------- */

typedef void (*range_fn)(void *ctx, int64_t lo, int64_t hi);
typedef struct { range_fn fn; void *ctx; int64_t lo, hi; } range_job;

static void *range_thread(void *p) {
    range_job *j = (range_job *)p;
    j->fn(j->ctx, j->lo, j->hi);
    return NULL;
}

static void parallel_for(int64_t n, int nthreads, range_fn fn, void *ctx) {
    if (nthreads < 1) nthreads = 1;
    if (nthreads > 256) nthreads = 256;
    if ((int64_t)nthreads > n) nthreads = (int)(n > 0 ? n : 1);
    if (nthreads == 1) { fn(ctx, 0, n); return; }
    pthread_t th[256];
    range_job jobs[256];
    for (int i = 0; i < nthreads; ++i) {
        jobs[i].fn = fn; jobs[i].ctx = ctx;
        jobs[i].lo = n * i / nthreads; jobs[i].hi = n * (i + 1) / nthreads;
    }
    for (int i = 1; i < nthreads; ++i) pthread_create(&th[i], NULL, range_thread, &jobs[i]);
    range_thread(&jobs[0]);
    for (int i = 1; i < nthreads; ++i) pthread_join(th[i], NULL);
}

/* dot product of two bf16 rows of length K with stride 1, fp64, k ascending */
static double dot_bf16(const uint16_t *a, const uint16_t *b, int64_t K) {
    double s = 0.0;
    for (int64_t k = 0; k < K; ++k) s += oracle_bf16_to_f64(a[k]) * oracle_bf16_to_f64(b[k]);
    return s;
}

static int64_t row_of(const int64_t *rows, int64_t i) { return rows ? rows[i] : i; }

/* ------------------------------------------------------------------------- */
/* gate_up + SiluAndMul                                                      */
/* ------------------------------------------------------------------------- */

typedef struct {
    const uint16_t *x, *w; int64_t H, I, j0, j1; const int64_t *rows;
    uint16_t *h; double *g, *u;
} hid_ctx;

static void hid_range(void *p, int64_t lo, int64_t hi) {
    hid_ctx *c = (hid_ctx *)p;
    int64_t width = c->j1 - c->j0;
    for (int64_t e = lo; e < hi; ++e) {
        int64_t i = e / width, jj = e % width, j = c->j0 + jj;
        const uint16_t *xr = c->x + row_of(c->rows, i) * c->H;
        double g = dot_bf16(xr, c->w + j * c->H, c->H);            /* gate row j      */
        double u = dot_bf16(xr, c->w + (c->I + j) * c->H, c->H);   /* up row I + j    */
        double hv = oracle_silu(g) * u;
        c->h[i * width + jj] = oracle_f64_to_bf16_rne(hv);
        if (c->g) c->g[i * width + jj] = g;
        if (c->u) c->u[i * width + jj] = u;
    }
}

void oracle_swiglu_hidden(const uint16_t *x, int64_t T, int64_t H, int64_t I,
                          const uint16_t *w_gate_up, int64_t j_begin, int64_t j_end,
                          const int64_t *rows, int64_t n_rows,
                          uint16_t *h, double *g_out, double *u_out, int nthreads) {
    (void)T;
    hid_ctx c = {x, w_gate_up, H, I, j_begin, j_end, rows, h, g_out, u_out};
    parallel_for(n_rows * (j_end - j_begin), nthreads, hid_range, &c);
}

/* ------------------------------------------------------------------------- */
/* down projection over an intermediate slice [j0, j1)                       */
/* acc[i, n] = sum_{j in [j0,j1)} h[i, j - j0] * W_down[n, j]                 */
/* ------------------------------------------------------------------------- */

typedef struct {
    const uint16_t *h, *wd; int64_t H, I, j0, j1; double *acc;
} down_ctx;

static void down_range(void *p, int64_t lo, int64_t hi) {
    down_ctx *c = (down_ctx *)p;
    int64_t width = c->j1 - c->j0;
    for (int64_t e = lo; e < hi; ++e) {
        int64_t i = e / c->H, n = e % c->H;
        const uint16_t *hr = c->h + i * width;
        const uint16_t *wr = c->wd + n * c->I + c->j0;
        c->acc[e] = dot_bf16(hr, wr, width);
    }
}

static void down_slice(const uint16_t *h, int64_t n_rows, int64_t H, int64_t I,
                       const uint16_t *w_down, int64_t j0, int64_t j1, double *acc, int nthreads) {
    down_ctx c = {h, w_down, H, I, j0, j1, acc};
    parallel_for(n_rows * H, nthreads, down_range, &c);
}

void oracle_mlp_forward(const uint16_t *x, int64_t T, int64_t H, int64_t I,
                        const uint16_t *w_gate_up, const uint16_t *w_down,
                        const int64_t *rows, int64_t n_rows,
                        uint16_t *y, double *y_f64, uint16_t *h_out, int nthreads) {
    uint16_t *h = h_out ? h_out : (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(n_rows * I));
    double *acc = (double *)malloc(sizeof(double) * (size_t)(n_rows * H));
    oracle_swiglu_hidden(x, T, H, I, w_gate_up, 0, I, rows, n_rows, h, NULL, NULL, nthreads);
    down_slice(h, n_rows, H, I, w_down, 0, I, acc, nthreads);
    for (int64_t e = 0; e < n_rows * H; ++e) {
        if (y) y[e] = oracle_f64_to_bf16_rne(acc[e]);
        if (y_f64) y_f64[e] = acc[e];
    }
    free(acc);
    if (!h_out) free(h);
}

int oracle_shard_partial(const uint16_t *x, int64_t T, int64_t H, int64_t I,
                         const uint16_t *w_gate_up, const uint16_t *w_down,
                         int tp, int rank, const int64_t *rows, int64_t n_rows,
                         double *p_f64, void *p_round, int dtype, int nthreads) {
    if (tp <= 0 || rank < 0 || rank >= tp || I % tp != 0) return -1;
    int64_t s = I / tp, j0 = (int64_t)rank * s, j1 = j0 + s;
    uint16_t *h = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(n_rows * s));
    double *acc = (double *)malloc(sizeof(double) * (size_t)(n_rows * H));
    /* the shard's gate rows [j0, j1) and up rows I + [j0, j1) */
    oracle_swiglu_hidden(x, T, H, I, w_gate_up, j0, j1, rows, n_rows, h, NULL, NULL, nthreads);
    /* the shard's down columns [j0, j1) */
    down_slice(h, n_rows, H, I, w_down, j0, j1, acc, nthreads);
    for (int64_t e = 0; e < n_rows * H; ++e) {
        if (p_f64) p_f64[e] = acc[e];
        if (p_round) {
            if (dtype == 0) ((uint16_t *)p_round)[e] = oracle_f64_to_bf16_rne(acc[e]);
            else ((float *)p_round)[e] = (float)acc[e]; /* IEEE round-to-nearest-even */
        }
    }
    free(acc);
    free(h);
    return 0;
}

/* The summed partials of shards [rank_first, rank_first + rank_count) of tp: the
 * reduce-scatter's sum (Kimi-K3 PR, section "Change"; prhub section "关键源码片段",
 * stack(partials).sum(0)) taken over the shards' fp64 partials before any rounding,
 * r ascending, then rounded once.  This is the sum a GEMM epilogue that reduces
 * the partials itself produces: no partial is rounded to a storage dtype. */
int oracle_shard_group_sum(const uint16_t *x, int64_t T, int64_t H, int64_t I,
                           const uint16_t *w_gate_up, const uint16_t *w_down,
                           int tp, int rank_first, int rank_count,
                           const int64_t *rows, int64_t n_rows,
                           double *out_f64, void *out_round, int dtype, int nthreads) {
    if (tp <= 0 || I % tp != 0 || rank_first < 0 || rank_count < 1 || rank_first + rank_count > tp)
        return -1;
    double *sum = (double *)calloc((size_t)(n_rows * H), sizeof(double));
    double *part = (double *)malloc(sizeof(double) * (size_t)(n_rows * H));
    for (int r = rank_first; r < rank_first + rank_count; ++r) {
        oracle_shard_partial(x, T, H, I, w_gate_up, w_down, tp, r, rows, n_rows, part, NULL, 0, nthreads);
        for (int64_t e = 0; e < n_rows * H; ++e) sum[e] += part[e];
    }
    for (int64_t e = 0; e < n_rows * H; ++e) {
        if (out_f64) out_f64[e] = sum[e];
        if (out_round) {
            if (dtype == 0) ((uint16_t *)out_round)[e] = oracle_f64_to_bf16_rne(sum[e]);
            else ((float *)out_round)[e] = (float)sum[e];
        }
    }
    free(part);
    free(sum);
    return 0;
}

void oracle_shard_sum(const void *partials, int dtype, int n_parts, int64_t T, int64_t H,
                      uint16_t *out) {
    int64_t plane = T * H;
    for (int64_t e = 0; e < plane; ++e) {
        double s = 0.0;
        for (int r = 0; r < n_parts; ++r) {
            if (dtype == 0) s += oracle_bf16_to_f64(((const uint16_t *)partials)[r * plane + e]);
            else s += (double)((const float *)partials)[r * plane + e];
        }
        out[e] = oracle_f64_to_bf16_rne(s);
    }
}

/* ------------------------------------------------------------------------- */
/* merged q_a / kv_a projection                                              */
/* ------------------------------------------------------------------------- */

/* Rank r holds q_a rows [r*q/tp, (r+1)*q/tp) then kv_a rows [r*kv/tp, (r+1)*kv/tp);
 * the gather concatenates the ranks' local outputs in rank order. */
int oracle_rank_major_to_logical(int64_t q_dim, int64_t kv_dim, int tp, int64_t *logical_of_gathered) {
    if (tp <= 0 || q_dim % tp != 0 || kv_dim % tp != 0) return -1;
    int64_t qs = q_dim / tp, ks = kv_dim / tp, w = qs + ks;
    for (int r = 0; r < tp; ++r)
        for (int64_t l = 0; l < w; ++l)
            logical_of_gathered[r * w + l] = (l < qs) ? r * qs + l : q_dim + r * ks + (l - qs);
    return 0;
}

typedef struct {
    const uint16_t *x, *w; int64_t H, C; const int64_t *rows; double *acc;
} proj_ctx;

static void proj_range(void *p, int64_t lo, int64_t hi) {
    proj_ctx *c = (proj_ctx *)p;
    for (int64_t e = lo; e < hi; ++e) {
        int64_t i = e / c->C, col = e % c->C;
        c->acc[e] = dot_bf16(c->x + row_of(c->rows, i) * c->H, c->w + col * c->H, c->H);
    }
}

int oracle_merged_proj(const uint16_t *x, int64_t T, int64_t H, const uint16_t *w,
                       int64_t q_dim, int64_t kv_dim, int tp,
                       const int64_t *rows, int64_t n_rows,
                       uint16_t *out_logical, uint16_t *out_rank_major, double *out_f64,
                       int nthreads) {
    (void)T;
    int64_t C = q_dim + kv_dim;
    int64_t *map = (int64_t *)malloc(sizeof(int64_t) * (size_t)C);
    if (oracle_rank_major_to_logical(q_dim, kv_dim, tp, map) != 0) { free(map); return -1; }
    double *acc = (double *)malloc(sizeof(double) * (size_t)(n_rows * C));
    proj_ctx c = {x, w, H, C, rows, acc};
    parallel_for(n_rows * C, nthreads, proj_range, &c);
    for (int64_t i = 0; i < n_rows; ++i) {
        for (int64_t col = 0; col < C; ++col) {
            double v = acc[i * C + col];
            if (out_logical) out_logical[i * C + col] = oracle_f64_to_bf16_rne(v);
            if (out_f64) out_f64[i * C + col] = v;
        }
        if (out_rank_major)
            for (int64_t g = 0; g < C; ++g)
                out_rank_major[i * C + g] = oracle_f64_to_bf16_rne(acc[i * C + map[g]]);
    }
    free(acc);
    free(map);
    return 0;
}

int oracle_reorder(const uint16_t *rank_major, uint16_t *logical, int64_t T,
                   int64_t q_dim, int64_t kv_dim, int tp) {
    int64_t C = q_dim + kv_dim;
    int64_t *map = (int64_t *)malloc(sizeof(int64_t) * (size_t)C);
    if (oracle_rank_major_to_logical(q_dim, kv_dim, tp, map) != 0) { free(map); return -1; }
    for (int64_t t = 0; t < T; ++t)
        for (int64_t g = 0; g < C; ++g) logical[t * C + map[g]] = rank_major[t * C + g];
    free(map);
    return 0;
}
