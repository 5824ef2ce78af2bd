/*
 * FP64 CPU oracle for the BF16 attention leaf.  TEST INFRASTRUCTURE ONLY:
 * only the tests, the smoke check and the bench's CPU-baseline leg may load
 * this file's library.  It shares no code with the CUDA path.
 *
 * What it computes (page "Audit SGLang interfaces and refresh validated kernel
 * solutions"):
 *   - definitions/dense_attention/noncausal_dense_attention_h32_d128.json and
 *     ..._h32_d64.json, field "reference": for Q [B,Nq,H,D], K,V [B,Nk,H,D],
 *     scores = einsum(bqhd,bkhd->bhqk)(Q,K) * D^-0.5, probabilities =
 *     softmax over k, O = einsum(bhqk,bkhd->bqhd)(probabilities, V).  No mask;
 *     the description allows cross attention (Nq != Nk).
 *   - definitions/block_causal_attention/prefix_cached_block_causal_h32_d128
 *     .json, field "reference": keys = cat(K_prefix, K_current) and values =
 *     cat(V_prefix, V_current) along the token axis, then the same attention
 *     with every key visible and scale 128^-0.5.
 *
 * Arithmetic: every bf16 input is widened exactly to double; the score row is
 * formed in double, the softmax is the naive two-pass form (max, then
 * exp(s - max), sum, weighted sum of V, divide), and the result is returned
 * unrounded in double.  The definitions evaluate in FP32 and round the output
 * to bf16; the oracle keeps FP64 and leaves rounding to the comparison.
 *
 * Parallelism: OpenMP over independent output rows (b, i, h) only.  No
 * blocking, no fusion, no online softmax.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>
#ifdef _OPENMP
#include <omp.h>
#endif

/* bf16 is the top half of an IEEE binary32; widening is exact. */
static double bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/*
 * One output row: O[b, i, h, :] for query row i of batch b and head h, over
 * Nk keys of K/V laid out [B, Nk, H, D].  `s` is caller scratch of Nk doubles,
 * `qd` of D doubles, `acc` of D doubles.
 */
static void attention_row(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                          double *o_row, int64_t b, int64_t i, int64_t h,
                          int64_t Nq, int64_t Nk, int64_t H, int64_t D,
                          double *s, double *qd, double *acc)
{
    const double scale = pow((double)D, -0.5);
    const uint16_t *q = Q + ((b * Nq + i) * H + h) * D;
    for (int64_t d = 0; d < D; ++d)
        qd[d] = bf16_to_double(q[d]);

    /* Pass 1: scores s_j = (q . k_j) * D^-0.5 and their maximum. */
    double m = -INFINITY;
    for (int64_t j = 0; j < Nk; ++j) {
        const uint16_t *k = K + ((b * Nk + j) * H + h) * D;
        double dot = 0.0;
        for (int64_t d = 0; d < D; ++d)
            dot += qd[d] * bf16_to_double(k[d]);
        s[j] = dot * scale;
        if (s[j] > m)
            m = s[j];
    }

    /* Pass 2: w_j = exp(s_j - m), l = sum w_j, o = sum w_j v_j / l. */
    double l = 0.0;
    for (int64_t d = 0; d < D; ++d)
        acc[d] = 0.0;
    for (int64_t j = 0; j < Nk; ++j) {
        const double w = exp(s[j] - m);
        const uint16_t *v = V + ((b * Nk + j) * H + h) * D;
        l += w;
        for (int64_t d = 0; d < D; ++d)
            acc[d] += w * bf16_to_double(v[d]);
    }
    for (int64_t d = 0; d < D; ++d)
        o_row[d] = acc[d] / l;
}

static int check_shape(int B, int Nq, int Nk, int H, int D)
{
    return (B >= 1 && Nq >= 1 && Nk >= 1 && H >= 1 && D >= 1) ? 0 : -2;
}

/*
 * Rows listed by flat index r = (b * Nq + i) * H + h; output [nrows, D].
 * The full-output entry points below call this with every row.
 */
int oracle_dense_attention_rows(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                                double *O_rows, int B, int Nq, int Nk, int H, int D,
                                const int64_t *rows, int64_t nrows)
{
    if (!Q || !K || !V || !O_rows || (nrows > 0 && !rows))
        return -1;
    if (check_shape(B, Nq, Nk, H, D))
        return -2;
    const int64_t total = (int64_t)B * Nq * H;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= total)
            return -2;
    int failed = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)Nk);
        double *qd = (double *)malloc(sizeof(double) * (size_t)D);
        double *acc = (double *)malloc(sizeof(double) * (size_t)D);
        if (!s || !qd || !acc) {
#pragma omp atomic write
            failed = 1;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (int64_t r = 0; r < nrows; ++r) {
                const int64_t flat = rows[r];
                const int64_t h = flat % H;
                const int64_t i = (flat / H) % Nq;
                const int64_t b = flat / ((int64_t)H * Nq);
                attention_row(Q, K, V, O_rows + r * D, b, i, h, Nq, Nk, H, D, s, qd, acc);
            }
        }
        free(s);
        free(qd);
        free(acc);
    }
    return failed ? -3 : 0;
}

/* Full output O [B, Nq, H, D] of dense (self or cross) attention. */
int oracle_dense_attention(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                           double *O, int B, int Nq, int Nk, int H, int D)
{
    if (!Q || !K || !V || !O)
        return -1;
    if (check_shape(B, Nq, Nk, H, D))
        return -2;
    const int64_t total = (int64_t)B * Nq * H;
    int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)total);
    if (!rows)
        return -3;
    for (int64_t r = 0; r < total; ++r)
        rows[r] = r;
    int rc = oracle_dense_attention_rows(Q, K, V, O, B, Nq, Nk, H, D, rows, total);
    free(rows);
    return rc;
}

/*
 * cat(X_prefix, X_current) along the token axis: [B,Np,H,D] ++ [B,Nc,H,D]
 * -> [B,Np+Nc,H,D], prefix tokens first (torch.cat(..., dim=1)).
 */
static uint16_t *concat_tokens(const uint16_t *Xp, const uint16_t *Xc,
                               int64_t B, int64_t Np, int64_t Nc, int64_t H, int64_t D)
{
    const int64_t row = H * D, Nall = Np + Nc;
    uint16_t *out = (uint16_t *)malloc(sizeof(uint16_t) * (size_t)(B * Nall * row));
    if (!out)
        return NULL;
    for (int64_t b = 0; b < B; ++b) {
        if (Np > 0)
            memcpy(out + b * Nall * row, Xp + b * Np * row, sizeof(uint16_t) * (size_t)(Np * row));
        memcpy(out + (b * Nall + Np) * row, Xc + b * Nc * row, sizeof(uint16_t) * (size_t)(Nc * row));
    }
    return out;
}

/*
 * Prefix-cached full-visibility attention, rows listed as in
 * oracle_dense_attention_rows.  Np may be 0 (then the keys are the current
 * keys alone); Nc >= 1.
 */
int oracle_prefix_attention_rows(const uint16_t *Q, const uint16_t *K_prefix,
                                 const uint16_t *V_prefix, const uint16_t *K_current,
                                 const uint16_t *V_current, double *O_rows, int B, int Nq,
                                 int Np, int Nc, int H, int D, const int64_t *rows,
                                 int64_t nrows)
{
    if (!Q || !K_current || !V_current || !O_rows || (Np > 0 && (!K_prefix || !V_prefix)))
        return -1;
    if (Np < 0 || check_shape(B, Nq, Nc, H, D))
        return -2;
    uint16_t *keys = concat_tokens(K_prefix, K_current, B, Np, Nc, H, D);
    uint16_t *values = concat_tokens(V_prefix, V_current, B, Np, Nc, H, D);
    int rc = -3;
    if (keys && values)
        rc = oracle_dense_attention_rows(Q, keys, values, O_rows, B, Nq, Np + Nc, H, D,
                                         rows, nrows);
    free(keys);
    free(values);
    return rc;
}

/* Full output O [B, Nq, H, D] of the prefix-cached form. */
int oracle_prefix_attention(const uint16_t *Q, const uint16_t *K_prefix,
                            const uint16_t *V_prefix, const uint16_t *K_current,
                            const uint16_t *V_current, double *O, int B, int Nq, int Np,
                            int Nc, int H, int D)
{
    if (!Q || !O)
        return -1;
    if (check_shape(B, Nq, Nc, H, D))
        return -2;
    const int64_t total = (int64_t)B * Nq * H;
    int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)total);
    if (!rows)
        return -3;
    for (int64_t r = 0; r < total; ++r)
        rows[r] = r;
    int rc = oracle_prefix_attention_rows(Q, K_prefix, V_prefix, K_current, V_current, O,
                                          B, Nq, Np, Nc, H, D, rows, total);
    free(rows);
    return rc;
}

/* Threads the parallel regions use (0 leaves the OpenMP default). */
void oracle_set_threads(int n)
{
#ifdef _OPENMP
    if (n > 0)
        omp_set_num_threads(n);
#else
    (void)n;
#endif
}

int oracle_max_threads(void)
{
#ifdef _OPENMP
    return omp_get_max_threads();
#else
    return 1;
#endif
}
