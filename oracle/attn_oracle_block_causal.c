/*
 * FP64 CPU oracle, block-causal form.  TEST INFRASTRUCTURE ONLY, like
 * attn_oracle.c (built into the same library); shares no code with the CUDA
 * path.
 *
 * What it computes (page "Audit SGLang interfaces and refresh validated kernel
 * solutions", definitions/block_causal_attention/prefix_cached_block_causal_
 * h32_d128_prefix0.json, field "reference"): for Q, K, V [B, N, H, D] and
 * image_ids [N] (shared by the batch; -1 marks a text token), query i sees key
 * j iff j <= i (causal), or image_ids[i] == image_ids[j] with image_ids[i] >= 0
 * (tokens of one image see each other).  Scores q_i . k_j * D^-0.5 over the
 * visible keys, softmax, weighted sum of V.  The definition fills masked
 * scores with -inf before its softmax; here they are left out of both passes,
 * which is the same result.
 *
 * Arithmetic as in attn_oracle.c: exact bf16 -> double, naive two-pass
 * softmax, unrounded FP64 output; OpenMP over output rows only.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

/* bf16 is the top half of an IEEE binary32; widening is exact. */
static double bc_bf16_to_double(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

static int visible(const int32_t *image_ids, int64_t i, int64_t j)
{
    return j <= i || (image_ids[i] >= 0 && image_ids[j] == image_ids[i]);
}

/* One output row O[b, i, h, :]; `s` holds N doubles, `qd` and `acc` D each. */
static void block_causal_row(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                             const int32_t *image_ids, double *o_row, int64_t b, int64_t i,
                             int64_t h, int64_t N, int64_t H, int64_t D, double *s,
                             double *qd, double *acc)
{
    const double scale = pow((double)D, -0.5);
    const uint16_t *q = Q + ((b * N + i) * H + h) * D;
    for (int64_t d = 0; d < D; ++d)
        qd[d] = bc_bf16_to_double(q[d]);

    /* Pass 1: scores of the visible keys and their maximum. */
    double mx = -INFINITY;
    for (int64_t j = 0; j < N; ++j) {
        if (!visible(image_ids, i, j))
            continue;
        const uint16_t *kr = K + ((b * N + j) * H + h) * D;
        double dot = 0.0;
        for (int64_t d = 0; d < D; ++d)
            dot += qd[d] * bc_bf16_to_double(kr[d]);
        s[j] = dot * scale;
        if (s[j] > mx)
            mx = s[j];
    }

    /* Pass 2: weights exp(s_j - max) of the visible keys, normalised sum of V. */
    double total = 0.0;
    for (int64_t d = 0; d < D; ++d)
        acc[d] = 0.0;
    for (int64_t j = 0; j < N; ++j) {
        if (!visible(image_ids, i, j))
            continue;
        const double wj = exp(s[j] - mx);
        const uint16_t *vr = V + ((b * N + j) * H + h) * D;
        total += wj;
        for (int64_t d = 0; d < D; ++d)
            acc[d] += wj * bc_bf16_to_double(vr[d]);
    }
    for (int64_t d = 0; d < D; ++d)
        o_row[d] = acc[d] / total;
}

/* Rows listed by flat index r = (b * N + i) * H + h; output [nrows, D]. */
int oracle_block_causal_attention_rows(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                                       const int32_t *image_ids, double *O_rows, int B, int N,
                                       int H, int D, const int64_t *rows, int64_t nrows)
{
    if (!Q || !K || !V || !image_ids || !O_rows || (nrows > 0 && !rows))
        return -1;
    if (B < 1 || N < 1 || H < 1 || D < 1)
        return -2;
    const int64_t total = (int64_t)B * N * H;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= total)
            return -2;
    int failed = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)N);
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
                const int64_t i = (flat / H) % N;
                const int64_t b = flat / ((int64_t)H * N);
                block_causal_row(Q, K, V, image_ids, O_rows + r * D, b, i, h, N, H, D, s, qd,
                                 acc);
            }
        }
        free(s);
        free(qd);
        free(acc);
    }
    return failed ? -3 : 0;
}

/* Full output O [B, N, H, D]. */
int oracle_block_causal_attention(const uint16_t *Q, const uint16_t *K, const uint16_t *V,
                                  const int32_t *image_ids, double *O, int B, int N, int H, int D)
{
    if (!Q || !K || !V || !image_ids || !O)
        return -1;
    if (B < 1 || N < 1 || H < 1 || D < 1)
        return -2;
    const int64_t total = (int64_t)B * N * H;
    int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)total);
    if (!rows)
        return -3;
    for (int64_t r = 0; r < total; ++r)
        rows[r] = r;
    int rc = oracle_block_causal_attention_rows(Q, K, V, image_ids, O, B, N, H, D, rows, total);
    free(rows);
    return rc;
}
