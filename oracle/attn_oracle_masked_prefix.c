/*
 * FP64 CPU oracle, masked prefix-cached form.  TEST INFRASTRUCTURE ONLY, like
 * attn_oracle.c (built into the same library); shares no code with the CUDA
 * path.
 *
 * What it computes: the earlier ("old") form of the page "Audit SGLang
 * interfaces and refresh validated kernel solutions",
 * definitions/block_causal_attention/prefix_cached_block_causal_h32_d128.json,
 * field "reference" as it stood before the audit.  Inputs Q, K_current,
 * V_current [B, Nq, H, D], K_prefix, V_prefix [B, Np, H, D], image_ids [Nall]
 * (Nall = Np + Nq, shared by the batch, -1 = text), key_valid [B, Nall] and a
 * runtime sm_scale.  Keys and values are cat(prefix, current) on the token
 * axis; query i sits at position Np + i.  Key j is visible to query i of batch
 * b iff (j <= Np + i, or image_ids[Np + i] >= 0 and image_ids[j] ==
 * image_ids[Np + i]) and key_valid[b, j].  Scores q . k_j * sm_scale over the
 * visible keys, softmax, weighted sum of V.  The definition asserts that every
 * query sees a key; here a row without one makes the call fail (-4).
 *
 * Arithmetic as in attn_oracle.c: exact bf16 -> double, naive two-pass
 * softmax, unrounded FP64 output; OpenMP over output rows only.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double mp_bf16(uint16_t bits)
{
    uint32_t u = (uint32_t)bits << 16;
    float f;
    memcpy(&f, &u, sizeof f);
    return (double)f;
}

/* Key row j of cat(prefix, current) for batch b and head h. */
static const uint16_t *mp_key_row(const uint16_t *Xc, const uint16_t *Xp, int64_t b, int64_t j,
                                  int64_t h, int64_t Nq, int64_t Np, int64_t H, int64_t D)
{
    if (j < Np)
        return Xp + ((b * Np + j) * H + h) * D;
    return Xc + ((b * Nq + (j - Np)) * H + h) * D;
}

static int mp_visible(const int32_t *image_ids, const uint8_t *key_valid, int64_t b, int64_t qpos,
                      int64_t j, int64_t Nall)
{
    const int causal_or_image =
        j <= qpos || (image_ids[qpos] >= 0 && image_ids[j] == image_ids[qpos]);
    return causal_or_image && key_valid[b * Nall + j] != 0;
}

static int masked_prefix_row(const uint16_t *Q, const uint16_t *Kc, const uint16_t *Vc,
                             const uint16_t *Kp, const uint16_t *Vp, const int32_t *image_ids,
                             const uint8_t *key_valid, double scale, double *o_row, int64_t b,
                             int64_t i, int64_t h, int64_t Nq, int64_t Np, int64_t H, int64_t D,
                             double *s, double *qd, double *acc)
{
    const int64_t Nall = Np + Nq, qpos = Np + i;
    const uint16_t *q = Q + ((b * Nq + i) * H + h) * D;
    for (int64_t d = 0; d < D; ++d)
        qd[d] = mp_bf16(q[d]);

    /* Pass 1: scores of the visible keys and their maximum. */
    double top = -INFINITY;
    int64_t seen = 0;
    for (int64_t j = 0; j < Nall; ++j) {
        if (!mp_visible(image_ids, key_valid, b, qpos, j, Nall))
            continue;
        const uint16_t *kr = mp_key_row(Kc, Kp, b, j, h, Nq, Np, H, D);
        double dot = 0.0;
        for (int64_t d = 0; d < D; ++d)
            dot += qd[d] * mp_bf16(kr[d]);
        s[j] = dot * scale;
        if (s[j] > top)
            top = s[j];
        ++seen;
    }
    if (seen == 0)
        return -4;

    /* Pass 2: exp(s_j - top) over the visible keys, normalised weighted sum of V. */
    double denom = 0.0;
    for (int64_t d = 0; d < D; ++d)
        acc[d] = 0.0;
    for (int64_t j = 0; j < Nall; ++j) {
        if (!mp_visible(image_ids, key_valid, b, qpos, j, Nall))
            continue;
        const double e = exp(s[j] - top);
        const uint16_t *vr = mp_key_row(Vc, Vp, b, j, h, Nq, Np, H, D);
        denom += e;
        for (int64_t d = 0; d < D; ++d)
            acc[d] += e * mp_bf16(vr[d]);
    }
    for (int64_t d = 0; d < D; ++d)
        o_row[d] = acc[d] / denom;
    return 0;
}

/* Rows listed by flat index r = (b * Nq + i) * H + h; output [nrows, D]. */
int oracle_masked_prefix_attention_rows(const uint16_t *Q, const uint16_t *K_current,
                                        const uint16_t *V_current, const uint16_t *K_prefix,
                                        const uint16_t *V_prefix, const int32_t *image_ids,
                                        const uint8_t *key_valid, float sm_scale,
                                        double *O_rows, int B, int Nq, int Np, int H, int D,
                                        const int64_t *rows, int64_t nrows)
{
    if (!Q || !K_current || !V_current || !image_ids || !key_valid || !O_rows ||
        (Np > 0 && (!K_prefix || !V_prefix)) || (nrows > 0 && !rows))
        return -1;
    if (B < 1 || Nq < 1 || Np < 0 || H < 1 || D < 1)
        return -2;
    const int64_t total = (int64_t)B * Nq * H, Nall = (int64_t)Np + Nq;
    for (int64_t r = 0; r < nrows; ++r)
        if (rows[r] < 0 || rows[r] >= total)
            return -2;
    int failed = 0, empty = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)Nall);
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
                if (masked_prefix_row(Q, K_current, V_current, K_prefix, V_prefix, image_ids,
                                      key_valid, (double)sm_scale, O_rows + r * D, b, i, h, Nq,
                                      Np, H, D, s, qd, acc) != 0) {
#pragma omp atomic write
                    empty = 1;
                }
            }
        }
        free(s);
        free(qd);
        free(acc);
    }
    return failed ? -3 : (empty ? -4 : 0);
}

/* Full output O [B, Nq, H, D]. */
int oracle_masked_prefix_attention(const uint16_t *Q, const uint16_t *K_current,
                                   const uint16_t *V_current, const uint16_t *K_prefix,
                                   const uint16_t *V_prefix, const int32_t *image_ids,
                                   const uint8_t *key_valid, float sm_scale, double *O, int B,
                                   int Nq, int Np, int H, int D)
{
    if (!Q || !O)
        return -1;
    if (B < 1 || Nq < 1 || H < 1 || D < 1)
        return -2;
    const int64_t total = (int64_t)B * Nq * H;
    int64_t *rows = (int64_t *)malloc(sizeof(int64_t) * (size_t)total);
    if (!rows)
        return -3;
    for (int64_t r = 0; r < total; ++r)
        rows[r] = r;
    int rc = oracle_masked_prefix_attention_rows(Q, K_current, V_current, K_prefix, V_prefix,
                                                 image_ids, key_valid, sm_scale, O, B, Nq, Np, H,
                                                 D, rows, total);
    free(rows);
    return rc;
}
