/*
 * attn_oracle.c -- plain, slow, fp64 reference for the fused attention forward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference arm may load this library.  The CUDA
 * product path never calls it and shares no code, header or table with it.
 *
 * What it computes (the plain definition, no blocking and no online rescaling):
 *   "PipeThreader: Software-Defined Pipelining for Efficient DNN Execution",
 *   section A2, paragraph "FlashAttention-3" with Fig. 7: the operator graph
 *   takes Q, K, V; MatMulQK gives acc_s = Q K^T; Softmax turns acc_s into P;
 *   MatMulPV multiplies P by V to give the output O.
 * The pages leave scale, mask, layout, grouped heads and the log-sum-exp open;
 * this file takes these readings:
 *   - scores are multiplied by `scale` before the mask and the softmax;
 *   - causal means key j is visible to query i iff j <= i (top-left aligned);
 *   - query head h uses key/value head h / (H_q / H_kv) (grouped heads);
 *   - LSE_i is the natural log of sum_{j visible} exp(scale * q_i . k_j);
 *   - tensors are contiguous [B, H, S, D]; LSE is [B, H_q, S_q].
 *
 * Inputs are bf16 bit patterns (uint16); each is widened to double exactly
 * (a bf16 is the top half of an IEEE float).  All arithmetic is fp64.
 * Parallelism is OpenMP over independent output rows only.
 *
 * Return codes: 0 ok, 1 invalid argument.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bf16_bits_to_double(uint16_t bits)
{
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

static int check_dims(int B, int Hq, int Hkv, int Sq, int Skv, int D)
{
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Skv <= 0 || D <= 0)
        return 1;
    if (Hq % Hkv != 0)
        return 1;
    return 0;
}

/* Number of keys row i may see: all S_kv keys, or keys 0..i when causal. */
static int64_t visible_keys(int64_t i, int Skv, int causal)
{
    if (!causal)
        return Skv;
    return (i + 1 < (int64_t)Skv) ? (i + 1) : (int64_t)Skv;
}

/*
 * One output row.  `flat_row` indexes [B, H_q, S_q].  `s` is scratch of S_kv
 * doubles.  Writes D values of O to `o_row`, and the LSE to `*lse_out`.
 * If `p_row` is non-null the S_kv softmax probabilities (0 for masked keys)
 * are written there too.
 */
static void one_row(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                    int Hq, int Hkv, int Sq, int Skv, int D, int causal,
                    double scale, int64_t flat_row, double *s, double *o_row,
                    double *lse_out, double *p_row)
{
    int64_t i = flat_row % Sq;
    int64_t bh = flat_row / Sq;
    int64_t h = bh % Hq;
    int64_t b = bh / Hq;
    int64_t hkv = h / (Hq / Hkv);

    const uint16_t *qi = q + ((b * Hq + h) * (int64_t)Sq + i) * D;
    const uint16_t *kb = k + (b * Hkv + hkv) * (int64_t)Skv * D;
    const uint16_t *vb = v + (b * Hkv + hkv) * (int64_t)Skv * D;
    int64_t nvis = visible_keys(i, Skv, causal);

    /* acc_s = scale * q_i . k_j over the visible keys */
    double m = -INFINITY;
    for (int64_t j = 0; j < nvis; ++j) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += bf16_bits_to_double(qi[d]) * bf16_bits_to_double(kb[j * D + d]);
        s[j] = scale * dot;
        if (s[j] > m)
            m = s[j];
    }
    /* softmax: p_j = exp(s_j - m) / l */
    double l = 0.0;
    for (int64_t j = 0; j < nvis; ++j) {
        s[j] = exp(s[j] - m);
        l += s[j];
    }
    /* O = P V */
    for (int d = 0; d < D; ++d)
        o_row[d] = 0.0;
    for (int64_t j = 0; j < nvis; ++j) {
        double pj = s[j] / l;
        for (int d = 0; d < D; ++d)
            o_row[d] += pj * bf16_bits_to_double(vb[j * D + d]);
    }
    *lse_out = m + log(l);
    if (p_row) {
        for (int64_t j = 0; j < Skv; ++j)
            p_row[j] = (j < nvis) ? s[j] / l : 0.0;
    }
}

/* Full forward: o [B,H_q,S_q,D] fp64, lse [B,H_q,S_q] fp64. */
int oracle_attn_fwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                    double *o, double *lse, int B, int Hq, int Hkv, int Sq,
                    int Skv, int D, int causal, double scale)
{
    if (check_dims(B, Hq, Hkv, Sq, Skv, D) || !q || !k || !v || !o || !lse)
        return 1;
    int64_t nrows = (int64_t)B * Hq * Sq;
    int bad = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)Skv);
        if (!s) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 16)
            for (int64_t r = 0; r < nrows; ++r)
                one_row(q, k, v, Hq, Hkv, Sq, Skv, D, causal, scale, r, s,
                        o + r * D, lse + r, NULL);
            free(s);
        }
    }
    return bad ? 1 : 0;
}

/*
 * Selected rows only: rows[n] are flat indices into [B, H_q, S_q]; writes
 * o_rows [n, D] and lse_rows [n].  Used to check full-size runs on a sample.
 */
int oracle_attn_rows(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                     const int64_t *rows, int64_t n, double *o_rows,
                     double *lse_rows, int B, int Hq, int Hkv, int Sq, int Skv,
                     int D, int causal, double scale)
{
    if (check_dims(B, Hq, Hkv, Sq, Skv, D) || !q || !k || !v || !rows ||
        !o_rows || !lse_rows || n < 0)
        return 1;
    int64_t nrows = (int64_t)B * Hq * Sq;
    for (int64_t t = 0; t < n; ++t)
        if (rows[t] < 0 || rows[t] >= nrows)
            return 1;
    int bad = 0;
#pragma omp parallel
    {
        double *s = (double *)malloc(sizeof(double) * (size_t)Skv);
        if (!s) {
#pragma omp atomic write
            bad = 1;
        } else {
#pragma omp for schedule(dynamic, 4)
            for (int64_t t = 0; t < n; ++t)
                one_row(q, k, v, Hq, Hkv, Sq, Skv, D, causal, scale, rows[t],
                        s, o_rows + t * D, lse_rows + t, NULL);
            free(s);
        }
    }
    return bad ? 1 : 0;
}

/*
 * Full probability matrix P [B, H_q, S_q, S_kv] (masked keys give 0) along
 * with O and LSE.  Meant for tiny sizes (row-sum and brute-force checks).
 */
int oracle_attn_probs(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                      double *p, double *o, double *lse, int B, int Hq,
                      int Hkv, int Sq, int Skv, int D, int causal, double scale)
{
    if (check_dims(B, Hq, Hkv, Sq, Skv, D) || !q || !k || !v || !p || !o ||
        !lse)
        return 1;
    int64_t nrows = (int64_t)B * Hq * Sq;
    double *s = (double *)malloc(sizeof(double) * (size_t)Skv);
    if (!s)
        return 1;
    for (int64_t r = 0; r < nrows; ++r)
        one_row(q, k, v, Hq, Hkv, Sq, Skv, D, causal, scale, r, s, o + r * D,
                lse + r, p + r * Skv);
    free(s);
    return 0;
}

/* Threads OpenMP will use (reported next to the CPU baseline's timing). */
int oracle_num_threads(void)
{
#ifdef _OPENMP
    extern int omp_get_max_threads(void);
    return omp_get_max_threads();
#else
    return 1;
#endif
}
