/*
 * attn_bwd_oracle.c -- plain, slow, fp64 reference for the attention backward.
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite, the smoke check and the
 * benchmark's CPU-baseline / reference arm may load this library.  The CUDA
 * product path never calls it and shares no code, header or table with it.
 *
 * What it computes: the gradients of L = sum_{b,h,i,d} O[b,h,i,d] dO[b,h,i,d]
 * with respect to Q, K and V, where O is the attention forward of
 * "PipeThreader: Software-Defined Pipelining for Efficient DNN Execution",
 * section A2, paragraph "FlashAttention-3" and Fig. 7 (acc_s = Q K^T ->
 * Softmax -> P -> P V = O), with the forward oracle's readings (scale before
 * the mask, causal j <= i, query head h on key/value head h / (H_q / H_kv),
 * [B, H, S, D] layout).  The backward pass itself is the subject of
 * "GPU软件流水线与Warp Specialization优化技术解析", section 3.2, which names
 * no formulas; these are the chain rule through the definition, per row i of
 * one query head:
 *   P_ij  = exp(s_ij - m_i) / l_i                (the forward's softmax)
 *   O_i   = sum_j P_ij v_j
 *   dP_ij = dO_i . v_j
 *   D_i   = dO_i . O_i  (= sum_j P_ij dP_ij)
 *   dS_ij = P_ij (dP_ij - D_i)
 *   dQ_i  = scale sum_j dS_ij k_j
 *   dK_j += scale dS_ij q_i      (summed over rows and over the query heads
 *   dV_j += P_ij dO_i             sharing the key/value head)
 * No blocking, no recomputation tricks: every row is formed from scratch.
 *
 * Two input forms: bf16 bit patterns (uint16, widened exactly, as the GPU
 * path consumes them) and fp64 arrays (for finite-difference checks of the
 * gradients against the forward definition, which needs perturbations far
 * below bf16 resolution).  All arithmetic is fp64.  Parallelism is OpenMP
 * over independent key/value heads (or independent rows) only.
 *
 * Return codes: 0 ok, 1 invalid argument.
 */
#include <math.h>
#include <stdint.h>
#include <stdlib.h>
#include <string.h>

static double bwd_bf16_to_double(uint16_t bits)
{
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

static int bwd_check_dims(int B, int Hq, int Hkv, int Sq, int Skv, int D)
{
    if (B <= 0 || Hq <= 0 || Hkv <= 0 || Sq <= 0 || Skv <= 0 || D <= 0)
        return 1;
    if (Hq % Hkv != 0)
        return 1;
    return 0;
}

static int64_t bwd_visible(int64_t i, int Skv, int causal)
{
    if (!causal)
        return Skv;
    return (i + 1 < (int64_t)Skv) ? (i + 1) : (int64_t)Skv;
}

static double *widen(const uint16_t *x, size_t n)
{
    double *y = (double *)malloc(sizeof(double) * (n ? n : 1));
    if (!y)
        return NULL;
    for (size_t t = 0; t < n; ++t)
        y[t] = bwd_bf16_to_double(x[t]);
    return y;
}

/*
 * Softmax row of query row i of head h (batch b): p[j] for j < nvis (the
 * rest 0), the output row o[D] and D_i = dO_i . O_i.  Returns nvis.
 */
static int64_t bwd_row(const double *q, const double *k, const double *v,
                       const double *dout, int Hq, int Hkv, int Sq, int Skv,
                       int D, int causal, double scale, int64_t b, int64_t h,
                       int64_t i, double *p, double *o, double *delta)
{
    int64_t hkv = h / (Hq / Hkv);
    const double *qi = q + ((b * Hq + h) * (int64_t)Sq + i) * D;
    const double *doi = dout + ((b * Hq + h) * (int64_t)Sq + i) * D;
    const double *kb = k + (b * Hkv + hkv) * (int64_t)Skv * D;
    const double *vb = v + (b * Hkv + hkv) * (int64_t)Skv * D;
    int64_t nvis = bwd_visible(i, Skv, causal);
    double m = -INFINITY;
    for (int64_t j = 0; j < nvis; ++j) {
        double dot = 0.0;
        for (int d = 0; d < D; ++d)
            dot += qi[d] * kb[j * D + d];
        p[j] = scale * dot;
        if (p[j] > m)
            m = p[j];
    }
    double l = 0.0;
    for (int64_t j = 0; j < nvis; ++j) {
        p[j] = exp(p[j] - m);
        l += p[j];
    }
    for (int64_t j = 0; j < nvis; ++j)
        p[j] /= l;
    for (int64_t j = nvis; j < Skv; ++j)
        p[j] = 0.0;
    for (int d = 0; d < D; ++d)
        o[d] = 0.0;
    for (int64_t j = 0; j < nvis; ++j)
        for (int d = 0; d < D; ++d)
            o[d] += p[j] * vb[j * D + d];
    double dl = 0.0;
    for (int d = 0; d < D; ++d)
        dl += doi[d] * o[d];
    *delta = dl;
    return nvis;
}

/*
 * All gradients for fp64 inputs.  q, dout, dq: [B, H_q, S_q, D]; k, v, dk,
 * dv: [B, H_kv, S_kv, D].
 */
int oracle_attn_bwd_f64(const double *q, const double *k, const double *v,
                        const double *dout, double *dq, double *dk, double *dv,
                        int B, int Hq, int Hkv, int Sq, int Skv, int D,
                        int causal, double scale)
{
    if (bwd_check_dims(B, Hq, Hkv, Sq, Skv, D) || !q || !k || !v || !dout ||
        !dq || !dk || !dv)
        return 1;
    int64_t groups = (int64_t)B * Hkv;
    int bad = 0;
#pragma omp parallel
    {
        double *p = (double *)malloc(sizeof(double) * (size_t)Skv);
        double *o = (double *)malloc(sizeof(double) * (size_t)D);
        /* every thread takes part in the loop; one without scratch only
         * records the failure */
#pragma omp for schedule(dynamic, 1)
        for (int64_t g = 0; g < groups; ++g) {
            if (!p || !o) {
#pragma omp atomic write
                bad = 1;
                continue;
            }
            {
                int64_t b = g / Hkv;
                int64_t hkv = g % Hkv;
                double *dkb = dk + g * (int64_t)Skv * D;
                double *dvb = dv + g * (int64_t)Skv * D;
                const double *kb = k + g * (int64_t)Skv * D;
                const double *vb = v + g * (int64_t)Skv * D;
                memset(dkb, 0, sizeof(double) * (size_t)Skv * D);
                memset(dvb, 0, sizeof(double) * (size_t)Skv * D);
                int rep = Hq / Hkv;
                for (int64_t h = hkv * rep; h < (hkv + 1) * rep; ++h) {
                    for (int64_t i = 0; i < Sq; ++i) {
                        double delta;
                        int64_t nvis = bwd_row(q, k, v, dout, Hq, Hkv, Sq, Skv,
                                               D, causal, scale, b, h, i, p, o,
                                               &delta);
                        int64_t row = (b * Hq + h) * (int64_t)Sq + i;
                        const double *qi = q + row * D;
                        const double *doi = dout + row * D;
                        double *dqi = dq + row * D;
                        for (int d = 0; d < D; ++d)
                            dqi[d] = 0.0;
                        for (int64_t j = 0; j < nvis; ++j) {
                            double dp = 0.0;
                            for (int d = 0; d < D; ++d)
                                dp += doi[d] * vb[j * D + d];
                            double ds = p[j] * (dp - delta);
                            for (int d = 0; d < D; ++d) {
                                dqi[d] += scale * ds * kb[j * D + d];
                                dkb[j * D + d] += scale * ds * qi[d];
                                dvb[j * D + d] += p[j] * doi[d];
                            }
                        }
                    }
                }
            }
        }
        free(p);
        free(o);
    }
    return bad ? 1 : 0;
}

/* The same for bf16 inputs (the GPU path's operands). */
int oracle_attn_bwd(const uint16_t *q, const uint16_t *k, const uint16_t *v,
                    const uint16_t *dout, double *dq, double *dk, double *dv,
                    int B, int Hq, int Hkv, int Sq, int Skv, int D, int causal,
                    double scale)
{
    if (bwd_check_dims(B, Hq, Hkv, Sq, Skv, D) || !q || !k || !v || !dout ||
        !dq || !dk || !dv)
        return 1;
    size_t nq = (size_t)B * Hq * Sq * D, nk = (size_t)B * Hkv * Skv * D;
    double *qd = widen(q, nq), *kd = widen(k, nk), *vd = widen(v, nk),
           *dod = widen(dout, nq);
    int rc = 1;
    if (qd && kd && vd && dod)
        rc = oracle_attn_bwd_f64(qd, kd, vd, dod, dq, dk, dv, B, Hq, Hkv, Sq,
                                 Skv, D, causal, scale);
    free(qd);
    free(kd);
    free(vd);
    free(dod);
    return rc;
}

/*
 * The forward for fp64 inputs: o [B, H_q, S_q, D], lse [B, H_q, S_q].  The
 * finite-difference checks differentiate L = sum O dO through this.
 */
int oracle_attn_fwd_f64(const double *q, const double *k, const double *v,
                        double *o, double *lse, int B, int Hq, int Hkv, int Sq,
                        int Skv, int D, int causal, double scale)
{
    if (bwd_check_dims(B, Hq, Hkv, Sq, Skv, D) || !q || !k || !v || !o || !lse)
        return 1;
    int64_t nrows = (int64_t)B * Hq * Sq;
    double *s = (double *)malloc(sizeof(double) * (size_t)Skv);
    if (!s)
        return 1;
    for (int64_t r = 0; r < nrows; ++r) {
        int64_t i = r % Sq, bh = r / Sq, h = bh % Hq, b = bh / Hq;
        int64_t hkv = h / (Hq / Hkv);
        const double *qi = q + r * D;
        const double *kb = k + (b * Hkv + hkv) * (int64_t)Skv * D;
        const double *vb = v + (b * Hkv + hkv) * (int64_t)Skv * D;
        int64_t nvis = bwd_visible(i, Skv, causal);
        double m = -INFINITY;
        for (int64_t j = 0; j < nvis; ++j) {
            double dot = 0.0;
            for (int d = 0; d < D; ++d)
                dot += qi[d] * kb[j * D + d];
            s[j] = scale * dot;
            if (s[j] > m)
                m = s[j];
        }
        double l = 0.0;
        for (int64_t j = 0; j < nvis; ++j) {
            s[j] = exp(s[j] - m);
            l += s[j];
        }
        for (int d = 0; d < D; ++d) {
            double acc = 0.0;
            for (int64_t j = 0; j < nvis; ++j)
                acc += s[j] / l * vb[j * D + d];
            o[r * D + d] = acc;
        }
        lse[r] = m + log(l);
    }
    free(s);
    return 0;
}

/*
 * dQ of selected query rows (flat indices into [B, H_q, S_q]) for bf16
 * inputs: dq_rows [n, D].  Each row needs only its own softmax row.
 */
int oracle_attn_bwd_dq_rows(const uint16_t *q, const uint16_t *k,
                            const uint16_t *v, const uint16_t *dout,
                            const int64_t *rows, int64_t n, double *dq_rows,
                            int B, int Hq, int Hkv, int Sq, int Skv, int D,
                            int causal, double scale)
{
    if (bwd_check_dims(B, Hq, Hkv, Sq, Skv, D) || !q || !k || !v || !dout ||
        !rows || !dq_rows || n < 0)
        return 1;
    int64_t nrows = (int64_t)B * Hq * Sq;
    for (int64_t t = 0; t < n; ++t)
        if (rows[t] < 0 || rows[t] >= nrows)
            return 1;
    size_t nq = (size_t)B * Hq * Sq * D, nk = (size_t)B * Hkv * Skv * D;
    double *qd = widen(q, nq), *kd = widen(k, nk), *vd = widen(v, nk),
           *dod = widen(dout, nq);
    int bad = !(qd && kd && vd && dod);
    if (!bad) {
#pragma omp parallel
        {
            double *p = (double *)malloc(sizeof(double) * (size_t)Skv);
            double *o = (double *)malloc(sizeof(double) * (size_t)D);
#pragma omp for schedule(dynamic, 1)
            for (int64_t t = 0; t < n; ++t) {
                if (!p || !o) {
#pragma omp atomic write
                    bad = 1;
                    continue;
                }
                {
                    int64_t r = rows[t];
                    int64_t i = r % Sq, bh = r / Sq, h = bh % Hq, b = bh / Hq;
                    int64_t hkv = h / (Hq / Hkv);
                    const double *kb = kd + (b * Hkv + hkv) * (int64_t)Skv * D;
                    const double *vb = vd + (b * Hkv + hkv) * (int64_t)Skv * D;
                    const double *doi = dod + r * D;
                    double delta;
                    int64_t nvis = bwd_row(qd, kd, vd, dod, Hq, Hkv, Sq, Skv, D,
                                           causal, scale, b, h, i, p, o, &delta);
                    double *out = dq_rows + t * D;
                    for (int d = 0; d < D; ++d)
                        out[d] = 0.0;
                    for (int64_t j = 0; j < nvis; ++j) {
                        double dp = 0.0;
                        for (int d = 0; d < D; ++d)
                            dp += doi[d] * vb[j * D + d];
                        double ds = p[j] * (dp - delta);
                        for (int d = 0; d < D; ++d)
                            out[d] += scale * ds * kb[j * D + d];
                    }
                }
            }
            free(p);
            free(o);
        }
    }
    free(qd);
    free(kd);
    free(vd);
    free(dod);
    return bad ? 1 : 0;
}

/*
 * dK and dV of selected key rows (flat indices into [B, H_kv, S_kv]) for
 * bf16 inputs: dk_rows, dv_rows [n, D].  Every query row of the key's group
 * contributes, so each needed group's softmax rows are all formed once.
 */
int oracle_attn_bwd_dkv_rows(const uint16_t *q, const uint16_t *k,
                             const uint16_t *v, const uint16_t *dout,
                             const int64_t *rows, int64_t n, double *dk_rows,
                             double *dv_rows, int B, int Hq, int Hkv, int Sq,
                             int Skv, int D, int causal, double scale)
{
    if (bwd_check_dims(B, Hq, Hkv, Sq, Skv, D) || !q || !k || !v || !dout ||
        !rows || !dk_rows || !dv_rows || n < 0)
        return 1;
    int64_t nkrows = (int64_t)B * Hkv * Skv;
    for (int64_t t = 0; t < n; ++t)
        if (rows[t] < 0 || rows[t] >= nkrows)
            return 1;
    size_t nq = (size_t)B * Hq * Sq * D, nk = (size_t)B * Hkv * Skv * D;
    double *qd = widen(q, nq), *kd = widen(k, nk), *vd = widen(v, nk),
           *dod = widen(dout, nq);
    int bad = !(qd && kd && vd && dod);
    if (!bad) {
        memset(dk_rows, 0, sizeof(double) * (size_t)n * D);
        memset(dv_rows, 0, sizeof(double) * (size_t)n * D);
        int rep = Hq / Hkv;
        /* one query row at a time, in parallel; each thread sums into its own
         * copy of the requested rows, merged at the end */
        int64_t nqrows = (int64_t)B * Hq * Sq;
#pragma omp parallel
        {
            double *p = (double *)malloc(sizeof(double) * (size_t)Skv);
            double *o = (double *)malloc(sizeof(double) * (size_t)D);
            double *dk_loc = (double *)calloc((size_t)n * D + 1, sizeof(double));
            double *dv_loc = (double *)calloc((size_t)n * D + 1, sizeof(double));
            const int have = p && o && dk_loc && dv_loc;
#pragma omp for schedule(dynamic, 8)
            for (int64_t r = 0; r < nqrows; ++r) {
                if (!have) {
#pragma omp atomic write
                    bad = 1;
                    continue;
                }
                {
                    int64_t i = r % Sq, bh = r / Sq, h = bh % Hq, b = bh / Hq;
                    int64_t g = b * Hkv + h / rep;
                    int needed = 0;
                    for (int64_t t = 0; t < n && !needed; ++t)
                        needed = (rows[t] / Skv == g);
                    if (!needed)
                        continue;
                    double delta;
                    int64_t nvis = bwd_row(qd, kd, vd, dod, Hq, Hkv, Sq, Skv, D,
                                           causal, scale, b, h, i, p, o, &delta);
                    const double *qi = qd + r * D;
                    const double *doi = dod + r * D;
                    const double *vb = vd + g * (int64_t)Skv * D;
                    for (int64_t t = 0; t < n; ++t) {
                        if (rows[t] / Skv != g)
                            continue;
                        int64_t j = rows[t] % Skv;
                        if (j >= nvis)
                            continue;
                        double dp = 0.0;
                        for (int d = 0; d < D; ++d)
                            dp += doi[d] * vb[j * D + d];
                        double ds = p[j] * (dp - delta);
                        for (int d = 0; d < D; ++d) {
                            dk_loc[t * D + d] += scale * ds * qi[d];
                            dv_loc[t * D + d] += p[j] * doi[d];
                        }
                    }
                }
            }
            if (have) {
#pragma omp critical
                {
                    for (int64_t x = 0; x < n * D; ++x) {
                        dk_rows[x] += dk_loc[x];
                        dv_rows[x] += dv_loc[x];
                    }
                }
            }
            free(p);
            free(o);
            free(dk_loc);
            free(dv_loc);
        }
    }
    free(qd);
    free(kd);
    free(vd);
    free(dod);
    return bad ? 1 : 0;
}
