/*
 * chunk_scan_oracle.c -- plain, slow, fp64 reference for the Mamba2 chunk
 * scan (intra-chunk part).
 *
 * TEST INFRASTRUCTURE ONLY.  Only the test suite and the benchmark's
 * CPU-baseline arm may load this library.  The CUDA product path never calls
 * it and shares no code, header or table with it.
 *
 * What it computes: "PipeThreader: Software-Defined Pipelining for Efficient
 * DNN Execution", section 2 (running example, Mamba2 ChunkScan, Fig. 6(a)):
 * the function loads cb, dA and dt, multiplies cb by the exponential product
 * of dA and dt, and accumulates the matrix product of the result with x into
 * acc_o (of size (M, N), with X of size (K, N)).  The page does not spell the
 * product out; this file takes Mamba2's structured state-space reading (the
 * model the page cites), for chunk c of length Q, head h, rows m and
 * reduction index k of the chunk:
 *   out[m, :] = sum_{k <= m} cb[m, k] * exp(dA_cs[m] - dA_cs[k]) * dt[k] * x[k, :]
 * where dA_cs is the within-chunk cumulative sum of dA, cb = C B^T of the
 * chunk (given), and heads h share the cb of group h / (H / G).
 * Layouts: cb [B, nchunks, G, Q, Q] fp32; dA_cs, dt [B, H, nchunks, Q] fp32;
 * x, out [B, L, H, P] (L = nchunks * Q), x as bf16 bit patterns widened
 * exactly, out fp64.  All arithmetic is fp64; OpenMP over output rows.
 *
 * Return codes: 0 ok, 1 invalid argument.
 */
#include <math.h>
#include <stdint.h>
#include <string.h>

static double cs_bf16_to_double(uint16_t bits)
{
    uint32_t w = ((uint32_t)bits) << 16;
    float f;
    memcpy(&f, &w, sizeof f);
    return (double)f;
}

static int cs_check(int B, int L, int H, int G, int P, int Q)
{
    if (B <= 0 || L <= 0 || H <= 0 || G <= 0 || P <= 0 || Q <= 0)
        return 1;
    if (H % G != 0 || L % Q != 0)
        return 1;
    return 0;
}

/* One output row: batch b, position l, head h; writes P values. */
static void cs_row(const float *cb, const float *dA_cs, const float *dt,
                   const uint16_t *x, int L, int H, int G, int P, int Q,
                   int64_t b, int64_t l, int64_t h, double *out_row)
{
    int64_t nch = L / Q;
    int64_t c = l / Q;
    int64_t m = l % Q;
    int64_t g = h / (H / G);
    const float *cb_row = cb + (((b * nch + c) * G + g) * (int64_t)Q + m) * Q;
    const float *da = dA_cs + ((b * H + h) * nch + c) * (int64_t)Q;
    const float *dtc = dt + ((b * H + h) * nch + c) * (int64_t)Q;
    for (int n = 0; n < P; ++n)
        out_row[n] = 0.0;
    for (int64_t k = 0; k <= m; ++k) {
        double w = (double)cb_row[k] * exp((double)da[m] - (double)da[k]) * (double)dtc[k];
        const uint16_t *xk = x + ((b * L + c * Q + k) * H + h) * (int64_t)P;
        for (int n = 0; n < P; ++n)
            out_row[n] += w * cs_bf16_to_double(xk[n]);
    }
}

/* Full output: out [B, L, H, P] fp64. */
int oracle_chunk_scan(const float *cb, const float *dA_cs, const float *dt,
                      const uint16_t *x, double *out, int B, int L, int H,
                      int G, int P, int Q)
{
    if (cs_check(B, L, H, G, P, Q) || !cb || !dA_cs || !dt || !x || !out)
        return 1;
    int64_t rows = (int64_t)B * L * H;
#pragma omp parallel for schedule(dynamic, 64)
    for (int64_t r = 0; r < rows; ++r) {
        int64_t h = r % H, bl = r / H, l = bl % L, b = bl / L;
        cs_row(cb, dA_cs, dt, x, L, H, G, P, Q, b, l, h, out + r * P);
    }
    return 0;
}

/*
 * Selected rows (flat indices into [B, L, H]): out_rows [n, P].  Used to
 * check full-size runs on a sample.
 */
int oracle_chunk_scan_rows(const float *cb, const float *dA_cs,
                           const float *dt, const uint16_t *x,
                           const int64_t *rows, int64_t n, double *out_rows,
                           int B, int L, int H, int G, int P, int Q)
{
    if (cs_check(B, L, H, G, P, Q) || !cb || !dA_cs || !dt || !x || !rows ||
        !out_rows || n < 0)
        return 1;
    int64_t total = (int64_t)B * L * H;
    for (int64_t t = 0; t < n; ++t)
        if (rows[t] < 0 || rows[t] >= total)
            return 1;
#pragma omp parallel for schedule(dynamic, 16)
    for (int64_t t = 0; t < n; ++t) {
        int64_t r = rows[t];
        int64_t h = r % H, bl = r / H, l = bl % L, b = bl / L;
        cs_row(cb, dA_cs, dt, x, L, H, G, P, Q, b, l, h, out_rows + t * P);
    }
    return 0;
}
