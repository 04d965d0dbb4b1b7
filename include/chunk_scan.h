/*
 * chunk_scan.h -- C ABI of the Mamba2 chunk scan (intra-chunk part) on GB300.
 *
 * The operation: "PipeThreader: Software-Defined Pipelining for Efficient DNN
 * Execution", section 2 (running example, Mamba2 ChunkScan, Fig. 6(a)):
 * cb is multiplied by the exponential product of dA and dt, and its matrix
 * product with x is accumulated into acc_o.  The page leaves the product
 * implicit; this library takes Mamba2's structured state-space reading: for
 * chunk c (length Q), head h of group g = h / (H / G), row m of the chunk,
 *
 *     out[b, c*Q + m, h, :] = sum_{k <= m} cb[b, c, g, m, k]
 *                              * exp(dA_cs[b, h, c, m] - dA_cs[b, h, c, k])
 *                              * dt[b, h, c, k] * x[b, c*Q + k, h, :]
 *
 * where dA_cs is the within-chunk running sum of dA.  The scaled cb is
 * rounded to bf16 before the product (fp32 accumulation); out is bf16.
 *
 *   cb      [B, L/Q, G, Q, Q] fp32, device, read
 *   dA_cs   [B, H, L/Q, Q]    fp32, device, read
 *   dt      [B, H, L/Q, Q]    fp32, device, read
 *   x       [B, L, H, P]      bf16, device, read
 *   out     [B, L, H, P]      bf16, device, written
 *   P = 64, Q = 128 or 256, L a multiple of Q, H a multiple of G.
 *
 * All buffers are caller-owned and 16-byte aligned; nothing is allocated.
 * Returns once the kernel is queued on `stream`.  Errors: ATTN_ERR_INVALID_ARG
 * for null pointers, sizes <= 0, H % G or L % Q not 0; ATTN_ERR_UNSUPPORTED
 * for other P or Q, sizes beyond the kernel's limits or a device that is not
 * sm_103; ATTN_ERR_MISALIGNED; ATTN_ERR_CUDA.  A kernel wait that runs out is
 * reported by attn_device_status (include/attn.h).
 */
#ifndef ATTN_GB300_CHUNK_SCAN_H
#define ATTN_GB300_CHUNK_SCAN_H

#include "attn.h"

#ifdef __cplusplus
extern "C" {
#endif

attn_status_t chunk_scan_fwd(const float *cb, const float *dA_cs, const float *dt, const void *x,
                             void *out, int B, int L, int H, int G, int P, int Q,
                             attn_stream_t stream);

/*
 * chunk_scan_fwd with host inputs and output: copies cb, dA_cs, dt and x from
 * host memory into the caller's device buffers (the *_dev arguments, same
 * shapes as chunk_scan_fwd's), runs the scan and copies out back to host
 * memory, ordered after the work already queued on `stream` and before the
 * work queued on it afterwards.  Inputs of 32 MiB or more are split into
 * chunks of consecutive batch entries (one per entry, at most 32),
 * pipelined on the internal streams attn_fwd_host uses: one chunk's inputs
 * go up while another's output comes back, so the host link carries both
 * directions at once.
 * Every output element is computed the same way as in one chunk_scan_fwd
 * call, so the results are bit-identical to it.  Host buffers should be
 * page-locked for the copies to be asynchronous.  Returns once everything
 * is queued; the host output is valid once `stream` has been synchronised.
 * Argument rules and errors as chunk_scan_fwd for the device buffers;
 * ATTN_ERR_INVALID_ARG for a null host pointer.  Nothing is queued when a
 * check fails.
 */
attn_status_t chunk_scan_fwd_host(const float *cb_host, const float *dA_cs_host,
                                  const float *dt_host, const void *x_host, void *out_host,
                                  float *cb_dev, float *dA_cs_dev, float *dt_dev, void *x_dev,
                                  void *out_dev, int B, int L, int H, int G, int P, int Q,
                                  attn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_CHUNK_SCAN_H */
