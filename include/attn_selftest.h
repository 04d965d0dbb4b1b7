/*
 * attn_selftest.h -- GPU checks of the attention kernel's building blocks.
 *
 * Each call runs one CTA that uses the same TMA tensor maps (128-byte
 * swizzle), shared-memory matrix descriptors, instruction descriptors and
 * tensor-memory layouts as the fused kernel, on a single 128-row tile, so a
 * wrong encoding shows up as a wrong number in a small, checkable product.
 * They correspond to the two tensor-core steps of the fused operation
 * ("PipeThreader: Software-Defined Pipelining for Efficient DNN Execution",
 * section A2, Fig. 7: mma_qk and mma_pv).
 *
 * Same conventions as attn.h: device buffers owned by the caller, 16-byte
 * aligned, asynchronous on `stream`, status codes from attn_status_t.
 */
#ifndef ATTN_GB300_SELFTEST_H
#define ATTN_GB300_SELFTEST_H

#include "attn.h"

#ifdef __cplusplus
extern "C" {
#endif

/*
 * s = q k^T on the tensor cores.
 *   q [128, D] bf16 row-major (device), k [128, D] bf16 row-major (device),
 *   s [128, 128] fp32 row-major (device, written); D in {64, 128}.
 * q and k go through TMA into shared memory, the product through
 * tcgen05.mma (both operands K-major from shared memory) into tensor memory,
 * and back to global memory through tcgen05.ld.
 */
attn_status_t attn_selftest_qk(const void *q, const void *k, float *s, int D,
                               attn_stream_t stream);

/*
 * o = p v on the tensor cores with p taken from tensor memory.
 *   p [128, 128] bf16 row-major (device), v [128, D] bf16 row-major (device),
 *   o [128, D] fp32 row-major (device, written); D in {64, 128}.
 * Each thread writes its row of p into tensor memory with tcgen05.st as
 * packed bf16 pairs, v goes through TMA into shared memory (used MN-major),
 * and the product is read back with tcgen05.ld.
 */
attn_status_t attn_selftest_pv(const void *p, const void *v, float *o, int D,
                               attn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_SELFTEST_H */
