/*
 * attn_testing.h -- test hook for the kernel's failure detection.
 *
 * Every wait inside the fused kernel gives up after a time budget; the CTA
 * then stops, lets its own copies and tensor-core work finish, frees its
 * tensor memory, and records ATTN_ERR_TIMEOUT in the device status word
 * (attn_device_status in attn.h).  The pages describe no failure handling;
 * this hook exists so that path can be tested without faulting the GPU.
 *
 * attn_fwd_timeout_test runs the same computation as attn_fwd (same
 * arguments and buffers) in the diagnostic instantiation of the kernel, with
 * one difference: the first softmax warpgroup of every CTA that reaches KV
 * block `drop_block` does not signal that its probabilities are ready, so
 * the tensor-core issuer's wait for them runs out after `wait_budget_ns`.
 * A CTA whose sequence has fewer blocks completes normally.  Outputs of a
 * timed-out CTA are unspecified.  `wait_budget_ns` must lie in
 * [1 ms, 2 s]; `drop_block` must be >= 0 (else ATTN_ERR_INVALID_ARG).
 * For tests only.
 */
#ifndef ATTN_GB300_TESTING_H
#define ATTN_GB300_TESTING_H

#include "attn.h"

#ifdef __cplusplus
extern "C" {
#endif

attn_status_t attn_fwd_timeout_test(const void *q, const void *k, const void *v, void *o,
                                    float *lse, int B, int H_q, int H_kv, int S_q, int S_kv,
                                    int D, int causal, float scale, int drop_block,
                                    unsigned long long wait_budget_ns, attn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_TESTING_H */
