/*
 * attn_testing.h -- test hooks for the kernel's failure detection.
 *
 * Every wait inside the fused kernel gives up after a time budget; the CTA
 * then stops, lets its own copies and tensor-core work finish, frees its
 * tensor memory, and records ATTN_ERR_TIMEOUT in the device status word
 * (attn_device_status in attn.h).  The pages describe no failure handling;
 * these hooks exist so that path can be tested without faulting the GPU.
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
 *
 * attn_fwd_tail_timeout_test does the same for the split tail of attn_fwd (see
 * attn.h: the last round's tiles split across a cluster of two CTAs).  The
 * call runs the split-tail launch with one difference: no CTA of a pair
 * sends its partner the partial result it has staged, so each CTA's bounded
 * wait for the partner's partial runs out after `wait_budget_ns`.  Both
 * CTAs unwind, reach the cluster barrier at exit and return; the status word
 * reads ATTN_ERR_TIMEOUT.  Returns ATTN_ERR_UNSUPPORTED (nothing launched) when
 * attn_fwd would not split the tail for these sizes on this device;
 * `wait_budget_ns` must lie in [1 ms, 2 s].  Outputs are unspecified.
 * For tests only.
 *
 * attn_bwd_timeout_test runs attn_bwd (same arguments and buffers; the
 * path that computes dQ inside the dK/dV kernel) with one difference: in
 * every dK/dV CTA that reaches work item `drop_item` (its query blocks with
 * work, counted from 0 in the order it walks them), the first elementwise
 * warpgroup does not signal that the item's first half block of P^T and
 * dS^T is stored, so the tensor-core issuer's wait for it runs out after
 * `wait_budget_ns`.  Every role of the CTA unwinds (the dQ read-out warps
 * included), the status word reads ATTN_ERR_TIMEOUT and the gradients are
 * unspecified.  `drop_item` must be >= 0 and `wait_budget_ns` in [1 ms,
 * 2 s] (else ATTN_ERR_INVALID_ARG).  For tests only.
 *
 * attn_fwd_tail_pairs returns how many tiles attn_fwd splits across CTA
 * pairs for these sizes on the current device (0 when the tail is not
 * split), or -1 for invalid sizes or a device that cannot be queried.
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

attn_status_t attn_fwd_tail_timeout_test(const void *q, const void *k, const void *v, void *o,
                                         float *lse, int B, int H_q, int H_kv, int S_q, int S_kv,
                                         int D, int causal, float scale,
                                         unsigned long long wait_budget_ns, attn_stream_t stream);

attn_status_t attn_bwd_timeout_test(const void *q, const void *k, const void *v, const void *o,
                                    const float *lse, const void *dout, void *dq, void *dk,
                                    void *dv, void *workspace, size_t workspace_bytes, int B,
                                    int H_q, int H_kv, int S_q, int S_kv, int D, int causal,
                                    float scale, int drop_item, unsigned long long wait_budget_ns,
                                    attn_stream_t stream);

int attn_fwd_tail_pairs(int B, int H_q, int H_kv, int S_q, int S_kv, int D, int causal);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_TESTING_H */
