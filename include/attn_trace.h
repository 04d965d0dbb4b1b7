/*
 * attn_trace.h -- timeline trace of the fused attention forward.
 *
 * The same computation as attn_fwd (include/attn.h), run by an instantiation
 * of the kernel that also stamps the SM cycle counter (clock64, comparable
 * within one CTA) when each warp role passes its hand-off points for each KV
 * block of the first tile a CTA works on; a warpgroup's slot keeps the latest
 * of its four warps: the two softmax warpgroups (S ready, S in registers, P
 * stored), the tensor-core issuer (each GEMM issued), the correction
 * warpgroup (O ready, epilogue start) and the TMA producer (each K / V load
 * issued).  The stamps collect in shared memory and are copied out when the
 * CTA ends.  This is the per-unit, per-step timeline that "PipeThreader:
 * Software-Defined Pipelining for Efficient DNN Execution" (section A2, Fig.
 * 6(d) and the profiler paragraph) uses to judge a pipelined schedule,
 * recorded from the running kernel instead of estimated.
 *
 *   trace         device buffer of uint64, [trace_ctas][20][trace_blocks],
 *                 caller-owned, 8-byte aligned; slots of events that do not
 *                 happen are left untouched (clear it first)
 *   trace_ctas    CTAs traced: those with index < trace_ctas in the
 *                 persistent grid (at most one CTA per SM)
 *   trace_blocks  KV blocks recorded per event, 1..128 (blocks beyond are
 *                 skipped)
 *
 * Event rows (index into the middle dimension): 0-2 softmax 0 wake / loaded /
 * done, 3-5 softmax 1 wake / loaded / done, 6 PV_0 issued, 7 S_0 issued,
 * 8 PV_1 issued, 9 S_1 issued, 10-11 correction 0 / 1 done, 12 K load issued,
 * 13 V load issued, 14 epilogue of sub-tile j starts (j = 0, 1), 15 end of the
 * first tile's epilogue (slot 0), 16-19 issue of PV_0 / S_0 / PV_1 / S_1
 * begins (its waits passed).  Other arguments and return codes as attn_fwd,
 * plus ATTN_ERR_INVALID_ARG for a null trace, non-positive counts or
 * trace_blocks > 128.
 */
#ifndef ATTN_GB300_TRACE_H
#define ATTN_GB300_TRACE_H

#include "attn.h"

#ifdef __cplusplus
extern "C" {
#endif

attn_status_t attn_fwd_trace(const void *q, const void *k, const void *v, void *o, float *lse,
                             int B, int H_q, int H_kv, int S_q, int S_kv, int D, int causal,
                             float scale, unsigned long long *trace, int trace_ctas,
                             int trace_blocks, attn_stream_t stream);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_TRACE_H */
