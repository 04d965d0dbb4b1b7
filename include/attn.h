/*
 * attn.h -- C ABI of the GB300 (sm_103a) fused attention forward.
 *
 * The operation ("PipeThreader: Software-Defined Pipelining for Efficient DNN
 * Execution", section A2, paragraph "FlashAttention-3" and Fig. 7): from Q, K
 * and V, MatMulQK gives acc_s = Q K^T, Softmax turns acc_s into P, MatMulPV
 * gives O = P V, all fused into one kernel.  This library computes, for each
 * batch b, query head h and query row i,
 *
 *     s_ij   = scale * sum_d Q[b,h,i,d] * K[b,g,j,d]     g = h / (H_q / H_kv)
 *     A_i    = { j < S_kv }            (non-causal)
 *              { j < S_kv, j <= i }    (causal: top-left aligned lower triangle)
 *     O[b,h,i,:] = sum_{j in A_i} exp(s_ij) V[b,g,j,:] / sum_{j in A_i} exp(s_ij)
 *     LSE[b,h,i] = ln sum_{j in A_i} exp(s_ij)
 *
 * The kernel follows the Blackwell warp-role split described in "GPU软件流水线与
 * Warp Specialization优化技术解析", section 3.1 (Flash Attention forward,
 * Blackwell): loads and tensor-core GEMMs in their own warps, the softmax of
 * two query sub-tiles in two warpgroups, the accumulator rescale in a third.
 *
 * Layout: Q, O are contiguous row-major [B, H_q, S_q, D] bf16; K, V are
 * contiguous [B, H_kv, S_kv, D] bf16; LSE is contiguous [B, H_q, S_q] fp32.
 * Arithmetic: bf16 operands, fp32 accumulation and softmax statistics, the
 * probabilities P rounded to bf16 before the second GEMM, O rounded to bf16.
 *
 * Ownership: every buffer belongs to the caller.  The library allocates no
 * memory and keeps no per-call state; it caches, per device, only the
 * architecture check and the kernels' shared-memory attribute.
 *
 * Errors: arguments are checked on the host before anything is launched; a
 * rejected call returns a status other than ATTN_OK and touches no memory.
 * There is no CPU fallback: a device that is not compute capability 10.3
 * gives ATTN_ERR_UNSUPPORTED.
 */
#ifndef ATTN_GB300_H
#define ATTN_GB300_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* A CUDA stream (cudaStream_t / CUstream); NULL is the legacy default stream. */
typedef void *attn_stream_t;

typedef enum {
  ATTN_OK = 0,
  ATTN_ERR_INVALID_ARG = 1, /* null pointer, a size <= 0, H_q % H_kv != 0, scale not finite */
  ATTN_ERR_UNSUPPORTED = 2, /* D not 64 or 128, size beyond the kernel's limits, not sm_103 */
  ATTN_ERR_MISALIGNED = 3,  /* a device pointer not 16-byte aligned */
  ATTN_ERR_CUDA = 4,        /* a CUDA runtime or driver call failed */
  ATTN_ERR_TIMEOUT = 5      /* a kernel wait ran out of time (see attn_device_status) */
} attn_status_t;

/*
 * Fused attention forward on device buffers, asynchronous on `stream`.
 *
 *   q    [B, H_q, S_q, D]  bf16, device, read
 *   k    [B, H_kv, S_kv, D] bf16, device, read
 *   v    [B, H_kv, S_kv, D] bf16, device, read
 *   o    [B, H_q, S_q, D]  bf16, device, written
 *   lse  [B, H_q, S_q]     fp32, device, written (natural log)
 *   D in {64, 128}; H_q a multiple of H_kv; every size >= 1;
 *   causal 0 or 1; scale any finite value, negative and zero included (the
 *   scores are multiplied by it before the mask and the softmax; 1/sqrt(D)
 *   is the usual choice).
 *
 * All pointers must be 16-byte aligned and must not alias o/lse with inputs.
 * Returns once the kernel is queued; no synchronisation happens inside.
 *
 * Scheduling: 256-row tiles on a persistent grid of one CTA per SM.  When
 * the last round of tiles would leave more than half of the SMs idle, the
 * grid runs as clusters of two CTAs and each tile of that round is split
 * across a pair: each CTA takes half of its KV blocks and the first merges
 * the second's partial result (received through distributed shared memory)
 * by their log-sum-exps.  The results are deterministic for given sizes.
 */
attn_status_t attn_fwd(const void *q, const void *k, const void *v, void *o, float *lse,
                       int B, int H_q, int H_kv, int S_q, int S_kv, int D, int causal,
                       float scale, attn_stream_t stream);

/*
 * The same computation with host inputs and outputs: copies q/k/v from host
 * memory into the caller's device buffers q_dev/k_dev/v_dev, runs attn_fwd
 * into o_dev/lse_dev, and copies o/lse back to host memory, ordered after
 * the work already queued on `stream` and before the work queued on it
 * afterwards.  Inputs of 32 MiB or more are split into chunks of
 * consecutive (batch, kv-head) row groups, each a contiguous slice of every
 * tensor: 8 even chunks when the copies are expected to take longer than the
 * kernels, else about 16, the first and the last of a single row group when
 * the others hold two or more (those two copies are the ones nothing
 * overlaps).  A chunk's inputs go up on one internal stream, its kernel runs on
 * one of three internal compute streams and its outputs come back on another,
 * so each chunk's copies overlap the other chunks' kernels.  The internal
 * streams and events are created on first use, once per device, and kept;
 * concurrent callers on one device queue their chunks one call at a time.
 * The results are those of attn_fwd on each chunk: bit-identical to one
 * attn_fwd call on the whole, except in the rows of tiles that one of the
 * two splits across a CTA pair (see attn_fwd), which agree to within the
 * rounding of that merge.  Host buffers should be page-locked for
 * the copies to be asynchronous.  Returns once everything is queued; the
 * host outputs are valid once `stream` has been synchronised.  Same argument
 * rules as attn_fwd for the device buffers; host pointers must be non-null.
 */
attn_status_t attn_fwd_host(const void *q_host, const void *k_host, const void *v_host,
                            void *o_host, float *lse_host, void *q_dev, void *k_dev,
                            void *v_dev, void *o_dev, float *lse_dev, int B, int H_q, int H_kv,
                            int S_q, int S_kv, int D, int causal, float scale,
                            attn_stream_t stream);

/*
 * Split-KV ("FlashDecoding") forward: the same result as attn_fwd, computed
 * with the KV axis cut into `num_splits` ranges that run as separate CTAs,
 * followed by a merge of their partial results, L = ln sum_s exp(L_s),
 * O = sum_s exp(L_s - L) O_s.  The FlashDecoding microbenchmark of
 * "PipeThreader: Software-Defined Pipelining for Efficient DNN Execution",
 * section A4, is this operator at decoding shapes (S_q = 1): there a single
 * query row per head leaves the GPU idle unless the keys are split.
 *
 *   workspace        caller-owned device scratch, 256-byte aligned, of at
 *                    least attn_splitkv_workspace_bytes(B, H_q, S_q, D, s)
 *                    bytes for the split count s actually used; it holds the
 *                    partial O (fp32) and LSE of every split
 *   num_splits       1..128, or <= 0 for attn_splitkv_default_splits(...)
 *
 * Other arguments, layouts and errors as attn_fwd; additionally
 * ATTN_ERR_INVALID_ARG for a null or too small workspace,
 * ATTN_ERR_MISALIGNED for a workspace not 256-byte aligned,
 * ATTN_ERR_UNSUPPORTED for num_splits > 128.  Two kernels are queued on
 * `stream`; the workspace must not be shared with concurrent calls.
 */
attn_status_t attn_fwd_splitkv(const void *q, const void *k, const void *v, void *o, float *lse,
                               void *workspace, size_t workspace_bytes, int B, int H_q, int H_kv,
                               int S_q, int S_kv, int D, int causal, float scale, int num_splits,
                               attn_stream_t stream);

/* Workspace bytes attn_fwd_splitkv needs for `num_splits` splits (0 if the
 * arguments are invalid). */
size_t attn_splitkv_workspace_bytes(int B, int H_q, int S_q, int D, int num_splits);

/* The split count attn_fwd_splitkv uses when given num_splits <= 0 for these
 * sizes on the current device (0 if the arguments are invalid). */
int attn_splitkv_default_splits(int B, int H_q, int H_kv, int S_q, int S_kv, int causal);

/*
 * attn_fwd_splitkv without a caller workspace, for callers that cannot
 * allocate device memory: an engine that gives all device memory to its own
 * pool at start-up and allows no further allocations, a plugin loaded into a
 * program that exposes no allocator to it, or a latency-critical path where
 * an allocation call could block on the device.  The paper has no
 * counterpart of this entry point; it is an interface convenience.
 *
 * The partial results go to a scratch array of fixed size,
 * attn_splitkv_noalloc_capacity() = 16 MiB, that is part of the library's
 * device image: every GPU that loads the library holds it until the process
 * exits.  A call allocates nothing (no cudaMalloc, cudaFree or allocating
 * library routine).  The first call on a device looks up the array's device
 * address once (cudaGetSymbolAddress with that device current) and caches
 * it; make that first call before any stream capture.  The cached address
 * belongs to the device's current context: after cudaDeviceReset on that
 * device it no longer points at the array, and this entry point must not be
 * called again in that process (use attn_fwd_splitkv with a workspace).
 *
 * All calls on a device share the one array, which keeps the last call's
 * contents; every partial a call reads is written by that same call, so
 * nothing needs clearing.  Calls whose GPU work overlaps (different streams
 * without ordering) race on the array: order them, e.g. on one stream.
 *
 * Same arguments and results as attn_fwd_splitkv minus the workspace; a call
 * whose partial results would exceed the array (see
 * attn_splitkv_workspace_bytes for the split count used) returns
 * ATTN_ERR_UNSUPPORTED without launching anything: use attn_fwd_splitkv with
 * a workspace, or fewer splits.
 */
attn_status_t attn_fwd_splitkv_noalloc(const void *q, const void *k, const void *v, void *o,
                                       float *lse, int B, int H_q, int H_kv, int S_q, int S_kv,
                                       int D, int causal, float scale, int num_splits,
                                       attn_stream_t stream);

/* Bytes of the built-in scratch array attn_fwd_splitkv_noalloc uses. */
size_t attn_splitkv_noalloc_capacity(void);

/*
 * Backward of attn_fwd: the gradients of L = sum(O * dO) with respect to Q, K
 * and V, given the forward's O and LSE and the upstream gradient dO.  With
 * P_ij = exp(scale q_i . k_j - LSE_i) (0 where masked), D_i = dO_i . O_i,
 * dP_ij = dO_i . v_j and dS_ij = P_ij (dP_ij - D_i):
 *
 *     dV_j = sum_i P_ij dO_i,   dK_j = scale sum_i dS_ij q_i,
 *     dQ_i = scale sum_j dS_ij k_j,
 *
 * where dK_j and dV_j also sum over the H_q / H_kv query heads sharing key /
 * value head j's head.  The backward on Blackwell is the subject of "GPU软件
 * 流水线与Warp Specialization优化技术解析", section 3.2; the pages give no
 * formulas, these are the chain rule through the forward's definition.
 *
 *   q, k, v     as for attn_fwd (device, read)
 *   o, lse      attn_fwd's outputs for the same q, k, v, causal, scale (read)
 *   dout        [B, H_q, S_q, D] bf16, device, read
 *   dq          [B, H_q, S_q, D] bf16, device, written
 *   dk, dv      [B, H_kv, S_kv, D] bf16, device, written
 *   workspace   caller-owned device scratch, 256-byte aligned, of at least
 *               attn_bwd_workspace_bytes(B, H_q, H_kv, S_q, D) bytes (per-row
 *               D_i and LSE, and an fp32 dQ accumulator; no need to clear it)
 *
 * Arithmetic: bf16 operands, fp32 accumulation; P and dS are rounded to
 * bf16 before the GEMMs that consume them.  dQ is computed in the same
 * kernel as dK and dV: each (key block, query block) pair adds its fp32
 * partial dS K into the accumulator in the workspace with atomic adds in L2,
 * and a last kernel scales and rounds it to bf16.  The order of those adds
 * varies from run to run, so dQ may differ in its last bit between runs
 * (dK and dV do not); attn_bwd_deterministic gives reproducible bits (there
 * dQ has a kernel of its own that recomputes S and dP per query block).
 * Three kernels are queued on
 * `stream`; the workspace must not be shared with concurrent calls.  Errors
 * as attn_fwd, plus ATTN_ERR_INVALID_ARG for a null dout / dq / dk / dv /
 * workspace or a too small workspace, and ATTN_ERR_MISALIGNED for a workspace
 * not 256-byte aligned.
 */
attn_status_t attn_bwd(const void *q, const void *k, const void *v, const void *o,
                       const float *lse, const void *dout, void *dq, void *dk, void *dv,
                       void *workspace, size_t workspace_bytes, int B, int H_q, int H_kv,
                       int S_q, int S_kv, int D, int causal, float scale, attn_stream_t stream);

/*
 * attn_bwd with bit-reproducible results: dQ by its own kernel, which
 * recomputes S and dP per query block (two more GEMMs per block pair than
 * attn_bwd), with no atomic adds.  Arguments, workspace and
 * errors as attn_bwd.
 */
attn_status_t attn_bwd_deterministic(const void *q, const void *k, const void *v, const void *o,
                                     const float *lse, const void *dout, void *dq, void *dk,
                                     void *dv, void *workspace, size_t workspace_bytes, int B,
                                     int H_q, int H_kv, int S_q, int S_kv, int D, int causal,
                                     float scale, attn_stream_t stream);

/* Workspace bytes attn_bwd and attn_bwd_deterministic need (0 if the
 * arguments are invalid): 4 (D + 2) bytes per query row, rows padded to a
 * multiple of 128 per (batch, kv-head) group. */
size_t attn_bwd_workspace_bytes(int B, int H_q, int H_kv, int S_q, int D);

/*
 * attn_bwd with host inputs and outputs, pipelined as attn_fwd_host is:
 * copies q, k, v, o, lse and dout from host memory into the caller's device
 * buffers (the *_dev arguments, same shapes as attn_bwd's), runs the backward
 * and copies dq, dk and dv back to host memory, ordered after the work
 * already queued on `stream` and before the work queued on it afterwards.
 * Inputs of 32 MiB or more are split into chunks of consecutive (batch,
 * kv-head) row groups as in attn_fwd_host; a chunk's inputs go up on one internal
 * stream, its three kernels run on one of three internal compute streams with
 * its own slice of `workspace`, and its gradients come back on another, so
 * each chunk's copies overlap the other chunks' kernels.  Every gradient
 * element is computed by the same tiles in the same order as in one
 * attn_bwd call, so dK and dV are bit-identical to it and dQ is up to the
 * order of its atomic adds (see attn_bwd).  Host buffers
 * should be page-locked for the copies to be asynchronous.  Returns once
 * everything is queued; the host gradients are valid once `stream` has
 * been synchronised.  Argument rules and errors as attn_bwd for the device
 * buffers and the workspace (the same size, attn_bwd_workspace_bytes);
 * ATTN_ERR_INVALID_ARG for a null host pointer.  Nothing is queued when a
 * check fails.
 */
attn_status_t attn_bwd_host(const void *q_host, const void *k_host, const void *v_host,
                            const void *o_host, const float *lse_host, const void *dout_host,
                            void *dq_host, void *dk_host, void *dv_host, void *q_dev,
                            void *k_dev, void *v_dev, void *o_dev, float *lse_dev,
                            void *dout_dev, void *dq_dev, void *dk_dev, void *dv_dev,
                            void *workspace, size_t workspace_bytes, int B, int H_q, int H_kv,
                            int S_q, int S_kv, int D, int causal, float scale,
                            attn_stream_t stream);

/* Static English description of a status code (never NULL). */
const char *attn_status_string(attn_status_t status);

/*
 * Reads the device-side status words of the current device (forward,
 * backward and self-test kernels): ATTN_OK, or ATTN_ERR_TIMEOUT if a launch
 * since the last reset gave up on a wait (that launch's outputs are then
 * unspecified).  Synchronises the device.  With
 * reset != 0 the word is cleared afterwards.
 */
attn_status_t attn_device_status(int *status_out, int reset);

/* Library version, major * 10000 + minor * 100 + patch. */
int attn_version(void);

#ifdef __cplusplus
}
#endif

#endif /* ATTN_GB300_H */
