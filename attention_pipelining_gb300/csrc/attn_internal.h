// attn_internal.h -- declarations shared by the translation units of the
// CUDA library (kernel launchers, the C ABI, the self-tests).
#pragma once

#include <cstdint>
#include <cuda.h>
#include <cuda_runtime.h>

#include "attn.h"

namespace attnpipe {

// Everything the fused kernel reads, passed as one __grid_constant__ block.
struct AttnParams {
  // Row groups: the H_q / H_kv query heads that share a KV head form one
  // group of R = (H_q / H_kv) * S_q rows (row rho = head-in-group * S_q +
  // position); a group's rows are contiguous in the [B, H_q, S_q, D] layout.
  CUtensorMap tm_q;  // Q as [B*H_kv, R, D], box {64, 128, 1}, 128-byte swizzle (load)
  CUtensorMap tm_k;  // K as [B*H_kv, S_kv, D], box {64, 128, 1} (load)
  CUtensorMap tm_v;  // V as [B*H_kv, S_kv, D], box {64, 128, 1} (load)
  CUtensorMap tm_o;  // O as [B*H_kv, R, D], box {64, 32, 1}, 128-byte swizzle (store)
  void* o;           // [B, H_q, S_q, D] bf16 (row rho of group z at (z * R + rho) * D)
  float* lse;        // [B, H_q, S_q]
  int B, H_q, H_kv, S_q, S_kv, causal;
  int rows_per_group;       // R
  long long total_rows;     // B * H_q * S_q
  // Work tiles: one tile = 256 rows of one row group x one KV split.  The
  // grid is persistent (at most one CTA per SM); CTA c takes tiles c, then
  // 2G-1-c, then 2G+c, ... (G = gridDim.x, a snake over rounds of G tiles)
  // from the list ordered as below, so the longest tiles go first and the
  // CTAs' total work evens out.
  //   non-causal: group-major (the tiles running at once share K/V heads
  //               in L2), query tiles last-to-first, then split;
  //   causal:     by cost rank (longest first), then group, then split.  A
  //               rank names one query tile of a group: with lpt_heads > 0
  //               (S_q a multiple of 256) rank -> position block
  //               nh - 1 - rank / lpt_heads of head rank % lpt_heads (nh =
  //               S_q / 256), otherwise query tile n_m_tiles - 1 - rank.
  int n_m_tiles;            // ceil(R / 256)
  int groups;               // B * H_kv
  int num_tiles;            // n_m_tiles * groups * kv_splits
  int lpt_heads;            // H_q / H_kv when causal and S_q % 256 == 0, else 0
  // Split KV: split s of a query tile covers KV blocks
  // [s * kv_blocks_per_split, (s + 1) * kv_blocks_per_split).  With
  // kv_splits > 1 a tile writes a partial result instead of O and LSE:
  // o_part [kv_splits, total_rows, D] fp32 (normalised within the split) and
  // lse_part [kv_splits, total_rows] fp32 (-inf for a row with no key in it).
  int kv_splits;
  int kv_blocks_per_split;
  float* o_part;
  float* lse_part;
  // Split tail (set at launch; 0 = off): when the last round of the grid
  // holds tail_pairs <= G / 2 tiles (list entries tail_base = R * G ..),
  // the grid runs as clusters of two CTAs and cluster i takes tail tile
  // tail_base + i, each CTA one half of its KV blocks.  Each CTA of the pair
  // writes the merged O and LSE of one 128-row sub-tile and sends its partial
  // result for the other one to its partner, one bulk copy into the partner's
  // shared memory (a tile with one sub-tile: the second CTA sends, the first
  // writes).  Off in split-KV launches.
  int tail_base;
  int tail_pairs;
  float scale_log2;  // |scale| * log2(e) > 0: the softmax runs in base 2
  int neg_scores;    // 1 for a negative scale: the QK GEMM computes -Q K^T
  unsigned long long timeout_ns;  // budget of any single wait inside the kernel
  // Timeline trace (the trace instantiation only): SM clock stamps of the
  // first tile of each CTA with index < trace_ctas, layout [cta][event][block].
  unsigned long long* trace;
  int trace_ctas;
  int trace_blocks;
  // Test of the timeout path (diagnostic instantiation only): when >= 0, the
  // first softmax warpgroup does not signal "P ready" for this KV block, so
  // the tensor-core issuer's bounded wait runs out.  -1 in normal use.
  int fault_drop_block;
  // Test of the split tail's exchange (split-tail instantiation only): when
  // non-zero, no CTA of a pair issues the bulk copy of its staged partial,
  // so every receiving CTA's bounded wait for it runs out.  0 in normal use.
  int fault_drop_xfer;
};

// Everything the backward kernels read.  Q and dO are viewed as [B*H_kv,
// R, D] (row groups, as in the forward), K and V as [B*H_kv, S_kv, D].  The
// per-row vectors live in a padded per-group layout [groups, Rp] with Rp = R
// rounded up to 128, so every 128-row block of them is 16-byte aligned.
struct BwdParams {
  CUtensorMap tm_q, tm_k, tm_v, tm_do;
  void* dq;           // [B, H_q, S_q, D] bf16
  void* dk;           // [B, H_kv, S_kv, D] bf16
  void* dv;           // [B, H_kv, S_kv, D] bf16
  float* nlse2;       // [groups, Rp]: -LSE * log2(e) (workspace; negated so the
                      // kernels' products and sums map onto packed fma / add)
  float* ndelta;      // [groups, Rp]: -D_i = -(dO_i . O_i) (workspace)
  // [groups, Rp, D] fp32 dQ accumulator (workspace): set for the fused path
  // (the dK/dV kernel adds dS K into it, a last kernel scales and rounds it
  // into dq); nullptr for the three-kernel path (dQ by its own kernel)
  float* dq_acc;
  int B, H_q, H_kv, S_q, S_kv, causal;
  int R, Rp, groups;
  float scale, scale_log2;
  unsigned long long timeout_ns;
  // Test of the timeout path: when >= 0, the first elementwise warpgroup of
  // the dK/dV kernel does not signal "P^T, dS^T stored" for half 0 of this
  // work item (query block) of each CTA, so the issuer's bounded wait runs
  // out.  -1 in normal use.
  int fault_drop_item;
};

// Queues the backward on `stream`: with p.dq_acc set (D = 128) prep (which
// also clears dq_acc), dK/dV with dQ, and the dQ conversion; otherwise prep,
// dK/dV and dQ.
cudaError_t launch_attn_bwd(const BwdParams& p, int D, const void* o, const void* dout,
                            const float* lse, cudaStream_t stream);

// Reads (and optionally clears) the backward kernels' status word.
cudaError_t read_bwd_status(int* status, bool reset);

// Everything the chunk-scan kernel reads.  x and out are [B, L, H, P] bf16
// (P = 64), cb [B, L / Q, G, Q, Q] fp32, dA_cs and dt [B, H, L / Q, Q] fp32.
struct ChunkScanParams {
  CUtensorMap tm_x;   // x as a 4-D map {P, H, L, B}, box {64, 1, 64, 1}, 128-byte swizzle
  CUtensorMap tm_cb;  // cb as a 3-D map {Q, Q, B * nchunks * G}, box {32, 128, 1} fp32, 128-byte swizzle
  CUtensorMap tm_out; // out as a 4-D map {P, H, L, B}, box {64, 1, 128, 1}, 128-byte swizzle
  const float* dA_cs;
  const float* dt;
  void* out;
  int B, L, H, G, Q, nchunks;
  int HB;             // heads per CTA (divides H / G); 0 = chosen at launch
  unsigned long long timeout_ns;
};

// Queues the chunk-scan kernel on `stream`.
cudaError_t launch_chunk_scan(const ChunkScanParams& p, cudaStream_t stream);

// Reads (and optionally clears) the chunk-scan kernel's status word.
cudaError_t read_chunk_scan_status(int* status, bool reset);

// Events stamped by the trace instantiation, one slot per KV block j.
enum TraceEvent : int {
  kEvSm0Wake = 0,   // softmax 0: S_0(j) ready (wait returned)
  kEvSm0Loaded,     // softmax 0: S_0(j) in registers
  kEvSm0Done,       // softmax 0: P_0(j) stored, about to signal
  kEvSm1Wake,
  kEvSm1Loaded,
  kEvSm1Done,
  kEvMmaPV0,        // tensor-core issuer: O_0 += P_0(j) V_j issued
  kEvMmaS0,         // S_0(j) = Q_0 K_j^T issued
  kEvMmaPV1,
  kEvMmaS1,
  kEvCorr0,         // correction: O_0 ready for block j (j >= 1)
  kEvCorr1,
  kEvLoadK,         // producer: K_j load issued
  kEvLoadV,         // producer: V_j load issued
  kEvEpilogue,      // correction: epilogue of sub-tile j (j = 0, 1) starts
  kEvEnd,           // j = 0: the first tile's epilogue has stored O
  kEvMmaPV0Begin,   // tensor-core issuer: waits for PV_0(j) passed, issue begins
  kEvMmaS0Begin,
  kEvMmaPV1Begin,
  kEvMmaS1Begin,
  kNumTraceEvents
};
constexpr int kMaxTraceBlocks = 128;  // KV blocks a trace records per event, at most

// Encodes a 3-D bf16 tensor map over a contiguous [outer, rows, D] array with
// a {64, box_rows, 1} box and 128-byte swizzle.  Returns false on failure.
bool encode_bf16_map_3d(CUtensorMap* map, const void* base, uint64_t D, uint64_t rows,
                        uint64_t outer, uint32_t box_rows);

// Queues the fused kernel (D = 64 or 128) on min(p.num_tiles, SM count) CTAs.
// With p.trace set or p.fault_drop_block >= 0, the diagnostic instantiation
// (timeline stamps, timeout test) runs instead.
cudaError_t launch_attn_fwd(const AttnParams& p, int D, cudaStream_t stream);

// Queues the merge of split-KV partial results into O (bf16) and LSE.
cudaError_t launch_splitkv_combine(const float* o_part, const float* lse_part, void* o, float* lse,
                                   long long rows, int D, int splits, cudaStream_t stream);

// The number of tiles a launch of these parameters on the current device
// splits across CTA pairs (0: none), or -1 if the device cannot be queried.
int fwd_tail_pairs(const AttnParams& p, int D);

// Reads (and optionally clears) the device status word of the current device.
cudaError_t read_device_status(int* status, bool reset);

// Reads (and optionally clears) the self-test kernels' status word.
cudaError_t read_selftest_status(int* status, bool reset);

// Self-test launchers (one CTA each).
cudaError_t launch_selftest_qk(const CUtensorMap& tq, const CUtensorMap& tk, float* s, int D,
                               cudaStream_t stream);
cudaError_t launch_selftest_pv(const uint16_t* p, const CUtensorMap& tv, float* o, int D,
                               cudaStream_t stream);

// Host-side pieces of the C ABI (attn_api.cu) used by more than one file.
attn_status_t validate(const void* q, const void* k, const void* v, const void* o, const void* lse,
                       int B, int H_q, int H_kv, int S_q, int S_kv, int D, int causal,
                       float scale);
int default_splits(int B, int H_q, int H_kv, int S_q, int S_kv, int causal);
size_t splitkv_bytes(int B, int H_q, int S_q, int D, int splits);
attn_status_t splitkv_impl(const void* q, const void* k, const void* v, void* o, float* lse,
                           void* workspace, size_t workspace_bytes, int B, int H_q, int H_kv,
                           int S_q, int S_kv, int D, int causal, float scale, int num_splits,
                           attn_stream_t stream);

constexpr unsigned long long kDefaultTimeoutNs = 2000000000ull;  // 2 s per wait
constexpr int kMaxSplits = 128;  // most KV splits of the split-KV forward

}  // namespace attnpipe
