// attn_bwd_sm103.cu -- attention backward for sm_103a (GB300).
//
// The gradients of the forward of "PipeThreader: Software-Defined Pipelining
// for Efficient DNN Execution" (section A2, Fig. 7): with P the forward's
// softmax rows, D_i = dO_i . O_i, dP = dO V^T and dS = P o (dP - D),
//   dV = P^T dO,   dK = scale dS^T Q,   dQ = scale dS K
// (summed over the query heads that share a key/value head).  The backward
// is the subject of "GPU软件流水线与Warp Specialization优化技术解析", section
// 3.2 (Flash Attention backward on Blackwell: loads, tensor-core GEMMs and
// the elementwise work in separate warp groups).
//
// Two paths of three kernels each.  The default one (attn_bwd):
//   prep     D_i and the base-2 LSE per row, into a padded per-group
//            layout, and zeros for an fp32 dQ accumulator;
//   dK/dV    one CTA per (row group, 128 keys): over the group's query
//            blocks, S^T = K Q^T and dP^T = V dO^T on the tensor core, P^T
//            and dS^T by two elementwise warpgroups (64 queries each), then
//            dV += P^T dO and dK += dS^T Q accumulate in tensor memory, and
//            dQ^T = K^T dS^T per half block, which a fourth warpgroup reads
//            out and adds into the accumulator in L2 (kFuse);
//   convert  dq = bf16(scale * accumulator).
// The deterministic one (attn_bwd_deterministic) runs prep, dK/dV without
// dQ, and
//   dQ       one CTA per (row group, 128 query rows): over the key blocks,
//            S = Q K^T and dP = dO V^T, dS by the elementwise warpgroups (64
//            keys each), dQ += dS K in tensor memory.
// P needs no running max in the backward (the forward's LSE normalises it),
// so the elementwise work splits over columns with no exchange.
//
// Each 128 x 128 block runs as two halves of 64 columns, so the elementwise
// warps work on one half while the tensor core computes the other.
//
// 384 threads (512 with the fused dQ): warps 0-7 elementwise (warpgroup w
// takes columns 32w..32w+31 of each half, thread = TMEM lane = the tile's
// row), warp 8 tensor-core issuer and warp 9 TMA producer (warp-wide, one
// elected lane issues), warps 10-11 idle, warps 12-15 the dQ read-out.
// Every wait is bounded; a timeout raises a CTA-wide abort flag and the
// device status word records ATTN_ERR_TIMEOUT.
#include <cmath>
#include <cstdint>
#include <type_traits>
#include <mutex>

#include "attn_internal.h"
#include "attn_tiles.cuh"
#include "ptx.cuh"

namespace attnpipe {

__device__ int g_bwd_status = 0;

namespace {

constexpr int kThreadsB = 384;
constexpr int kThreadsFused = 512;  // the dK/dV kernel with dQ: + the dQ read-out warpgroup
constexpr int kRows = 128;       // rows of a tile: keys (dK/dV kernel) or queries (dQ kernel)
constexpr uint32_t kAll = 0xffffffffu;

__device__ __forceinline__ bool warp_wait_b(uint64_t* bar, uint32_t parity,
                                            volatile int* abort_flag, uint64_t budget) {
  const bool ok = mbar_wait(bar, parity, abort_flag, budget);
  return __all_sync(kAll, ok);
}

__device__ __forceinline__ void drain_wait_b(uint64_t* bar, uint32_t parity, uint64_t budget) {
  volatile int never = 0;
  mbar_wait(bar, parity, &never, budget);
}

__device__ __forceinline__ float u2f_b(uint32_t x) { return __uint_as_float(x); }

// Adds x to the fp32 at `addr` in global memory, performed in L2 (no
// return value; relaxed, device scope).
__device__ __forceinline__ void red_add_f32(float* addr, float x) {
  asm volatile("red.relaxed.gpu.global.add.f32 [%0], %1;" ::"l"(addr), "f"(x) : "memory");
}

// Adds `bytes` of fp32 from shared memory into global memory element by
// element (performed in L2), tracked by the issuing thread's bulk groups like
// a store.  Both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_reduce_add_f32(float* gdst, uint32_t ssrc, uint32_t bytes) {
  asm volatile("cp.reduce.async.bulk.global.shared::cta.bulk_group.add.f32 [%0], [%1], %2;"
               ::"l"(gdst), "r"(ssrc), "r"(bytes)
               : "memory");
}

// The work of a 128 x 128 block is done in two halves h = 0, 1 of 64
// columns, so the elementwise warpgroups work on one half while the tensor
// core runs the other half's GEMMs.

// C[tmem, 128 x 64 fp32] = A B_h^T: A a [128 x D] tile, B_h rows 64h..64h+63
// of a [128 x D] tile, both K-major (given as tile descriptors; the half's
// rows start 64 rows = 8 KB into each 128-byte-swizzled slab).
template <int D>
__device__ __forceinline__ void issue_qk_half(uint32_t c_tmem, uint64_t a_desc, uint64_t b_desc,
                                              int h) {
  constexpr uint32_t idesc = make_idesc_bf16_f32(128, 64, false, false);
  const uint64_t b_half = b_desc + (uint64_t)((h * 64 * 128) >> 4);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = (uint64_t)(((kk >> 2) * kSlabBytes + (kk & 3) * 32) >> 4);
    mma_ss(c_tmem, a_desc + off, b_half + off, idesc, kk > 0 ? 1u : 0u);
  }
}

// The same product with A in tensor memory: a [128 x D] bf16 tile copied
// there once (row i in lane i, elements 2c and 2c + 1 in column c, as the
// tensor core reads an A operand).  Only B is then read from shared memory,
// so these N = 64 products run at the tensor core's rate instead of at the
// rate shared memory can feed both operands.
template <int D>
__device__ __forceinline__ void issue_qk_half_ts(uint32_t c_tmem, uint32_t a_tmem, uint64_t b_desc,
                                                 int h) {
  constexpr uint32_t idesc = make_idesc_bf16_f32(128, 64, false, false);
  const uint64_t b_half = b_desc + (uint64_t)((h * 64 * 128) >> 4);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = (uint64_t)(((kk >> 2) * kSlabBytes + (kk & 3) * 32) >> 4);
    mma_ts(c_tmem, a_tmem + kk * 8, b_half + off, idesc, kk > 0 ? 1u : 0u);
  }
}

// Copies a [128 x D] bf16 tile from shared memory (the TMA 128-byte swizzle:
// 16-byte piece c of row r at piece c ^ (r % 8) of its 64-column slab) into
// tensor memory as an A operand (D / 2 columns from `t_col`); thread = row
// = lane of the warp's quadrant (lane_base).  Whole warp.
template <int D>
__device__ __forceinline__ void copy_tile_to_tmem(const uint8_t* tile, uint32_t t_col, int row) {
  const uint32_t base = smem_u32(tile) + (uint32_t)row * 128u;
#pragma unroll
  for (int sl = 0; sl < D / 64; ++sl) {
    uint32_t w[32];
#pragma unroll
    for (int c = 0; c < 8; ++c) {
      uint32_t a, b, cc, d;
      asm volatile("ld.shared.v4.b32 {%0, %1, %2, %3}, [%4];"
                   : "=r"(a), "=r"(b), "=r"(cc), "=r"(d)
                   : "r"(base + (uint32_t)(sl * kSlabBytes) + 16u * (uint32_t)(c ^ (row & 7))));
      w[4 * c + 0] = a;
      w[4 * c + 1] = b;
      w[4 * c + 2] = cc;
      w[4 * c + 3] = d;
    }
    tmem_st_x32(t_col + sl * 32, w);
  }
}

// Acc[tmem, 128 x D fp32] (+)= A_h B_h: A_h [128 x 64] bf16 in tensor memory,
// two per column, written by the elementwise warpgroups (warpgroup w's 32
// elements at columns 32w .. 32w + 15 from `a_tmem`); B_h rows 64h..64h+63
// of a [128 x D] tile used MN-major (D contiguous), given its MN-major tile
// descriptor.  `accumulate` = false overwrites Acc.
template <int D>
__device__ __forceinline__ void issue_pv_half(uint32_t d_tmem, uint32_t a_tmem, uint64_t b_desc,
                                              int h, bool accumulate) {
  constexpr uint32_t idesc = make_idesc_bf16_f32(128, D, false, true);
#pragma unroll
  for (int kk = 0; kk < 4; ++kk) {
    mma_ts(d_tmem, a_tmem + (kk >> 1) * 32 + (kk & 1) * 8,
           b_desc + (uint64_t)(((4 * h + kk) * 2048) >> 4), idesc,
           (accumulate || kk > 0) ? 1u : 0u);
  }
}

// dQ^T[tmem, D x 64 fp32] = K^T dS^T_h: M = the head dimension, N = the
// half's 64 queries, K = the block's 128 keys.  A is the K tile used
// MN-major (its rows are keys, the head dimension contiguous; at D = 128
// the two 64-column slabs along M one slab apart), B the half's dS^T buffer
// used MN-major (rows are keys, 64 queries contiguous).  Per K step of 16
// keys both starts advance 16 rows = 2048 bytes.  Overwrites the
// accumulator.  Row d lands in tensor-memory lane d for D = 128; for M = 64
// rows 16 q .. 16 q + 15 land in lanes 32 q .. 32 q + 15 (measured on
// GB300 with a one-MMA probe: the other 16 lanes of each quadrant are not
// part of the result).
template <int D>
__device__ __forceinline__ void issue_dqt_half(uint32_t d_tmem, uint64_t k_desc_mn,
                                               uint64_t ds_desc_mn) {
  constexpr uint32_t idesc = make_idesc_bf16_f32(D, 64, true, true);
#pragma unroll
  for (int kk = 0; kk < kRows / 16; ++kk) {
    const uint64_t off = (uint64_t)((kk * 2048) >> 4);
    mma_ss(d_tmem, k_desc_mn + off, ds_desc_mn + off, idesc, kk > 0 ? 1u : 0u);
  }
}

template <int D>
struct BwdCfg {
  static constexpr int kTileBytes = TileShape<D>::kBytes;
  // dK/dV kernel: K, V, then a ring of (Q, dO, base-2 LSE, D) stages
  static constexpr int kQStages = (D == 128) ? 2 : 4;
  static constexpr int kVecBytes = kRows * 4;                 // one [128] fp32 vector
  static constexpr int kQStageBytes = 2 * kTileBytes + 2 * kVecBytes;
  static constexpr int kOffK = 0;
  static constexpr int kOffV = kTileBytes;
  static constexpr int kOffQRing = 2 * kTileBytes;
  // dK/dV kernel with dQ (kFuse): dS^T of one half block, [128 keys x 64
  // queries] bf16 in the 128-byte swizzle (one slab), the B operand of
  // dQ^T = K^T dS^T (MN-major)
  static constexpr int kDsBytes = kRows * 64 * 2;
  static constexpr int kOffDsT = kOffQRing + kQStages * kQStageBytes;
  // ... and at D = 64 two staging buffers for a half block's dQ partial,
  // [64 queries][64] fp32 each (the accumulator's own row layout), which one
  // bulk reduction adds into it
  static constexpr int kDqStageBytes = (D == 64) ? 64 * D * 4 : 0;
  static constexpr int kOffDqStage = kOffDsT + kDsBytes;
  static constexpr int kOffBarKV = kOffDqStage + 2 * kDqStageBytes;
  // kv_full, q_full[S], q_empty[S], sp_full[2], ps_ready[2], acc_done, drain,
  // kt_ready (K and V copied into tensor memory; D = 64), then with kFuse
  // dq_full[2], dq_free[2], ds_free
  static constexpr int kNumBarsKV = 2 * kQStages + 8 + 5;
  // dK/dV kernel at D = 64: K and V as tensor-memory A operands too (D / 2
  // columns each after the two accumulators; at D = 128 there is no room)
  static constexpr bool kKVinTmem = (D == 64);
  static constexpr int kOffMiscKV = kOffBarKV + kNumBarsKV * 8;
  static constexpr int kSmemKV = kOffMiscKV + 16 + 1024;
  // dQ kernel: Q, dO, then a ring of (K, V) stages
  static constexpr int kKVStages = (D == 128) ? 2 : 4;
  static constexpr int kOffQ = 0;
  static constexpr int kOffDO = kTileBytes;
  static constexpr int kOffKVRing = 2 * kTileBytes;
  static constexpr int kOffBarQ = kOffKVRing + kKVStages * 2 * kTileBytes;
  // q_full, kv_full[S], kv_empty[S], sp_full[2], ds_ready[2], acc_done, drain,
  // qt_ready (Q and dO copied into tensor memory)
  static constexpr int kNumBarsQ = 2 * kKVStages + 8;
  static constexpr int kOffMiscQ = kOffBarQ + kNumBarsQ * 8;
  static constexpr int kSmemQ = kOffMiscQ + 16 + 1024;
  // tensor memory: S (or S^T) [0,128), dP [128,256), accumulators after;
  // the dQ kernel keeps Q and dO as A operands (D / 2 columns each) after its
  // one accumulator.  The dK/dV kernel places the two halves as slots of
  // 128 columns instead: half h's S^T at 128 h, its dP^T at 128 h + 64 (and,
  // with kFuse, the half's dQ^T over the dP^T columns once they are read).
  static constexpr uint32_t kTmS = 0, kTmDP = 128, kTmAcc0 = 256, kTmAcc1 = 256 + D;
  static constexpr uint32_t kTmQt = 256 + D, kTmDOt = 256 + D + D / 2;
  static_assert(kTmDOt + D / 2 <= 512, "tensor memory budget of the dQ kernel");
  static constexpr uint32_t kTmKt = 256 + 2 * D, kTmVt = 256 + 2 * D + D / 2;
  static_assert(!kKVinTmem || (kTmKt < kTmVt && kTmVt + D / 2 <= 512),
                "tensor memory budget of the dK/dV kernel");
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kSmemKV <= 227 * 1024 && kSmemQ <= 227 * 1024, "shared memory budget");
};

// Does query block [r0, r0 + 128) of a row group hold a row that sees a key
// of the block starting at kv0?  (Rows are head-in-group * S_q + position.)
__device__ __forceinline__ bool qblock_sees(const BwdParams& p, int r0, int kv0) {
  if (!p.causal) return true;
  const int last = min(r0 + kRows, p.R) - 1;
  if (r0 / p.S_q != last / p.S_q) return true;  // spans two heads: some row has a late position
  return last % p.S_q >= kv0;
}

// Causal grids: CTA idx -> (cost rank, row group), the costliest ranks first,
// in bands of kRankBand ranks; within a band the CTAs of one row group are
// adjacent.  The CTAs that run at once (one per SM) then cover a few row
// groups and share those groups' tiles in L2, instead of every group's (a
// rank-major order over 32 groups at 16K rows reads 256 MB of Q and dO per
// sweep, twice the L2).
constexpr int kRankBand = 16;

__device__ __forceinline__ void banded_rank(int idx, int n_ranks, int groups, int& rank,
                                            int& zkv) {
  const int full = n_ranks / kRankBand;  // whole bands
  const int per_band = groups * kRankBand;
  if (idx < full * per_band) {
    const int band = idx / per_band;
    const int rem = idx - band * per_band;
    zkv = rem / kRankBand;
    rank = band * kRankBand + (rem - zkv * kRankBand);
  } else {
    const int tail = n_ranks - full * kRankBand;  // ranks of the last, partial band
    const int rem = idx - full * per_band;
    zkv = rem / tail;
    rank = full * kRankBand + (rem - zkv * tail);
  }
}

}  // namespace

// ---------------------------------------------------------------- prep

// D_i = dO_i . O_i and LSE_i * log2(e), per row of the padded per-group
// layout [groups, Rp] (rows R..Rp-1 of a group get 0); with the fused dQ
// also zeros for the row's D fp32 accumulators.  A warp takes
// kPrepRowsPerWarp consecutive rows; a lane reads 16 bytes of O and of dO
// per row, and every load of the warp's rows is issued before any product,
// so each thread keeps several loads in flight (the kernel streams O and dO
// from HBM).
constexpr int kPrepRowsPerWarp = 8;

template <int D>
__global__ void __launch_bounds__(256) attn_bwd_prep_kernel(const BwdParams p,
                                                            const uint16_t* __restrict__ o,
                                                            const uint16_t* __restrict__ dout,
                                                            const float* __restrict__ lse) {
  constexpr int kLanesPerRow = D * 2 / 16;             // 16-byte pieces of a row
  constexpr int kRowsPerLoad = 32 / kLanesPerRow;      // rows one warp-wide load covers
  constexpr int kLoads = kPrepRowsPerWarp / kRowsPerLoad;
  const long long row0 = ((long long)blockIdx.x * 8 + (threadIdx.x >> 5)) * kPrepRowsPerWarp;
  const int lane = threadIdx.x & 31;
  const int sub = lane / kLanesPerRow;                 // row of a load
  const int piece = lane % kLanesPerRow;               // 16-byte piece within the row
  const long long total = (long long)p.groups * p.Rp;
  uint4 a[kLoads], b[kLoads];
#pragma unroll
  for (int i = 0; i < kLoads; ++i) {
    const long long row = row0 + i * kRowsPerLoad + sub;
    a[i] = make_uint4(0u, 0u, 0u, 0u);
    b[i] = make_uint4(0u, 0u, 0u, 0u);
    if (row < total) {
      const long long z = row / p.Rp;
      const int rho = (int)(row - z * p.Rp);
      if (rho < p.R) {
        const long long src = (z * p.R + rho) * D + piece * 8;
        a[i] = *reinterpret_cast<const uint4*>(o + src);
        b[i] = *reinterpret_cast<const uint4*>(dout + src);
      }
    }
  }
#pragma unroll
  for (int i = 0; i < kLoads; ++i) {
    const uint32_t av[4] = {a[i].x, a[i].y, a[i].z, a[i].w};
    const uint32_t bv[4] = {b[i].x, b[i].y, b[i].z, b[i].w};
    float acc = 0.f;
#pragma unroll
    for (int t = 0; t < 4; ++t) {
      acc += __uint_as_float(av[t] << 16) * __uint_as_float(bv[t] << 16);
      acc += __uint_as_float(av[t] & 0xffff0000u) * __uint_as_float(bv[t] & 0xffff0000u);
    }
    // sum over the row's lanes (a contiguous group of kLanesPerRow lanes)
#pragma unroll
    for (int off = kLanesPerRow / 2; off > 0; off >>= 1) acc += __shfl_xor_sync(kAll, acc, off);
    const long long row = row0 + i * kRowsPerLoad + sub;
    if (p.dq_acc != nullptr && row < total) {
      float4* acc = reinterpret_cast<float4*>(p.dq_acc + row * D + piece * 8);
      acc[0] = make_float4(0.f, 0.f, 0.f, 0.f);
      acc[1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
    if (piece == 0 && row < total) {
      const long long z = row / p.Rp;
      const int rho = (int)(row - z * p.Rp);
      if (rho < p.R) {
        p.ndelta[row] = -acc;
        p.nlse2[row] = -(lse[z * p.R + rho] * 1.4426950408889634f);
      } else {
        p.ndelta[row] = 0.f;
        p.nlse2[row] = 0.f;
      }
    }
  }
}

// dq = bf16(scale * dq_acc) over the rows of every group (padding rows
// skipped); one thread per 8 elements.
template <int D>
__global__ void __launch_bounds__(256) attn_bwd_dq_convert_kernel(const BwdParams p) {
  constexpr int kPieces = D / 8;
  const long long i = (long long)blockIdx.x * 256 + threadIdx.x;
  const long long total = (long long)p.groups * p.R * kPieces;
  if (i >= total) return;
  const long long row = i / kPieces;   // z * R + rho
  const int piece = (int)(i - row * kPieces);
  const long long z = row / p.R;
  const long long rho = row - z * p.R;
  const float4* src = reinterpret_cast<const float4*>(p.dq_acc + (z * p.Rp + rho) * D + piece * 8);
  const float4 a = src[0], b = src[1];
  const float sc = p.scale;
  uint4 out;
  out.x = pack_bf16x2(a.x * sc, a.y * sc);
  out.y = pack_bf16x2(a.z * sc, a.w * sc);
  out.z = pack_bf16x2(b.x * sc, b.y * sc);
  out.w = pack_bf16x2(b.z * sc, b.w * sc);
  *reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.dq) + row * D + piece * 8) = out;
}

// ---------------------------------------------------------------- dK, dV

// kFuse: dQ too.  Per half block the tensor core also computes
// dQ^T = K^T dS^T (dS^T from a shared buffer the elementwise warps write)
// into the half's dP^T columns, and warps 12-15 read it out and add it into
// the fp32 accumulator p.dq_acc in L2 (red.global.add); dS^T for dK then
// sits in tensor memory next to P^T.  512 threads.
template <int D, bool kFuse>
__global__ void __launch_bounds__(kFuse ? kThreadsFused : kThreadsB, 1)
    attn_bwd_dkdv_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw_b[];
  uint8_t* smem = align_smem_1024(smem_raw_b);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBarKV);
  uint64_t* kv_full = bars;
  uint64_t* q_full = bars + 1;
  uint64_t* q_empty = q_full + C::kQStages;
  uint64_t* sp_full = q_empty + C::kQStages;   // [half]: S^T, dP^T of the half computed
  uint64_t* ps_ready = sp_full + 2;            // [half]: P^T, dS^T of the half stored
  uint64_t* acc_done = sp_full + 4;
  uint64_t* drain = sp_full + 5;
  uint64_t* kt_ready = sp_full + 6;            // K and V copied into tensor memory (D = 64)
  uint64_t* dq_full = sp_full + 7;             // [half]: dQ^T of the half computed (kFuse)
  uint64_t* dq_free = sp_full + 9;             // [half]: dQ^T of the half read out (kFuse)
  uint64_t* ds_free = sp_full + 11;            // the GEMMs reading the dS^T buffer are done
  uint8_t* sDsT = smem + C::kOffDsT;
  uint32_t* sTmemBase = reinterpret_cast<uint32_t*>(smem + C::kOffMiscKV);
  volatile int* sAbort = reinterpret_cast<volatile int*>(smem + C::kOffMiscKV + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t budget = p.timeout_ns;

  // CTA -> (key block, row group): with the causal mask the first key
  // blocks carry the most query blocks, so they go first (in bands, see
  // banded_rank); without it the blocks of one group are adjacent (they
  // share their Q and dO tiles in L2)
  const int n_kvb = (p.S_kv + kRows - 1) / kRows;
  int kvb, zkv;
  if (p.causal) {
    banded_rank((int)blockIdx.x, n_kvb, p.groups, kvb, zkv);
  } else {
    zkv = blockIdx.x / n_kvb;
    kvb = blockIdx.x - zkv * n_kvb;
  }
  const int kv0 = kvb * kRows;              // first key of the block
  const int n_qb = (p.R + kRows - 1) / kRows;
  // the order every role walks the query blocks in: with kFuse and no mask
  // rotated by the key block, so the CTAs running at once add into
  // different dQ rows (with the causal mask each key block starts at its own
  // diagonal anyway)
  const int rot = (kFuse && !p.causal) ? kvb % n_qb : 0;
  auto qb_at = [&](int i) { return i + rot < n_qb ? i + rot : i + rot - n_qb; };
  // The query blocks with work (items n = 0 .. n_work - 1), walked by every
  // role in the same order.  With the causal mask and S_q a multiple of 128
  // no block spans two heads, and block pb of a head sees keys kv0 .. when
  // its last position pb * 128 + 127 >= kv0, i.e. pb >= kvb: the items are
  // those blocks of each head in turn, found without a scan (a scan's
  // division per skipped block cost a short CTA tens of microseconds).
  // Otherwise (a ragged S_q) the blocks are scanned with qblock_sees.
  const bool by_head = p.causal && (p.S_q % kRows == 0);
  const int nqh = by_head ? p.S_q / kRows : 1;             // position blocks per head
  const int per_head = by_head ? (nqh > kvb ? nqh - kvb : 0) : 0;
  int n_work = 0;
  if (!p.causal) {
    n_work = n_qb;
  } else if (by_head) {
    n_work = (p.R / p.S_q) * per_head;
  } else {
    for (int qb = 0; qb < n_qb; ++qb) n_work += qblock_sees(p, qb * kRows, kv0) ? 1 : 0;
  }
  // first row of item n's query block; `cursor` is the caller's scan
  // position (the ragged causal case only; items are asked for in order)
  auto item_r0 = [&](int n, int& cursor) -> int {
    if (!p.causal) return qb_at(n) * kRows;
    if (by_head) {
      const int h = n / per_head;
      return (h * nqh + kvb + (n - h * per_head)) * kRows;
    }
    while (cursor < n_qb - 1 && !qblock_sees(p, cursor * kRows, kv0)) ++cursor;
    return (cursor++) * kRows;
  };

  if (threadIdx.x == 0) {
    mbar_init(kv_full, 1);
    for (int s = 0; s < C::kQStages; ++s) {
      mbar_init(&q_full[s], 1);
      mbar_init(&q_empty[s], 1);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(&sp_full[h], 1);
      mbar_init(&ps_ready[h], 2 * 128);
    }
    mbar_init(acc_done, 1);
    mbar_init(drain, 1);
    mbar_init(kt_ready, 2 * 128);
    for (int h = 0; h < 2; ++h) {
      mbar_init(&dq_full[h], 1);
      mbar_init(&dq_free[h], 128);
    }
    mbar_init(ds_free, 1);
    *sAbort = 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc(sTmemBase, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *sTmemBase;
  uint8_t* sK = smem + C::kOffK;
  uint8_t* sV = smem + C::kOffV;
  auto stage_q = [&](int s) { return smem + C::kOffQRing + s * C::kQStageBytes; };
  auto stage_do = [&](int s) { return stage_q(s) + C::kTileBytes; };
  auto stage_lse = [&](int s) {
    return reinterpret_cast<float*>(stage_q(s) + 2 * C::kTileBytes);
  };
  auto stage_delta = [&](int s) {
    return reinterpret_cast<float*>(stage_q(s) + 2 * C::kTileBytes + C::kVecBytes);
  };

  if (warp < 8) {
    // -------------------------------------------------------- elementwise
    // half h of a block is queries 64h .. 64h + 63; warpgroup w takes
    // queries 64h + 32w .. 64h + 32w + 31 of it
    const int w = warp >> 2;
    const int r = (warp & 3) * 32 + lane;          // key row within the block
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int key = kv0 + r;
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = f2_pack(sl2, sl2);
    bool ok = true;
    if constexpr (C::kKVinTmem) {
      // K (warpgroup 0) and V (warpgroup 1) into tensor memory, the A
      // operands of every S^T and dP^T product of this CTA
      if (n_work > 0) {
        ok = warp_wait_b(kv_full, 0, sAbort, budget);
        if (ok) {
          copy_tile_to_tmem<D>(w == 0 ? sK : sV, tmem + lane_base + (w == 0 ? C::kTmKt : C::kTmVt), r);
          tmem_st_wait();
          tc_fence_before_sync();
          mbar_arrive(kt_ready);
        }
      }
    }
    int cursor = 0;
    for (int n = 0; n < n_work && ok; ++n) {
      const int r0 = item_r0(n, cursor);
      const int s = n % C::kQStages;
      // masking: rows past R, keys past S_kv, and (causal) keys after a row's
      // position; a block needs none when every row sees every key
      bool masked = (r0 + kRows > p.R) || (kv0 + kRows > p.S_kv);
      int base_pos = 0;
      if (p.causal) {
        base_pos = r0 % p.S_q;
        const bool one_head = (base_pos + kRows <= p.S_q);
        masked = masked || !(one_head && base_pos >= kv0 + kRows - 1);
      }
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        if (!warp_wait_b(&sp_full[h], n & 1, sAbort, budget)) { ok = false; break; }
        // the stage's LSE and D vectors arrived with its tiles: observe that
        // phase here too before reading them
        if (h == 0 && !warp_wait_b(&q_full[s], (n / C::kQStages) & 1, sAbort, budget)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        const int col0 = 64 * h + 32 * w;            // first query of this thread's slice
        const uint32_t cS = 128 * h + 32 * w;        // its S^T columns (dP^T: + 64)
        uint32_t sv[32], dp[32];
        tmem_ld_x32(tmem + lane_base + cS, sv);
        tmem_ld_x32(tmem + lane_base + cS + 64, dp);
        const float4* lse4 = reinterpret_cast<const float4*>(stage_lse(s) + col0);
        const float4* dl4 = reinterpret_cast<const float4*>(stage_delta(s) + col0);
        tmem_ld_wait();
        reg_after_wait(sv);
        reg_after_wait(dp);
        uint32_t pk[16], dk[16];
        // The masked and unmasked bodies are separate code paths, so the
        // common (unmasked) one carries no per-element mask arithmetic.
        auto body = [&](auto masked_tag) {
          constexpr bool kMasked = decltype(masked_tag)::value;
#pragma unroll
          for (int i4 = 0; i4 < 8; ++i4) {
            const float4 l4 = lse4[i4];              // -LSE * log2(e) of 4 queries
            const float4 d4 = dl4[i4];               // -D of the same queries
            const int c = 4 * i4;                    // first element of the four
            // x = s * scale * log2(e) - LSE * log2(e), two lanes per instruction
            float x[4];
            f2_unpack(f2_fma(f2_pack(u2f_b(sv[c]), u2f_b(sv[c + 1])), sl2x2, f2_pack(l4.x, l4.y)),
                      x[0], x[1]);
            f2_unpack(f2_fma(f2_pack(u2f_b(sv[c + 2]), u2f_b(sv[c + 3])), sl2x2,
                             f2_pack(l4.z, l4.w)), x[2], x[3]);
            float pr[4];
#pragma unroll
            for (int e = 0; e < 4; ++e) {
              float pv = ex2_approx(x[e]);
              if constexpr (kMasked) {
                const int rho = r0 + col0 + c + e;
                bool vis = (rho < p.R) && (key < p.S_kv);
                if (p.causal) {
                  int pos;
                  if (p.S_q >= kRows) {
                    pos = base_pos + col0 + c + e;
                    if (pos >= p.S_q) pos -= p.S_q;
                  } else {
                    pos = rho % p.S_q;
                  }
                  vis = vis && (key <= pos);
                }
                pv = vis ? pv : 0.f;
              }
              pr[e] = pv;
            }
            // dS = P (dP - D)
            const uint64_t ds01 = f2_mul(f2_pack(pr[0], pr[1]),
                                         f2_add(f2_pack(u2f_b(dp[c]), u2f_b(dp[c + 1])),
                                                f2_pack(d4.x, d4.y)));
            const uint64_t ds23 = f2_mul(f2_pack(pr[2], pr[3]),
                                         f2_add(f2_pack(u2f_b(dp[c + 2]), u2f_b(dp[c + 3])),
                                                f2_pack(d4.z, d4.w)));
            float d0, d1, d2, d3;
            f2_unpack(ds01, d0, d1);
            f2_unpack(ds23, d2, d3);
            pk[2 * i4] = pack_bf16x2(pr[0], pr[1]);
            pk[2 * i4 + 1] = pack_bf16x2(pr[2], pr[3]);
            dk[2 * i4] = pack_bf16x2(d0, d1);
            dk[2 * i4 + 1] = pack_bf16x2(d2, d3);
          }
        };
        if (masked)
          body(std::true_type{});
        else
          body(std::false_type{});
        // P^T of the slice: 16 columns from its S^T columns (this
        // warpgroup's own, already read)
        tmem_st_x16(tmem + lane_base + cS, pk);
        if constexpr (kFuse) {
          // dS^T of the slice into the shared buffer (row = key, this
          // warpgroup's 32 queries = 16-byte pieces 4w .. 4w + 3 of the
          // swizzled row), once the previous half's GEMMs have read it
          const int nh = 2 * n + h;
          if (nh > 0 && !warp_wait_b(ds_free, (nh - 1) & 1, sAbort, budget)) {
            ok = false;
            break;
          }
          const uint32_t row = smem_u32(sDsT) + (uint32_t)r * 128u;
#pragma unroll
          for (int j = 0; j < 4; ++j)
            st_shared_v4(row + 16u * (uint32_t)((4 * w + j) ^ (r & 7)), dk[4 * j], dk[4 * j + 1],
                         dk[4 * j + 2], dk[4 * j + 3]);
          fence_proxy_async_smem();  // the tensor core reads it through the async proxy
          // and into the slice's own S^T columns 16-31 (dK's A operand): the
          // half's dP^T columns take dQ^T
          tmem_st_x16(tmem + lane_base + cS + 16, dk);
        } else {
          // dS^T over the slice's dP^T columns, likewise
          tmem_st_x16(tmem + lane_base + cS + 64, dk);
        }
        tmem_st_wait();
        tc_fence_before_sync();
        if (!(w == 0 && h == 0 && n == p.fault_drop_item)) mbar_arrive(&ps_ready[h]);
      }
    }
    // ---------------------------------------------------------- epilogue
    // warpgroup w writes columns [D/2 w, D/2 (w + 1)) of dV and dK
    bool have_acc = ok && n_work > 0;
    if (have_acc) {
      if (!warp_wait_b(acc_done, 0, sAbort, budget)) { ok = false; have_acc = false; }
      tc_fence_after_sync();
    }
    const bool row_ok = key < p.S_kv;
    uint16_t* dk_row = static_cast<uint16_t*>(p.dk) + ((size_t)zkv * p.S_kv + key) * D;
    uint16_t* dv_row = static_cast<uint16_t*>(p.dv) + ((size_t)zkv * p.S_kv + key) * D;
#pragma unroll
    for (int which = 0; which < 2; ++which) {  // 0: dV, 1: dK
      uint16_t* dst = which ? dk_row : dv_row;
      const float mult = which ? p.scale : 1.f;
      const uint32_t acc = tmem + lane_base + (which ? C::kTmAcc1 : C::kTmAcc0) + (D / 2) * w;
#pragma unroll
      for (int ch = 0; ch < D / 64; ++ch) {
        uint32_t v[32];
        if (have_acc) {
          tmem_ld_x32(acc + ch * 32, v);
          tmem_ld_wait();
          reg_after_wait(v);
        } else {
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] = 0u;  // no query sees these keys
        }
        if (row_ok && ok) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + (D / 2) * w + ch * 32);
#pragma unroll
          for (int qd = 0; qd < 4; ++qd) {
            uint4 val;
            val.x = pack_bf16x2(u2f_b(v[qd * 8 + 0]) * mult, u2f_b(v[qd * 8 + 1]) * mult);
            val.y = pack_bf16x2(u2f_b(v[qd * 8 + 2]) * mult, u2f_b(v[qd * 8 + 3]) * mult);
            val.z = pack_bf16x2(u2f_b(v[qd * 8 + 4]) * mult, u2f_b(v[qd * 8 + 5]) * mult);
            val.w = pack_bf16x2(u2f_b(v[qd * 8 + 6]) * mult, u2f_b(v[qd * 8 + 7]) * mult);
            d4[qd] = val;
          }
        }
      }
    }
  } else if (warp == 8) {
    // -------------------------------------------------------- tensor-core issuer
    const bool leader = elect_one();
    const uint64_t dK = kmajor_tile_desc(smem_u32(sK));
    const uint64_t dV = kmajor_tile_desc(smem_u32(sV));
    // half h's slot: S^T (then P^T) at 128 h, dP^T (then dQ^T) at 128 h + 64
    const uint32_t tS = tmem, tDP = tmem + 64;
    const uint32_t tdV = tmem + C::kTmAcc0, tdK = tmem + C::kTmAcc1;
    bool ok = n_work > 0 &&
              warp_wait_b(C::kKVinTmem ? kt_ready : kv_full, 0, sAbort, budget);
    // S^T and dP^T of half h of work item n (its Q / dO stage is loaded);
    // at D = 64 K and V are read from tensor memory
    auto issue_sp = [&](int n, int h) {
      const int s = n % C::kQStages;
      if (leader) {
        if constexpr (C::kKVinTmem) {
          issue_qk_half_ts<D>(tS + 128 * h, tmem + C::kTmKt, kmajor_tile_desc(smem_u32(stage_q(s))), h);
          issue_qk_half_ts<D>(tDP + 128 * h, tmem + C::kTmVt, kmajor_tile_desc(smem_u32(stage_do(s))), h);
        } else {
          issue_qk_half<D>(tS + 128 * h, dK, kmajor_tile_desc(smem_u32(stage_q(s))), h);
          issue_qk_half<D>(tDP + 128 * h, dV, kmajor_tile_desc(smem_u32(stage_do(s))), h);
        }
        tc_commit(&sp_full[h]);
      }
    };
    if (ok && warp_wait_b(&q_full[0], 0, sAbort, budget)) {
      tc_fence_after_sync();
      issue_sp(0, 0);
      issue_sp(0, 1);
    } else {
      ok = false;
    }
    for (int n = 0; n < n_work && ok; ++n) {
      const int s = n % C::kQStages;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        if (!warp_wait_b(&ps_ready[h], n & 1, sAbort, budget)) { ok = false; break; }
        tc_fence_after_sync();
        if (leader) {
          if constexpr (kFuse) {
            // dQ^T = K^T dS^T first, so its read-out overlaps the next two;
            // it is the only reader of the dS^T buffer
            issue_dqt_half<D>(tDP + 128 * h, mnmajor_tile_desc<D>(smem_u32(sK)),
                              mnmajor_tile_desc<64>(smem_u32(sDsT)));
            tc_commit(&dq_full[h]);
            tc_commit(ds_free);
          }
          // dV += P^T dO and dK += dS^T Q over this half's 64 queries; with
          // kFuse dS^T sits in the S^T columns next to P^T (columns 16-31 of
          // each warpgroup's 32), otherwise over the dP^T columns
          issue_pv_half<D>(tdV, tS + 128 * h, mnmajor_tile_desc<D>(smem_u32(stage_do(s))), h,
                           n > 0 || h > 0);
          issue_pv_half<D>(tdK, kFuse ? tS + 128 * h + 16 : tDP + 128 * h,
                           mnmajor_tile_desc<D>(smem_u32(stage_q(s))), h, n > 0 || h > 0);
          if (h == 1) tc_commit(&q_empty[s]);  // both halves read: the stage is free
        }
        // the next item's half h overwrites what these GEMMs read: issued
        // after them by the same thread, it runs after them
        if (n + 1 < n_work) {
          if (h == 0) {
            if (!warp_wait_b(&q_full[(n + 1) % C::kQStages], ((n + 1) / C::kQStages) & 1,
                             sAbort, budget)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
          }
          if constexpr (kFuse) {
            // ... and over this half's dQ^T once it has been read out
            if (!warp_wait_b(&dq_free[h], n & 1, sAbort, budget)) { ok = false; break; }
            tc_fence_after_sync();
          }
          issue_sp(n + 1, h);
        }
      }
    }
    if (ok && leader) tc_commit(acc_done);
    if (leader) {
      tc_commit(drain);
      drain_wait_b(drain, 0, budget);
    }
    __syncwarp();
  } else if (warp == 9) {
    // -------------------------------------------------------- TMA producer
    const bool leader = elect_one();
    const uint64_t pol_kv = l2_policy_evict_first();
    const uint64_t pol_q = l2_policy_evict_last();
    int issued = 0;
    bool ok = n_work > 0;
    if (ok && leader) {
      mbar_arrive_expect_tx(kv_full, 2 * C::kTileBytes);
      tma_load_tile<D>(sK, &p.tm_k, kv_full, kv0, zkv, pol_kv);
      tma_load_tile<D>(sV, &p.tm_v, kv_full, kv0, zkv, pol_kv);
    }
    int cursor = 0;
    for (int n = 0; n < n_work && ok; ++n) {
      const int r0 = item_r0(n, cursor);
      const int s = issued % C::kQStages;
      const int round = issued / C::kQStages;
      if (round > 0 && !warp_wait_b(&q_empty[s], (round - 1) & 1, sAbort, budget)) {
        ok = false;
        break;
      }
      if (leader) {
        mbar_arrive_expect_tx(&q_full[s], 2 * C::kTileBytes + 2 * C::kVecBytes);
        tma_load_tile<D>(stage_q(s), &p.tm_q, &q_full[s], r0, zkv, pol_q);
        tma_load_tile<D>(stage_do(s), &p.tm_do, &q_full[s], r0, zkv, pol_q);
        const size_t vo = (size_t)zkv * p.Rp + r0;
        bulk_load(stage_lse(s), p.nlse2 + vo, C::kVecBytes, &q_full[s]);
        bulk_load(stage_delta(s), p.ndelta + vo, C::kVecBytes, &q_full[s]);
      }
      ++issued;
    }
    if (leader) {
      if (n_work > 0) drain_wait_b(kv_full, 0, budget);
      const int first = issued > C::kQStages ? issued - C::kQStages : 0;
      for (int t = first; t < issued; ++t)
        drain_wait_b(&q_full[t % C::kQStages], (t / C::kQStages) & 1, budget);
    }
    __syncwarp();
  } else if (kFuse && warp >= 12) {
    // -------------------------------------------------------- dQ read-out
    // thread = TMEM lane = head dimension d (D = 64: lanes 0-15 of each
    // quadrant, d = 16 q + lane); per half block it takes the 64 queries'
    // dQ^T values of its d and adds them into rows r0 + 64 h + j of the
    // group's fp32 accumulator (a warp's lanes cover 128 or 64 contiguous
    // bytes of a row)
    const bool has_d = (D == 128) || lane < 16;
    const int d = (D == 128) ? (warp & 3) * 32 + lane : (warp & 3) * 16 + (lane & 15);
    // D = 64: a warp's red would carry 64 bytes only, and the L2 takes
    // requests at a bounded rate whatever their size; instead the half's
    // values go to a staging buffer and one thread adds all 16 KB with a
    // bulk reduction (one bulk group per half block; two buffers)
    float* sStage = reinterpret_cast<float*>(smem + C::kOffDqStage);
    int nh = 0;
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    bool ok = true;
    int cursor = 0;
    for (int n = 0; n < n_work && ok; ++n) {
      const int r0 = item_r0(n, cursor);
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        if constexpr (D == 64) {
          // the bulk reduction that read this half's staging buffer two
          // halves ago is done (one bulk group per half)
          if (threadIdx.x == 12 * 32) tma_store_wait_read<1>();
        }
        const bool got = warp_wait_b(&dq_full[h], n & 1, sAbort, budget);
        if constexpr (D == 64) {
          // the four warps agree (they meet at named barriers below, which
          // no warp may skip); this also orders the buffer's reuse
          if (barrier_or(1, 128, !got)) { ok = false; break; }
        } else {
          if (!got) { ok = false; break; }
        }
        tc_fence_after_sync();
        uint32_t v0[32], v1[32];
        tmem_ld_x32(tmem + lane_base + 128 * h + 64, v0);
        tmem_ld_x32(tmem + lane_base + 128 * h + 96, v1);
        tmem_ld_wait();
        reg_after_wait(v0);
        reg_after_wait(v1);
        tc_fence_before_sync();
        mbar_arrive(&dq_free[h]);            // the columns may be overwritten
        const int q0 = r0 + 64 * h;
        if constexpr (D == 128) {
          const int rows = p.R - q0;           // rows past R are padding: skipped
          float* dst = p.dq_acc + ((size_t)zkv * p.Rp + q0) * D + d;
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (j < rows) red_add_f32(dst + (size_t)j * D, u2f_b(v0[j]));
#pragma unroll
          for (int j = 0; j < 32; ++j)
            if (32 + j < rows) red_add_f32(dst + (size_t)(32 + j) * D, u2f_b(v1[j]));
        } else {
          float* stg = sStage + (nh & 1) * 64 * D;
          if (has_d) {
#pragma unroll
            for (int j = 0; j < 32; ++j) stg[j * D + d] = u2f_b(v0[j]);
#pragma unroll
            for (int j = 0; j < 32; ++j) stg[(32 + j) * D + d] = u2f_b(v1[j]);
          }
          fence_proxy_async_smem();            // the bulk copy reads through the async proxy
          named_barrier_sync(1, 128);
          if (threadIdx.x == 12 * 32) {
            const int rows = min(64, p.R - q0);  // rows past R are padding: skipped
            if (rows > 0)
              bulk_reduce_add_f32(p.dq_acc + ((size_t)zkv * p.Rp + q0) * D, smem_u32(stg),
                                  (uint32_t)rows * D * 4);
            tma_store_commit();                // one group per half, possibly empty
          }
          ++nh;
        }
      }
    }
    // every bulk reduction has read its buffer and reached global memory
    if (D == 64 && threadIdx.x == 12 * 32) tma_store_wait_all();
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 8) tmem_dealloc(tmem, C::kTmemCols);
  if (threadIdx.x == 0 && *sAbort) atomicCAS(&g_bwd_status, 0, (int)ATTN_ERR_TIMEOUT);
}

// ---------------------------------------------------------------- dQ

template <int D>
__global__ void __launch_bounds__(kThreadsB, 1) attn_bwd_dq_kernel(const __grid_constant__ BwdParams p) {
  using C = BwdCfg<D>;
  extern __shared__ uint8_t smem_raw_b[];
  uint8_t* smem = align_smem_1024(smem_raw_b);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBarQ);
  uint64_t* q_full = bars;
  uint64_t* kv_full = bars + 1;
  uint64_t* kv_empty = kv_full + C::kKVStages;
  uint64_t* sp_full = kv_empty + C::kKVStages;  // [half]: S, dP of the half computed
  uint64_t* ds_ready = sp_full + 2;             // [half]: dS of the half stored
  uint64_t* acc_done = sp_full + 4;
  uint64_t* drain = sp_full + 5;
  uint64_t* qt_ready = sp_full + 6;             // Q and dO copied into tensor memory
  uint32_t* sTmemBase = reinterpret_cast<uint32_t*>(smem + C::kOffMiscQ);
  volatile int* sAbort = reinterpret_cast<volatile int*>(smem + C::kOffMiscQ + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t budget = p.timeout_ns;

  // CTA -> (query block, row group): with the causal mask by cost rank,
  // longest first (with S_q a multiple of 128 a rank is one position block
  // of one head of the group, so the group's heads interleave), in bands
  // (see banded_rank); without it group-major, query blocks last to first
  const int n_qb = (p.R + kRows - 1) / kRows;
  int qb, zkv;
  if (p.causal) {
    int rank;
    banded_rank((int)blockIdx.x, n_qb, p.groups, rank, zkv);
    const int hr = p.R / p.S_q;  // heads per group
    if (p.S_q % kRows == 0) {
      const int nh = p.S_q / kRows;
      qb = (rank % hr) * nh + (nh - 1 - rank / hr);
    } else {
      qb = n_qb - 1 - rank;
    }
  } else {
    zkv = blockIdx.x / n_qb;
    qb = n_qb - 1 - (blockIdx.x - zkv * n_qb);
  }
  const int r0 = qb * kRows;
  int kv_end = p.S_kv;
  if (p.causal) {
    const int last = min(r0 + kRows, p.R) - 1;
    kv_end = min(p.S_kv, (r0 / p.S_q == last / p.S_q) ? last % p.S_q + 1 : p.S_q);
  }
  const int n_kb = (kv_end + kRows - 1) / kRows;   // >= 1: every row sees key 0

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    for (int s = 0; s < C::kKVStages; ++s) {
      mbar_init(&kv_full[s], 1);
      mbar_init(&kv_empty[s], 1);
    }
    for (int h = 0; h < 2; ++h) {
      mbar_init(&sp_full[h], 1);
      mbar_init(&ds_ready[h], 2 * 128);
    }
    mbar_init(acc_done, 1);
    mbar_init(drain, 1);
    mbar_init(qt_ready, 2 * 128);
    *sAbort = 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc(sTmemBase, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *sTmemBase;
  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sDO = smem + C::kOffDO;
  auto stage_k = [&](int s) { return smem + C::kOffKVRing + s * 2 * C::kTileBytes; };
  auto stage_v = [&](int s) { return stage_k(s) + C::kTileBytes; };

  if (warp < 8) {
    // -------------------------------------------------------- elementwise
    const int w = warp >> 2;                       // key columns 64w .. 64w + 63
    const int r = (warp & 3) * 32 + lane;          // query row within the block
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const int rho = r0 + r;
    const bool row_ok = rho < p.R;
    const size_t vo = (size_t)zkv * p.Rp + rho;    // in the padded layout (rho < Rp)
    const uint64_t nlse2x2 = f2_pack(p.nlse2[vo], p.nlse2[vo]);  // -LSE * log2(e), twice
    const uint64_t ndl2 = f2_pack(p.ndelta[vo], p.ndelta[vo]);    // -D_i, twice
    const int pos = rho % p.S_q;
    const int key_limit = p.causal ? min(p.S_kv, pos + 1) : p.S_kv;
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = f2_pack(sl2, sl2);
    // Q (warpgroup 0) and dO (warpgroup 1) into tensor memory, the A
    // operands of every S and dP product of this CTA
    bool ok = warp_wait_b(q_full, 0, sAbort, budget);
    if (ok) {
      copy_tile_to_tmem<D>(w == 0 ? sQ : sDO, tmem + lane_base + (w == 0 ? C::kTmQt : C::kTmDOt), r);
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(qt_ready);
    }
    for (int j = 0; j < n_kb && ok; ++j) {
      const int kb0 = j * kRows;
      const bool masked = !row_ok || (kb0 + kRows > key_limit);
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        if (!warp_wait_b(&sp_full[h], j & 1, sAbort, budget)) { ok = false; break; }
        tc_fence_after_sync();
        // half h is keys 64h .. 64h + 63 of the block; this warpgroup's
        // slice is keys 64h + 32w .. 64h + 32w + 31
        const int col0 = 64 * h + 32 * w;
        uint32_t sv[32], dp[32];
        tmem_ld_x32(tmem + lane_base + C::kTmS + col0, sv);
        tmem_ld_x32(tmem + lane_base + C::kTmDP + col0, dp);
        tmem_ld_wait();
        reg_after_wait(sv);
        reg_after_wait(dp);
        uint32_t dk[16];
        // separate masked and unmasked code paths, as in the dK/dV kernel
        auto body = [&](auto masked_tag) {
          constexpr bool kMasked = decltype(masked_tag)::value;
#pragma unroll
          for (int i = 0; i < 16; ++i) {
            const int c = 2 * i;
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(u2f_b(sv[c]), u2f_b(sv[c + 1])), sl2x2, nlse2x2), x0, x1);
            float p0 = ex2_approx(x0), p1 = ex2_approx(x1);
            if constexpr (kMasked) {
              p0 = (row_ok && kb0 + col0 + c < key_limit) ? p0 : 0.f;
              p1 = (row_ok && kb0 + col0 + c + 1 < key_limit) ? p1 : 0.f;
            }
            float d0, d1;
            f2_unpack(f2_mul(f2_pack(p0, p1),
                             f2_add(f2_pack(u2f_b(dp[c]), u2f_b(dp[c + 1])), ndl2)), d0, d1);
            dk[i] = pack_bf16x2(d0, d1);
          }
        };
        if (masked)
          body(std::true_type{});
        else
          body(std::false_type{});
        // dS of the slice: 16 columns from col0 of the S region (this
        // warpgroup's own, already-read columns)
        tmem_st_x16(tmem + lane_base + C::kTmS + col0, dk);
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(&ds_ready[h]);
      }
    }
    // ---------------------------------------------------------- epilogue
    if (ok && warp_wait_b(acc_done, 0, sAbort, budget)) {
      tc_fence_after_sync();
      uint16_t* dst = static_cast<uint16_t*>(p.dq) + ((size_t)zkv * p.R + rho) * D + (D / 2) * w;
      const uint32_t acc = tmem + lane_base + C::kTmAcc0 + (D / 2) * w;
#pragma unroll
      for (int ch = 0; ch < D / 64; ++ch) {
        uint32_t v[32];
        tmem_ld_x32(acc + ch * 32, v);
        tmem_ld_wait();
        reg_after_wait(v);
        if (row_ok) {
          uint4* d4 = reinterpret_cast<uint4*>(dst + ch * 32);
          const float mult = p.scale;
#pragma unroll
          for (int qd = 0; qd < 4; ++qd) {
            uint4 val;
            val.x = pack_bf16x2(u2f_b(v[qd * 8 + 0]) * mult, u2f_b(v[qd * 8 + 1]) * mult);
            val.y = pack_bf16x2(u2f_b(v[qd * 8 + 2]) * mult, u2f_b(v[qd * 8 + 3]) * mult);
            val.z = pack_bf16x2(u2f_b(v[qd * 8 + 4]) * mult, u2f_b(v[qd * 8 + 5]) * mult);
            val.w = pack_bf16x2(u2f_b(v[qd * 8 + 6]) * mult, u2f_b(v[qd * 8 + 7]) * mult);
            d4[qd] = val;
          }
        }
      }
    }
  } else if (warp == 8) {
    // -------------------------------------------------------- tensor-core issuer
    const bool leader = elect_one();
    const uint64_t dQd = kmajor_tile_desc(smem_u32(sQ));
    const uint64_t dOd = kmajor_tile_desc(smem_u32(sDO));
    const uint32_t tS = tmem + C::kTmS, tDP = tmem + C::kTmDP, tdQ = tmem + C::kTmAcc0;
    const uint32_t tQt = tmem + C::kTmQt, tDOt = tmem + C::kTmDOt;
    (void)dQd;
    (void)dOd;
    bool ok = warp_wait_b(qt_ready, 0, sAbort, budget);
    // S and dP of half h of key block j (its K / V stage is loaded), with Q
    // and dO read from tensor memory
    auto issue_sp = [&](int j, int h) {
      const int s = j % C::kKVStages;
      if (leader) {
        issue_qk_half_ts<D>(tS + 64 * h, tQt, kmajor_tile_desc(smem_u32(stage_k(s))), h);
        issue_qk_half_ts<D>(tDP + 64 * h, tDOt, kmajor_tile_desc(smem_u32(stage_v(s))), h);
        tc_commit(&sp_full[h]);
      }
    };
    if (ok && warp_wait_b(&kv_full[0], 0, sAbort, budget)) {
      tc_fence_after_sync();
      issue_sp(0, 0);
      issue_sp(0, 1);
    } else {
      ok = false;
    }
    for (int j = 0; j < n_kb && ok; ++j) {
      const int s = j % C::kKVStages;
#pragma unroll 1
      for (int h = 0; h < 2; ++h) {
        if (!warp_wait_b(&ds_ready[h], j & 1, sAbort, budget)) { ok = false; break; }
        tc_fence_after_sync();
        if (leader) {
          // dQ += dS K over this half's 64 keys
          issue_pv_half<D>(tdQ, tS + 64 * h, mnmajor_tile_desc<D>(smem_u32(stage_k(s))), h,
                           j > 0 || h > 0);
          if (h == 1) tc_commit(&kv_empty[s]);  // both halves read: the stage is free
        }
        // the next block's half h overwrites the dS these GEMMs read
        if (j + 1 < n_kb) {
          if (h == 0) {
            if (!warp_wait_b(&kv_full[(j + 1) % C::kKVStages], ((j + 1) / C::kKVStages) & 1,
                             sAbort, budget)) {
              ok = false;
              break;
            }
            tc_fence_after_sync();
          }
          issue_sp(j + 1, h);
        }
      }
    }
    if (ok && leader) tc_commit(acc_done);
    if (leader) {
      tc_commit(drain);
      drain_wait_b(drain, 0, budget);
    }
    __syncwarp();
  } else if (warp == 9) {
    // -------------------------------------------------------- TMA producer
    const bool leader = elect_one();
    const uint64_t pol_q = l2_policy_evict_first();
    const uint64_t pol_kv = l2_policy_evict_last();
    if (leader) {
      mbar_arrive_expect_tx(q_full, 2 * C::kTileBytes);
      tma_load_tile<D>(sQ, &p.tm_q, q_full, r0, zkv, pol_q);
      tma_load_tile<D>(sDO, &p.tm_do, q_full, r0, zkv, pol_q);
    }
    int issued = 0;
    for (int j = 0; j < n_kb; ++j) {
      const int s = j % C::kKVStages;
      const int round = j / C::kKVStages;
      if (round > 0 && !warp_wait_b(&kv_empty[s], (round - 1) & 1, sAbort, budget)) break;
      if (leader) {
        mbar_arrive_expect_tx(&kv_full[s], 2 * C::kTileBytes);
        tma_load_tile<D>(stage_k(s), &p.tm_k, &kv_full[s], j * kRows, zkv, pol_kv);
        tma_load_tile<D>(stage_v(s), &p.tm_v, &kv_full[s], j * kRows, zkv, pol_kv);
      }
      ++issued;
    }
    if (leader) {
      drain_wait_b(q_full, 0, budget);
      const int first = issued > C::kKVStages ? issued - C::kKVStages : 0;
      for (int t = first; t < issued; ++t)
        drain_wait_b(&kv_full[t % C::kKVStages], (t / C::kKVStages) & 1, budget);
    }
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 8) tmem_dealloc(tmem, C::kTmemCols);
  if (threadIdx.x == 0 && *sAbort) atomicCAS(&g_bwd_status, 0, (int)ATTN_ERR_TIMEOUT);
}

namespace {

std::mutex g_bwd_mu;
bool g_bwd_attr[2][64] = {};  // [D == 128][device]

template <int D, bool kFuse>
cudaError_t set_dkdv_attr() {
  return cudaFuncSetAttribute(attn_bwd_dkdv_kernel<D, kFuse>,
                              cudaFuncAttributeMaxDynamicSharedMemorySize, BwdCfg<D>::kSmemKV);
}

template <int D>
cudaError_t launch_bwd_d(const BwdParams& p, const void* o, const void* dout, const float* lse,
                         cudaStream_t stream) {
  using C = BwdCfg<D>;
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lk(g_bwd_mu);
    if (!g_bwd_attr[D == 128][dev]) {
      err = set_dkdv_attr<D, false>();
      if (err != cudaSuccess) return err;
      err = set_dkdv_attr<D, true>();
      if (err != cudaSuccess) return err;
      err = cudaFuncSetAttribute(attn_bwd_dq_kernel<D>,
                                 cudaFuncAttributeMaxDynamicSharedMemorySize, C::kSmemQ);
      if (err != cudaSuccess) return err;
      g_bwd_attr[D == 128][dev] = true;
    }
  }
  const long long prep_rows = (long long)p.groups * p.Rp;
  const long long prep_rows_per_block = 8 * kPrepRowsPerWarp;
  attn_bwd_prep_kernel<D><<<(unsigned)((prep_rows + prep_rows_per_block - 1) / prep_rows_per_block),
                            256, 0, stream>>>(
      p, static_cast<const uint16_t*>(o), static_cast<const uint16_t*>(dout), lse);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const unsigned grid_kv = (unsigned)((p.S_kv + kRows - 1) / kRows) * (unsigned)p.groups;
  if (p.dq_acc != nullptr) {
    attn_bwd_dkdv_kernel<D, true><<<grid_kv, kThreadsFused, C::kSmemKV, stream>>>(p);
    err = cudaGetLastError();
    if (err != cudaSuccess) return err;
    const long long pieces = (long long)p.groups * p.R * (D / 8);
    attn_bwd_dq_convert_kernel<D><<<(unsigned)((pieces + 255) / 256), 256, 0, stream>>>(p);
    return cudaGetLastError();
  }
  attn_bwd_dkdv_kernel<D, false><<<grid_kv, kThreadsB, C::kSmemKV, stream>>>(p);
  err = cudaGetLastError();
  if (err != cudaSuccess) return err;
  const unsigned grid_q = (unsigned)((p.R + kRows - 1) / kRows) * (unsigned)p.groups;
  attn_bwd_dq_kernel<D><<<grid_q, kThreadsB, C::kSmemQ, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_bwd(const BwdParams& p, int D, const void* o, const void* dout,
                            const float* lse, cudaStream_t stream) {
  if (D == 128) return launch_bwd_d<128>(p, o, dout, lse, stream);
  if (D == 64) return launch_bwd_d<64>(p, o, dout, lse, stream);
  return cudaErrorInvalidValue;
}

cudaError_t read_bwd_status(int* status, bool reset) {
  cudaError_t err = cudaMemcpyFromSymbol(status, g_bwd_status, sizeof(int));
  if (err != cudaSuccess) return err;
  if (reset) {
    const int zero = 0;
    err = cudaMemcpyToSymbol(g_bwd_status, &zero, sizeof(int));
  }
  return err;
}

}  // namespace attnpipe
