// attn_fwd_sm103.cu -- fused attention forward for sm_103a (GB300).
//
// The operation is the FlashAttention forward of "PipeThreader: Software-
// Defined Pipelining for Efficient DNN Execution" (section A2, paragraph
// "FlashAttention-3", Fig. 7): per KV block j, load_k -> mma_qk -> softmax ->
// rescale -> load_v -> mma_pv, with the KV (reduction) axis tiled so the
// stages of consecutive blocks overlap.  The warp roles follow the Blackwell
// schedule in "GPU软件流水线与Warp Specialization优化技术解析", section 3.1:
// the variable-latency loads and the tensor-core GEMMs each own a warp, the
// softmax of two query sub-tiles runs in two warpgroups that ping-pong on the
// tensor core, and the accumulator rescale runs in a third warpgroup.
//
// One CTA = one (batch, query head, 256-row query tile) = two 128-row
// sub-tiles t = 0, 1.  512 threads:
//   warps 0-3   softmax warpgroup for sub-tile 0 (thread = query row)
//   warps 4-7   softmax warpgroup for sub-tile 1
//   warps 8-11  correction warpgroup: rescales O_t in tensor memory when a
//               row max moved, then the epilogue (O / l -> bf16 -> TMA
//               store, LSE store)
//   warp  12    tensor-core issuer (one thread issues every tcgen05.mma)
//   warp  13    TMA producer: Q_0, Q_1 once, then K_j, V_j through a ring
//   warps 14-15 idle (they complete warpgroup 3 for setmaxnreg)
//
// Tensor memory (512 columns x 128 lanes, lane = query row of the sub-tile):
//   [0,128) S_0, [128,256) S_1, [256,256+D) O_0, [256+D,256+2D) O_1.
// P_t (bf16, two per column) overwrites the first 64 columns of S_t once the
// softmax has read S_t into registers.  The next S_t GEMM is issued after the
// PV GEMM that reads P_t, by the same thread; tcgen05.mma operations issued
// by one thread execute in issue order.
//
// Every wait is bounded (see ptx.cuh); a timeout raises a CTA-wide abort
// flag, every role unwinds to the teardown, and the device status word
// records ATTN_ERR_TIMEOUT.  No trap, no assert.
#include <cmath>
#include <cstdint>
#include <type_traits>

#include "attn_internal.h"
#include "attn_tiles.cuh"
#include "ptx.cuh"

namespace attnpipe {

__device__ int g_attn_status = 0;

namespace {

constexpr int kThreads = 512;
constexpr int kBlockM = 128;  // rows per query sub-tile
constexpr int kBlockN = 128;  // keys per KV block
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P may grow to 2^8 before O is rescaled
constexpr uint32_t kFull = 0xffffffffu;
// Register split across the four warpgroups (setmaxnreg): softmax x2,
// correction, load/MMA.  The kernel launches with 128 registers per thread
// (launch bounds 512 x 1), and the split must fit in that pool.
constexpr int kRegsSoftmax = 160, kRegsCorrection = 88, kRegsLoadMma = 104;
static_assert((2 * kRegsSoftmax + kRegsCorrection + kRegsLoadMma) * 128 <= 65536 &&
                  kRegsCorrection <= 128 && kRegsLoadMma <= 128,
              "setmaxnreg split exceeds the launch register pool");

template <int D>
struct Cfg {
  static constexpr int kHalves = TileShape<D>::kSlabs;  // 128-byte swizzle slabs across D
  static constexpr int kHalfBytes = kSlabBytes;          // one [128 rows x 64 cols] bf16 slab
  static constexpr int kTileBytes = TileShape<D>::kBytes; // one 128-row tile of Q, K or V
  static constexpr int kStages = (D == 128) ? 4 : 8;   // K/V ring depth
  // shared memory, offsets from a 1024-byte aligned base
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kOffQ + 2 * kTileBytes;
  static constexpr int kOffBar = kOffKV + kStages * kTileBytes;
  // kv_full[S], kv_empty[S], q_full[2], s_full[2], p_full[2], stats[2],
  // pv_done[2], drain[1], fin[2]
  static constexpr int kNumBars = 2 * kStages + 13;
  static constexpr int kOffScale = kOffBar + kNumBars * 8;   // float [2][128]
  static constexpr int kOffRowSum = kOffScale + 2 * 128 * 4;  // float [2][128], fp32 sum of p
  static constexpr int kOffRowSumP = kOffRowSum + 2 * 128 * 4; // float [2][128], sum of bf16(p)
  static constexpr int kOffRowMax = kOffRowSumP + 2 * 128 * 4; // float [2][128]
  static constexpr int kOffMisc = kOffRowMax + 2 * 128 * 4;    // tmem base, abort flag
  static constexpr int kSmemBytes = kOffMisc + 16 + 1024;     // + slack to align the base
  // tensor memory columns
  static constexpr uint32_t kTmS0 = 0, kTmS1 = 128, kTmO0 = 256, kTmO1 = 256 + D;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
};

// Warp-uniform bounded wait: every lane waits, the warp agrees on the result.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t budget) {
  const bool ok = mbar_wait(bar, parity, abort_flag, budget);
  return __all_sync(kFull, ok);
}

// Waits for a phase while ignoring the abort flag: used only at teardown to
// let copies and tensor-core work already in flight land before exit.
__device__ __forceinline__ void drain_wait(uint64_t* bar, uint32_t parity, uint64_t budget) {
  volatile int never = 0;
  mbar_wait(bar, parity, &never, budget);
}

__device__ __forceinline__ float u2f(uint32_t x) { return __uint_as_float(x); }
__device__ __forceinline__ uint32_t f2u(float x) { return __float_as_uint(x); }

}  // namespace

template <int D, bool kTrace>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(const __grid_constant__ AttnParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sKV = smem + C::kOffKV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* kv_full = bars;
  uint64_t* kv_empty = bars + C::kStages;
  uint64_t* q_full = bars + 2 * C::kStages;
  uint64_t* s_full = q_full + 2;
  uint64_t* p_full = q_full + 4;
  uint64_t* stats = q_full + 6;
  uint64_t* pv_done = q_full + 8;
  uint64_t* drain = q_full + 10;
  uint64_t* fin = q_full + 11;
  float* sScale = reinterpret_cast<float*>(smem + C::kOffScale);
  float* sRowSum = reinterpret_cast<float*>(smem + C::kOffRowSum);
  float* sRowSumP = reinterpret_cast<float*>(smem + C::kOffRowSumP);
  float* sRowMax = reinterpret_cast<float*>(smem + C::kOffRowMax);
  uint32_t* sTmemBase = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* sAbort = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // grid = (query tiles x KV splits, H_kv, B).  A CTA works on 256 rows of
  // one row group (the query heads sharing KV head g of batch b, see
  // AttnParams); the tiles of one group are adjacent in launch order, so the
  // CTAs resident at once share few K/V heads in L2, and within a group the
  // longest causal tiles launch first.
  const int R = p.rows_per_group;
  const int split = blockIdx.x % p.kv_splits;
  const int m0 = ((int)(gridDim.x / p.kv_splits) - 1 - (int)(blockIdx.x / p.kv_splits)) * (2 * kBlockM);
  const int b = blockIdx.z;
  const int zkv = b * p.H_kv + blockIdx.y;  // row group = K/V head index
  // keys any row of this tile may see: row rho is query position rho % S_q,
  // and with the causal mask it sees keys <= its position
  int kv_end = p.S_kv;
  if (p.causal) {
    const int last = min(m0 + 2 * kBlockM, R) - 1;
    kv_end = min(p.S_kv, (m0 / p.S_q == last / p.S_q) ? last % p.S_q + 1 : p.S_q);
  }
  const int n_total = (kv_end + kBlockN - 1) / kBlockN;
  // sub-tile 1 holds rows m0 + 128 .. m0 + 255; when none of them exists
  // (short row groups, e.g. one decoding token per head, or a ragged last
  // tile) every role skips it and the tile costs half
  const bool has_sub1 = (m0 + kBlockM) < R;
  const int jb = split * p.kv_blocks_per_split;  // first KV block of this CTA
  const int n_blocks = min(n_total - jb, p.kv_blocks_per_split);
  if (n_blocks <= 0) {
    // split-KV only: no key of this split is visible to any row of the tile,
    // so its partial result is empty (weight 0 in the merge)
    for (int idx = threadIdx.x; idx < 2 * kBlockM; idx += kThreads) {
      const int rho = m0 + idx;
      if (rho < R) {
        const size_t row = (size_t)split * p.total_rows + (size_t)zkv * R + rho;
        p.lse_part[row] = -INFINITY;
        float4* dst = reinterpret_cast<float4*>(p.o_part + row * D);
        for (int c = 0; c < D / 4; ++c) dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    return;
  }
  const uint64_t budget = p.timeout_ns;
  // trace stamps (compiled only into the trace instantiation)
  const int cta_lin = blockIdx.x + gridDim.x * (blockIdx.y + gridDim.y * blockIdx.z);
  const bool traced = kTrace && cta_lin < p.trace_ctas;
  // The stamp is the SM cycle counter; a slot written by several warps keeps
  // the latest stamp (a barrier completes when its last warp arrives).
  auto stamp = [&](int ev, int j) {
    if constexpr (kTrace) {
      if (traced && j < p.trace_blocks)
        atomicMax(&p.trace[((size_t)cta_lin * kNumTraceEvents + ev) * p.trace_blocks + j],
                  (unsigned long long)clock64());
    }
  };

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&q_full[t], 1);
      mbar_init(&s_full[t], 1);
      // p_full[t]: P_t(j) stored by the softmax (128 arrivals) and O_t
      // rescaled for block j by the correction warpgroup (128 arrivals)
      mbar_init(&p_full[t], 2 * kBlockM);
      // stats[t]: one phase per block j >= 1 (the rescale factor alpha);
      // fin[t]: one phase, the final row sums and max.  Keeping them apart
      // means a waiter is never two phases behind on either barrier.
      mbar_init(&stats[t], kBlockM);
      mbar_init(&fin[t], kBlockM);
      mbar_init(&pv_done[t], 1);
    }
    mbar_init(drain, 1);
    *sAbort = 0;
    fence_mbar_init();
  }
  if (warp == 13 && lane == 0) {
    tma_prefetch_map(&p.tm_q);
    tma_prefetch_map(&p.tm_k);
    tma_prefetch_map(&p.tm_v);
    tma_prefetch_map(&p.tm_o);
  }
  if (warp == 12) {
    tmem_alloc(sTmemBase, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *sTmemBase;
  const int wg = warp >> 2;

  if (wg < 2) {
    // ------------------------------------------------------------ softmax
    // (warpgroup 1 has nothing to do when the tile has no sub-tile 1)
    if (wg == 0 || has_sub1) {
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kRegsSoftmax) : "memory");
    const int t = wg;
    const int r = (warp & 3) * 32 + lane;                 // row within the sub-tile
    const uint32_t tS = tmem + ((uint32_t)((warp & 3) * 32) << 16) + (t ? C::kTmS1 : C::kTmS0);
    const int rho = m0 + t * kBlockM + r;                  // row in the row group
    const int pos = rho % p.S_q;                           // its query position
    // smallest query position in this sub-tile (0 if it spans two heads)
    const int sub_first = m0 + t * kBlockM;
    const int min_pos = (sub_first / p.S_q == (sub_first + kBlockM - 1) / p.S_q) ? sub_first % p.S_q : 0;
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = f2_pack(sl2, sl2);
    const int key_limit = p.causal ? min(p.S_kv, pos + 1) : p.S_kv;
    // Two row sums: l_run of the fp32 probabilities (for the LSE), and lp_run
    // of the bf16-rounded probabilities that the PV GEMM actually consumes,
    // so O is normalised by the same weights it was accumulated with.
    float m_run = -INFINITY;
    float l_run = 0.f;
    float lp_run = 0.f;
    bool ok = true;
    for (int j = 0; j < n_blocks; ++j) {
      if (!warp_wait(&s_full[t], j & 1, sAbort, budget)) { ok = false; break; }
      tc_fence_after_sync();
      if (lane == 0) stamp(t ? kEvSm1Wake : kEvSm0Wake, j);
      uint32_t s[128];
      {
        uint32_t (&s0)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[0]);
        uint32_t (&s1)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[32]);
        uint32_t (&s2)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[64]);
        uint32_t (&s3)[32] = *reinterpret_cast<uint32_t(*)[32]>(&s[96]);
        tmem_ld_x32(tS + 0, s0);
        tmem_ld_x32(tS + 32, s1);
        tmem_ld_x32(tS + 64, s2);
        tmem_ld_x32(tS + 96, s3);
        tmem_ld_wait();
        reg_after_wait(s0);
        reg_after_wait(s1);
        reg_after_wait(s2);
        reg_after_wait(s3);
      }
      if (lane == 0) stamp(t ? kEvSm1Loaded : kEvSm0Loaded, j);
      const int kv0 = (jb + j) * kBlockN;
      const bool masked = (kv0 + kBlockN > p.S_kv) || (p.causal && kv0 + kBlockN - 1 > min_pos);
      const int lim = key_limit - kv0;  // columns c < lim are visible to this row
      float m_use = m_run;
      float alpha = 1.f;
      uint64_t l2[2] = {0, 0};                  // packed fp32 partial sums of p
      float lp[4] = {0.f, 0.f, 0.f, 0.f};       // partial sums of bf16(p)
      // The unmasked and masked bodies are separate code paths so the common
      // (unmasked) one carries no per-element predication.
      auto body = [&](auto masked_tag) {
        constexpr bool kMasked = decltype(masked_tag)::value;
        if constexpr (kMasked) {
          // keys this row may not see drop out of the max
#pragma unroll
          for (int c = 0; c < 128; ++c)
            if (c >= lim) s[c] = f2u(-INFINITY);
        }
        // row max of the raw scores (4 independent chains of 3-input max)
        float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
        for (int c = 0; c < 128; c += 8) {
#pragma unroll
          for (int i = 0; i < 4; ++i) mx[i] = max3(mx[i], u2f(s[c + 2 * i]), u2f(s[c + 2 * i + 1]));
        }
        const float mblk = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
        // scale >= 0, so the max of the scaled scores is the scaled max; a row
        // whose keys are all masked here leaves the running max unchanged
        const float m_new = (mblk == -INFINITY) ? m_run : fmaxf(m_run, mblk * sl2);
        if (j == 0) {
          m_use = m_new;
        } else if (m_new - m_run > kRescaleThreshold) {
          m_use = m_new;
          alpha = ex2_approx(m_run - m_new);
        }
        if (j > 0) {
          sScale[t * kBlockM + r] = alpha;
          mbar_arrive(&stats[t]);
        }
        const uint64_t neg_m2 = f2_pack(-m_use, -m_use);
#pragma unroll
        for (int ch = 0; ch < 8; ++ch) {
          uint32_t pk[8];
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            const int c = ch * 16 + 2 * i;
            // x = s * scale * log2(e) - m, two lanes per instruction
            float x0, x1;
            f2_unpack(f2_fma(f2_pack(u2f(s[c]), u2f(s[c + 1])), sl2x2, neg_m2), x0, x1);
            float p0 = ex2_approx(x0);
            float p1 = ex2_approx(x1);
            if constexpr (kMasked) {  // (also covers scale = 0, where -inf * 0 is NaN)
              p0 = (c < lim) ? p0 : 0.f;
              p1 = (c + 1 < lim) ? p1 : 0.f;
            }
            l2[i & 1] = f2_add(l2[i & 1], f2_pack(p0, p1));
            pk[i] = pack_bf16x2(p0, p1);
            add_bf16x2_to_f32(lp[(2 * i) & 3], lp[(2 * i + 1) & 3], pk[i]);
          }
          tmem_st_x8(tS + ch * 8, pk);
        }
      };
      if (masked)
        body(std::true_type{});
      else
        body(std::false_type{});
      float la, lb;
      f2_unpack(f2_add(l2[0], l2[1]), la, lb);
      l_run = l_run * alpha + (la + lb);
      lp_run = lp_run * alpha + ((lp[0] + lp[1]) + (lp[2] + lp[3]));
      tmem_st_wait();
      tc_fence_before_sync();
      if (lane == 0) stamp(t ? kEvSm1Done : kEvSm0Done, j);
      bool signal = true;
      if constexpr (kTrace) signal = !(t == 0 && j == p.fault_drop_block);
      if (signal) mbar_arrive(&p_full[t]);
      m_run = m_use;
    }
    if (ok) {
      sRowSum[t * kBlockM + r] = l_run;
      sRowSumP[t * kBlockM + r] = lp_run;
      sRowMax[t * kBlockM + r] = m_run;
      mbar_arrive(&fin[t]);
    }
    }
  } else if (wg == 2) {
    // ------------------------------------------------------------ correction + epilogue
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kRegsCorrection) : "memory");
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    bool ok = true;
    // Block 0 needs no rescale.  For block j >= 1 the softmax's alpha arrives
    // on stats[t]; it is published after the softmax saw S_t(j), whose commit
    // follows PV_t(j-1), so O_t already holds every earlier block.
    const int n_sub = has_sub1 ? 2 : 1;
    mbar_arrive(&p_full[0]);
    if (has_sub1) mbar_arrive(&p_full[1]);
    for (int j = 1; j < n_blocks && ok; ++j) {
      for (int t = 0; t < n_sub; ++t) {
        if (!warp_wait(&stats[t], (j - 1) & 1, sAbort, budget)) { ok = false; break; }
        const float alpha = sScale[t * kBlockM + r];
        tc_fence_after_sync();
        if (__any_sync(kFull, alpha != 1.f)) {
          const uint32_t tO = tmem + lane_base + (t ? C::kTmO1 : C::kTmO0);
#pragma unroll
          for (int ch = 0; ch < D / 32; ++ch) {
            uint32_t o[32];
            tmem_ld_x32(tO + ch * 32, o);
            tmem_ld_wait();
            reg_after_wait(o);
#pragma unroll
            for (int i = 0; i < 32; ++i) o[i] = f2u(u2f(o[i]) * alpha);
            tmem_st_x32(tO + ch * 32, o);
          }
          tmem_st_wait();
        }
        tc_fence_before_sync();
        if (lane == 0) stamp(t ? kEvCorr1 : kEvCorr0, j);
        mbar_arrive(&p_full[t]);
      }
    }
    for (int t = 0; t < n_sub && ok; ++t) {
      if (!warp_wait(&fin[t], 0, sAbort, budget)) { ok = false; break; }
      if (!warp_wait(&pv_done[t], 0, sAbort, budget)) { ok = false; break; }
      tc_fence_after_sync();
      if (lane == 0) stamp(kEvEpilogue, t);
      const float l = sRowSum[t * kBlockM + r];
      const float m = sRowMax[t * kBlockM + r];
      const float lp = sRowSumP[t * kBlockM + r];
      // a row with no visible key (possible only within one KV split) has
      // l = 0: its partial result is O = 0, LSE = -inf
      const bool empty = !(lp > 0.f);
      const float inv_l = empty ? 0.f : 1.f / lp;
      const float lse_row = empty ? -INFINITY : (m + log2f(l)) * 0.69314718055994530942f;
      const uint32_t tO = tmem + lane_base + (t ? C::kTmO1 : C::kTmO0);
      const int rho = m0 + t * kBlockM + r;
      if (p.o_part != nullptr) {
        // split-KV partial: fp32 O normalised within the split, and its LSE.
        // The tensor-memory loads are warp-wide; only the stores depend on
        // whether the row exists.
        const size_t row = (size_t)split * p.total_rows + (size_t)zkv * R + rho;
        float4* dst = reinterpret_cast<float4*>(p.o_part + row * D);
#pragma unroll
        for (int ch = 0; ch < D / 32; ++ch) {
          uint32_t o[32];
          tmem_ld_x32(tO + ch * 32, o);
          tmem_ld_wait();
          reg_after_wait(o);
          if (rho < R) {
#pragma unroll
            for (int qd = 0; qd < 8; ++qd)
              dst[ch * 8 + qd] = make_float4(u2f(o[qd * 4 + 0]) * inv_l, u2f(o[qd * 4 + 1]) * inv_l,
                                             u2f(o[qd * 4 + 2]) * inv_l, u2f(o[qd * 4 + 3]) * inv_l);
          }
        }
        if (rho < R) p.lse_part[row] = lse_row;
        continue;
      }
      uint8_t* stage = sQ + t * C::kTileBytes;  // Q_t is no longer read: reuse it
#pragma unroll
      for (int ch = 0; ch < D / 32; ++ch) {
        uint32_t o[32];
        tmem_ld_x32(tO + ch * 32, o);
        tmem_ld_wait();
        reg_after_wait(o);
#pragma unroll
        for (int qd = 0; qd < 4; ++qd) {
          const int c16 = ch * 4 + qd;     // 16-byte chunk index along the row
          const int half = c16 >> 3;
          const int cc = c16 & 7;
          uint4 val;
          val.x = pack_bf16x2(u2f(o[qd * 8 + 0]) * inv_l, u2f(o[qd * 8 + 1]) * inv_l);
          val.y = pack_bf16x2(u2f(o[qd * 8 + 2]) * inv_l, u2f(o[qd * 8 + 3]) * inv_l);
          val.z = pack_bf16x2(u2f(o[qd * 8 + 4]) * inv_l, u2f(o[qd * 8 + 5]) * inv_l);
          val.w = pack_bf16x2(u2f(o[qd * 8 + 6]) * inv_l, u2f(o[qd * 8 + 7]) * inv_l);
          *reinterpret_cast<uint4*>(stage + half * C::kHalfBytes + r * 128 + ((cc ^ (r & 7)) << 4)) = val;
        }
      }
      if (rho < R) p.lse[(size_t)zkv * R + rho] = lse_row;
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
#pragma unroll
        for (int hf = 0; hf < C::kHalves; ++hf) {
          tma_store_3d(&p.tm_o, stage + hf * C::kHalfBytes + q4 * 32 * 128, hf * 64,
                       m0 + t * kBlockM + q4 * 32, zkv);
        }
        tma_store_commit();
      }
      __syncwarp();
    }
    if (lane == 0) tma_store_wait_all();
    __syncwarp();
  } else {
    // ------------------------------------------------------------ warpgroup 3
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kRegsLoadMma) : "memory");
    if (warp == 12 && lane == 0) {
      // tensor-core issuer: one thread, no warp-wide votes, so it needs as
      // few issue slots as possible next to the busy softmax warps
      const uint64_t dq0 = kmajor_tile_desc(smem_u32(sQ));
      const uint64_t dq1 = kmajor_tile_desc(smem_u32(sQ + C::kTileBytes));
      const uint64_t dk0 = kmajor_tile_desc(smem_u32(sKV));
      const uint64_t dv0 = mnmajor_tile_desc<D>(smem_u32(sKV));
      constexpr uint64_t kStageDesc = C::kTileBytes >> 4;  // start-address step per ring stage
      const uint32_t tS0 = tmem + C::kTmS0, tS1 = tmem + C::kTmS1;
      const uint32_t tO0 = tmem + C::kTmO0, tO1 = tmem + C::kTmO1;
      do {
        if (!mbar_wait(&kv_full[0], 0, sAbort, budget)) break;
        if (!mbar_wait(&q_full[0], 0, sAbort, budget)) break;
        tc_fence_after_sync();
        issue_qk_gemm<D>(tS0, dq0, dk0);
        tc_commit(&s_full[0]);
        stamp(kEvMmaS0, 0);
        if (has_sub1) {
          if (!mbar_wait(&q_full[1], 0, sAbort, budget)) break;
          tc_fence_after_sync();
          issue_qk_gemm<D>(tS1, dq1, dk0);
          tc_commit(&s_full[1]);
          stamp(kEvMmaS1, 0);
        }
        tc_commit(&kv_empty[0]);
        int sv = 1 % C::kStages, sk = 2 % C::kStages;   // ring stages of V_j and K_{j+1}
        for (int j = 0; j < n_blocks; ++j) {
          const bool more = (j + 1) < n_blocks;
          // V_j lives in ring slot 2j+1, K_{j+1} in slot 2j+2.  Both loads were
          // issued long before; waiting for them here, while the softmax is
          // still busy, keeps them off the path from "P ready" to the GEMMs.
          const uint32_t v_par = ((2 * j + 1) / C::kStages) & 1;
          const uint32_t k_par = ((2 * j + 2) / C::kStages) & 1;
          if (!mbar_wait(&kv_full[sv], v_par, sAbort, budget)) break;
          if (more && !mbar_wait(&kv_full[sk], k_par, sAbort, budget)) break;
          const uint64_t dv = dv0 + (uint64_t)sv * kStageDesc;
          const uint64_t dk = dk0 + (uint64_t)sk * kStageDesc;
          // sub-tile 0: O_0 += P_0 V_j, then S_0 = Q_0 K_{j+1}^T
          if (!mbar_wait(&p_full[0], j & 1, sAbort, budget)) break;
          tc_fence_after_sync();
          stamp(kEvMmaPV0Begin, j);
          issue_pv_gemm<D>(tO0, tS0, dv, j > 0);
          if (!more) tc_commit(&pv_done[0]);  // the epilogue waits for the last PV only
          stamp(kEvMmaPV0, j);
          if (more) {
            stamp(kEvMmaS0Begin, j + 1);
            issue_qk_gemm<D>(tS0, dq0, dk);
            tc_commit(&s_full[0]);
            stamp(kEvMmaS0, j + 1);
          }
          // sub-tile 1: O_1 += P_1 V_j, then S_1 = Q_1 K_{j+1}^T
          if (has_sub1) {
            if (!mbar_wait(&p_full[1], j & 1, sAbort, budget)) break;
            tc_fence_after_sync();
            stamp(kEvMmaPV1Begin, j);
            issue_pv_gemm<D>(tO1, tS1, dv, j > 0);
            if (!more) tc_commit(&pv_done[1]);
            stamp(kEvMmaPV1, j);
            if (more) {
              stamp(kEvMmaS1Begin, j + 1);
              issue_qk_gemm<D>(tS1, dq1, dk);
              tc_commit(&s_full[1]);
              stamp(kEvMmaS1, j + 1);
            }
          }
          // release the ring slots last: off the critical path
          tc_commit(&kv_empty[sv]);
          if (more) tc_commit(&kv_empty[sk]);
          sv = (sv + 2) % C::kStages;
          sk = (sk + 2) % C::kStages;
        }
      } while (0);
      // let every tensor-core op this thread issued finish before teardown
      tc_commit(drain);
      drain_wait(drain, 0, budget);
    } else if (warp == 13 && lane == 0) {
      // TMA producer (one thread)
      const uint64_t pol_q = l2_policy_evict_first();
      const uint64_t pol_kv = l2_policy_evict_last();
      for (int t = 0; t < (has_sub1 ? 2 : 1); ++t) {
        mbar_arrive_expect_tx(&q_full[t], C::kTileBytes);
        tma_load_tile<D>(sQ + t * C::kTileBytes, &p.tm_q, &q_full[t], m0 + t * kBlockM, zkv, pol_q);
      }
      int issued = 0;
      for (int idx = 0; idx < 2 * n_blocks; ++idx) {
        const int slot = idx % C::kStages;
        const int round = idx / C::kStages;
        if (round > 0 && !mbar_wait(&kv_empty[slot], (round - 1) & 1, sAbort, budget)) break;
        mbar_arrive_expect_tx(&kv_full[slot], C::kTileBytes);
        const CUtensorMap* map = (idx & 1) ? &p.tm_v : &p.tm_k;
        tma_load_tile<D>(sKV + slot * C::kTileBytes, map, &kv_full[slot],
                         (jb + (idx >> 1)) * kBlockN, zkv, pol_kv);
        stamp((idx & 1) ? kEvLoadV : kEvLoadK, idx >> 1);
        issued = idx + 1;
      }
      // every copy issued must land before the CTA exits (on the normal path
      // these phases completed long ago)
      drain_wait(&q_full[0], 0, budget);
      if (has_sub1) drain_wait(&q_full[1], 0, budget);
      const int first = issued > C::kStages ? issued - C::kStages : 0;
      for (int idx = first; idx < issued; ++idx)
        drain_wait(&kv_full[idx % C::kStages], (idx / C::kStages) & 1, budget);
    }
    __syncwarp();
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 12) tmem_dealloc(tmem, C::kTmemCols);
  if (threadIdx.x == 0) stamp(kEvEnd, 0);
  if (threadIdx.x == 0 && *sAbort) atomicCAS(&g_attn_status, 0, (int)ATTN_ERR_TIMEOUT);
}

namespace {

template <int D, bool kTrace>
cudaError_t launch_d(const AttnParams& p, int n_m_tiles, cudaStream_t stream) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    err = cudaFuncSetAttribute(attn_fwd_kernel<D, kTrace>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::kSmemBytes);
    if (err != cudaSuccess) return err;
    attr_set[dev] = true;
  }
  dim3 grid(n_m_tiles * p.kv_splits, p.H_kv, p.B);
  attn_fwd_kernel<D, kTrace><<<grid, kThreads, Cfg<D>::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd(const AttnParams& p, int D, int n_m_tiles, cudaStream_t stream) {
  if (p.trace || p.fault_drop_block >= 0) {
    if (D == 128) return launch_d<128, true>(p, n_m_tiles, stream);
    if (D == 64) return launch_d<64, true>(p, n_m_tiles, stream);
    return cudaErrorInvalidValue;
  }
  if (D == 128) return launch_d<128, false>(p, n_m_tiles, stream);
  if (D == 64) return launch_d<64, false>(p, n_m_tiles, stream);
  return cudaErrorInvalidValue;
}

cudaError_t read_device_status(int* status, bool reset) {
  cudaError_t err = cudaMemcpyFromSymbol(status, g_attn_status, sizeof(int));
  if (err != cudaSuccess) return err;
  if (reset) {
    const int zero = 0;
    err = cudaMemcpyToSymbol(g_attn_status, &zero, sizeof(int));
  }
  return err;
}

}  // namespace attnpipe
