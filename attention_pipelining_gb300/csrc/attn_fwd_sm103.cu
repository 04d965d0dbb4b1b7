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
constexpr int kRegsSoftmax = 168, kRegsCorrection = 88, kRegsLoadMma = 88;
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
  // o_corr[2], pv_done[2], drain[1]
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

template <int D>
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
  uint64_t* o_corr = q_full + 8;
  uint64_t* pv_done = q_full + 10;
  uint64_t* drain = q_full + 12;
  float* sScale = reinterpret_cast<float*>(smem + C::kOffScale);
  float* sRowSum = reinterpret_cast<float*>(smem + C::kOffRowSum);
  float* sRowSumP = reinterpret_cast<float*>(smem + C::kOffRowSumP);
  float* sRowMax = reinterpret_cast<float*>(smem + C::kOffRowMax);
  uint32_t* sTmemBase = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* sAbort = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int h = blockIdx.x;
  const int b = blockIdx.y;
  const int m0 = (gridDim.z - 1 - blockIdx.z) * (2 * kBlockM);  // heaviest tiles launch first
  const int hkv = h / (p.H_q / p.H_kv);
  const int zq = b * p.H_q + h;
  const int zkv = b * p.H_kv + hkv;
  const int kv_end = p.causal ? min(p.S_kv, m0 + 2 * kBlockM) : p.S_kv;
  const int n_blocks = (kv_end + kBlockN - 1) / kBlockN;
  const uint64_t budget = p.timeout_ns;

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kStages; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&q_full[t], 1);
      mbar_init(&s_full[t], 1);
      mbar_init(&p_full[t], kBlockM);
      mbar_init(&stats[t], kBlockM);
      mbar_init(&o_corr[t], kBlockM);
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
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kRegsSoftmax) : "memory");
    const int t = wg;
    const int r = (warp & 3) * 32 + lane;                 // row within the sub-tile
    const uint32_t tS = tmem + ((uint32_t)((warp & 3) * 32) << 16) + (t ? C::kTmS1 : C::kTmS0);
    const int row = m0 + t * kBlockM + r;                  // query row in the sequence
    const int row_first = m0 + t * kBlockM;
    const float sl2 = p.scale_log2;
    const int key_limit = p.causal ? min(p.S_kv, row + 1) : p.S_kv;
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
      const int kv0 = j * kBlockN;
      const bool masked = (kv0 + kBlockN > p.S_kv) || (p.causal && kv0 + kBlockN - 1 > row_first);
      const int lim = key_limit - kv0;  // columns c < lim are visible to this row
      // row max of the raw scores (8 independent chains)
      float mx[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) mx[i] = -INFINITY;
      if (masked) {
#pragma unroll
        for (int c = 0; c < 128; ++c) mx[c & 7] = fmaxf(mx[c & 7], c < lim ? u2f(s[c]) : -INFINITY);
      } else {
#pragma unroll
        for (int c = 0; c < 128; ++c) mx[c & 7] = fmaxf(mx[c & 7], u2f(s[c]));
      }
      const float mblk = fmaxf(fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3])),
                               fmaxf(fmaxf(mx[4], mx[5]), fmaxf(mx[6], mx[7])));
      const float m_new = fmaxf(m_run, mblk * sl2);
      float m_use = m_run;
      float alpha = 1.f;
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
      const float neg_m = -m_use;
      float ls[8], lp[8];
#pragma unroll
      for (int i = 0; i < 8; ++i) ls[i] = lp[i] = 0.f;
#pragma unroll
      for (int ch = 0; ch < 4; ++ch) {
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) {
          const int c = ch * 32 + 2 * i;
          float p0 = ex2_approx(fmaf(u2f(s[c]), sl2, neg_m));
          float p1 = ex2_approx(fmaf(u2f(s[c + 1]), sl2, neg_m));
          if (masked) {
            p0 = (c < lim) ? p0 : 0.f;
            p1 = (c + 1 < lim) ? p1 : 0.f;
          }
          ls[i & 7] += p0 + p1;
          pk[i] = pack_bf16x2(p0, p1);
          lp[i & 7] += u2f(pk[i] << 16) + u2f(pk[i] & 0xffff0000u);
        }
        tmem_st_x16(tS + ch * 16, pk);
      }
      l_run = l_run * alpha + (((ls[0] + ls[1]) + (ls[2] + ls[3])) + ((ls[4] + ls[5]) + (ls[6] + ls[7])));
      lp_run = lp_run * alpha + (((lp[0] + lp[1]) + (lp[2] + lp[3])) + ((lp[4] + lp[5]) + (lp[6] + lp[7])));
      tmem_st_wait();
      tc_fence_before_sync();
      mbar_arrive(&p_full[t]);
      m_run = m_use;
    }
    if (ok) {
      sRowSum[t * kBlockM + r] = l_run;
      sRowSumP[t * kBlockM + r] = lp_run;
      sRowMax[t * kBlockM + r] = m_run;
      mbar_arrive(&stats[t]);
    }
  } else if (wg == 2) {
    // ------------------------------------------------------------ correction + epilogue
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kRegsCorrection) : "memory");
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    bool ok = true;
    for (int j = 1; j < n_blocks && ok; ++j) {
      for (int t = 0; t < 2; ++t) {
        if (!warp_wait(&stats[t], (j - 1) & 1, sAbort, budget)) { ok = false; break; }
        const float alpha = sScale[t * kBlockM + r];
        if (!warp_wait(&pv_done[t], (j - 1) & 1, sAbort, budget)) { ok = false; break; }
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
        mbar_arrive(&o_corr[t]);
      }
    }
    for (int t = 0; t < 2 && ok; ++t) {
      if (!warp_wait(&stats[t], (n_blocks - 1) & 1, sAbort, budget)) { ok = false; break; }
      if (!warp_wait(&pv_done[t], (n_blocks - 1) & 1, sAbort, budget)) { ok = false; break; }
      tc_fence_after_sync();
      const float l = sRowSum[t * kBlockM + r];
      const float m = sRowMax[t * kBlockM + r];
      const float inv_l = 1.f / sRowSumP[t * kBlockM + r];
      const uint32_t tO = tmem + lane_base + (t ? C::kTmO1 : C::kTmO0);
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
      const int grow = m0 + t * kBlockM + r;
      if (grow < p.S_q) {
        p.lse[(size_t)zq * p.S_q + grow] = (m + log2f(l)) * 0.69314718055994530942f;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
#pragma unroll
        for (int hf = 0; hf < C::kHalves; ++hf) {
          tma_store_3d(&p.tm_o, stage + hf * C::kHalfBytes + q4 * 32 * 128, hf * 64,
                       m0 + t * kBlockM + q4 * 32, zq);
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
    if (warp == 12) {
      // tensor-core issuer
      const uint32_t sQ_addr = smem_u32(sQ);
      const uint32_t sKV_addr = smem_u32(sKV);
      auto issue_qk = [&](int t, int slot) {
        issue_qk_gemm<D>(tmem + (t ? C::kTmS1 : C::kTmS0), sQ_addr + t * C::kTileBytes,
                         sKV_addr + slot * C::kTileBytes);
      };
      auto issue_pv = [&](int t, int slot, bool acc) {
        issue_pv_gemm<D>(tmem + (t ? C::kTmO1 : C::kTmO0), tmem + (t ? C::kTmS1 : C::kTmS0),
                         sKV_addr + slot * C::kTileBytes, acc);
      };
      do {
        if (!warp_wait(&kv_full[0], 0, sAbort, budget)) break;
        if (!warp_wait(&q_full[0], 0, sAbort, budget)) break;
        tc_fence_after_sync();
        if (lane == 0) {
          issue_qk(0, 0);
          tc_commit(&s_full[0]);
        }
        __syncwarp();
        if (!warp_wait(&q_full[1], 0, sAbort, budget)) break;
        tc_fence_after_sync();
        if (lane == 0) {
          issue_qk(1, 0);
          tc_commit(&s_full[1]);
          tc_commit(&kv_empty[0]);
        }
        __syncwarp();
        bool ok = true;
        for (int j = 0; j < n_blocks && ok; ++j) {
          const int iv = 2 * j + 1;
          const int sv = iv % C::kStages;
          const int ik = 2 * j + 2;
          const int sk = ik % C::kStages;
          const bool more = (j + 1) < n_blocks;
          if (!warp_wait(&kv_full[sv], (iv / C::kStages) & 1, sAbort, budget)) { ok = false; break; }
          // sub-tile 0: O_0 += P_0 V_j, then S_0 = Q_0 K_{j+1}^T
          if (!warp_wait(&p_full[0], j & 1, sAbort, budget)) { ok = false; break; }
          if (j > 0 && !warp_wait(&o_corr[0], (j - 1) & 1, sAbort, budget)) { ok = false; break; }
          tc_fence_after_sync();
          if (lane == 0) {
            issue_pv(0, sv, j > 0);
            tc_commit(&pv_done[0]);
          }
          __syncwarp();
          if (more) {
            if (!warp_wait(&kv_full[sk], (ik / C::kStages) & 1, sAbort, budget)) { ok = false; break; }
            tc_fence_after_sync();
            if (lane == 0) {
              issue_qk(0, sk);
              tc_commit(&s_full[0]);
            }
            __syncwarp();
          }
          // sub-tile 1: O_1 += P_1 V_j, then S_1 = Q_1 K_{j+1}^T
          if (!warp_wait(&p_full[1], j & 1, sAbort, budget)) { ok = false; break; }
          if (j > 0 && !warp_wait(&o_corr[1], (j - 1) & 1, sAbort, budget)) { ok = false; break; }
          tc_fence_after_sync();
          if (lane == 0) {
            issue_pv(1, sv, j > 0);
            tc_commit(&pv_done[1]);
            tc_commit(&kv_empty[sv]);
            if (more) {
              issue_qk(1, sk);
              tc_commit(&s_full[1]);
              tc_commit(&kv_empty[sk]);
            }
          }
          __syncwarp();
        }
      } while (0);
      // let every tensor-core op this thread issued finish before teardown
      if (lane == 0) {
        tc_commit(drain);
        drain_wait(drain, 0, budget);
      }
      __syncwarp();
    } else if (warp == 13) {
      // TMA producer
      const uint64_t pol_q = l2_policy_evict_first();
      const uint64_t pol_kv = l2_policy_evict_last();
      if (lane == 0) {
        for (int t = 0; t < 2; ++t) {
          mbar_arrive_expect_tx(&q_full[t], C::kTileBytes);
          tma_load_tile<D>(sQ + t * C::kTileBytes, &p.tm_q, &q_full[t], m0 + t * kBlockM, zq, pol_q);
        }
      }
      __syncwarp();
      int issued = 0;
      bool ok = true;
      for (int idx = 0; idx < 2 * n_blocks; ++idx) {
        const int slot = idx % C::kStages;
        const int round = idx / C::kStages;
        if (round > 0 && !warp_wait(&kv_empty[slot], (round - 1) & 1, sAbort, budget)) {
          ok = false;
          break;
        }
        if (lane == 0) {
          mbar_arrive_expect_tx(&kv_full[slot], C::kTileBytes);
          const CUtensorMap* map = (idx & 1) ? &p.tm_v : &p.tm_k;
          tma_load_tile<D>(sKV + slot * C::kTileBytes, map, &kv_full[slot], (idx >> 1) * kBlockN, zkv,
                           pol_kv);
        }
        __syncwarp();
        issued = idx + 1;
      }
      (void)ok;
      if (lane == 0) {
        // every copy this warp issued must land before the CTA exits (on the
        // normal path these phases completed long ago)
        drain_wait(&q_full[0], 0, budget);
        drain_wait(&q_full[1], 0, budget);
        const int first = issued > C::kStages ? issued - C::kStages : 0;
        for (int idx = first; idx < issued; ++idx)
          drain_wait(&kv_full[idx % C::kStages], (idx / C::kStages) & 1, budget);
      }
      __syncwarp();
    }
  }

  // ------------------------------------------------------------ teardown
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 12) tmem_dealloc(tmem, C::kTmemCols);
  if (threadIdx.x == 0 && *sAbort) atomicCAS(&g_attn_status, 0, (int)ATTN_ERR_TIMEOUT);
}

namespace {

template <int D>
cudaError_t launch_d(const AttnParams& p, int n_m_tiles, cudaStream_t stream) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!attr_set[dev]) {
    err = cudaFuncSetAttribute(attn_fwd_kernel<D>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               Cfg<D>::kSmemBytes);
    if (err != cudaSuccess) return err;
    attr_set[dev] = true;
  }
  dim3 grid(p.H_q, p.B, n_m_tiles);
  attn_fwd_kernel<D><<<grid, kThreads, Cfg<D>::kSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

}  // namespace

cudaError_t launch_attn_fwd(const AttnParams& p, int D, int n_m_tiles, cudaStream_t stream) {
  if (D == 128) return launch_d<128>(p, n_m_tiles, stream);
  if (D == 64) return launch_d<64>(p, n_m_tiles, stream);
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
