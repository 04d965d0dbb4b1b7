// chunk_scan_sm103.cu -- Mamba2 chunk scan (intra-chunk part) for sm_103a.
//
// "PipeThreader: Software-Defined Pipelining for Efficient DNN Execution",
// section 2 (running example, Mamba2 ChunkScan, Fig. 6): load cb, dA and dt,
// multiply cb by the exponential product of dA and dt, and accumulate the
// matrix product with x into acc_o, the reduction axis (the chunk's keys)
// tiled so the loads, the exponentials and the tensor-core products of
// consecutive slices overlap.  Per chunk c, head h, row m of the chunk:
//   out[m, :] = sum_{k <= m} cb[m, k] exp(dA_cs[m] - dA_cs[k]) dt[k] x[k, :]
//
// One CTA = (batch, chunk, 128-row tile of the chunk, block of HB heads of
// one group), 768 threads.  The CTA's slices (64 keys of one head) are
// numbered gs = 0, 1, ... head by head:
//   warps 0-15  four scaling warpgroups; warpgroup w takes slices gs = w,
//               w + 4, ...: thread = row of the tile, it scales its row's 64
//               keys of cb (kept in shared memory for all the CTA's heads)
//               by the decay and dt, rounds to bf16 and stores them into the
//               slice's A slot in tensor memory (a ring of eight slots; two
//               consecutive slices share one full/free barrier pair);
//   warps 16-19 output warpgroup: per head, reads the accumulator from tensor
//               memory, rounds to bf16 into a staging tile in shared memory
//               and writes it with one TMA store;
//   warp 20     tensor-core issuer: per pair of slices, 8 tcgen05.mma (M = 128,
//               N = 64, K = 16) of the A slices (tensor memory) with the x
//               slices (shared memory, MN-major) into one of four 128 x 64
//               fp32 accumulators (heads rotate over them);
//   warps 22-23 vectors and key factors, heads alternating between the two
//               warps: per head, loads dA_cs and dt of the keys the tile's
//               rows see (1-D bulk copies, into a ring of 4 heads of 256
//               keys or 8 of 128, as far ahead as the ring allows) and
//               computes the per-key factors of the decay and the mask of
//               portions where dA_cs rises (see below);
//   warp 21     TMA producer: the tile's cb once (3-D map, 32-key boxes;
//               one barrier per 64-key slice, issued along with the first
//               head's x slices), then per head its x slices (4-D map over
//               [B, L, H, P])
//               through a ring of eight slots (two slices per full/free
//               barrier pair), with the head two ahead prefetched into L2.
// Every wait is bounded; a timeout raises a CTA-wide abort flag and the
// device status word records ATTN_ERR_TIMEOUT.
#include <cmath>
#include <cstdint>
#include <mutex>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attnpipe {

__device__ int g_cs_status = 0;

namespace {

constexpr int kCsScaleGroups = 4;  // scaling warpgroups
constexpr int kCsOutWarp0 = 4 * kCsScaleGroups;  // first warp of the output warpgroup
constexpr int kCsMmaWarp = kCsOutWarp0 + 4;
constexpr int kCsProdWarp = kCsMmaWarp + 1;
constexpr int kCsVecWarp = kCsProdWarp + 1;
constexpr int kCsVecWarps = 2;     // vector warps, heads alternating between them
constexpr int kCsThreads = (kCsVecWarp + kCsVecWarps) * 32;
constexpr int kCsRows = 128;       // rows of a CTA's tile
constexpr int kCsSlice = 64;       // keys per slice of the reduction axis
constexpr int kCsPortion = 16;     // keys per portion (one decay pivot)
constexpr int kCsP = 64;           // head width
constexpr int kCsMaxQ = 256;       // longest chunk
constexpr int kCsBox = 32;         // keys per cb box (128 bytes of fp32)
constexpr int kCsRing = 8;         // A slices in tensor memory
constexpr int kCsPairs = kCsRing / 2;  // slices go in pairs (gs, gs + 1), gs even
constexpr int kCsRingX = 8;        // x slices in shared memory
constexpr int kCsPairsX = kCsRingX / 2;
constexpr int kCsRingV = 4;        // heads' vectors in shared memory (256 keys each)
constexpr int kCsRingVMax = kCsRingV * (kCsMaxQ / kCsRows);  // heads of 128 keys in the same space
constexpr int kCsAcc = 4;          // accumulators in tensor memory
constexpr uint32_t kCsAll = 0xffffffffu;

// shared memory, offsets from a 1024-byte aligned base
constexpr int kCsBoxBytes = kCsRows * kCsBox * 4;                    // 16 KB
constexpr int kCsOffCb = 0;                                          // [Q / 32 boxes]
constexpr int kCsSliceBytesX = kCsSlice * kCsP * 2;                  // 8 KB
constexpr int kCsOffX = kCsOffCb + (kCsMaxQ / kCsBox) * kCsBoxBytes; // [ring]
constexpr int kCsStageBytes = kCsRows * kCsP * 2;                    // 16 KB
constexpr int kCsOffStage = kCsOffX + kCsRingX * kCsSliceBytesX;     // one tile
// The vector ring holds, per head, dA_cs and dt of the keys the tile's rows
// see (nkeys = 128 or 256; rows see keys up to the tile's last row) and
// their key factors: 4 heads of 256 keys or 8 of 128 in the same space.
constexpr int kCsVecRegion = kCsRingV * 2 * kCsMaxQ * 4;             // dA_cs, dt
constexpr int kCsOffVec = kCsOffStage + kCsStageBytes;               // [ring][2][nkeys]
constexpr int kCsOffKf = kCsOffVec + kCsVecRegion;                   // [ring][nkeys] key factors
constexpr int kCsOffMask = kCsOffKf + kCsRingV * kCsMaxQ * 4;        // [ring] rise masks
constexpr int kCsOffBar = kCsOffMask + kCsRingVMax * 4;
// cb_full[Q / 64], pair_full[R / 2], pair_free[R / 2], xp_full[RX / 2],
// xp_free[RX / 2], v_full[RV], v_free[RV], kf_full[RV], acc_full[ACC],
// acc_free[ACC], drain
constexpr int kCsCbSlices = kCsMaxQ / kCsSlice;  // cb arrives slice by slice
constexpr int kCsNumBars =
    kCsCbSlices + 2 * kCsPairs + 2 * kCsPairsX + 3 * kCsRingVMax + 2 * kCsAcc + 1;
constexpr int kCsOffMisc = kCsOffBar + kCsNumBars * 8;
constexpr int kCsSmemBytes = kCsOffMisc + 16 + 1024;
static_assert(kCsSmemBytes <= 227 * 1024, "shared memory budget");
// tensor memory: accumulators in columns [0, 256), A slices (64 bf16 keys =
// 32 columns each) in [256, 512)
constexpr uint32_t kCsTmemCols = 512;
constexpr uint32_t kCsTmemA = kCsAcc * kCsP;
static_assert(kCsTmemA + kCsRing * (kCsSlice / 2) <= kCsTmemCols, "tensor memory budget");
constexpr uint32_t kCsBarOut = 1;  // named barrier of the output warpgroup

__device__ __forceinline__ bool cs_warp_wait(uint64_t* bar, uint32_t parity,
                                             volatile int* abort_flag, uint64_t budget) {
  const bool ok = mbar_wait(bar, parity, abort_flag, budget);
  return __all_sync(kCsAll, ok);
}

__device__ __forceinline__ void cs_drain_wait(uint64_t* bar, uint32_t parity, uint64_t budget) {
  volatile int never = 0;
  mbar_wait(bar, parity, &never, budget);
}

}  // namespace

__global__ void __launch_bounds__(kCsThreads, 1) chunk_scan_kernel(const __grid_constant__ ChunkScanParams p) {
  extern __shared__ uint8_t smem_raw_cs[];
  uint8_t* smem = align_smem_1024(smem_raw_cs);
  uint8_t* sCb = smem + kCsOffCb;
  uint8_t* sX = smem + kCsOffX;
  uint8_t* sStage = smem + kCsOffStage;
  uint8_t* sVec = smem + kCsOffVec;
  float* sKfAll = reinterpret_cast<float*>(smem + kCsOffKf);
  uint32_t* sMask = reinterpret_cast<uint32_t*>(smem + kCsOffMask);
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kCsOffBar);
  uint64_t* cb_full = bars;  // [slice]: the cb boxes of keys 64s .. 64s + 63 landed
  // Slices gs and gs + 1 (gs even, the same head: a head has an even
  // number of slices) share the barriers of pair gs / 2: its A slices in
  // slot pair (gs / 2) % kCsPairs (pair_full: 128 arrivals of each slice's
  // warpgroup), its x slices in x slot pair (gs / 2) % kCsPairsX (xp_full:
  // one arrival with its bytes per slice); the matching _free barriers say
  // the products that read them are done.
  uint64_t* pair_full = bars + kCsCbSlices;
  uint64_t* pair_free = pair_full + kCsPairs;
  uint64_t* xp_full = pair_free + kCsPairs;
  uint64_t* xp_free = xp_full + kCsPairsX;
  uint64_t* v_full = xp_free + kCsPairsX;
  uint64_t* v_free = v_full + kCsRingVMax;
  uint64_t* kf_full = v_free + kCsRingVMax;  // the head's key factors and rise mask written
  uint64_t* acc_full = kf_full + kCsRingVMax;
  uint64_t* acc_free = acc_full + kCsAcc;
  uint64_t* drain = acc_free + kCsAcc;
  uint32_t* sTmemBase = reinterpret_cast<uint32_t*>(smem + kCsOffMisc);
  volatile int* sAbort = reinterpret_cast<volatile int*>(smem + kCsOffMisc + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t budget = p.timeout_ns;

  // CTA -> (b, c, tile, head block): the head blocks and tiles of one chunk
  // are adjacent, so the CTAs of a chunk read its cb and x from L2
  const int tiles = p.Q / kCsRows;
  const int hblocks = p.H / p.HB;
  int idx = blockIdx.x;
  const int hb = idx % hblocks;
  idx /= hblocks;
  const int mt = idx % tiles;
  idx /= tiles;
  const int c = idx % p.nchunks;
  const int b = idx / p.nchunks;
  const int h0 = hb * p.HB;                    // first head of the block
  const int g = h0 / (p.H / p.G);              // the block's group (HB divides H / G)
  const int m0 = mt * kCsRows;                 // first row of the tile within the chunk
  const int n_slices = (m0 + kCsRows) / kCsSlice;  // keys 0 .. m0 + 127 are visible to some row
  const int log_ns = (n_slices == 4) ? 2 : 1;      // n_slices is 2 or 4 (Q = 128 or 256)
  const int total = p.HB * n_slices;           // slices of the CTA
  const int nkeys = n_slices * kCsSlice;       // keys some row of the tile sees
  const int log_rv = (nkeys == kCsMaxQ) ? 2 : 3;  // heads in the vector ring: 4 or 8
  const int ringv = 1 << log_rv;

  if (threadIdx.x == 0) {
    for (int i = 0; i < kCsCbSlices; ++i) mbar_init(&cb_full[i], 1);
    for (int i = 0; i < kCsPairs; ++i) {
      mbar_init(&pair_full[i], 2 * 128);
      mbar_init(&pair_free[i], 1);
    }
    for (int i = 0; i < kCsPairsX; ++i) {
      mbar_init(&xp_full[i], 2);
      mbar_init(&xp_free[i], 1);
    }
    for (int i = 0; i < kCsRingVMax; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_free[i], 128 * n_slices);  // every slice's warpgroup
      mbar_init(&kf_full[i], 32);
    }
    for (int i = 0; i < kCsAcc; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_free[i], 128);
    }
    mbar_init(drain, 1);
    *sAbort = 0;
    fence_mbar_init();
  }
  if (warp == kCsMmaWarp) {
    tmem_alloc(sTmemBase, kCsTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *sTmemBase;

  if (warp < kCsOutWarp0) {
    // ---------------------------------------------------------- scaling
    const int w = warp >> 2;                   // warpgroup
    // Tensor-memory lanes 32q .. 32q + 31 (q = warp % 4, the warp's
    // scheduler) hold the tile's row block (q + j) % 4 for head j: the rows
    // near the diagonal cost the most, and rotating the blocks over the
    // heads spreads them over the four schedulers.
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const float l2e = 1.4426950408889634f;
    const uint64_t nl2e2 = f2_pack(-l2e, -l2e);
    bool ok = true;
    uint32_t cb_seen = 0;                      // cb slices this warp has seen land
    for (int gs = w; gs < total && ok; gs += kCsScaleGroups) {
      const int j = gs >> log_ns;              // head of the block
      const int s = gs & (n_slices - 1);       // slice of the head
      const int vs = j & (ringv - 1);
      const int slot = gs % kCsRing;
      const int pr = gs >> 1;                  // pair
      if (!((cb_seen >> s) & 1u)) {
        ok = cs_warp_wait(&cb_full[s], 0, sAbort, budget);
        cb_seen |= 1u << s;
      }
      ok = ok && cs_warp_wait(&kf_full[vs], (j >> log_rv) & 1, sAbort, budget);
      ok = ok && (pr < kCsPairs || cs_warp_wait(&pair_free[pr % kCsPairs],
                                                ((pr / kCsPairs) - 1) & 1, sAbort, budget));
      tc_fence_after_sync();                   // the slot's last products are done before it is rewritten
      const float* sDA = reinterpret_cast<const float*>(sVec) + vs * 2 * nkeys;
      const float* sDT = sDA + nkeys;
      const float* sKf = sKfAll + vs * nkeys + s * kCsSlice;
      const uint32_t rises = sMask[vs] >> (s * (kCsSlice / kCsPortion));
      const int r = ((warp + j) & 3) * 32 + lane;  // row of the tile
      const int m = m0 + r;                      // row of the chunk
      const int row0 = m0 + ((warp + j) & 3) * 32;  // the warp's first row
      if (ok) {
        const float da_raw = sDA[m];
        const float da_m = da_raw * l2e;
        const uint64_t dam2 = f2_pack(da_m, da_m);
        const uint32_t a_col = tmem + lane_base + kCsTmemA + slot * (kCsSlice / 2);
        // the four portions unrolled: their loads and products interleave
#pragma unroll
        for (int pi = 0; pi < kCsSlice / kCsPortion; ++pi) {
          const int k0 = s * kCsSlice + pi * kCsPortion;   // first key of the portion
          const float* cb_row = reinterpret_cast<const float*>(
              sCb + (2 * s + (pi >> 1)) * kCsBoxBytes + r * 128);
          uint32_t pk[kCsPortion / 2];
          const float dap = sDA[k0 + kCsPortion - 1];
          if (k0 > row0 + 31) {
            // every key after every row of the warp
#pragma unroll
            for (int q = 0; q < kCsPortion / 2; ++q) pk[q] = 0u;
          } else if (!((rises >> pi) & 1u) && k0 + kCsPortion - 1 <= row0 && da_raw <= dap) {
            // every key at or before the row: row factor times key factors
            const float rowf = ex2_approx((da_raw - dap) * l2e);
            const uint64_t rf2 = f2_pack(rowf, rowf);
#pragma unroll
            for (int q = 0; q < kCsPortion / 4; ++q) {
              const int cq = (pi & 1) * 4 + q;  // 16-byte chunk of the 128-byte cb row
              const float4 cv = *reinterpret_cast<const float4*>(
                  reinterpret_cast<const uint8_t*>(cb_row) + ((cq ^ (r & 7)) << 4));
              const float4 kv = *reinterpret_cast<const float4*>(sKf + pi * kCsPortion + 4 * q);
              float v0, v1, v2, v3;
              f2_unpack(f2_mul(f2_mul(f2_pack(kv.x, kv.y), rf2), f2_pack(cv.x, cv.y)), v0, v1);
              f2_unpack(f2_mul(f2_mul(f2_pack(kv.z, kv.w), rf2), f2_pack(cv.z, cv.w)), v2, v3);
              pk[2 * q] = pack_bf16x2(v0, v1);
              pk[2 * q + 1] = pack_bf16x2(v2, v3);
            }
          } else {
            // the diagonal band, or a decay that rises: one exponential per
            // (row, key); keys after the row drop out by a select, since the
            // decay may be inf there
            const bool diag = (k0 + kCsPortion - 1 > row0);
#pragma unroll
            for (int q = 0; q < kCsPortion / 4; ++q) {
              const int k = k0 + 4 * q;
              const int cq = (pi & 1) * 4 + q;
              const float4 cv = *reinterpret_cast<const float4*>(
                  reinterpret_cast<const uint8_t*>(cb_row) + ((cq ^ (r & 7)) << 4));
              const float4 da = *reinterpret_cast<const float4*>(sDA + k);
              const float4 dtv = *reinterpret_cast<const float4*>(sDT + k);
              float e0, e1, e2, e3;
              f2_unpack(f2_fma(f2_pack(da.x, da.y), nl2e2, dam2), e0, e1);
              f2_unpack(f2_fma(f2_pack(da.z, da.w), nl2e2, dam2), e2, e3);
              const uint64_t w01 = f2_mul(f2_mul(f2_pack(ex2_approx(e0), ex2_approx(e1)),
                                                 f2_pack(cv.x, cv.y)), f2_pack(dtv.x, dtv.y));
              const uint64_t w23 = f2_mul(f2_mul(f2_pack(ex2_approx(e2), ex2_approx(e3)),
                                                 f2_pack(cv.z, cv.w)), f2_pack(dtv.z, dtv.w));
              float v0, v1, v2, v3;
              f2_unpack(w01, v0, v1);
              f2_unpack(w23, v2, v3);
              if (diag) {
                v0 = (k + 0 <= m) ? v0 : 0.f;
                v1 = (k + 1 <= m) ? v1 : 0.f;
                v2 = (k + 2 <= m) ? v2 : 0.f;
                v3 = (k + 3 <= m) ? v3 : 0.f;
              }
              pk[2 * q] = pack_bf16x2(v0, v1);
              pk[2 * q + 1] = pack_bf16x2(v2, v3);
            }
          }
          // keys 2i, 2i + 1 of the portion in column i
          tmem_st_x8(a_col + pi * (kCsPortion / 2), pk);
        }
        tmem_st_wait();
        tc_fence_before_sync();
        mbar_arrive(&pair_full[pr % kCsPairs]);
        mbar_arrive(&v_free[vs]);              // this slice no longer reads the head's vectors
      }
    }
  } else if (warp < kCsMmaWarp) {
    // ---------------------------------------------------------- output
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const bool issuer = (warp == kCsOutWarp0) && elect_one();
    const uint64_t pol_out = l2_policy_evict_first();  // nothing here reads it again
    bool ok = true;
    for (int j = 0; j < p.HB; ++j) {
      const int a = j % kCsAcc;
      ok = ok && cs_warp_wait(&acc_full[a], (j / kCsAcc) & 1, sAbort, budget);
      const int r = ((warp + j) & 3) * 32 + lane;  // the tile row in this lane for head j
      uint8_t* stage = sStage;
      // the store of head j - 1 is done reading the staging tile
      if (issuer) tma_store_wait_read<0>();
      __syncwarp();
      named_barrier_sync(kCsBarOut, 128);
      if (ok) {
        tc_fence_after_sync();
#pragma unroll
        for (int half = 0; half < 2; ++half) {
          uint32_t v[32];
          tmem_ld_x32(tmem + lane_base + a * kCsP + half * 32, v);
          tmem_ld_wait();
          reg_after_wait(v);
          if (half == 1) {
            tc_fence_before_sync();
            mbar_arrive(&acc_free[a]);         // the accumulator may take head j + 4
          }
#pragma unroll
          for (int q = 0; q < 4; ++q) {        // 16-byte chunks 4 * half + q of the row
            const int chunk = (4 * half + q) ^ (r & 7);
            *reinterpret_cast<uint4*>(stage + r * 128 + chunk * 16) = make_uint4(
                pack_bf16x2(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1])),
                pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3])),
                pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5])),
                pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7])));
          }
        }
        fence_proxy_async_smem();              // the staging writes before the TMA store reads them
      }
      named_barrier_sync(kCsBarOut, 128);
      if (issuer && ok) {
        tma_store_4d_hint(&p.tm_out, stage, 0, h0 + j, c * p.Q + m0, b, pol_out);
        tma_store_commit();
      }
    }
    if (issuer) tma_store_wait_all();
  } else if (warp == kCsMmaWarp) {
    // ---------------------------------------------------------- tensor-core issuer
    const bool leader = elect_one();
    constexpr uint32_t idesc = make_idesc_bf16_f32(128, kCsP, false, true);
    bool ok = true;
    for (int pr = 0; 2 * pr < total && ok; ++pr) {
      const int j = (2 * pr) >> log_ns;
      const int s0 = (2 * pr) & (n_slices - 1);  // first slice of the pair within its head
      const int a = j % kCsAcc;
      const int ps = pr % kCsPairs, px = pr % kCsPairsX;
      // accumulator a must have been read out (head j - 4)
      if (s0 == 0 && j >= kCsAcc &&
          !cs_warp_wait(&acc_free[a], ((j / kCsAcc) - 1) & 1, sAbort, budget)) {
        ok = false;
        break;
      }
      if (!cs_warp_wait(&pair_full[ps], (pr / kCsPairs) & 1, sAbort, budget) ||
          !cs_warp_wait(&xp_full[px], (pr / kCsPairsX) & 1, sAbort, budget)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      if (leader) {
#pragma unroll
        for (int i = 0; i < 2; ++i) {
          const uint32_t a_tmem = tmem + kCsTmemA + (2 * ps + i) * (kCsSlice / 2);
          // the x slice is a single 64-wide slab: the leading offset is unused
          const uint64_t b_desc =
              make_smem_desc_sw128(smem_u32(sX + (2 * px + i) * kCsSliceBytesX), 1024, 1024);
#pragma unroll
          for (int kk = 0; kk < kCsSlice / 16; ++kk) {
            mma_ts(tmem + a * kCsP, a_tmem + kk * 8, b_desc + (uint64_t)((kk * 2048) >> 4),
                   idesc, (s0 + i > 0 || kk > 0) ? 1u : 0u);
          }
        }
        tc_commit(&pair_free[ps]);
        tc_commit(&xp_free[px]);
        if (s0 + 2 == n_slices) tc_commit(&acc_full[a]);
      }
    }
    if (leader) {
      tc_commit(drain);
      cs_drain_wait(drain, 0, budget);
    }
    __syncwarp();
  } else if (warp >= kCsVecWarp) {
    // ---------------------------------------------------------- key factors
    // Per head, kf[k] = exp(dA_cs[k | 15] - dA_cs[k]) dt[k] (k | 15 is the
    // last key of k's 16-key portion) and a mask with bit i set where
    // portion i has a key whose factor would exceed 1.  For a row m at or
    // after k | 15,
    //   exp(dA_cs[m] - dA_cs[k]) = exp(dA_cs[m] - dA_cs[k | 15]) exp(dA_cs[k | 15] - dA_cs[k]),
    // and where both exponents are <= 0 (dA_cs does not rise, as with
    // dt > 0 and A < 0) both factors lie in [0, 1]: a portion wholly at or
    // before a row then costs one exponential per row and one per key
    // instead of one per (row, key).
    // It also loads each head's dA_cs and dt (1-D bulk copies, the keys
    // 0 .. nkeys - 1 the tile's rows see) into a ring of 4 or 8 slots, as far
    // ahead of the head it works on as the slots allow.  Warp v takes the
    // heads j = v, v + 2, ... (so the even slots or the odd ones).
    const float l2e = 1.4426950408889634f;
    const bool leader = elect_one();
    const int v = warp - kCsVecWarp;
    bool ok = true;
    int issued = v;                            // next head of this warp to load
    auto issue = [&](int jn) {
      const int vs = jn & (ringv - 1);
      if (leader) {
        const size_t off = (((size_t)b * p.H + h0 + jn) * p.nchunks + c) * p.Q;
        float* dst = reinterpret_cast<float*>(sVec) + vs * 2 * nkeys;
        mbar_arrive_expect_tx(&v_full[vs], 2 * nkeys * 4);
        bulk_load(dst, p.dA_cs + off, nkeys * 4, &v_full[vs]);
        bulk_load(dst + nkeys, p.dt + off, nkeys * 4, &v_full[vs]);
      }
      __syncwarp();
    };
    for (int j = v; j < p.HB && ok; j += kCsVecWarps) {
      const int vs = j & (ringv - 1);
      // issue every later head of this warp whose slot is free (without
      // waiting), and head j itself in any case (waiting for its slot if
      // need be)
      while (ok && issued < p.HB) {
        const int jn = issued;
        if (jn >= ringv) {
          bool free_now = mbar_test_wait(&v_free[jn & (ringv - 1)], ((jn >> log_rv) - 1) & 1);
          free_now = __all_sync(kCsAll, free_now);
          if (!free_now) {
            if (jn > j) break;
            ok = cs_warp_wait(&v_free[jn & (ringv - 1)], ((jn >> log_rv) - 1) & 1, sAbort,
                              budget);
            if (!ok) break;
          }
        }
        issue(jn);
        issued += kCsVecWarps;
      }
      if (!ok || !cs_warp_wait(&v_full[vs], (j >> log_rv) & 1, sAbort, budget)) {
        ok = false;
        break;
      }
      const float* sDA = reinterpret_cast<const float*>(sVec) + vs * 2 * nkeys;
      const float* sDT = sDA + nkeys;
      float* sKf = sKfAll + vs * nkeys;
      uint32_t mask = 0;
      // every load first, then the arithmetic and the stores, so the
      // 32-key groups overlap (a store to sKf could otherwise alias a
      // later load)
      float dak[kCsMaxQ / 32], dap[kCsMaxQ / 32], dtk[kCsMaxQ / 32];
#pragma unroll
      for (int i = 0; i < kCsMaxQ / 32; ++i) {
        if (32 * i < nkeys) {
          const int k = 32 * i + lane;
          dak[i] = sDA[k];
          dap[i] = sDA[k | (kCsPortion - 1)];
          dtk[i] = sDT[k];
        }
      }
#pragma unroll
      for (int i = 0; i < kCsMaxQ / 32; ++i) {
        if (32 * i < nkeys) {
          sKf[32 * i + lane] = ex2_approx((dap[i] - dak[i]) * l2e) * dtk[i];
          const uint32_t bal = __ballot_sync(kCsAll, !(dap[i] <= dak[i]));
          mask |= ((bal & 0xffffu) ? 1u : 0u) << (2 * i);
          mask |= ((bal >> 16) ? 1u : 0u) << (2 * i + 1);
        }
      }
      if (lane == 0) sMask[vs] = mask;
      __syncwarp();
      mbar_arrive(&kf_full[vs]);
    }
    // every copy this warp issued lands before the CTA exits (the last
    // loads into its slots: heads issued - ringv .. issued - 2 of its parity)
    if (leader) {
      for (int j = issued - kCsVecWarps; j >= v && j >= issued - ringv; j -= kCsVecWarps)
        cs_drain_wait(&v_full[j & (ringv - 1)], (j >> log_rv) & 1, budget);
    }
    __syncwarp();
  } else {
    // ---------------------------------------------------------- TMA producer
    const bool leader = elect_one();
    // The keys 0 .. 127 of a chunk's x are read by the CTAs of both row
    // tiles, the first tile's CTA running ahead (half the slices per head):
    // its reads stay in L2 for the second's (evict last), the second
    // tile's, the last ones, go first (as does the output).  On 8 x 8192
    // this took the DRAM reads from 985 MB (everything evict first) to
    // 682 MB, against 638 MB read once.
    const uint64_t pol_x = (mt + 1 < tiles) ? l2_policy_evict_last() : l2_policy_evict_first();
    const uint64_t pol_cb = l2_policy_evict_last();
    bool ok = true;
    int gs = 0;
    int cb_issued = 0;                         // cb slices whose loads were issued
    const int zc = (b * p.nchunks + c) * p.G + g;
    for (int j = 0; j < p.HB && ok; ++j) {
      const int h = h0 + j;
      if (leader) {
        // the x slices and vectors of the head two ahead into L2, so that
        // their loads into the rings wait on L2 rather than on DRAM
        for (int jj = (j == 0 ? 1 : j + 2); jj <= j + 2 && jj < p.HB; ++jj) {
          for (int s = 0; s < n_slices; ++s)
            tma_prefetch_4d(&p.tm_x, 0, h0 + jj, c * p.Q + s * kCsSlice, b);
          const size_t off = (((size_t)b * p.H + h0 + jj) * p.nchunks + c) * p.Q;
          bulk_prefetch_l2(p.dA_cs + off, nkeys * 4);
          bulk_prefetch_l2(p.dt + off, nkeys * 4);
        }
      }
      for (int s = 0; s < n_slices; ++s, ++gs) {
        const int pr = gs >> 1;
        const int px = pr % kCsPairsX;
        if ((gs & 1) == 0 && pr >= kCsPairsX &&
            !cs_warp_wait(&xp_free[px], ((pr / kCsPairsX) - 1) & 1, sAbort, budget)) {
          ok = false;
          break;
        }
        if (j == 0) {
          // the tile's cb for slice s (two 32-key boxes) just ahead of the
          // first head's x slice s: the first slices can start before the
          // whole cb has arrived
          if (leader) {
            mbar_arrive_expect_tx(&cb_full[s], 2 * kCsBoxBytes);
            for (int i = 2 * s; i < 2 * s + 2; ++i)
              tma_load_3d(sCb + i * kCsBoxBytes, &p.tm_cb, &cb_full[s], i * kCsBox, m0, zc,
                          pol_cb);
          }
          ++cb_issued;
        }
        if (leader) {
          mbar_arrive_expect_tx(&xp_full[px], kCsSliceBytesX);
          tma_load_4d(sX + (2 * px + (gs & 1)) * kCsSliceBytesX, &p.tm_x, &xp_full[px], 0, h,
                      c * p.Q + s * kCsSlice, b, pol_x);
        }
      }
    }
    // every copy issued lands before the CTA exits (the producer stops only
    // before the first slice of a pair, so every x pair it started is whole)
    if (leader) {
      for (int i = 0; i < cb_issued; ++i) cs_drain_wait(&cb_full[i], 0, budget);
      const int np = gs / 2;                   // pairs with both x slices issued
      for (int pr = np > kCsPairsX ? np - kCsPairsX : 0; pr < np; ++pr)
        cs_drain_wait(&xp_full[pr % kCsPairsX], (pr / kCsPairsX) & 1, budget);
    }
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == kCsMmaWarp) tmem_dealloc(tmem, kCsTmemCols);
  if (threadIdx.x == 0 && *sAbort) atomicCAS(&g_cs_status, 0, (int)ATTN_ERR_TIMEOUT);
}

namespace {
std::mutex g_cs_mu;
bool g_cs_attr[64] = {};
int g_cs_sms[64] = {};

// Heads per CTA: the largest of 32, 16, 8, 4, 2, 1 that divides the group
// size and still gives every SM at least three CTAs.  A CTA loads its tile's
// cb once for all its heads, so larger blocks load it less often; too few
// CTAs leave SMs idle.
int choose_head_block(const ChunkScanParams& p, int sms) {
  const int group = p.H / p.G;
  const long long tiles = (long long)p.B * p.nchunks * (p.Q / kCsRows) * p.G;
  int hb = 32;
  while (hb > 1 && (group % hb != 0 || tiles * (group / hb) < 3ll * sms)) hb >>= 1;
  return hb;
}
}  // namespace

cudaError_t launch_chunk_scan(const ChunkScanParams& params, cudaStream_t stream) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  int sms = 0;
  {
    std::lock_guard<std::mutex> lk(g_cs_mu);
    if (!g_cs_attr[dev]) {
      err = cudaFuncSetAttribute(chunk_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kCsSmemBytes);
      if (err != cudaSuccess) return err;
      err = cudaDeviceGetAttribute(&g_cs_sms[dev], cudaDevAttrMultiProcessorCount, dev);
      if (err != cudaSuccess) return err;
      g_cs_attr[dev] = true;
    }
    sms = g_cs_sms[dev];
  }
  ChunkScanParams p = params;
  if (p.HB <= 0) p.HB = choose_head_block(p, sms);
  if ((p.H / p.G) % p.HB != 0) return cudaErrorInvalidValue;
  const long long ctas = (long long)p.B * p.nchunks * (p.Q / kCsRows) * (p.H / p.HB);
  if (ctas <= 0 || ctas >= (1ll << 31)) return cudaErrorInvalidValue;
  chunk_scan_kernel<<<(unsigned)ctas, kCsThreads, kCsSmemBytes, stream>>>(p);
  return cudaGetLastError();
}

cudaError_t read_chunk_scan_status(int* status, bool reset) {
  cudaError_t err = cudaMemcpyFromSymbol(status, g_cs_status, sizeof(int));
  if (err != cudaSuccess) return err;
  if (reset) {
    const int zero = 0;
    err = cudaMemcpyToSymbol(g_cs_status, &zero, sizeof(int));
  }
  return err;
}

}  // namespace attnpipe
