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
// one group), 640 threads:
//   warps 0-15 four elementwise warpgroups, thread = row of the tile; for
//              each head and each 64-key slice, warpgroup w scales keys
//              16w .. 16w + 15 of its row of cb (kept in shared memory for
//              all the CTA's heads) by exp2 of the decay and dt into bf16,
//              written into a ring of 128-byte-swizzled K-major A slices;
//              after each head they also store the previous head's output;
//   warp 16    tensor-core issuer: per slice, 4 tcgen05.mma (M = 128,
//              N = 64, K = 16) of the A slice with the x slice (MN-major)
//              into one of two 128 x 64 fp32 accumulators in tensor memory
//              (heads alternate between them);
//   warp 17    TMA producer: the tile's cb once (3-D map, 32-key boxes), then
//              per head its dA_cs and dt vectors (1-D bulk copies) and its x
//              slices (4-D map over [B, L, H, P]) through rings.
// The rings and the two accumulators let the next head's loads and scaling
// overlap the current head's products and the previous head's output.
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

constexpr int kCsThreads = 640;
constexpr int kCsEwGroups = 4;     // elementwise warpgroups
constexpr int kCsRows = 128;       // rows of a CTA's tile
constexpr int kCsSlice = 64;       // keys per slice of the reduction axis
constexpr int kCsEwKeys = kCsSlice / kCsEwGroups;  // keys of a slice per thread
constexpr int kCsP = 64;           // head width
constexpr int kCsMaxQ = 256;       // longest chunk
constexpr int kCsBox = 32;         // keys per cb box (128 bytes of fp32)
constexpr int kCsRingA = 3;        // A slices in flight
constexpr int kCsRingX = 3;        // x slices in flight
constexpr int kCsRingV = 2;        // heads' vectors in flight
constexpr uint32_t kCsAll = 0xffffffffu;

// shared memory, offsets from a 1024-byte aligned base
constexpr int kCsBoxBytes = kCsRows * kCsBox * 4;                    // 16 KB
constexpr int kCsOffCb = 0;                                          // [Q / 32 boxes]
constexpr int kCsSliceBytesA = kCsRows * kCsSlice * 2;               // 16 KB
constexpr int kCsOffA = kCsOffCb + (kCsMaxQ / kCsBox) * kCsBoxBytes; // [ring]
constexpr int kCsSliceBytesX = kCsSlice * kCsP * 2;                  // 8 KB
constexpr int kCsOffX = kCsOffA + kCsRingA * kCsSliceBytesA;         // [ring]
constexpr int kCsVecBytes = 2 * kCsMaxQ * 4;                         // dA_cs, dt of one head
constexpr int kCsOffVec = kCsOffX + kCsRingX * kCsSliceBytesX;       // [ring]
constexpr int kCsOffBar = kCsOffVec + kCsRingV * kCsVecBytes;
// cb_full, a_full[RA], a_free[RA], x_full[RX], x_free[RX], v_full[RV],
// v_free[RV], acc_full[2], acc_free[2], drain
constexpr int kCsNumBars = 1 + 2 * kCsRingA + 2 * kCsRingX + 2 * kCsRingV + 4 + 1;
constexpr int kCsOffMisc = kCsOffBar + kCsNumBars * 8;
constexpr int kCsSmemBytes = kCsOffMisc + 16 + 1024;
constexpr uint32_t kCsTmemCols = 128;                                // two accumulators
static_assert(kCsSmemBytes <= 227 * 1024, "shared memory budget");

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
  uint8_t* sA = smem + kCsOffA;
  uint8_t* sX = smem + kCsOffX;
  uint8_t* sVec = smem + kCsOffVec;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kCsOffBar);
  uint64_t* cb_full = bars;
  uint64_t* a_full = bars + 1;
  uint64_t* a_free = a_full + kCsRingA;
  uint64_t* x_full = a_free + kCsRingA;
  uint64_t* x_free = x_full + kCsRingX;
  uint64_t* v_full = x_free + kCsRingX;
  uint64_t* v_free = v_full + kCsRingV;
  uint64_t* acc_full = v_free + kCsRingV;   // [2]
  uint64_t* acc_free = acc_full + 2;        // [2]
  uint64_t* drain = acc_free + 2;
  uint32_t* sTmemBase = reinterpret_cast<uint32_t*>(smem + kCsOffMisc);
  volatile int* sAbort = reinterpret_cast<volatile int*>(smem + kCsOffMisc + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t budget = p.timeout_ns;

  // CTA -> (b, c, tile, head block): the head blocks and tiles of one chunk
  // are adjacent, so the CTAs of a chunk read its cb from L2
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
  const int n_boxes = 2 * n_slices;

  if (threadIdx.x == 0) {
    mbar_init(cb_full, 1);
    for (int i = 0; i < kCsRingA; ++i) {
      mbar_init(&a_full[i], kCsEwGroups * 128);
      mbar_init(&a_free[i], 1);
    }
    for (int i = 0; i < kCsRingX; ++i) {
      mbar_init(&x_full[i], 1);
      mbar_init(&x_free[i], 1);
    }
    for (int i = 0; i < kCsRingV; ++i) {
      mbar_init(&v_full[i], 1);
      mbar_init(&v_free[i], kCsEwGroups * 128);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(&acc_full[i], 1);
      mbar_init(&acc_free[i], kCsEwGroups * 128);
    }
    mbar_init(drain, 1);
    *sAbort = 0;
    fence_mbar_init();
  }
  if (warp == 16) {
    tmem_alloc(sTmemBase, kCsTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *sTmemBase;

  if (warp < 4 * kCsEwGroups) {
    // ---------------------------------------------------------- elementwise
    const int w = warp >> 2;
    const int r = (warp & 3) * 32 + lane;      // row of the tile
    const int m = m0 + r;                      // row of the chunk
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const float l2e = 1.4426950408889634f;
    const uint64_t nl2e2 = f2_pack(-l2e, -l2e);
    bool ok = cs_warp_wait(cb_full, 0, sAbort, budget);
    // stores the output rows of head j from accumulator j & 1
    auto epilogue = [&](int j) -> bool {
      if (!cs_warp_wait(&acc_full[j & 1], (j >> 1) & 1, sAbort, budget)) return false;
      tc_fence_after_sync();
      uint32_t v[16];
      tmem_ld_x16(tmem + lane_base + (j & 1) * kCsP + kCsEwKeys * w, v);
      tmem_ld_wait();
      reg_after_wait(v);
      tc_fence_before_sync();
      mbar_arrive(&acc_free[j & 1]);           // the accumulator may take head j + 2
      uint4* dst = reinterpret_cast<uint4*>(
          static_cast<uint16_t*>(p.out) +
          ((((size_t)b * p.L + (size_t)c * p.Q + m) * p.H + h0 + j) * kCsP) + kCsEwKeys * w);
#pragma unroll
      for (int q = 0; q < kCsEwKeys / 8; ++q) {
        uint4 val;
        val.x = pack_bf16x2(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1]));
        val.y = pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3]));
        val.z = pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5]));
        val.w = pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7]));
        dst[q] = val;
      }
      return true;
    };
    int gs = 0;                                // A slices produced so far
    for (int j = 0; j < p.HB && ok; ++j) {
      const int vs = j % kCsRingV;
      if (!cs_warp_wait(&v_full[vs], (j / kCsRingV) & 1, sAbort, budget)) { ok = false; break; }
      const float* sDA = reinterpret_cast<const float*>(sVec + vs * kCsVecBytes);
      const float* sDT = sDA + kCsMaxQ;
      const float da_m = sDA[m] * l2e;
      const uint64_t dam2 = f2_pack(da_m, da_m);
      for (int s = 0; s < n_slices; ++s, ++gs) {
        const int slot = gs % kCsRingA;
        if (gs >= kCsRingA &&
            !cs_warp_wait(&a_free[slot], ((gs / kCsRingA) - 1) & 1, sAbort, budget)) {
          ok = false;
          break;
        }
        const int k0 = s * kCsSlice + kCsEwKeys * w;  // first key of this thread's 16
        const bool diag = (k0 + kCsEwKeys - 1 > m0);   // keys after some row of the tile
        // row r of the cb box holding these keys: 16-byte chunks in the
        // 128-byte swizzle, this thread's 4 chunks from (w % 2) * 4
        const uint8_t* cb_row = sCb + (2 * s + (w >> 1)) * kCsBoxBytes + r * 128;
        uint32_t pk[kCsEwKeys / 2];
#pragma unroll
        for (int q = 0; q < kCsEwKeys / 4; ++q) {
          const int k = k0 + 4 * q;
          const int cq = (w & 1) * 4 + q;
          const float4 cv = *reinterpret_cast<const float4*>(cb_row + ((cq ^ (r & 7)) << 4));
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
          if (diag) {  // keys after the row drop out (select: the decay may be inf there)
            v0 = (k + 0 <= m) ? v0 : 0.f;
            v1 = (k + 1 <= m) ? v1 : 0.f;
            v2 = (k + 2 <= m) ? v2 : 0.f;
            v3 = (k + 3 <= m) ? v3 : 0.f;
          }
          pk[2 * q] = pack_bf16x2(v0, v1);
          pk[2 * q + 1] = pack_bf16x2(v2, v3);
        }
        uint8_t* row_base = sA + slot * kCsSliceBytesA + r * 128;
#pragma unroll
        for (int q = 0; q < kCsEwKeys / 8; ++q) {
          const int chunk = ((kCsEwKeys / 8) * w + q) ^ (r & 7);
          *reinterpret_cast<uint4*>(row_base + chunk * 16) =
              make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
        }
        fence_proxy_async_smem();  // generic-proxy writes before the tensor core reads them
        mbar_arrive(&a_full[slot]);
      }
      if (!ok) break;
      mbar_arrive(&v_free[vs]);                // this head's vectors are no longer read
      // the previous head's output, while the tensor core works on this one
      if (j > 0 && !epilogue(j - 1)) { ok = false; break; }
    }
    if (ok && p.HB > 0) epilogue(p.HB - 1);
  } else if (warp == 16) {
    // ---------------------------------------------------------- tensor-core issuer
    const bool leader = elect_one();
    constexpr uint32_t idesc = make_idesc_bf16_f32(128, kCsP, false, true);
    bool ok = true;
    int gs = 0;                                // slices consumed (A and x rings advance together)
    for (int j = 0; j < p.HB && ok; ++j) {
      // accumulator j & 1 must have been read out (head j - 2)
      if (j >= 2 && !cs_warp_wait(&acc_free[j & 1], ((j >> 1) - 1) & 1, sAbort, budget)) {
        ok = false;
        break;
      }
      for (int s = 0; s < n_slices; ++s, ++gs) {
        const int sa = gs % kCsRingA, sx = gs % kCsRingX;
        if (!cs_warp_wait(&a_full[sa], (gs / kCsRingA) & 1, sAbort, budget) ||
            !cs_warp_wait(&x_full[sx], (gs / kCsRingX) & 1, sAbort, budget)) {
          ok = false;
          break;
        }
        tc_fence_after_sync();
        if (leader) {
          const uint64_t a_desc = make_smem_desc_sw128(smem_u32(sA + sa * kCsSliceBytesA), 16, 1024);
          // the x slice is a single 64-wide slab: the leading offset is unused
          const uint64_t b_desc =
              make_smem_desc_sw128(smem_u32(sX + sx * kCsSliceBytesX), 1024, 1024);
#pragma unroll
          for (int kk = 0; kk < kCsSlice / 16; ++kk) {
            mma_ss(tmem + (j & 1) * kCsP, a_desc + (uint64_t)((kk * 32) >> 4),
                   b_desc + (uint64_t)((kk * 2048) >> 4), idesc, (s > 0 || kk > 0) ? 1u : 0u);
          }
          tc_commit(&a_free[sa]);
          tc_commit(&x_free[sx]);
          if (s + 1 == n_slices) tc_commit(&acc_full[j & 1]);
        }
      }
    }
    if (leader) {
      tc_commit(drain);
      cs_drain_wait(drain, 0, budget);
    }
    __syncwarp();
  } else if (warp == 17) {
    // ---------------------------------------------------------- TMA producer
    const bool leader = elect_one();
    const uint64_t pol_x = l2_policy_evict_first();
    const uint64_t pol_cb = l2_policy_evict_last();
    bool ok = true;
    int gs = 0, issued_v = 0;
    if (leader) {
      mbar_arrive_expect_tx(cb_full, n_boxes * kCsBoxBytes);
      const int zc = (b * p.nchunks + c) * p.G + g;
      for (int i = 0; i < n_boxes; ++i)
        tma_load_3d(sCb + i * kCsBoxBytes, &p.tm_cb, cb_full, i * kCsBox, m0, zc, pol_cb);
    }
    for (int j = 0; j < p.HB && ok; ++j) {
      const int h = h0 + j;
      const int vs = j % kCsRingV;
      if (j >= kCsRingV &&
          !cs_warp_wait(&v_free[vs], ((j / kCsRingV) - 1) & 1, sAbort, budget)) {
        ok = false;
        break;
      }
      if (leader) {
        const size_t vec_off = (((size_t)b * p.H + h) * p.nchunks + c) * p.Q;
        float* dst = reinterpret_cast<float*>(sVec + vs * kCsVecBytes);
        mbar_arrive_expect_tx(&v_full[vs], 2 * p.Q * 4);
        bulk_load(dst, p.dA_cs + vec_off, p.Q * 4, &v_full[vs]);
        bulk_load(dst + kCsMaxQ, p.dt + vec_off, p.Q * 4, &v_full[vs]);
      }
      ++issued_v;
      for (int s = 0; s < n_slices; ++s, ++gs) {
        const int sx = gs % kCsRingX;
        if (gs >= kCsRingX &&
            !cs_warp_wait(&x_free[sx], ((gs / kCsRingX) - 1) & 1, sAbort, budget)) {
          ok = false;
          break;
        }
        if (leader) {
          mbar_arrive_expect_tx(&x_full[sx], kCsSliceBytesX);
          tma_load_4d(sX + sx * kCsSliceBytesX, &p.tm_x, &x_full[sx], 0, h,
                      c * p.Q + s * kCsSlice, b, pol_x);
        }
      }
    }
    // every copy issued lands before the CTA exits
    if (leader) {
      cs_drain_wait(cb_full, 0, budget);
      const int first_v = issued_v > kCsRingV ? issued_v - kCsRingV : 0;
      for (int j = first_v; j < issued_v; ++j)
        cs_drain_wait(&v_full[j % kCsRingV], (j / kCsRingV) & 1, budget);
      const int first_x = gs > kCsRingX ? gs - kCsRingX : 0;
      for (int t = first_x; t < gs; ++t)
        cs_drain_wait(&x_full[t % kCsRingX], (t / kCsRingX) & 1, budget);
    }
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 16) tmem_dealloc(tmem, kCsTmemCols);
  if (threadIdx.x == 0 && *sAbort) atomicCAS(&g_cs_status, 0, (int)ATTN_ERR_TIMEOUT);
}

namespace {
std::mutex g_cs_mu;
bool g_cs_attr[64] = {};
}  // namespace

cudaError_t launch_chunk_scan(const ChunkScanParams& p, cudaStream_t stream) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lk(g_cs_mu);
    if (!g_cs_attr[dev]) {
      err = cudaFuncSetAttribute(chunk_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 kCsSmemBytes);
      if (err != cudaSuccess) return err;
      g_cs_attr[dev] = true;
    }
  }
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
