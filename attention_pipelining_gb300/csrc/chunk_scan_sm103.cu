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
// One CTA = (batch, chunk, head, 128-row tile of the chunk), 384 threads:
//   warps 0-7  two elementwise warpgroups, thread = row of the tile; for each
//              64-key slice warpgroup w scales keys 32w .. 32w + 31 of its
//              row (cb read from global, the decay by exp2) into bf16 and
//              writes them into the slice's 128-byte-swizzled K-major A tile;
//   warp 8     tensor-core issuer: per slice, 4 tcgen05.mma (M = 128, N = 64,
//              K = 16) of A (shared memory) with x (shared memory, MN-major)
//              into a 128 x 64 fp32 accumulator in tensor memory;
//   warp 9     TMA producer: the chunk's dA_cs and dt vectors (1-D bulk
//              copies) and the x slices (4-D tensor map over [B, L, H, P]).
// Slices of the A tile are handed over one at a time (an mbarrier per
// slice), so the tensor core works on slice s while slice s + 1 is scaled.
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

constexpr int kCsThreads = 384;
constexpr int kCsRows = 128;     // rows of a CTA's tile
constexpr int kCsSlice = 64;     // keys per slice of the reduction axis
constexpr int kCsP = 64;         // head width
constexpr int kCsMaxQ = 256;     // longest chunk
constexpr int kCsMaxSlices = kCsMaxQ / kCsSlice;
constexpr uint32_t kCsAll = 0xffffffffu;

// shared memory, offsets from a 1024-byte aligned base
constexpr int kCsOffA = 0;                                   // [slices][128 x 64] bf16 K-major
constexpr int kCsSliceBytesA = kCsRows * kCsSlice * 2;        // 16 KB
constexpr int kCsOffX = kCsOffA + kCsMaxSlices * kCsSliceBytesA;  // [slices][64 x 64] bf16
constexpr int kCsSliceBytesX = kCsSlice * kCsP * 2;           // 8 KB
constexpr int kCsOffVec = kCsOffX + kCsMaxSlices * kCsSliceBytesX;  // dA_cs [Q], dt [Q] fp32
constexpr int kCsOffBar = kCsOffVec + 2 * kCsMaxQ * 4;
// vec_full, x_full[S], a_ready[S], acc_done, drain
constexpr int kCsNumBars = 3 + 2 * kCsMaxSlices;
constexpr int kCsOffMisc = kCsOffBar + kCsNumBars * 8;
constexpr int kCsSmemBytes = kCsOffMisc + 16 + 1024;
constexpr uint32_t kCsTmemCols = 64;

__device__ __forceinline__ bool cs_warp_wait(uint64_t* bar, uint32_t parity,
                                             volatile int* abort_flag, uint64_t budget) {
  const bool ok = mbar_wait(bar, parity, abort_flag, budget);
  return __all_sync(kCsAll, ok);
}

__device__ __forceinline__ void cs_drain_wait(uint64_t* bar, uint32_t parity, uint64_t budget) {
  volatile int never = 0;
  mbar_wait(bar, parity, &never, budget);
}

__device__ __forceinline__ float4 ldg_f4(const float* p) {
  return __ldg(reinterpret_cast<const float4*>(p));
}

}  // namespace

__global__ void __launch_bounds__(kCsThreads, 2) chunk_scan_kernel(const __grid_constant__ ChunkScanParams p) {
  extern __shared__ uint8_t smem_raw_cs[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw_cs) + 1023) &
                                             ~static_cast<uintptr_t>(1023));
  uint8_t* sA = smem + kCsOffA;
  uint8_t* sX = smem + kCsOffX;
  float* sDA = reinterpret_cast<float*>(smem + kCsOffVec);
  float* sDT = sDA + kCsMaxQ;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + kCsOffBar);
  uint64_t* vec_full = bars;
  uint64_t* x_full = bars + 1;
  uint64_t* a_ready = x_full + kCsMaxSlices;
  uint64_t* acc_done = a_ready + kCsMaxSlices;
  uint64_t* drain = acc_done + 1;
  uint32_t* sTmemBase = reinterpret_cast<uint32_t*>(smem + kCsOffMisc);
  volatile int* sAbort = reinterpret_cast<volatile int*>(smem + kCsOffMisc + 4);
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t budget = p.timeout_ns;

  // CTA -> (b, c, h, tile): the tiles and heads of one chunk are adjacent, so
  // the heads of a group read their shared cb from L2
  const int tiles = p.Q / kCsRows;
  int idx = blockIdx.x;
  const int mt = idx % tiles;
  idx /= tiles;
  const int h = idx % p.H;
  idx /= p.H;
  const int c = idx % p.nchunks;
  const int b = idx / p.nchunks;
  const int g = h / (p.H / p.G);
  const int m0 = mt * kCsRows;                 // first row of the tile within the chunk
  const int n_slices = (m0 + kCsRows) / kCsSlice;  // keys 0 .. m0 + 127 are visible to some row

  if (threadIdx.x == 0) {
    mbar_init(vec_full, 1);
    for (int s = 0; s < kCsMaxSlices; ++s) {
      mbar_init(&x_full[s], 1);
      mbar_init(&a_ready[s], 2 * 128);
    }
    mbar_init(acc_done, 1);
    mbar_init(drain, 1);
    *sAbort = 0;
    fence_mbar_init();
  }
  if (warp == 8) {
    tmem_alloc(sTmemBase, kCsTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = *sTmemBase;
  const size_t vec_off = (((size_t)b * p.H + h) * p.nchunks + c) * p.Q;

  if (warp < 8) {
    // ---------------------------------------------------------- elementwise
    const int w = warp >> 2;
    const int r = (warp & 3) * 32 + lane;      // row of the tile
    const int m = m0 + r;                      // row of the chunk
    const uint32_t lane_base = (uint32_t)((warp & 3) * 32) << 16;
    const float* cb_row =
        p.cb + ((((size_t)b * p.nchunks + c) * p.G + g) * p.Q + m) * (size_t)p.Q;
    bool ok = cs_warp_wait(vec_full, 0, sAbort, budget);
    const float l2e = 1.4426950408889634f;
    const float da_m = ok ? sDA[m] * l2e : 0.f;
    // exponent (dA_cs[m] - dA_cs[k]) * log2(e) as da_m - dA_cs[k] * log2(e),
    // two keys per instruction
    const uint64_t dam2 = f2_pack(da_m, da_m);
    const uint64_t nl2e2 = f2_pack(-l2e, -l2e);
    for (int s = 0; s < n_slices && ok; ++s) {
      const int k0 = s * kCsSlice + 32 * w;    // first key of this thread's 32
      const bool diag = (k0 + 31 > m0);        // the slice may hold keys after some row
      uint32_t pk[16];
#pragma unroll
      for (int q = 0; q < 8; ++q) {
        const int k = k0 + 4 * q;
        const float4 cv = ldg_f4(cb_row + k);
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
      // row r of slice s: 16-byte chunks 4w .. 4w + 3, 128-byte swizzle
      uint8_t* row_base = sA + s * kCsSliceBytesA + r * 128;
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int chunk = (4 * w + q) ^ (r & 7);
        *reinterpret_cast<uint4*>(row_base + chunk * 16) =
            make_uint4(pk[4 * q], pk[4 * q + 1], pk[4 * q + 2], pk[4 * q + 3]);
      }
      fence_proxy_async_smem();   // generic-proxy writes before the tensor core reads them
      mbar_arrive(&a_ready[s]);
    }
    // ---------------------------------------------------------- epilogue
    if (ok && cs_warp_wait(acc_done, 0, sAbort, budget)) {
      tc_fence_after_sync();
      uint32_t v[32];
      tmem_ld_x32(tmem + lane_base + 32 * w, v);
      tmem_ld_wait();
      reg_after_wait(v);
      uint4* dst = reinterpret_cast<uint4*>(
          static_cast<uint16_t*>(p.out) +
          ((((size_t)b * p.L + (size_t)c * p.Q + m) * p.H + h) * kCsP) + 32 * w);
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        uint4 val;
        val.x = pack_bf16x2(__uint_as_float(v[8 * q + 0]), __uint_as_float(v[8 * q + 1]));
        val.y = pack_bf16x2(__uint_as_float(v[8 * q + 2]), __uint_as_float(v[8 * q + 3]));
        val.z = pack_bf16x2(__uint_as_float(v[8 * q + 4]), __uint_as_float(v[8 * q + 5]));
        val.w = pack_bf16x2(__uint_as_float(v[8 * q + 6]), __uint_as_float(v[8 * q + 7]));
        dst[q] = val;
      }
    }
  } else if (warp == 8) {
    // ---------------------------------------------------------- tensor-core issuer
    const bool leader = elect_one();
    constexpr uint32_t idesc = make_idesc_bf16_f32(128, kCsP, false, true);
    bool ok = true;
    for (int s = 0; s < n_slices && ok; ++s) {
      if (!cs_warp_wait(&a_ready[s], 0, sAbort, budget) ||
          !cs_warp_wait(&x_full[s], 0, sAbort, budget)) {
        ok = false;
        break;
      }
      tc_fence_after_sync();
      if (leader) {
        const uint64_t a_desc = make_smem_desc_sw128(smem_u32(sA + s * kCsSliceBytesA), 16, 1024);
        // the x slice is a single 64-wide slab: the leading offset is unused
        const uint64_t b_desc = make_smem_desc_sw128(smem_u32(sX + s * kCsSliceBytesX), 1024, 1024);
#pragma unroll
        for (int kk = 0; kk < kCsSlice / 16; ++kk) {
          mma_ss(tmem, a_desc + (uint64_t)((kk * 32) >> 4), b_desc + (uint64_t)((kk * 2048) >> 4),
                 idesc, (s > 0 || kk > 0) ? 1u : 0u);
        }
      }
    }
    if (ok && leader) tc_commit(acc_done);
    if (leader) {
      tc_commit(drain);
      cs_drain_wait(drain, 0, budget);
    }
    __syncwarp();
  } else if (warp == 9) {
    // ---------------------------------------------------------- TMA producer
    const bool leader = elect_one();
    if (leader) {
      mbar_arrive_expect_tx(vec_full, 2 * p.Q * 4);
      bulk_load(sDA, p.dA_cs + vec_off, p.Q * 4, vec_full);
      bulk_load(sDT, p.dt + vec_off, p.Q * 4, vec_full);
      const uint64_t pol = l2_policy_evict_first();
      for (int s = 0; s < n_slices; ++s) {
        mbar_arrive_expect_tx(&x_full[s], kCsSliceBytesX);
        tma_load_4d(sX + s * kCsSliceBytesX, &p.tm_x, &x_full[s], 0, h,
                    c * p.Q + s * kCsSlice, b, pol);
      }
      // all copies land before the CTA exits
      cs_drain_wait(vec_full, 0, budget);
      for (int s = 0; s < n_slices; ++s) cs_drain_wait(&x_full[s], 0, budget);
    }
    __syncwarp();
  }

  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 8) tmem_dealloc(tmem, kCsTmemCols);
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
  const long long ctas = (long long)p.B * p.nchunks * p.H * (p.Q / kCsRows);
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
