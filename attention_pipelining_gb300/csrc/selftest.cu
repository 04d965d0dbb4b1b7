// selftest.cu -- one-CTA kernels that run the fused kernel's building blocks
// (TMA tile loads, the QK^T and PV tensor-core steps, tensor-memory loads and
// stores) on a single tile so each encoding can be checked against a CPU
// product.  They use the very functions the fused kernel uses
// (attn_tiles.cuh, ptx.cuh).
#include <cstdint>

#include "attn_internal.h"
#include "attn_tiles.cuh"
#include "ptx.cuh"

namespace attnpipe {

namespace {

// Status word of the self-test kernels (ATTN_ERR_TIMEOUT after a timed-out wait).
__device__ int g_selftest_status = 0;

constexpr uint64_t kSelftestBudgetNs = 1000000000ull;  // 1 s per wait

struct SelftestSmem {
  uint64_t full;
  uint64_t mma_done;
  uint32_t tmem_base;
  int abort_flag;
};

// 128 threads: thread i owns row i (TMEM lane i).
template <int D>
__global__ void __launch_bounds__(128, 1)
    selftest_qk_kernel(const __grid_constant__ CUtensorMap tq, const __grid_constant__ CUtensorMap tk,
                       float* s_out) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align_smem_1024(smem_raw);
  uint8_t* sQ = base;
  uint8_t* sK = base + TileShape<D>::kBytes;
  SelftestSmem* ctl = reinterpret_cast<SelftestSmem*>(base + 2 * TileShape<D>::kBytes);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(&ctl->full, 1);
    mbar_init(&ctl->mma_done, 1);
    ctl->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&ctl->tmem_base, 128);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = ctl->tmem_base;
  volatile int* abort_flag = &ctl->abort_flag;

  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&ctl->full, 2 * TileShape<D>::kBytes);
    tma_load_tile<D>(sQ, &tq, &ctl->full, 0, 0, l2_policy_evict_first());
    tma_load_tile<D>(sK, &tk, &ctl->full, 0, 0, l2_policy_evict_first());
    if (mbar_wait(&ctl->full, 0, abort_flag, kSelftestBudgetNs)) {
      tc_fence_after_sync();
      issue_qk_gemm<D>(tmem, kmajor_tile_desc(smem_u32(sQ)), kmajor_tile_desc(smem_u32(sK)));
    }
    tc_commit(&ctl->mma_done);
  }
  __syncwarp();
  const bool ok = __all_sync(0xffffffffu, mbar_wait(&ctl->mma_done, 0, abort_flag, kSelftestBudgetNs));
  tc_fence_after_sync();
  if (ok && !*abort_flag) {
    const int row = threadIdx.x;
    const uint32_t taddr = tmem + ((uint32_t)(warp * 32) << 16);
#pragma unroll
    for (int c = 0; c < 128; c += 32) {
      uint32_t r[32];
      tmem_ld_x32(taddr + c, r);
      tmem_ld_wait();
      reg_after_wait(r);
#pragma unroll
      for (int i = 0; i < 32; ++i) s_out[row * 128 + c + i] = __uint_as_float(r[i]);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem, 128);
  if (threadIdx.x == 0 && *abort_flag) atomicCAS(&g_selftest_status, 0, (int)ATTN_ERR_TIMEOUT);
}

// 128 threads: thread i writes row i of P (bf16) into TMEM lane i, columns
// [0, 64), as packed pairs; O goes to columns [128, 128 + D).
template <int D>
__global__ void __launch_bounds__(128, 1)
    selftest_pv_kernel(const uint16_t* __restrict__ p_in, const __grid_constant__ CUtensorMap tv,
                       float* o_out) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* base = align_smem_1024(smem_raw);
  uint8_t* sV = base;
  SelftestSmem* ctl = reinterpret_cast<SelftestSmem*>(base + TileShape<D>::kBytes);
  const int warp = threadIdx.x >> 5;
  if (threadIdx.x == 0) {
    mbar_init(&ctl->full, 1);
    mbar_init(&ctl->mma_done, 1);
    ctl->abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0) {
    tmem_alloc(&ctl->tmem_base, 256);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  const uint32_t tmem = ctl->tmem_base;
  volatile int* abort_flag = &ctl->abort_flag;
  const int row = threadIdx.x;
  const uint32_t lane_addr = tmem + ((uint32_t)(warp * 32) << 16);

  if (threadIdx.x == 0) {
    mbar_arrive_expect_tx(&ctl->full, TileShape<D>::kBytes);
    tma_load_tile<D>(sV, &tv, &ctl->full, 0, 0, l2_policy_evict_first());
  }
  // P row -> TMEM columns [0, 64): column c holds keys 2c (low half) and 2c+1.
  const uint32_t* prow = reinterpret_cast<const uint32_t*>(p_in + row * 128);
#pragma unroll
  for (int c = 0; c < 64; c += 32) {
    uint32_t r[32];
#pragma unroll
    for (int i = 0; i < 32; ++i) r[i] = prow[c + i];
    tmem_st_x32(lane_addr + c, r);
  }
  tmem_st_wait();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();

  if (threadIdx.x == 0) {
    if (mbar_wait(&ctl->full, 0, abort_flag, kSelftestBudgetNs)) {
      tc_fence_after_sync();
      issue_pv_gemm<D>(tmem + 128, tmem, mnmajor_tile_desc<D>(smem_u32(sV)), false);
    }
    tc_commit(&ctl->mma_done);
  }
  __syncwarp();
  const bool ok = __all_sync(0xffffffffu, mbar_wait(&ctl->mma_done, 0, abort_flag, kSelftestBudgetNs));
  tc_fence_after_sync();
  if (ok && !*abort_flag) {
#pragma unroll
    for (int c = 0; c < D; c += 32) {
      uint32_t r[32];
      tmem_ld_x32(lane_addr + 128 + c, r);
      tmem_ld_wait();
      reg_after_wait(r);
#pragma unroll
      for (int i = 0; i < 32; ++i) o_out[row * D + c + i] = __uint_as_float(r[i]);
    }
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  if (warp == 0) tmem_dealloc(tmem, 256);
  if (threadIdx.x == 0 && *abort_flag) atomicCAS(&g_selftest_status, 0, (int)ATTN_ERR_TIMEOUT);
}

template <int D>
cudaError_t qk_d(const CUtensorMap& tq, const CUtensorMap& tk, float* s, cudaStream_t stream) {
  const int smem = 2 * TileShape<D>::kBytes + (int)sizeof(SelftestSmem) + 1024;
  cudaError_t err = cudaFuncSetAttribute(selftest_qk_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  selftest_qk_kernel<D><<<1, 128, smem, stream>>>(tq, tk, s);
  return cudaGetLastError();
}

template <int D>
cudaError_t pv_d(const uint16_t* p, const CUtensorMap& tv, float* o, cudaStream_t stream) {
  const int smem = TileShape<D>::kBytes + (int)sizeof(SelftestSmem) + 1024;
  cudaError_t err = cudaFuncSetAttribute(selftest_pv_kernel<D>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize, smem);
  if (err != cudaSuccess) return err;
  selftest_pv_kernel<D><<<1, 128, smem, stream>>>(p, tv, o);
  return cudaGetLastError();
}

}  // namespace

cudaError_t read_selftest_status(int* status, bool reset) {
  cudaError_t err = cudaMemcpyFromSymbol(status, g_selftest_status, sizeof(int));
  if (err != cudaSuccess) return err;
  if (reset) {
    const int zero = 0;
    err = cudaMemcpyToSymbol(g_selftest_status, &zero, sizeof(int));
  }
  return err;
}

cudaError_t launch_selftest_qk(const CUtensorMap& tq, const CUtensorMap& tk, float* s, int D,
                               cudaStream_t stream) {
  if (D == 128) return qk_d<128>(tq, tk, s, stream);
  if (D == 64) return qk_d<64>(tq, tk, s, stream);
  return cudaErrorInvalidValue;
}

cudaError_t launch_selftest_pv(const uint16_t* p, const CUtensorMap& tv, float* o, int D,
                               cudaStream_t stream) {
  if (D == 128) return pv_d<128>(p, tv, o, stream);
  if (D == 64) return pv_d<64>(p, tv, o, stream);
  return cudaErrorInvalidValue;
}

}  // namespace attnpipe
