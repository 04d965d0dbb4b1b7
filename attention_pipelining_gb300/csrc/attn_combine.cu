// attn_combine.cu -- merge of split-KV partial results.
//
// With the KV axis split into S ranges, range s gives, per query row, a
// partial output O_s normalised within the range and its log-sum-exp L_s
// (-inf when the row sees no key in the range).  The full result is
//   L = ln sum_s exp(L_s),   O = sum_s exp(L_s - L) O_s,
// the reduction step of the split ("FlashDecoding") form of the forward, one
// of the microbenchmark operators of "PipeThreader: Software-Defined
// Pipelining for Efficient DNN Execution", section A4 (experimental setup;
// decoding with batch x sequence = 1 x 1 and 32 x 1).  HBM-bound: one warp per
// row streams S x D partial values.
#include <cmath>
#include <cstdint>

#include "attn_internal.h"
#include "ptx.cuh"

namespace attnpipe {
namespace {

constexpr int kRowsPerBlock = 8;  // one warp per row

template <int D>
__global__ void __launch_bounds__(kRowsPerBlock * 32)
    splitkv_combine_kernel(const float* __restrict__ o_part, const float* __restrict__ lse_part,
                           uint16_t* __restrict__ o, float* __restrict__ lse, long long rows,
                           int splits) {
  const long long row = (long long)blockIdx.x * kRowsPerBlock + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (row >= rows) return;
  float m = -INFINITY;
  for (int s = 0; s < splits; ++s) m = fmaxf(m, lse_part[(long long)s * rows + row]);
  float sum = 0.f;
  if (m != -INFINITY) {
    for (int s = 0; s < splits; ++s) {
      const float x = lse_part[(long long)s * rows + row];
      if (x != -INFINITY) sum += expf(x - m);
    }
  }
  const float lse_row = (m == -INFINITY) ? -INFINITY : m + logf(sum);
  constexpr int kPer = D / 32;  // elements per lane: 4 (D = 128) or 2 (D = 64)
  float acc[kPer];
#pragma unroll
  for (int i = 0; i < kPer; ++i) acc[i] = 0.f;
  if (m != -INFINITY) {
    for (int s = 0; s < splits; ++s) {
      const float x = lse_part[(long long)s * rows + row];
      if (x == -INFINITY) continue;
      const float w = expf(x - lse_row);
      const float* src = o_part + ((long long)s * rows + row) * D + lane * kPer;
      if constexpr (kPer == 4) {
        const float4 v = *reinterpret_cast<const float4*>(src);
        acc[0] += w * v.x;
        acc[1] += w * v.y;
        acc[2] += w * v.z;
        acc[3] += w * v.w;
      } else {
        const float2 v = *reinterpret_cast<const float2*>(src);
        acc[0] += w * v.x;
        acc[1] += w * v.y;
      }
    }
  }
  uint32_t* dst = reinterpret_cast<uint32_t*>(o + row * D + lane * kPer);
#pragma unroll
  for (int i = 0; i < kPer; i += 2) dst[i / 2] = pack_bf16x2(acc[i], acc[i + 1]);
  if (lane == 0) lse[row] = lse_row;
}

}  // namespace

cudaError_t launch_splitkv_combine(const float* o_part, const float* lse_part, void* o, float* lse,
                                   long long rows, int D, int splits, cudaStream_t stream) {
  const long long blocks = (rows + kRowsPerBlock - 1) / kRowsPerBlock;
  if (blocks <= 0 || blocks > 0x7fffffffLL) return cudaErrorInvalidValue;
  if (D == 128)
    splitkv_combine_kernel<128><<<(unsigned)blocks, kRowsPerBlock * 32, 0, stream>>>(
        o_part, lse_part, static_cast<uint16_t*>(o), lse, rows, splits);
  else if (D == 64)
    splitkv_combine_kernel<64><<<(unsigned)blocks, kRowsPerBlock * 32, 0, stream>>>(
        o_part, lse_part, static_cast<uint16_t*>(o), lse, rows, splits);
  else
    return cudaErrorInvalidValue;
  return cudaGetLastError();
}

}  // namespace attnpipe
