// attn_tiles.cuh -- tile-level steps shared by the fused kernel and the
// self-test kernels: TMA loads of one 128-row bf16 tile and the two
// tensor-core GEMMs of the attention forward ("PipeThreader: Software-
// Defined Pipelining for Efficient DNN Execution", section A2, Fig. 7:
// load_k / load_v, mma_qk, mma_pv).
//
// Shared-memory tile layout: a [128 rows x D] bf16 tile is stored as D/64
// slabs of [128 rows x 64 columns]; each slab is 128 rows of 128 bytes in
// the 128-byte swizzle (16-byte chunk c of row r sits at chunk c ^ (r % 8)),
// exactly what one TMA load with 128-byte swizzle and a {64, 128} box writes.
// Slabs are 16 KB apart and 1024-byte aligned.
#pragma once

#include <cstdint>

#include "ptx.cuh"

namespace attnpipe {

constexpr int kTileRows = 128;
constexpr int kSlabBytes = kTileRows * 128;  // one [128 x 64] bf16 slab

template <int D>
struct TileShape {
  static_assert(D == 64 || D == 128, "head dim");
  static constexpr int kSlabs = D / 64;
  static constexpr int kBytes = kTileRows * D * 2;
};

// Loads rows [row0, row0 + 128) of slice z of a [*, rows, D] tensor map into
// `dst` (a tile as above); completion is counted on `bar`.  Rows outside the
// tensor are filled with zeros (and still counted).
template <int D>
__device__ __forceinline__ void tma_load_tile(uint8_t* dst, const CUtensorMap* map, uint64_t* bar,
                                              int row0, int z, uint64_t hint) {
#pragma unroll
  for (int s = 0; s < TileShape<D>::kSlabs; ++s)
    tma_load_3d(dst + s * kSlabBytes, map, bar, s * 64, row0, z, hint);
}

// Shared-memory descriptor of the start of a tile, for either operand use.
// The GEMM helpers below add constant offsets to its start-address field
// (bits 0-13, address >> 4), which never carries: shared addresses stay
// below 2^18.
__device__ __forceinline__ uint64_t kmajor_tile_desc(uint32_t smem_addr) {
  return make_smem_desc_sw128(smem_addr, 16, 1024);
}

template <int D>
__device__ __forceinline__ uint64_t mnmajor_tile_desc(uint32_t smem_addr) {
  // With D = 64 there is a single slab along N and the leading offset is
  // never used; it is set to the in-slab group stride so no field can point
  // past the tile.
  return make_smem_desc_sw128(smem_addr, (D == 64) ? 1024 : kSlabBytes, 1024);
}

// S[tmem, 128 x 128 fp32] = Q K^T (or -Q K^T) for one 128-row Q tile and one
// 128-row K tile, given their K-major tile descriptors.  Both operands are
// K-major (the head dimension is contiguous): per K step of 16 elements the
// start advances
// 32 bytes inside a swizzle row, and moves to the next slab every 64
// elements.  Stride between 8-row groups (SBO) is 1024 bytes; the leading
// offset is unused for swizzled K-major operands.  Issued by one thread.
template <int D>
__device__ __forceinline__ void issue_qk_gemm(uint32_t s_tmem, uint64_t q_desc, uint64_t k_desc,
                                              bool negate = false) {
  // with `negate`, the instruction descriptor's negate-A bit gives -Q K^T
  const uint32_t idesc =
      make_idesc_bf16_f32(128, 128, false, false) | (negate ? kIdescNegateA : 0u);
#pragma unroll
  for (int kk = 0; kk < D / 16; ++kk) {
    const uint64_t off = (uint64_t)(((kk >> 2) * kSlabBytes + (kk & 3) * 32) >> 4);
    mma_ss(s_tmem, q_desc + off, k_desc + off, idesc, kk > 0 ? 1u : 0u);
  }
}

// O[tmem, 128 x D fp32] (+)= P V with P [128 x 128] bf16 in tensor memory
// (row i in lane i, keys 2c and 2c+1 packed in column c) and V a
// [128 keys x D] tile used MN-major (D contiguous), given its MN-major tile
// descriptor.  Per K step of 16 keys the start advances 16 rows = 2048
// bytes; the 8-row groups along K are 1024 bytes apart (SBO); the 64-column
// slabs along N are one slab apart (LBO).  `accumulate` = false overwrites
// O.  Issued by one thread.
//
// With N > D (a multiple of 16 up to D + 64), B is [V | W]: the columns
// past D come from the 64-column atom at the descriptor's leading offset
// from V (the attention kernel's constant ones, which make those columns of
// O the row sums of P).
template <int D, int N = D>
__device__ __forceinline__ void issue_pv_gemm(uint32_t o_tmem, uint32_t p_tmem, uint64_t v_desc,
                                              bool accumulate) {
  static_assert(N % 16 == 0 && N >= D && N <= D + 64, "PV GEMM width");
  constexpr uint32_t idesc = make_idesc_bf16_f32(128, N, false, true);
#pragma unroll
  for (int kk = 0; kk < kTileRows / 16; ++kk) {
    mma_ts(o_tmem, p_tmem + kk * 8, v_desc + (uint64_t)((kk * 2048) >> 4), idesc,
           (accumulate || kk > 0) ? 1u : 0u);
  }
}

}  // namespace attnpipe
