// attn_noalloc.cu -- split-KV forward for callers that cannot allocate device
// memory.
//
// attn_fwd_splitkv needs a scratch buffer for the per-split partial results.
// Some callers have no way to provide one: an engine that hands all device
// memory to its own pool at start-up and forbids further allocations, a
// plugin loaded into a host program that exposes no allocator, or a
// latency-critical path where an allocation call could block on the device.
// This entry point serves them from a fixed scratch array that is part of the
// library image itself, so a call allocates nothing.
//
// The array lives in this file as a file-scope __device__ variable.  In host
// code its name only stands for a host-side shadow, not a device address, so
// the device address is fetched once per device with cudaGetSymbolAddress
// (with that device current) and cached.
#include <cstddef>
#include <cstdint>
#include <mutex>

#include "attn_internal.h"

namespace attnpipe {
namespace {

// 16 MiB: every GPU that loads the library holds it until the process exits.
constexpr size_t kNoAllocScratchBytes = size_t(16) << 20;
static __device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_scratch_mu;
void* g_scratch_dev_ptr[64] = {};  // device address of g_noalloc_scratch, per device

// Device address of the scratch array on the current device (nullptr on error).
void* scratch_on_current_device(attn_status_t* st) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) {
    *st = ATTN_ERR_CUDA;
    return nullptr;
  }
  if (dev < 0 || dev >= 64) {
    *st = ATTN_ERR_UNSUPPORTED;
    return nullptr;
  }
  std::lock_guard<std::mutex> lk(g_scratch_mu);
  if (g_scratch_dev_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr) {
      *st = ATTN_ERR_CUDA;
      return nullptr;
    }
    g_scratch_dev_ptr[dev] = ptr;
  }
  *st = ATTN_OK;
  return g_scratch_dev_ptr[dev];
}

}  // namespace
}  // namespace attnpipe

using namespace attnpipe;

extern "C" {

size_t attn_splitkv_noalloc_capacity(void) { return kNoAllocScratchBytes; }

attn_status_t attn_fwd_splitkv_noalloc(const void* q, const void* k, const void* v, void* o,
                                       float* lse, int B, int H_q, int H_kv, int S_q, int S_kv,
                                       int D, int causal, float scale, int num_splits,
                                       attn_stream_t stream) {
  attn_status_t st = validate(q, k, v, o, lse, B, H_q, H_kv, S_q, S_kv, D, causal, scale);
  if (st != ATTN_OK) return st;
  if (num_splits > kMaxSplits) return ATTN_ERR_UNSUPPORTED;
  const int splits =
      num_splits > 0 ? num_splits : default_splits(B, H_q, H_kv, S_q, S_kv, causal);
  // partial results that would not fit the built-in scratch are refused
  if (splitkv_bytes(B, H_q, S_q, D, splits) > kNoAllocScratchBytes) return ATTN_ERR_UNSUPPORTED;
  void* scratch = scratch_on_current_device(&st);
  if (st != ATTN_OK) return st;
  // Every partial the merge reads is written by the forward of the same call,
  // so nothing left in the array by an earlier call needs clearing.
  return splitkv_impl(q, k, v, o, lse, scratch, kNoAllocScratchBytes, B, H_q, H_kv, S_q, S_kv,
                      D, causal, scale, splits, stream);
}

}  // extern "C"
