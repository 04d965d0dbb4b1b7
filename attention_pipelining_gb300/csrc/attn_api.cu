// attn_api.cu -- the C ABI: argument checks, tensor-map encoding, launch.
//
// Host-side half of the boundary declared in include/attn.h.  Every check
// runs before anything touches the device; nothing here allocates memory.
#include <cmath>
#include <cstdint>
#include <cstring>
#include <mutex>

#include "attn_internal.h"

namespace attnpipe {
namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*,
                                   const cuuint64_t*, const cuuint64_t*, const cuuint32_t*,
                                   const cuuint32_t*, CUtensorMapInterleave, CUtensorMapSwizzle,
                                   CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn get_encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000,
                                         cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

// Per-device cache of "is this an sm_103 part": 0 unknown, 1 yes, 2 no.
int g_arch_ok[64] = {};
std::mutex g_arch_mu;

attn_status_t check_device() {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return ATTN_ERR_CUDA;
  if (dev < 0 || dev >= 64) return ATTN_ERR_UNSUPPORTED;
  {
    std::lock_guard<std::mutex> lk(g_arch_mu);
    if (g_arch_ok[dev] == 0) {
      int major = 0, minor = 0;
      if (cudaDeviceGetAttribute(&major, cudaDevAttrComputeCapabilityMajor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&minor, cudaDevAttrComputeCapabilityMinor, dev) != cudaSuccess)
        return ATTN_ERR_CUDA;
      g_arch_ok[dev] = (major == 10 && minor == 3) ? 1 : 2;
    }
    if (g_arch_ok[dev] != 1) return ATTN_ERR_UNSUPPORTED;
  }
  return ATTN_OK;
}

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }

}  // namespace

bool encode_bf16_map_3d(CUtensorMap* map, const void* base, uint64_t D, uint64_t rows,
                        uint64_t outer, uint32_t box_rows) {
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return false;
  cuuint64_t dims[3] = {D, rows, outer};
  cuuint64_t strides[2] = {D * 2, rows * D * 2};  // bytes, for dims 1 and 2
  cuuint32_t box[3] = {64, box_rows, 1};
  cuuint32_t estr[3] = {1, 1, 1};
  CUresult r = fn(map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(base), dims, strides,
                  box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
                  CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  return r == CUDA_SUCCESS;
}

// Pure argument checks (no CUDA calls), shared by both entry points.
static attn_status_t validate(const void* q, const void* k, const void* v, const void* o,
                              const void* lse, int B, int H_q, int H_kv, int S_q, int S_kv, int D,
                              int causal, float scale) {
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || H_q <= 0 || H_kv <= 0 || S_q <= 0 || S_kv <= 0 || D <= 0)
    return ATTN_ERR_INVALID_ARG;
  if (H_q % H_kv != 0) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale) || scale < 0.f) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  // grid is (ceil(S_q / 256), H_q, B); y and z are limited to 65535
  if (B > 65535 || H_q > 65535) return ATTN_ERR_UNSUPPORTED;
  // tensor-map extents must stay below 2^32 per dimension
  if ((int64_t)B * H_q >= (1ll << 31) || (int64_t)B * H_kv >= (1ll << 31))
    return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(o) || !aligned16(lse))
    return ATTN_ERR_MISALIGNED;
  return ATTN_OK;
}

}  // namespace attnpipe

using namespace attnpipe;

namespace attnpipe {

static attn_status_t fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int H_q, int H_kv, int S_q, int S_kv, int D, int causal,
                              float scale, unsigned long long* trace, int trace_ctas,
                              int trace_blocks, int fault_drop_block,
                              unsigned long long timeout_ns, attn_stream_t stream) {
  attn_status_t st = validate(q, k, v, o, lse, B, H_q, H_kv, S_q, S_kv, D, causal, scale);
  if (st != ATTN_OK) return st;
  st = check_device();
  if (st != ATTN_OK) return st;
  AttnParams p;
  std::memset(&p, 0, sizeof(p));
  if (!encode_bf16_map_3d(&p.tm_q, q, D, S_q, (uint64_t)B * H_q, 128) ||
      !encode_bf16_map_3d(&p.tm_k, k, D, S_kv, (uint64_t)B * H_kv, 128) ||
      !encode_bf16_map_3d(&p.tm_v, v, D, S_kv, (uint64_t)B * H_kv, 128) ||
      !encode_bf16_map_3d(&p.tm_o, o, D, S_q, (uint64_t)B * H_q, 32))
    return ATTN_ERR_CUDA;
  p.lse = lse;
  p.B = B;
  p.H_q = H_q;
  p.H_kv = H_kv;
  p.S_q = S_q;
  p.S_kv = S_kv;
  p.causal = causal;
  p.scale_log2 = (float)((double)scale * 1.4426950408889634);
  p.timeout_ns = timeout_ns;
  p.trace = trace;
  p.trace_ctas = trace_ctas;
  p.trace_blocks = trace_blocks;
  p.fault_drop_block = fault_drop_block;
  const int n_m_tiles = (S_q + 255) / 256;
  if (launch_attn_fwd(p, D, n_m_tiles, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

}  // namespace attnpipe

extern "C" {

attn_status_t attn_fwd(const void* q, const void* k, const void* v, void* o, float* lse, int B,
                       int H_q, int H_kv, int S_q, int S_kv, int D, int causal, float scale,
                       attn_stream_t stream) {
  return fwd_impl(q, k, v, o, lse, B, H_q, H_kv, S_q, S_kv, D, causal, scale, nullptr, 0, 0, -1,
                  kDefaultTimeoutNs, stream);
}

attn_status_t attn_fwd_trace(const void* q, const void* k, const void* v, void* o, float* lse,
                             int B, int H_q, int H_kv, int S_q, int S_kv, int D, int causal,
                             float scale, unsigned long long* trace, int trace_ctas,
                             int trace_blocks, attn_stream_t stream) {
  if (!trace || trace_ctas <= 0 || trace_blocks <= 0) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(trace) & 7u) != 0) return ATTN_ERR_MISALIGNED;
  return fwd_impl(q, k, v, o, lse, B, H_q, H_kv, S_q, S_kv, D, causal, scale, trace, trace_ctas,
                  trace_blocks, -1, kDefaultTimeoutNs, stream);
}

attn_status_t attn_fwd_timeout_test(const void* q, const void* k, const void* v, void* o,
                                    float* lse, int B, int H_q, int H_kv, int S_q, int S_kv,
                                    int D, int causal, float scale, int drop_block,
                                    unsigned long long wait_budget_ns, attn_stream_t stream) {
  if (drop_block < 0) return ATTN_ERR_INVALID_ARG;
  if (wait_budget_ns < 1000000ull || wait_budget_ns > kDefaultTimeoutNs)
    return ATTN_ERR_INVALID_ARG;
  return fwd_impl(q, k, v, o, lse, B, H_q, H_kv, S_q, S_kv, D, causal, scale, nullptr, 0, 0,
                  drop_block, wait_budget_ns, stream);
}

attn_status_t attn_fwd_host(const void* q_host, const void* k_host, const void* v_host,
                            void* o_host, float* lse_host, void* q_dev, void* k_dev, void* v_dev,
                            void* o_dev, float* lse_dev, int B, int H_q, int H_kv, int S_q,
                            int S_kv, int D, int causal, float scale, attn_stream_t stream) {
  if (!q_host || !k_host || !v_host || !o_host || !lse_host) return ATTN_ERR_INVALID_ARG;
  attn_status_t st =
      validate(q_dev, k_dev, v_dev, o_dev, lse_dev, B, H_q, H_kv, S_q, S_kv, D, causal, scale);
  if (st != ATTN_OK) return st;
  st = check_device();
  if (st != ATTN_OK) return st;
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  const size_t q_bytes = (size_t)B * H_q * S_q * D * 2;
  const size_t kv_bytes = (size_t)B * H_kv * S_kv * D * 2;
  const size_t lse_bytes = (size_t)B * H_q * S_q * sizeof(float);
  if (cudaMemcpyAsync(q_dev, q_host, q_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(k_dev, k_host, kv_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess ||
      cudaMemcpyAsync(v_dev, v_host, kv_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
    return ATTN_ERR_CUDA;
  st = attn_fwd(q_dev, k_dev, v_dev, o_dev, lse_dev, B, H_q, H_kv, S_q, S_kv, D, causal, scale,
                stream);
  if (st != ATTN_OK) return st;
  if (cudaMemcpyAsync(o_host, o_dev, q_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
      cudaMemcpyAsync(lse_host, lse_dev, lse_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

const char* attn_status_string(attn_status_t status) {
  switch (status) {
    case ATTN_OK: return "ok";
    case ATTN_ERR_INVALID_ARG: return "invalid argument";
    case ATTN_ERR_UNSUPPORTED: return "unsupported (head dim, size or device architecture)";
    case ATTN_ERR_MISALIGNED: return "pointer not 16-byte aligned";
    case ATTN_ERR_CUDA: return "CUDA runtime or driver call failed";
    case ATTN_ERR_TIMEOUT: return "a wait inside the kernel ran out of time";
  }
  return "unknown status";
}

attn_status_t attn_device_status(int* status_out, int reset) {
  if (!status_out) return ATTN_ERR_INVALID_ARG;
  attn_status_t st = check_device();
  if (st != ATTN_OK) return st;
  int main_status = 0, selftest_status = 0;
  if (read_device_status(&main_status, reset != 0) != cudaSuccess ||
      read_selftest_status(&selftest_status, reset != 0) != cudaSuccess)
    return ATTN_ERR_CUDA;
  *status_out = main_status != 0 ? main_status : selftest_status;
  return ATTN_OK;
}

int attn_version(void) { return 100; }

attn_status_t attn_selftest_qk(const void* q, const void* k, float* s, int D, attn_stream_t stream) {
  if (!q || !k || !s) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(q) || !aligned16(k) || !aligned16(s)) return ATTN_ERR_MISALIGNED;
  attn_status_t st = check_device();
  if (st != ATTN_OK) return st;
  CUtensorMap tq, tk;
  if (!encode_bf16_map_3d(&tq, q, D, 128, 1, 128) || !encode_bf16_map_3d(&tk, k, D, 128, 1, 128))
    return ATTN_ERR_CUDA;
  if (launch_selftest_qk(tq, tk, s, D, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

attn_status_t attn_selftest_pv(const void* p, const void* v, float* o, int D, attn_stream_t stream) {
  if (!p || !v || !o) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(p) || !aligned16(v) || !aligned16(o)) return ATTN_ERR_MISALIGNED;
  attn_status_t st = check_device();
  if (st != ATTN_OK) return st;
  CUtensorMap tv;
  if (!encode_bf16_map_3d(&tv, v, D, 128, 1, 128)) return ATTN_ERR_CUDA;
  if (launch_selftest_pv(static_cast<const uint16_t*>(p), tv, o, D,
                         static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

}  // extern "C"
