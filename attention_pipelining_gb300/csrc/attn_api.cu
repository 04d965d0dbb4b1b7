// attn_api.cu -- the C ABI: argument checks, tensor-map encoding, launch.
//
// Host-side half of the boundary declared in include/attn.h.  Every check
// runs before anything touches the device; nothing here allocates memory.
#include <cfloat>
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

// Pure argument checks (no CUDA calls), shared by the entry points.
attn_status_t validate(const void* q, const void* k, const void* v, const void* o,
                              const void* lse, int B, int H_q, int H_kv, int S_q, int S_kv, int D,
                              int causal, float scale) {
  if (!q || !k || !v || !o || !lse) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || H_q <= 0 || H_kv <= 0 || S_q <= 0 || S_kv <= 0 || D <= 0)
    return ATTN_ERR_INVALID_ARG;
  if (H_q % H_kv != 0) return ATTN_ERR_INVALID_ARG;
  if (causal != 0 && causal != 1) return ATTN_ERR_INVALID_ARG;
  if (!std::isfinite(scale)) return ATTN_ERR_INVALID_ARG;
  if (D != 64 && D != 128) return ATTN_ERR_UNSUPPORTED;
  // R = (H_q / H_kv) * S_q rows per K/V head must fit an int, and so must
  // the number of 256-row work tiles, ceil(R / 256) * B * H_kv
  if (B > 65535 || H_kv > 65535) return ATTN_ERR_UNSUPPORTED;
  if ((int64_t)(H_q / H_kv) * S_q >= (1ll << 30)) return ATTN_ERR_UNSUPPORTED;
  if ((((int64_t)(H_q / H_kv) * S_q + 255) / 256) * B * H_kv >= (1ll << 31))
    return ATTN_ERR_UNSUPPORTED;
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

// scale * log2(e), the factor the kernels apply to the raw scores (their
// softmax runs in base 2).  It is never zero: a masked score is an infinity,
// which must keep its sign after scaling.  A zero (or underflowing) scale
// runs as the smallest normal float of the same sign: then every scaled
// score of magnitude below 2^100 is under 2^-26, and its probability rounds
// to exactly 1, as with a zero scale.
static float scale_log2_of(float scale) {
  const float v = (float)((double)scale * 1.4426950408889634);
  if (v == 0.f) return std::signbit(scale) ? -FLT_MIN : FLT_MIN;
  return v;
}

// Fills the kernel parameters (tensor maps over the row-group view).
static attn_status_t make_params(AttnParams* p, const void* q, const void* k, const void* v,
                                 void* o, float* lse, int B, int H_q, int H_kv, int S_q, int S_kv,
                                 int D, int causal, float scale) {
  std::memset(p, 0, sizeof(*p));
  const int R = (H_q / H_kv) * S_q;
  if (!encode_bf16_map_3d(&p->tm_q, q, D, R, (uint64_t)B * H_kv, 128) ||
      !encode_bf16_map_3d(&p->tm_k, k, D, S_kv, (uint64_t)B * H_kv, 128) ||
      !encode_bf16_map_3d(&p->tm_v, v, D, S_kv, (uint64_t)B * H_kv, 128) ||
      !encode_bf16_map_3d(&p->tm_o, o, D, R, (uint64_t)B * H_kv, 32))
    return ATTN_ERR_CUDA;
  p->o = o;
  p->lse = lse;
  p->B = B;
  p->H_q = H_q;
  p->H_kv = H_kv;
  p->S_q = S_q;
  p->S_kv = S_kv;
  p->causal = causal;
  p->rows_per_group = R;
  p->total_rows = (long long)B * H_q * S_q;
  // The forward's softmax takes its row max over the raw scores and needs a
  // positive factor: a negative scale runs as -Q K^T (the QK GEMM negates
  // its A operand) times |scale|, the same scores.
  p->neg_scores = std::signbit(scale) ? 1 : 0;
  p->scale_log2 = scale_log2_of(std::fabs(scale));
  p->timeout_ns = kDefaultTimeoutNs;
  p->kv_splits = 1;
  p->kv_blocks_per_split = 1 << 30;
  p->fault_drop_block = -1;
  p->n_m_tiles = (R + 255) / 256;
  p->groups = B * H_kv;
  p->num_tiles = p->n_m_tiles * p->groups;  // times the split count, set by the split-KV path
  p->lpt_heads = (causal && S_q % 256 == 0) ? H_q / H_kv : 0;
  return ATTN_OK;
}

static int n_m_tiles_of(int H_q, int H_kv, int S_q) { return ((H_q / H_kv) * S_q + 255) / 256; }

// Work tiles of a call with `splits` KV splits; the kernel indexes them with
// an int.
static bool tiles_fit(int B, int H_q, int H_kv, int S_q, int splits) {
  return (int64_t)n_m_tiles_of(H_q, H_kv, S_q) * B * H_kv * splits < (1ll << 31);
}

static attn_status_t fwd_impl(const void* q, const void* k, const void* v, void* o, float* lse,
                              int B, int H_q, int H_kv, int S_q, int S_kv, int D, int causal,
                              float scale, unsigned long long* trace, int trace_ctas,
                              int trace_blocks, int fault_drop_block,
                              unsigned long long timeout_ns, attn_stream_t stream,
                              int fault_drop_xfer = 0) {
  attn_status_t st = validate(q, k, v, o, lse, B, H_q, H_kv, S_q, S_kv, D, causal, scale);
  if (st != ATTN_OK) return st;
  st = check_device();
  if (st != ATTN_OK) return st;
  AttnParams p;
  st = make_params(&p, q, k, v, o, lse, B, H_q, H_kv, S_q, S_kv, D, causal, scale);
  if (st != ATTN_OK) return st;
  p.timeout_ns = timeout_ns;
  p.trace = trace;
  p.trace_ctas = trace_ctas;
  p.trace_blocks = trace_blocks;
  p.fault_drop_block = fault_drop_block;
  p.fault_drop_xfer = fault_drop_xfer;
  // the hand-off test needs a launch that splits its tail
  if (fault_drop_xfer && fwd_tail_pairs(p, D) <= 0) return ATTN_ERR_UNSUPPORTED;
  if (launch_attn_fwd(p, D, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

// Split count used when the caller passes num_splits <= 0.  The split-KV
// forward is bound by streaming K and V, so the CTAs should fill whole waves
// of the GPU: with fewer query tiles than SMs, one wave of about one CTA per
// SM; otherwise the split count in 1..4 whose last wave is fullest.  Each
// split keeps at least two KV blocks.
int default_splits(int B, int H_q, int H_kv, int S_q, int S_kv, int causal) {
  int sms = 152;
  int dev = 0;
  if (cudaGetDevice(&dev) == cudaSuccess)
    cudaDeviceGetAttribute(&sms, cudaDevAttrMultiProcessorCount, dev);
  const long long tiles = (long long)n_m_tiles_of(H_q, H_kv, S_q) * H_kv * B;
  const int kv_blocks = ((causal ? (S_kv < S_q ? S_kv : S_q) : S_kv) + 127) / 128;
  long long want = 1;
  if (tiles < sms) {
    want = sms / tiles;
  } else {
    double best = 0.0;
    for (int s = 1; s <= 4; ++s) {
      const long long ctas = tiles * s;
      const long long waves = (ctas + sms - 1) / sms;
      const double fill = (double)ctas / (double)(waves * sms);
      if (fill > best + 1e-9) {
        best = fill;
        want = s;
      }
    }
  }
  const long long cap = kv_blocks / 2;
  if (want > cap) want = cap;
  if (want > kMaxSplits) want = kMaxSplits;
  return want < 1 ? 1 : (int)want;
}

size_t splitkv_bytes(int B, int H_q, int S_q, int D, int splits) {
  const size_t rows = (size_t)B * H_q * S_q;
  const size_t o_bytes = (size_t)splits * rows * D * sizeof(float);
  const size_t o_pad = (o_bytes + 255) & ~(size_t)255;
  return o_pad + (size_t)splits * rows * sizeof(float);
}

attn_status_t splitkv_impl(const void* q, const void* k, const void* v, void* o, float* lse,
                                  void* workspace, size_t workspace_bytes, int B, int H_q,
                                  int H_kv, int S_q, int S_kv, int D, int causal, float scale,
                                  int num_splits, attn_stream_t stream) {
  attn_status_t st = validate(q, k, v, o, lse, B, H_q, H_kv, S_q, S_kv, D, causal, scale);
  if (st != ATTN_OK) return st;
  if (!workspace) return ATTN_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ATTN_ERR_MISALIGNED;
  if (num_splits > kMaxSplits) return ATTN_ERR_UNSUPPORTED;
  st = check_device();
  if (st != ATTN_OK) return st;
  const int splits = num_splits > 0 ? num_splits
                                    : default_splits(B, H_q, H_kv, S_q, S_kv, causal);
  if (workspace_bytes < splitkv_bytes(B, H_q, S_q, D, splits)) return ATTN_ERR_INVALID_ARG;
  AttnParams p;
  st = make_params(&p, q, k, v, o, lse, B, H_q, H_kv, S_q, S_kv, D, causal, scale);
  if (st != ATTN_OK) return st;
  if (!tiles_fit(B, H_q, H_kv, S_q, splits)) return ATTN_ERR_UNSUPPORTED;
  const int kv_blocks = (S_kv + 127) / 128;
  p.kv_splits = splits;
  p.kv_blocks_per_split = (kv_blocks + splits - 1) / splits;
  p.num_tiles = p.n_m_tiles * p.groups * splits;
  const size_t rows = (size_t)B * H_q * S_q;
  const size_t o_bytes = (size_t)splits * rows * D * sizeof(float);
  p.o_part = static_cast<float*>(workspace);
  p.lse_part = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                        ((o_bytes + 255) & ~(size_t)255));
  cudaStream_t s = static_cast<cudaStream_t>(stream);
  if (launch_attn_fwd(p, D, s) != cudaSuccess) return ATTN_ERR_CUDA;
  if (launch_splitkv_combine(p.o_part, p.lse_part, o, lse, (long long)rows, D, splits, s) !=
      cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

// Rows of the per-group padded layout of the backward's row vectors.
static int64_t bwd_padded_rows(int H_q, int H_kv, int S_q) {
  const int64_t R = (int64_t)(H_q / H_kv) * S_q;
  return (R + 127) / 128 * 128;
}

// [groups, Rp] -LSE log2(e), [groups, Rp] -D_i, then [groups, Rp, D] the
// fused backward's fp32 dQ accumulator.
size_t bwd_workspace_bytes(int B, int H_q, int H_kv, int S_q, int D) {
  return (size_t)(D + 2) * B * H_kv * (size_t)bwd_padded_rows(H_q, H_kv, S_q) * sizeof(float);
}

// Every check of attn_bwd's arguments, the device's included.
static attn_status_t bwd_validate(const void* q, const void* k, const void* v, const void* o,
                                  const float* lse, const void* dout, const void* dq,
                                  const void* dk, const void* dv, const void* workspace,
                                  size_t workspace_bytes, int B, int H_q, int H_kv, int S_q,
                                  int S_kv, int D, int causal, float scale) {
  attn_status_t st = validate(q, k, v, o, lse, B, H_q, H_kv, S_q, S_kv, D, causal, scale);
  if (st != ATTN_OK) return st;
  if (!dout || !dq || !dk || !dv || !workspace) return ATTN_ERR_INVALID_ARG;
  if (!aligned16(dout) || !aligned16(dq) || !aligned16(dk) || !aligned16(dv))
    return ATTN_ERR_MISALIGNED;
  if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return ATTN_ERR_MISALIGNED;
  if (workspace_bytes < bwd_workspace_bytes(B, H_q, H_kv, S_q, D)) return ATTN_ERR_INVALID_ARG;
  // grids: key blocks x groups and query blocks x groups CTAs, in one dimension
  const int64_t R64 = (int64_t)(H_q / H_kv) * S_q;
  if (((S_kv + 127) / 128) * (int64_t)B * H_kv >= (1ll << 31) ||
      ((R64 + 127) / 128) * (int64_t)B * H_kv >= (1ll << 31))
    return ATTN_ERR_UNSUPPORTED;
  return check_device();
}

static attn_status_t bwd_impl(const void* q, const void* k, const void* v, const void* o,
                              const float* lse, const void* dout, void* dq, void* dk, void* dv,
                              void* workspace, size_t workspace_bytes, int B, int H_q, int H_kv,
                              int S_q, int S_kv, int D, int causal, float scale,
                              bool deterministic, attn_stream_t stream, int drop_item = -1,
                              unsigned long long timeout_ns = kDefaultTimeoutNs) {
  attn_status_t st = bwd_validate(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes,
                                  B, H_q, H_kv, S_q, S_kv, D, causal, scale);
  if (st != ATTN_OK) return st;
  BwdParams p;
  std::memset(&p, 0, sizeof(p));
  const int R = (H_q / H_kv) * S_q;
  if (!encode_bf16_map_3d(&p.tm_q, q, D, R, (uint64_t)B * H_kv, 128) ||
      !encode_bf16_map_3d(&p.tm_do, dout, D, R, (uint64_t)B * H_kv, 128) ||
      !encode_bf16_map_3d(&p.tm_k, k, D, S_kv, (uint64_t)B * H_kv, 128) ||
      !encode_bf16_map_3d(&p.tm_v, v, D, S_kv, (uint64_t)B * H_kv, 128))
    return ATTN_ERR_CUDA;
  p.dq = dq;
  p.dk = dk;
  p.dv = dv;
  const int64_t Rp = bwd_padded_rows(H_q, H_kv, S_q);
  p.nlse2 = static_cast<float*>(workspace);
  p.ndelta = p.nlse2 + (size_t)B * H_kv * Rp;
  // the fused dQ: accumulated in the workspace's third part
  p.dq_acc = deterministic ? nullptr : p.ndelta + (size_t)B * H_kv * Rp;
  p.B = B;
  p.H_q = H_q;
  p.H_kv = H_kv;
  p.S_q = S_q;
  p.S_kv = S_kv;
  p.causal = causal;
  p.R = R;
  p.Rp = (int)Rp;
  p.groups = B * H_kv;
  p.scale = scale;
  p.scale_log2 = scale_log2_of(scale);
  p.timeout_ns = timeout_ns;
  p.fault_drop_item = drop_item;
  if (launch_attn_bwd(p, D, o, dout, lse, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

// ---------------------------------------------------------------- host entry
//
// attn_fwd_host and attn_bwd_host: the row groups (b, h_kv) are cut into
// chunks of consecutive groups; a chunk is a contiguous slice of every tensor
// and a problem of its own (B = 1, its groups' heads).  Its inputs go up on
// one stream, its kernels run on one of three compute streams (so one chunk's
// last tiles overlap the next chunk's first), and its outputs come back on a
// third: the copies of the other chunks overlap each chunk's kernels.  The
// streams start after, and the caller's stream continues after, the whole.
// When the kernels take longer than the copies, 16 chunks (the first chunk's
// inputs and the last chunk's outputs, which nothing overlaps, are then
// small); when the copies take longer, 8 (fewer, larger copies).
constexpr int kHostChunks = 16;
// The chunk scan's copies always take far longer than its kernel, and its
// chunks are large (a batch entry of the 64 x 8192 workload is 147 MB): it
// takes up to kHostChunksMax chunks, so the unoverlapped first upload and
// last download are short.
constexpr int kHostChunksMax = 32;
// Compute streams: consecutive chunks' kernels run on different ones, so a
// chunk kernel that leaves SMs idle (a chunk of fewer tiles than SMs) shares
// the GPU with the next chunks'.
constexpr int kHostCompStreams = 3;
// Rates on GB300 that decide which side is longer: the forward's and the
// backward's dense rates and the host link's copy rate (measured, both
// directions).
constexpr double kHostKernelFlops = 1.5e15, kHostBwdFlops = 1.0e15, kHostLinkBytes = 1.9e11;
constexpr size_t kHostPipeMinBytes = size_t(32) << 20;  // smaller inputs: one chunk

struct HostPipe {
  bool ready = false;
  cudaStream_t up = nullptr, down = nullptr, comp[kHostCompStreams] = {};
  cudaEvent_t start = nullptr, done = nullptr;
  cudaEvent_t loaded[kHostChunksMax] = {}, computed[kHostChunksMax] = {};
};
static std::mutex g_pipe_mu;
static HostPipe g_pipe[64];

// Chunk boundaries of a host call over `units` row groups: chunk c holds
// units [bound[c], bound[c + 1]).
struct ChunkPlan {
  int n = 1;
  int bound[kHostChunksMax + 1] = {};
};

// One chunk below kHostPipeMinBytes of inputs, else 16 or 8 as above (never
// more than the units), evenly sized.  When the kernels are the longer side,
// the first and the last chunk hold one unit each and the units between keep
// the even chunks' size: the first upload and the last download are the two
// copies that nothing overlaps, and chunks that small everywhere would leave
// each kernel too few tiles.
static ChunkPlan host_plan(size_t in_bytes, size_t out_bytes, double kernel_s, int units) {
  ChunkPlan pl;
  pl.bound[0] = 0;
  pl.bound[1] = units;
  if (in_bytes < kHostPipeMinBytes) return pl;
  const bool kernel_longer = kernel_s > (double)(in_bytes + out_bytes) / kHostLinkBytes;
  const int want = kernel_longer ? kHostChunks : kHostChunks / 2;
  const int even = units < want ? units : want;
  const int size = units / even;  // units per even chunk
  const int inner = units - 2;
  const int n_in = size > 0 ? (inner + size - 1) / size : 0;
  if (kernel_longer && size >= 2 && n_in >= 1 && n_in + 2 <= kHostChunksMax) {
    pl.n = n_in + 2;
    pl.bound[1] = 1;
    for (int i = 1; i <= n_in; ++i) pl.bound[1 + i] = 1 + (int)((long long)inner * i / n_in);
    pl.bound[pl.n] = units;
    return pl;
  }
  pl.n = even;
  for (int c = 0; c <= even; ++c) pl.bound[c] = (int)((long long)units * c / even);
  return pl;
}

// The device's streams and events, made on first use (call with g_pipe_mu held).
static HostPipe* host_pipe(int dev) {
  HostPipe& hp = g_pipe[dev];
  if (hp.ready) return &hp;
  const unsigned sf = cudaStreamNonBlocking;
  const unsigned ef = cudaEventDisableTiming;
  bool ok = cudaStreamCreateWithFlags(&hp.up, sf) == cudaSuccess &&
            cudaStreamCreateWithFlags(&hp.down, sf) == cudaSuccess &&
            cudaEventCreateWithFlags(&hp.start, ef) == cudaSuccess &&
            cudaEventCreateWithFlags(&hp.done, ef) == cudaSuccess;
  for (int i = 0; ok && i < kHostCompStreams; ++i)
    ok = cudaStreamCreateWithFlags(&hp.comp[i], sf) == cudaSuccess;
  for (int c = 0; ok && c < kHostChunksMax; ++c)
    ok = cudaEventCreateWithFlags(&hp.loaded[c], ef) == cudaSuccess &&
         cudaEventCreateWithFlags(&hp.computed[c], ef) == cudaSuccess;
  if (!ok) return nullptr;  // (what was made stays cached for the process)
  hp.ready = true;
  return &hp;
}

// The pipe's streams start after the work queued on `s` so far ...
static bool pipe_fork(HostPipe* hp, cudaStream_t s) {
  bool ok = cudaEventRecord(hp->start, s) == cudaSuccess &&
            cudaStreamWaitEvent(hp->up, hp->start, 0) == cudaSuccess &&
            cudaStreamWaitEvent(hp->down, hp->start, 0) == cudaSuccess;
  for (int i = 0; ok && i < kHostCompStreams; ++i)
    ok = cudaStreamWaitEvent(hp->comp[i], hp->start, 0) == cudaSuccess;
  return ok;
}

// ... and `s` continues once every chunk's outputs are back (and so its
// kernels and inputs are done).
static bool pipe_join(HostPipe* hp, cudaStream_t s) {
  return cudaEventRecord(hp->done, hp->down) == cudaSuccess &&
         cudaStreamWaitEvent(s, hp->done, 0) == cudaSuccess;
}

static attn_status_t fwd_host_impl(const void* q_host, const void* k_host, const void* v_host,
                                   void* o_host, float* lse_host, void* q_dev, void* k_dev,
                                   void* v_dev, void* o_dev, float* lse_dev, int B, int H_q,
                                   int H_kv, int S_q, int S_kv, int D, int causal, float scale,
                                   cudaStream_t s) {
  const size_t q_bytes = (size_t)B * H_q * S_q * D * 2;
  const size_t kv_bytes = (size_t)B * H_kv * S_kv * D * 2;
  const size_t lse_bytes = (size_t)B * H_q * S_q * sizeof(float);
  const int groups = B * H_kv;
  const double flops = 4.0 * B * H_q * (double)S_q * S_kv * D * (causal ? 0.5 : 1.0);
  const ChunkPlan plan = host_plan(q_bytes + 2 * kv_bytes, q_bytes, flops / kHostKernelFlops, groups);
  const int chunks = plan.n;
  if (chunks <= 1) {
    if (cudaMemcpyAsync(q_dev, q_host, q_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(k_dev, k_host, kv_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess ||
        cudaMemcpyAsync(v_dev, v_host, kv_bytes, cudaMemcpyHostToDevice, s) != cudaSuccess)
      return ATTN_ERR_CUDA;
    attn_status_t st = fwd_impl(q_dev, k_dev, v_dev, o_dev, lse_dev, B, H_q, H_kv, S_q, S_kv, D,
                                causal, scale, nullptr, 0, 0, -1, kDefaultTimeoutNs, s);
    if (st != ATTN_OK) return st;
    if (cudaMemcpyAsync(o_host, o_dev, q_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess ||
        cudaMemcpyAsync(lse_host, lse_dev, lse_bytes, cudaMemcpyDeviceToHost, s) != cudaSuccess)
      return ATTN_ERR_CUDA;
    return ATTN_OK;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return ATTN_ERR_CUDA;
  // queued under the lock, so concurrent callers' chunks do not interleave
  std::lock_guard<std::mutex> lk(g_pipe_mu);
  HostPipe* hp = host_pipe(dev);
  if (!hp || !pipe_fork(hp, s)) return ATTN_ERR_CUDA;
  // past this point every exit joins the pipe, so `s` stays ordered after
  // whatever was already queued on the internal streams
  auto leave = [&](attn_status_t st) { pipe_join(hp, s); return st; };
  const int r = H_q / H_kv;
  const size_t q_group = (size_t)r * S_q * D * 2;     // bytes of one group's Q (and O)
  const size_t kv_group = (size_t)S_kv * D * 2;       // bytes of one group's K (and V)
  const size_t lse_group = (size_t)r * S_q;           // floats of one group's LSE
  for (int c = 0; c < chunks; ++c) {
    const int z0 = plan.bound[c];
    const int z1 = plan.bound[c + 1];
    const int ng = z1 - z0;
    const size_t qo = z0 * q_group, qn = ng * q_group;
    const size_t ko = z0 * kv_group, kn = ng * kv_group;
    const size_t lo = z0 * lse_group, ln = ng * lse_group;
    auto hb = [](const void* p, size_t off) { return static_cast<const char*>(p) + off; };
    auto db = [](void* p, size_t off) { return static_cast<char*>(p) + off; };
    if (cudaMemcpyAsync(db(q_dev, qo), hb(q_host, qo), qn, cudaMemcpyHostToDevice, hp->up) !=
            cudaSuccess ||
        cudaMemcpyAsync(db(k_dev, ko), hb(k_host, ko), kn, cudaMemcpyHostToDevice, hp->up) !=
            cudaSuccess ||
        cudaMemcpyAsync(db(v_dev, ko), hb(v_host, ko), kn, cudaMemcpyHostToDevice, hp->up) !=
            cudaSuccess ||
        cudaEventRecord(hp->loaded[c], hp->up) != cudaSuccess)
      return leave(ATTN_ERR_CUDA);
    cudaStream_t cs = hp->comp[c % kHostCompStreams];
    if (cudaStreamWaitEvent(cs, hp->loaded[c], 0) != cudaSuccess) return leave(ATTN_ERR_CUDA);
    attn_status_t st =
        fwd_impl(db(q_dev, qo), db(k_dev, ko), db(v_dev, ko), db(o_dev, qo), lse_dev + lo, 1,
                 ng * r, ng, S_q, S_kv, D, causal, scale, nullptr, 0, 0, -1, kDefaultTimeoutNs, cs);
    if (st != ATTN_OK) return leave(st);
    if (cudaEventRecord(hp->computed[c], cs) != cudaSuccess ||
        cudaStreamWaitEvent(hp->down, hp->computed[c], 0) != cudaSuccess ||
        cudaMemcpyAsync(db(o_host, qo), db(o_dev, qo), qn, cudaMemcpyDeviceToHost, hp->down) !=
            cudaSuccess ||
        cudaMemcpyAsync(lse_host + lo, lse_dev + lo, ln * sizeof(float), cudaMemcpyDeviceToHost,
                        hp->down) != cudaSuccess)
      return leave(ATTN_ERR_CUDA);
  }
  return pipe_join(hp, s) ? ATTN_OK : ATTN_ERR_CUDA;
}

static attn_status_t bwd_host_impl(const void* q_host, const void* k_host, const void* v_host,
                                   const void* o_host, const float* lse_host,
                                   const void* dout_host, void* dq_host, void* dk_host,
                                   void* dv_host, void* q_dev, void* k_dev, void* v_dev,
                                   void* o_dev, float* lse_dev, void* dout_dev, void* dq_dev,
                                   void* dk_dev, void* dv_dev, void* workspace,
                                   size_t workspace_bytes, int B, int H_q, int H_kv, int S_q,
                                   int S_kv, int D, int causal, float scale, cudaStream_t s) {
  const size_t q_bytes = (size_t)B * H_q * S_q * D * 2;
  const size_t kv_bytes = (size_t)B * H_kv * S_kv * D * 2;
  const size_t lse_bytes = (size_t)B * H_q * S_q * sizeof(float);
  const int groups = B * H_kv;
  const double flops = 2.5 * 4.0 * B * H_q * (double)S_q * S_kv * D * (causal ? 0.5 : 1.0);
  const ChunkPlan plan = host_plan(3 * q_bytes + 2 * kv_bytes + lse_bytes,
                                   q_bytes + 2 * kv_bytes, flops / kHostBwdFlops, groups);
  const int chunks = plan.n;
  auto up = [](void* dst, const void* src, size_t n, cudaStream_t st) {
    return cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, st) == cudaSuccess;
  };
  auto down = [](void* dst, const void* src, size_t n, cudaStream_t st) {
    return cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToHost, st) == cudaSuccess;
  };
  if (chunks <= 1) {
    if (!up(q_dev, q_host, q_bytes, s) || !up(k_dev, k_host, kv_bytes, s) ||
        !up(v_dev, v_host, kv_bytes, s) || !up(o_dev, o_host, q_bytes, s) ||
        !up(lse_dev, lse_host, lse_bytes, s) || !up(dout_dev, dout_host, q_bytes, s))
      return ATTN_ERR_CUDA;
    attn_status_t st = bwd_impl(q_dev, k_dev, v_dev, o_dev, lse_dev, dout_dev, dq_dev, dk_dev,
                                dv_dev, workspace, workspace_bytes, B, H_q, H_kv, S_q, S_kv, D,
                                causal, scale, false, s);
    if (st != ATTN_OK) return st;
    if (!down(dq_host, dq_dev, q_bytes, s) || !down(dk_host, dk_dev, kv_bytes, s) ||
        !down(dv_host, dv_dev, kv_bytes, s))
      return ATTN_ERR_CUDA;
    return ATTN_OK;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_pipe_mu);
  HostPipe* hp = host_pipe(dev);
  if (!hp || !pipe_fork(hp, s)) return ATTN_ERR_CUDA;
  // past this point every exit joins the pipe, so `s` stays ordered after
  // whatever was already queued on the internal streams
  auto leave = [&](attn_status_t st) { pipe_join(hp, s); return st; };
  const int r = H_q / H_kv;
  const size_t q_group = (size_t)r * S_q * D * 2;     // bytes of one group's Q (O, dO, dQ)
  const size_t kv_group = (size_t)S_kv * D * 2;       // bytes of one group's K (V, dK, dV)
  const size_t lse_group = (size_t)r * S_q;           // floats of one group's LSE
  // a chunk's workspace is its own slice: the per-group layout of a call on
  // ng groups takes 2 * ng padded row vectors (a multiple of 1024 bytes)
  const size_t ws_group = (size_t)(D + 2) * bwd_padded_rows(H_q, H_kv, S_q) * sizeof(float);
  auto hb = [](const void* p, size_t off) { return static_cast<const char*>(p) + off; };
  auto db = [](void* p, size_t off) { return static_cast<char*>(p) + off; };
  for (int c = 0; c < chunks; ++c) {
    const int z0 = plan.bound[c];
    const int z1 = plan.bound[c + 1];
    const int ng = z1 - z0;
    const size_t qo = z0 * q_group, qn = ng * q_group;
    const size_t ko = z0 * kv_group, kn = ng * kv_group;
    const size_t lo = z0 * lse_group, ln = ng * lse_group;
    if (!up(db(q_dev, qo), hb(q_host, qo), qn, hp->up) ||
        !up(db(k_dev, ko), hb(k_host, ko), kn, hp->up) ||
        !up(db(v_dev, ko), hb(v_host, ko), kn, hp->up) ||
        !up(db(o_dev, qo), hb(o_host, qo), qn, hp->up) ||
        !up(lse_dev + lo, lse_host + lo, ln * sizeof(float), hp->up) ||
        !up(db(dout_dev, qo), hb(dout_host, qo), qn, hp->up) ||
        cudaEventRecord(hp->loaded[c], hp->up) != cudaSuccess)
      return leave(ATTN_ERR_CUDA);
    cudaStream_t cs = hp->comp[c % kHostCompStreams];
    if (cudaStreamWaitEvent(cs, hp->loaded[c], 0) != cudaSuccess) return leave(ATTN_ERR_CUDA);
    attn_status_t st = bwd_impl(db(q_dev, qo), db(k_dev, ko), db(v_dev, ko), db(o_dev, qo),
                                lse_dev + lo, db(dout_dev, qo), db(dq_dev, qo), db(dk_dev, ko),
                                db(dv_dev, ko), db(workspace, z0 * ws_group), ng * ws_group, 1,
                                ng * r, ng, S_q, S_kv, D, causal, scale, false, cs);
    if (st != ATTN_OK) return leave(st);
    if (cudaEventRecord(hp->computed[c], cs) != cudaSuccess ||
        cudaStreamWaitEvent(hp->down, hp->computed[c], 0) != cudaSuccess ||
        !down(db(dq_host, qo), db(dq_dev, qo), qn, hp->down) ||
        !down(db(dk_host, ko), db(dk_dev, ko), kn, hp->down) ||
        !down(db(dv_host, ko), db(dv_dev, ko), kn, hp->down))
      return leave(ATTN_ERR_CUDA);
  }
  return pipe_join(hp, s) ? ATTN_OK : ATTN_ERR_CUDA;
}

// Every check of chunk_scan_fwd's arguments, the device's included.
static attn_status_t chunk_scan_validate(const void* cb, const void* dA_cs, const void* dt,
                                         const void* x, const void* out, int B, int L, int H,
                                         int G, int P, int Q) {
  if (!cb || !dA_cs || !dt || !x || !out) return ATTN_ERR_INVALID_ARG;
  if (B <= 0 || L <= 0 || H <= 0 || G <= 0 || P <= 0 || Q <= 0) return ATTN_ERR_INVALID_ARG;
  if (H % G != 0 || L % Q != 0) return ATTN_ERR_INVALID_ARG;
  if (P != 64 || (Q != 128 && Q != 256)) return ATTN_ERR_UNSUPPORTED;
  if ((int64_t)B * L * H >= (1ll << 31) || (int64_t)B * (L / Q) * H * (Q / 128) >= (1ll << 31) ||
      (int64_t)B * (L / Q) * G >= (1ll << 31))
    return ATTN_ERR_UNSUPPORTED;
  if (!aligned16(cb) || !aligned16(dA_cs) || !aligned16(dt) || !aligned16(x) || !aligned16(out))
    return ATTN_ERR_MISALIGNED;
  return check_device();
}

static attn_status_t chunk_scan_impl(const float* cb, const float* dA_cs, const float* dt,
                                     const void* x, void* out, int B, int L, int H, int G, int P,
                                     int Q, attn_stream_t stream) {
  attn_status_t st = chunk_scan_validate(cb, dA_cs, dt, x, out, B, L, H, G, P, Q);
  if (st != ATTN_OK) return st;
  EncodeTiledFn fn = get_encode_fn();
  if (!fn) return ATTN_ERR_CUDA;
  ChunkScanParams p;
  std::memset(&p, 0, sizeof(p));
  // x [B, L, H, P] as a 4-D map {P, H, L, B}: box {64, 1, 64, 1} = 64 rows of
  // one head, 128 bytes each
  cuuint64_t dims[4] = {(cuuint64_t)P, (cuuint64_t)H, (cuuint64_t)L, (cuuint64_t)B};
  cuuint64_t strides[3] = {(cuuint64_t)P * 2, (cuuint64_t)H * P * 2, (cuuint64_t)L * H * P * 2};
  cuuint32_t box[4] = {64, 1, 64, 1};
  cuuint32_t estr[4] = {1, 1, 1, 1};
  if (fn(&p.tm_x, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(x), dims, strides, box,
         estr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return ATTN_ERR_CUDA;
  // out [B, L, H, P] as the same 4-D map with 128 rows per box (one head's
  // rows of a 128-row tile)
  cuuint32_t obox[4] = {64, 1, 128, 1};
  if (fn(&p.tm_out, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, out, dims, strides, obox, estr,
         CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return ATTN_ERR_CUDA;
  // cb [B * nchunks * G, Q, Q] fp32 as a 3-D map: box {32, 128, 1} = 128 rows
  // of 32 keys (128 bytes each)
  cuuint64_t cdims[3] = {(cuuint64_t)Q, (cuuint64_t)Q, (cuuint64_t)B * (L / Q) * G};
  cuuint64_t cstrides[2] = {(cuuint64_t)Q * 4, (cuuint64_t)Q * Q * 4};
  cuuint32_t cbox[3] = {32, 128, 1};
  cuuint32_t cestr[3] = {1, 1, 1};
  if (fn(&p.tm_cb, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 3, const_cast<float*>(cb), cdims, cstrides,
         cbox, cestr, CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B,
         CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return ATTN_ERR_CUDA;
  p.HB = 0;  // heads per CTA: chosen at launch from the SM count
  p.dA_cs = dA_cs;
  p.dt = dt;
  p.out = out;
  p.B = B;
  p.L = L;
  p.H = H;
  p.G = G;
  p.Q = Q;
  p.nchunks = L / Q;
  p.timeout_ns = kDefaultTimeoutNs;
  if (launch_chunk_scan(p, static_cast<cudaStream_t>(stream)) != cudaSuccess)
    return ATTN_ERR_CUDA;
  return ATTN_OK;
}

// chunk_scan_fwd_host: the batch is cut into up to 32 chunks of consecutive batch
// entries (a contiguous slice of every tensor and a problem of its own),
// pipelined on the same streams as attn_fwd_host.  The kernel is far shorter
// than the copies here, so the gain is the uploads of one chunk overlapping
// the downloads of another (the host link carries both directions at once).
static attn_status_t chunk_scan_host_impl(const float* cb_host, const float* dA_host,
                                          const float* dt_host, const void* x_host,
                                          void* out_host, float* cb_dev, float* dA_dev,
                                          float* dt_dev, void* x_dev, void* out_dev, int B, int L,
                                          int H, int G, int P, int Q, cudaStream_t s) {
  const size_t nch = (size_t)(L / Q);
  const size_t cb_b = nch * G * Q * Q;     // floats of one batch entry's cb
  const size_t vec_b = (size_t)H * nch * Q;  // floats of its dA_cs (and of its dt)
  const size_t x_b = (size_t)L * H * P * 2;  // bytes of its x (and of its out)
  const size_t in_bytes = (size_t)B * (cb_b * 4 + 2 * vec_b * 4 + x_b);
  const size_t out_bytes = (size_t)B * x_b;
  const int chunks =
      in_bytes < kHostPipeMinBytes ? 1 : (B < kHostChunksMax ? B : kHostChunksMax);
  auto up = [](void* dst, const void* src, size_t n, cudaStream_t st) {
    return cudaMemcpyAsync(dst, src, n, cudaMemcpyHostToDevice, st) == cudaSuccess;
  };
  auto down = [](void* dst, const void* src, size_t n, cudaStream_t st) {
    return cudaMemcpyAsync(dst, src, n, cudaMemcpyDeviceToHost, st) == cudaSuccess;
  };
  if (chunks <= 1) {
    if (!up(cb_dev, cb_host, B * cb_b * 4, s) || !up(dA_dev, dA_host, B * vec_b * 4, s) ||
        !up(dt_dev, dt_host, B * vec_b * 4, s) || !up(x_dev, x_host, B * x_b, s))
      return ATTN_ERR_CUDA;
    attn_status_t st = chunk_scan_impl(cb_dev, dA_dev, dt_dev, x_dev, out_dev, B, L, H, G, P, Q, s);
    if (st != ATTN_OK) return st;
    return down(out_host, out_dev, out_bytes, s) ? ATTN_OK : ATTN_ERR_CUDA;
  }
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return ATTN_ERR_CUDA;
  std::lock_guard<std::mutex> lk(g_pipe_mu);
  HostPipe* hp = host_pipe(dev);
  if (!hp || !pipe_fork(hp, s)) return ATTN_ERR_CUDA;
  // past this point every exit joins the pipe, so `s` stays ordered after
  // whatever was already queued on the internal streams
  auto leave = [&](attn_status_t st) { pipe_join(hp, s); return st; };
  auto hb = [](const void* p, size_t off) { return static_cast<const char*>(p) + off; };
  auto db = [](void* p, size_t off) { return static_cast<char*>(p) + off; };
  for (int c = 0; c < chunks; ++c) {
    const int b0 = (int)((long long)B * c / chunks);
    const int b1 = (int)((long long)B * (c + 1) / chunks);
    const int nb = b1 - b0;
    const size_t co = b0 * cb_b * 4, cn = nb * cb_b * 4;
    const size_t vo = b0 * vec_b * 4, vn = nb * vec_b * 4;
    const size_t xo = b0 * x_b, xn = nb * x_b;
    if (!up(db(cb_dev, co), hb(cb_host, co), cn, hp->up) ||
        !up(db(dA_dev, vo), hb(dA_host, vo), vn, hp->up) ||
        !up(db(dt_dev, vo), hb(dt_host, vo), vn, hp->up) ||
        !up(db(x_dev, xo), hb(x_host, xo), xn, hp->up) ||
        cudaEventRecord(hp->loaded[c], hp->up) != cudaSuccess)
      return leave(ATTN_ERR_CUDA);
    cudaStream_t cs = hp->comp[c % kHostCompStreams];
    if (cudaStreamWaitEvent(cs, hp->loaded[c], 0) != cudaSuccess) return leave(ATTN_ERR_CUDA);
    attn_status_t st = chunk_scan_impl(cb_dev + b0 * cb_b, dA_dev + b0 * vec_b,
                                       dt_dev + b0 * vec_b, db(x_dev, xo), db(out_dev, xo), nb,
                                       L, H, G, P, Q, cs);
    if (st != ATTN_OK) return leave(st);
    if (cudaEventRecord(hp->computed[c], cs) != cudaSuccess ||
        cudaStreamWaitEvent(hp->down, hp->computed[c], 0) != cudaSuccess ||
        !down(db(out_host, xo), db(out_dev, xo), xn, hp->down))
      return leave(ATTN_ERR_CUDA);
  }
  return pipe_join(hp, s) ? ATTN_OK : ATTN_ERR_CUDA;
}

}  // namespace attnpipe

extern "C" {

attn_status_t chunk_scan_fwd(const float* cb, const float* dA_cs, const float* dt, const void* x,
                             void* out, int B, int L, int H, int G, int P, int Q,
                             attn_stream_t stream) {
  return chunk_scan_impl(cb, dA_cs, dt, x, out, B, L, H, G, P, Q, stream);
}

attn_status_t chunk_scan_fwd_host(const float* cb_host, const float* dA_cs_host,
                                  const float* dt_host, const void* x_host, void* out_host,
                                  float* cb_dev, float* dA_cs_dev, float* dt_dev, void* x_dev,
                                  void* out_dev, int B, int L, int H, int G, int P, int Q,
                                  attn_stream_t stream) {
  if (!cb_host || !dA_cs_host || !dt_host || !x_host || !out_host) return ATTN_ERR_INVALID_ARG;
  attn_status_t st = chunk_scan_validate(cb_dev, dA_cs_dev, dt_dev, x_dev, out_dev, B, L, H, G,
                                         P, Q);
  if (st != ATTN_OK) return st;
  return attnpipe::chunk_scan_host_impl(cb_host, dA_cs_host, dt_host, x_host, out_host, cb_dev,
                                        dA_cs_dev, dt_dev, x_dev, out_dev, B, L, H, G, P, Q,
                                        static_cast<cudaStream_t>(stream));
}

attn_status_t attn_bwd(const void* q, const void* k, const void* v, const void* o,
                       const float* lse, const void* dout, void* dq, void* dk, void* dv,
                       void* workspace, size_t workspace_bytes, int B, int H_q, int H_kv,
                       int S_q, int S_kv, int D, int causal, float scale, attn_stream_t stream) {
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, B, H_q, H_kv,
                  S_q, S_kv, D, causal, scale, false, stream);
}

attn_status_t attn_bwd_deterministic(const void* q, const void* k, const void* v, const void* o,
                                     const float* lse, const void* dout, void* dq, void* dk,
                                     void* dv, void* workspace, size_t workspace_bytes, int B,
                                     int H_q, int H_kv, int S_q, int S_kv, int D, int causal,
                                     float scale, attn_stream_t stream) {
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, B, H_q, H_kv,
                  S_q, S_kv, D, causal, scale, true, stream);
}

size_t attn_bwd_workspace_bytes(int B, int H_q, int H_kv, int S_q, int D) {
  if (B <= 0 || H_q <= 0 || H_kv <= 0 || S_q <= 0 || H_q % H_kv != 0) return 0;
  if (D != 64 && D != 128) return 0;
  return bwd_workspace_bytes(B, H_q, H_kv, S_q, D);
}

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
  if (!trace || trace_ctas <= 0 || trace_blocks <= 0 || trace_blocks > kMaxTraceBlocks)
    return ATTN_ERR_INVALID_ARG;
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

attn_status_t attn_fwd_tail_timeout_test(const void* q, const void* k, const void* v, void* o,
                                         float* lse, int B, int H_q, int H_kv, int S_q, int S_kv,
                                         int D, int causal, float scale,
                                         unsigned long long wait_budget_ns,
                                         attn_stream_t stream) {
  if (wait_budget_ns < 1000000ull || wait_budget_ns > kDefaultTimeoutNs)
    return ATTN_ERR_INVALID_ARG;
  return fwd_impl(q, k, v, o, lse, B, H_q, H_kv, S_q, S_kv, D, causal, scale, nullptr, 0, 0, -1,
                  wait_budget_ns, stream, 1);
}

attn_status_t attn_bwd_timeout_test(const void* q, const void* k, const void* v, const void* o,
                                    const float* lse, const void* dout, void* dq, void* dk,
                                    void* dv, void* workspace, size_t workspace_bytes, int B,
                                    int H_q, int H_kv, int S_q, int S_kv, int D, int causal,
                                    float scale, int drop_item, unsigned long long wait_budget_ns,
                                    attn_stream_t stream) {
  if (drop_item < 0) return ATTN_ERR_INVALID_ARG;
  if (wait_budget_ns < 1000000ull || wait_budget_ns > kDefaultTimeoutNs)
    return ATTN_ERR_INVALID_ARG;
  return bwd_impl(q, k, v, o, lse, dout, dq, dk, dv, workspace, workspace_bytes, B, H_q, H_kv,
                  S_q, S_kv, D, causal, scale, false, stream, drop_item, wait_budget_ns);
}

int attn_fwd_tail_pairs(int B, int H_q, int H_kv, int S_q, int S_kv, int D, int causal) {
  // the size rules of attn_fwd, with a stand-in address that is never used
  const void* a = reinterpret_cast<const void*>(static_cast<uintptr_t>(256));
  if (validate(a, a, a, a, a, B, H_q, H_kv, S_q, S_kv, D, causal, 1.f) != ATTN_OK) return -1;
  if (check_device() != ATTN_OK) return -1;
  AttnParams p;
  std::memset(&p, 0, sizeof(p));
  p.S_kv = S_kv;
  p.causal = causal;
  p.kv_splits = 1;
  p.n_m_tiles = n_m_tiles_of(H_q, H_kv, S_q);
  p.groups = B * H_kv;
  p.num_tiles = p.n_m_tiles * p.groups;
  return fwd_tail_pairs(p, D);
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
  return attnpipe::fwd_host_impl(q_host, k_host, v_host, o_host, lse_host, q_dev, k_dev, v_dev,
                                 o_dev, lse_dev, B, H_q, H_kv, S_q, S_kv, D, causal, scale,
                                 static_cast<cudaStream_t>(stream));
}

attn_status_t attn_bwd_host(const void* q_host, const void* k_host, const void* v_host,
                            const void* o_host, const float* lse_host, const void* dout_host,
                            void* dq_host, void* dk_host, void* dv_host, void* q_dev, void* k_dev,
                            void* v_dev, void* o_dev, float* lse_dev, void* dout_dev,
                            void* dq_dev, void* dk_dev, void* dv_dev, void* workspace,
                            size_t workspace_bytes, int B, int H_q, int H_kv, int S_q, int S_kv,
                            int D, int causal, float scale, attn_stream_t stream) {
  if (!q_host || !k_host || !v_host || !o_host || !lse_host || !dout_host || !dq_host ||
      !dk_host || !dv_host)
    return ATTN_ERR_INVALID_ARG;
  attn_status_t st = bwd_validate(q_dev, k_dev, v_dev, o_dev, lse_dev, dout_dev, dq_dev, dk_dev,
                                  dv_dev, workspace, workspace_bytes, B, H_q, H_kv, S_q, S_kv, D,
                                  causal, scale);
  if (st != ATTN_OK) return st;
  return attnpipe::bwd_host_impl(q_host, k_host, v_host, o_host, lse_host, dout_host, dq_host,
                                 dk_host, dv_host, q_dev, k_dev, v_dev, o_dev, lse_dev, dout_dev,
                                 dq_dev, dk_dev, dv_dev, workspace, workspace_bytes, B, H_q, H_kv,
                                 S_q, S_kv, D, causal, scale, static_cast<cudaStream_t>(stream));
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
  int main_status = 0, selftest_status = 0, bwd_status = 0, cs_status = 0;
  if (read_device_status(&main_status, reset != 0) != cudaSuccess ||
      read_selftest_status(&selftest_status, reset != 0) != cudaSuccess ||
      read_bwd_status(&bwd_status, reset != 0) != cudaSuccess ||
      read_chunk_scan_status(&cs_status, reset != 0) != cudaSuccess)
    return ATTN_ERR_CUDA;
  *status_out = main_status != 0 ? main_status
                : bwd_status != 0 ? bwd_status
                : cs_status != 0  ? cs_status
                                  : selftest_status;
  return ATTN_OK;
}

int attn_version(void) { return 100; }

size_t attn_splitkv_workspace_bytes(int B, int H_q, int S_q, int D, int num_splits) {
  if (B <= 0 || H_q <= 0 || S_q <= 0 || (D != 64 && D != 128) || num_splits <= 0 ||
      num_splits > kMaxSplits)
    return 0;
  return splitkv_bytes(B, H_q, S_q, D, num_splits);
}

int attn_splitkv_default_splits(int B, int H_q, int H_kv, int S_q, int S_kv, int causal) {
  if (B <= 0 || H_q <= 0 || H_kv <= 0 || S_q <= 0 || S_kv <= 0 || H_q % H_kv != 0) return 0;
  return default_splits(B, H_q, H_kv, S_q, S_kv, causal);
}

attn_status_t attn_fwd_splitkv(const void* q, const void* k, const void* v, void* o, float* lse,
                               void* workspace, size_t workspace_bytes, int B, int H_q, int H_kv,
                               int S_q, int S_kv, int D, int causal, float scale, int num_splits,
                               attn_stream_t stream) {
  return splitkv_impl(q, k, v, o, lse, workspace, workspace_bytes, B, H_q, H_kv, S_q, S_kv, D,
                      causal, scale, num_splits, stream);
}

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
