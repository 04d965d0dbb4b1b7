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
// The grid is persistent: at most one CTA per SM, each working through a list
// of tiles (see AttnParams for the order).  A tile is 256 query rows of one
// row group against one KV split, as two 128-row sub-tiles t = 0, 1.  Every
// role keeps its barrier phases running from tile to tile, so the next
// tile's loads and first GEMMs overlap the current tile's last blocks and its
// epilogue.  512 threads:
//   warps 0-3   softmax warpgroup for sub-tile 0 (thread = query row)
//   warps 4-7   softmax warpgroup for sub-tile 1
//   warps 8-11  correction warpgroup: rescales O_t in tensor memory when a
//               row max moved, then the epilogue (O / l -> bf16 -> global,
//               LSE)
//   warp  12    tensor-core issuer (one thread issues every tcgen05.mma)
//   warp  13    TMA producer: Q_0, Q_1 per tile, K_j, V_j through a ring
//   warps 14-15 idle (they complete warpgroup 3 for setmaxnreg)
//
// Tensor memory (512 columns x 128 lanes, lane = query row of the sub-tile):
//   [0,128) S_0, [128,256) S_1, [256,256+D) O_0, [256+D,256+2D) O_1.
// P_t (bf16, two per column) overwrites the first 64 columns of S_t once the
// softmax has read S_t into registers.  The next S_t GEMM is issued after the
// PV GEMM that reads P_t, by the same thread; tcgen05.mma operations issued
// by one thread execute in issue order.
//
// Hand-offs between tiles:
//   q_free[t]  the tile's last S_t GEMM has read Q_t: the producer may load
//              the next tile's Q_t into the same buffer;
//   p_full[t]  for block 0 of a tile, the correction's half of the arrivals
//              means "the previous tile's O_t has been read out of tensor
//              memory", so the first PV_t (which overwrites O_t) waits for it;
//   fin[2][t]  the final row statistics, double-buffered by tile parity so a
//              one-block tile cannot overwrite them before they are read.
//
// Split tail (the kTail instantiation, launched as clusters of two CTAs):
// when the grid's last round would leave more than half of the CTAs idle,
// each of its tiles is split across a CTA pair, half of the KV blocks each.
// Both halves run as ordinary tiles.  At the end each CTA writes one
// sub-tile (the first sub-tile 0, the second sub-tile 1; with one sub-tile,
// the first) and sends the other one's partial (normalised fp32 O and
// base-2 log-sum-exp) to its partner: it stages the partial in its own idle
// K/V ring and Q buffer, arms its xfer_full with the bytes it will receive
// and arrives on the partner's xfer_free; once its own xfer_free completes
// it sends the staged partial with two bulk copies (shared memory to the
// partner's shared memory, completing as transaction bytes on the partner's
// xfer_full); then it merges its sub-tile with the received partial by the
// two log-sum-exps and writes O and LSE.
// Cluster barriers at start (barriers initialised) and exit (no CTA leaves
// while its partner may still touch its shared memory) bracket the kernel.
//
// Every wait is bounded (see ptx.cuh); a timeout raises a CTA-wide abort
// flag, every role unwinds to the teardown, and the device status word
// records ATTN_ERR_TIMEOUT.  No trap, no assert.
#include <cmath>
#include <cstdint>
#include <mutex>
#include <type_traits>

#include "attn_internal.h"
#include "attn_tiles.cuh"
#include "ptx.cuh"

namespace attnpipe {

__device__ int g_attn_status = 0;

namespace {

constexpr int kThreads = 512;
constexpr uint32_t kBarCorrection = 1;  // named barrier of the correction warpgroup (split tail)
constexpr int kBlockM = 128;  // rows per query sub-tile
constexpr int kBlockN = 128;  // keys per KV block
constexpr float kRescaleThreshold = 8.0f;  // log2 units: P may grow to 2^8 before O is rescaled
// Split tail only for tiles of at least this many KV blocks: half a tile must
// save more than the exchange, the merge and the cluster start cost.  Measured
// on GB300 with the one-bulk-copy exchange: +2.8 % at 16 blocks per tile (4 x
// 16 heads x 2048, 128-dim), the same at 8; causal tiles are never split (the
// last round holds the shortest of them).
constexpr int kSplitTailMinBlocks = 16;
constexpr uint32_t kFull = 0xffffffffu;
// Pairs of probabilities out of every 8 whose exp2 runs on the FMA pipe
// (exp2_poly_x2) instead of MUFU, in unmasked blocks.  0: every exp2 on
// MUFU.  Measured on GB300 (grouped-query D = 64 workload, 828 TFLOP/s with
// 0): 1 pair 782, 2 pairs 747, 4 pairs 635 -- the softmax is bound by
// instruction issue, not by MUFU (whose exp2 rate on this part matches the
// tensor core's at D = 64), and each pair on the FMA pipe costs about ten
// issue slots instead of two.
#ifndef ATTN_POLY_PAIRS
#define ATTN_POLY_PAIRS 0
#endif
constexpr int kPolyPairs = ATTN_POLY_PAIRS;
// Register split across the four warpgroups (setmaxnreg): softmax x2,
// correction, load/MMA.  The kernel launches with 128 registers per thread
// (launch bounds 512 x 1), and the split must fit in that pool.
constexpr int kRegsSoftmax = 168, kRegsCorrection = 80, kRegsLoadMma = 96;
static_assert((2 * kRegsSoftmax + kRegsCorrection + kRegsLoadMma) * 128 <= 65536 &&
                  kRegsCorrection <= 128 && kRegsLoadMma <= 128,
              "setmaxnreg split exceeds the launch register pool");

template <int D>
struct Cfg {
  static constexpr int kTileBytes = TileShape<D>::kBytes; // one 128-row tile of Q, K or V
  // K/V ring: kSlots tile slots grouped into kPairs stages.  Stage s holds
  // one V tile in slot (2s - 1) mod kSlots and one K tile in slot 2s.
  static constexpr int kSlots = (D == 128) ? 4 : 8;
  static constexpr int kPairs = kSlots / 2;
  // shared memory, offsets from a 1024-byte aligned base
  static constexpr int kOffQ = 0;
  static constexpr int kOffKV = kOffQ + 2 * kTileBytes;
  static constexpr int kOffBar = kOffKV + kSlots * kTileBytes;
  // kv_full[P], kv_empty[P], q_full[2], s_full[2], p_full[2], stats[2],
  // pv_done[2], drain[1], fin[2][2], q_free[2], xfer_full, xfer_free
  static constexpr int kNumBars = 2 * kPairs + 19;
  static constexpr int kOffScale = kOffBar + kNumBars * 8;      // float [2][128]: alpha per row
  static constexpr int kOffRowSum = kOffScale + 2 * 128 * 4;    // float [2][2][128]: fp32 sum of p
  static constexpr int kOffRowSumP = kOffRowSum + 4 * 128 * 4;  // float [2][2][128]: sum of bf16(p)
  static constexpr int kOffRowMax = kOffRowSumP + 4 * 128 * 4;  // float [2][2][128]
  static constexpr int kOffMisc = kOffRowMax + 4 * 128 * 4;     // tmem base, abort flag
  // One region, 1024-byte aligned, used by one of two instantiations: the
  // trace instantiation's timeline stamps, uint64 [event][block]; or the
  // epilogue's O staging, one [32 rows x 64 columns] bf16 slab per
  // correction warp in the TMA 128-byte swizzle (4 x 4 KB)
  static constexpr int kOffTrace = (kOffMisc + 16 + 1023) / 1024 * 1024;
  static constexpr int kOffStage = kOffTrace;
  static constexpr int kStageBytes = 4 * 32 * 128;
  static constexpr int kTraceBytes = kNumTraceEvents * kMaxTraceBlocks * 8;
  static constexpr int kSmemEnd0 =
      (kOffTrace + (kTraceBytes > kStageBytes ? kTraceBytes : kStageBytes) + 1023) / 1024 * 1024;
  static constexpr int kOnesBytes = (D == 64) ? kSlabBytes : 0;  // one [128 x 64] bf16 atom of ones
  static constexpr int kSmemBytes = kSmemEnd0 + kOnesBytes + 1024;
  // split tail: a received partial (128 rows x D fp32) lands here in the
  // K/V ring, after the sender's own staged one
  static constexpr uint32_t kSplitIn = (uint32_t)kBlockM * D * 4;
  static_assert(2 * kSplitIn <= (uint32_t)(kSlots * kTileBytes), "split-tail partials in the ring");
  static_assert(2 * kBlockM * 4 <= 2 * kTileBytes, "split-tail log-sum-exps in the Q buffer");
  // Row sums on the tensor core (D = 64, where tensor memory has room): the
  // PV GEMM runs with N = D + 16 against [V | ones], so columns D .. D + 15
  // of O_t accumulate the sum of the bf16 probabilities the GEMM consumed,
  // with exactly O's weights and rescales.  The ones are a constant slab of
  // one 64-column atom in shared memory, reached from every V slot through
  // the descriptor's leading-dimension offset.
  static constexpr bool kSumCol = (D == 64);
  static constexpr int kOCols = D + (kSumCol ? 16 : 0);
  static constexpr int kOffOnes = kSmemEnd0;  // 1024-aligned, after the staging / trace region
  static_assert(kOffOnes % 1024 == 0 && kOffOnes - kOffKV < (1 << 18),
                "the ones atom's offset from every V slot fits the descriptor's LBO field");
  // tensor memory columns
  static constexpr uint32_t kTmS0 = 0, kTmS1 = 128, kTmO0 = 256, kTmO1 = 256 + kOCols;
  static constexpr uint32_t kTmemCols = 512;
  static_assert(kSmemBytes <= 227 * 1024, "shared memory budget");
  // a split tail tile's partial result, [sub-tile][row][D] fp32, fits in
  // the K/V ring, and its log-sum-exps [sub-tile][row] in the Q buffer
  static_assert(2 * 128 * D * 4 <= kSlots * kTileBytes && 2 * 128 * 4 <= 2 * kTileBytes,
                "split-tail partial does not fit");
};

// Warp-uniform bounded wait: every lane waits, the warp agrees on the result.
__device__ __forceinline__ bool warp_wait(uint64_t* bar, uint32_t parity, volatile int* abort_flag,
                                          uint64_t budget) {
  const bool ok = mbar_wait(bar, parity, abort_flag, budget);
  return __all_sync(kFull, ok);
}

// The same at cluster scope: for barriers the partner CTA arrives on.
__device__ __forceinline__ bool warp_wait_cluster(uint64_t* bar, uint32_t parity,
                                                  volatile int* abort_flag, uint64_t budget) {
  const bool ok = mbar_wait_cluster(bar, parity, abort_flag, budget);
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

// One work tile.
struct Tile {
  int m0;         // first row of the tile within its row group
  int zkv;        // row group = K/V head index b * H_kv + g
  int split;      // KV split
  int jb;         // first KV block the tile visits
  int n_blocks;   // KV blocks it visits (<= 0: a split with no visible key)
  bool has_sub1;  // rows m0 + 128 .. m0 + 255 exist in the row group
  int pair;       // -1: a whole tile; 0 / 1: the first / second KV half of a
                  // split tail tile, run by cluster ranks 0 / 1
};

// Index of the k-th tile of this CTA, or -1 when it has no k-th tile: round
// k covers list entries [k G, (k + 1) G), taken left to right in even rounds
// and right to left in odd ones.  With a split tail, the last round's
// tail_pairs tiles go one per CTA pair (c / 2), half c % 2 each (`pair`).
template <bool kTail>
__device__ __forceinline__ int tile_of(const AttnParams& p, int k, int& pair) {
  const long long G = gridDim.x;
  const long long c = blockIdx.x;
  const long long base = (long long)k * G;
  pair = -1;
  if (kTail && base >= p.tail_base) {
    if (base != p.tail_base || (c >> 1) >= p.tail_pairs) return -1;
    pair = (int)(c & 1);
    return (int)(p.tail_base + (c >> 1));
  }
  const long long idx = base + ((k & 1) ? (G - 1 - c) : c);
  return idx < (long long)p.num_tiles ? (int)idx : -1;
}

__device__ __forceinline__ Tile decode_tile(const AttnParams& p, int ti, int pair) {
  const int S = p.kv_splits;
  int m, zkv, split;
  if (p.causal) {
    // cost rank first (longest tiles first), then group, then split
    const int per_rank = p.groups * S;
    const int rank = ti / per_rank;
    const int rr = ti - rank * per_rank;
    zkv = rr / S;
    split = rr - zkv * S;
    if (p.lpt_heads > 0) {
      const int nh = p.S_q >> 8;  // query tiles per head
      m = (rank % p.lpt_heads) * nh + (nh - 1 - rank / p.lpt_heads);
    } else {
      m = p.n_m_tiles - 1 - rank;
    }
  } else {
    // group-major, query tiles last to first, then split
    const int per_group = p.n_m_tiles * S;
    zkv = ti / per_group;
    const int rr = ti - zkv * per_group;
    const int mr = rr / S;
    m = p.n_m_tiles - 1 - mr;
    split = rr - mr * S;
  }
  Tile t;
  t.m0 = m * (2 * kBlockM);
  t.zkv = zkv;
  t.split = split;
  // keys any row of this tile may see: row rho is query position rho % S_q,
  // and with the causal mask it sees keys <= its position
  const int R = p.rows_per_group;
  int kv_end = p.S_kv;
  if (p.causal) {
    const int last = min(t.m0 + 2 * kBlockM, R) - 1;
    kv_end = min(p.S_kv, (t.m0 / p.S_q == last / p.S_q) ? last % p.S_q + 1 : p.S_q);
  }
  const int n_total = (kv_end + kBlockN - 1) / kBlockN;
  t.jb = split * p.kv_blocks_per_split;
  t.n_blocks = min(n_total - t.jb, p.kv_blocks_per_split);
  // sub-tile 1 holds rows m0 + 128 .. m0 + 255; when none of them exists
  // (short row groups, e.g. one decoding token per head, or a ragged last
  // tile) every role skips it and the tile costs half
  t.has_sub1 = (t.m0 + kBlockM) < R;
  // a split tail tile: the first ceil(n / 2) blocks, or the rest
  t.pair = pair;
  if (pair >= 0) {
    const int n0 = (t.n_blocks + 1) >> 1;
    if (pair == 0) {
      t.n_blocks = n0;
    } else {
      t.jb += n0;
      t.n_blocks -= n0;
    }
  }
  return t;
}

}  // namespace

// kTail: the instantiation with the split tail (launched only when the tail
// is split; the other one carries none of its code)
template <int D, bool kTrace, bool kTail>
__global__ void __launch_bounds__(kThreads, 1) attn_fwd_kernel(const __grid_constant__ AttnParams p) {
  using C = Cfg<D>;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = align_smem_1024(smem_raw);
  uint8_t* sQ = smem + C::kOffQ;
  uint8_t* sKV = smem + C::kOffKV;
  uint64_t* bars = reinterpret_cast<uint64_t*>(smem + C::kOffBar);
  uint64_t* kv_full = bars;
  uint64_t* kv_empty = bars + C::kPairs;
  uint64_t* q_full = bars + 2 * C::kPairs;
  uint64_t* s_full = q_full + 2;
  uint64_t* p_full = q_full + 4;
  uint64_t* stats = q_full + 6;
  uint64_t* pv_done = q_full + 8;
  uint64_t* drain = q_full + 10;
  uint64_t* fin = q_full + 11;     // [buffer][sub-tile]
  uint64_t* q_free = q_full + 15;
  // split tail: the partner's partial result is in this CTA's shared
  // memory (one arrival with the expected bytes by this CTA, the bytes of
  // the partner's bulk copies), and the partner's receiving region is idle
  // (128 remote arrivals by the partner's correction warpgroup)
  uint64_t* xfer_full = q_full + 17;
  uint64_t* xfer_free = q_full + 18;
  float* sScale = reinterpret_cast<float*>(smem + C::kOffScale);
  float* sRowSum = reinterpret_cast<float*>(smem + C::kOffRowSum);
  float* sRowSumP = reinterpret_cast<float*>(smem + C::kOffRowSumP);
  float* sRowMax = reinterpret_cast<float*>(smem + C::kOffRowMax);
  uint32_t* sTmemBase = reinterpret_cast<uint32_t*>(smem + C::kOffMisc);
  volatile int* sAbort = reinterpret_cast<volatile int*>(smem + C::kOffMisc + 4);
  unsigned long long* sTrace = reinterpret_cast<unsigned long long*>(smem + C::kOffTrace);

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint64_t budget = p.timeout_ns;
  // trace stamps (compiled only into the trace instantiation): the first
  // tile of CTAs below trace_ctas.  The stamp is the SM cycle counter, kept
  // in shared memory while the kernel runs and copied out at the end.  One
  // thread stamps each event (lane 0 of the first warp of a warpgroup, the
  // elected lane of the issuer and the producer), with a plain store.
  const bool trace_cta = kTrace && (int)blockIdx.x < p.trace_ctas;
  auto stamp = [&](bool on, int ev, int j) {
    if constexpr (kTrace) {
      if (on && j < p.trace_blocks)
        sTrace[ev * kMaxTraceBlocks + j] = (unsigned long long)clock64();
    }
  };
  if constexpr (kTrace) {
    for (int i = threadIdx.x; i < kNumTraceEvents * kMaxTraceBlocks; i += kThreads) sTrace[i] = 0;
  }

  if (threadIdx.x == 0) {
    for (int i = 0; i < C::kPairs; ++i) {
      mbar_init(&kv_full[i], 1);
      mbar_init(&kv_empty[i], 1);
    }
    for (int t = 0; t < 2; ++t) {
      mbar_init(&q_full[t], 1);
      mbar_init(&q_free[t], 1);
      mbar_init(&s_full[t], 1);
      // p_full[t]: P_t(j) stored by the softmax (128 arrivals) and O_t
      // rescaled for block j, or for block 0 read out of the previous tile,
      // by the correction warpgroup (128 arrivals)
      mbar_init(&p_full[t], 2 * kBlockM);
      // stats[t]: one phase per block j >= 1 (the rescale factor alpha);
      // fin[.][t]: one phase per tile, the final row sums and max.  Keeping
      // them apart, and fin double-buffered, means no waiter is ever two
      // phases behind.
      mbar_init(&stats[t], kBlockM);
      mbar_init(&fin[t], kBlockM);
      mbar_init(&fin[2 + t], kBlockM);
      mbar_init(&pv_done[t], 1);
    }
    mbar_init(drain, 1);
    mbar_init(xfer_full, 1);
    mbar_init(xfer_free, kBlockM);
    *sAbort = 0;
    fence_mbar_init();
  }
  if constexpr (C::kSumCol) {
    // the constant ones atom of [V | ones] (bf16 1.0 = 0x3f80), written
    // before the tensor core reads it (async proxy: fenced below)
    uint4* ones = reinterpret_cast<uint4*>(smem + C::kOffOnes);
    for (int i = threadIdx.x; i < C::kOnesBytes / 16; i += kThreads)
      ones[i] = make_uint4(0x3f803f80u, 0x3f803f80u, 0x3f803f80u, 0x3f803f80u);
    fence_proxy_async_smem();
  }
  if (warp == 13 && lane == 0) {
    tma_prefetch_map(&p.tm_q);
    tma_prefetch_map(&p.tm_k);
    tma_prefetch_map(&p.tm_v);
    if (!kTrace) tma_prefetch_map(&p.tm_o);
  }
  if (warp == 12) {
    tmem_alloc(sTmemBase, C::kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  // the partner CTA's barriers are initialised before any remote arrival
  if (kTail) cluster_sync_all();
  const uint32_t tmem = *sTmemBase;
  const int wg = warp >> 2;
  const int R = p.rows_per_group;

  if (wg < 2) {
    // ------------------------------------------------------------ softmax
    asm volatile("setmaxnreg.inc.sync.aligned.u32 %0;\n" ::"n"(kRegsSoftmax) : "memory");
    const int t = wg;
    const int r = (warp & 3) * 32 + lane;                 // row within the sub-tile
    const uint32_t tS = tmem + ((uint32_t)((warp & 3) * 32) << 16) + (t ? C::kTmS1 : C::kTmS0);
    const float sl2 = p.scale_log2;
    const uint64_t sl2x2 = f2_pack(sl2, sl2);
    uint32_t nblk = 0;  // blocks of sub-tile t so far: the phase of s_full[t]
    uint32_t ntl = 0;   // tiles with sub-tile t so far: row-stat buffer, fin phase
    bool ok = true;
    for (int k = 0; ok; ++k) {
      int pr = -1;
      const int ti = tile_of<kTail>(p, k, pr);
      if (ti < 0) break;
      const Tile tl = decode_tile(p, ti, pr);
      // (warpgroup 1 has nothing to do when the tile has no sub-tile 1)
      if (tl.n_blocks <= 0 || (t == 1 && !tl.has_sub1)) continue;
      const bool tr = trace_cta && k == 0 && lane == 0 && (warp & 3) == 0;
      const int rho = tl.m0 + t * kBlockM + r;               // row in the row group
      const int pos = rho % p.S_q;                           // its query position
      // smallest query position in this sub-tile (0 if it spans two heads)
      const int sub_first = tl.m0 + t * kBlockM;
      const int min_pos =
          (sub_first / p.S_q == (sub_first + kBlockM - 1) / p.S_q) ? sub_first % p.S_q : 0;
      const int key_limit = p.causal ? min(p.S_kv, pos + 1) : p.S_kv;
      // Two row sums: l_run of the fp32 probabilities (for the LSE), and
      // lp_run of the bf16-rounded probabilities that the PV GEMM actually
      // consumes, so O is normalised by the same weights it was accumulated
      // with (with the sum column the tensor core accumulates the latter in
      // O_t itself, and lp_run stays unused).
      float m_run = -INFINITY;
      float l_run = 0.f;
      float lp_run = 0.f;
      for (int j = 0; j < tl.n_blocks; ++j) {
        if (!warp_wait(&s_full[t], nblk & 1, sAbort, budget)) { ok = false; break; }
        ++nblk;
        tc_fence_after_sync();
        stamp(tr, t ? kEvSm1Wake : kEvSm0Wake, j);
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
        stamp(tr, t ? kEvSm1Loaded : kEvSm0Loaded, j);
        const int kv0 = (tl.jb + j) * kBlockN;
        const bool masked = (kv0 + kBlockN > p.S_kv) || (p.causal && kv0 + kBlockN - 1 > min_pos);
        const int lim = key_limit - kv0;  // columns c < lim are visible to this row
        float m_use = m_run;
        float alpha = 1.f;
        uint64_t l2[2] = {0, 0};                  // packed fp32 partial sums of p
        float lp[4] = {0.f, 0.f, 0.f, 0.f};       // partial sums of bf16(p)
        // The unmasked and masked bodies are separate code paths so the
        // common (unmasked) one carries no per-element predication.
        auto body = [&](auto masked_tag) {
          constexpr bool kMasked = decltype(masked_tag)::value;
          if constexpr (kMasked) {
            // keys this row may not see drop out of the max
#pragma unroll
            for (int c = 0; c < 128; ++c)
              if (c >= lim) s[c] = f2u(-INFINITY);
          }
          // row max of the raw scores (4 independent chains of 3-input max)
          float mx[4] = {-INFINITY, -INFINITY, -INFINITY, -INFINITY};
#pragma unroll
          for (int c = 0; c < 128; c += 8) {
#pragma unroll
            for (int i = 0; i < 4; ++i) mx[i] = max3(mx[i], u2f(s[c + 2 * i]), u2f(s[c + 2 * i + 1]));
          }
          const float mblk = fmaxf(fmaxf(mx[0], mx[1]), fmaxf(mx[2], mx[3]));
          // scale_log2 > 0 (a negative scale negates S in the GEMM instead),
          // so the max of the scaled scores is the scaled max; a row whose
          // keys are all masked here leaves the running max unchanged
          const float m_new = (mblk == -INFINITY) ? m_run : fmaxf(m_run, mblk * sl2);
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
          // A masked score is -inf, and so is its x below (scale_log2 > 0),
          // so its p is exactly 0 -- unless the row has seen no key yet
          // (m_use = -inf, only possible inside one KV split): then subtract
          // 0 instead, which keeps x = -inf rather than -inf + inf.
          float m_sub = m_use;
          if constexpr (kMasked) m_sub = (m_use == -INFINITY) ? 0.f : m_use;
          const uint64_t neg_m2 = f2_pack(-m_sub, -m_sub);
#pragma unroll
          for (int ch = 0; ch < 8; ++ch) {
            uint32_t pk[8];
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const int c = ch * 16 + 2 * i;
              // x = s * scale * log2(e) - m, two lanes per instruction
              float x0, x1;
              f2_unpack(f2_fma(f2_pack(u2f(s[c]), u2f(s[c + 1])), sl2x2, neg_m2), x0, x1);
              float p0, p1;
              if (!kMasked && i >= 8 - kPolyPairs) {
                exp2_poly_x2(x0, x1, p0, p1);
              } else {
                p0 = ex2_approx(x0);
                p1 = ex2_approx(x1);
              }
              l2[i & 1] = f2_add(l2[i & 1], f2_pack(p0, p1));
              pk[i] = pack_bf16x2(p0, p1);
              if constexpr (!C::kSumCol)
                add_bf16x2_to_f32(lp[(2 * i) & 3], lp[(2 * i + 1) & 3], pk[i]);
            }
            tmem_st_x8(tS + ch * 8, pk);
          }
        };
        if (masked)
          body(std::true_type{});
        else
          body(std::false_type{});
        float la, lb;
        f2_unpack(f2_add(l2[0], l2[1]), la, lb);
        l_run = l_run * alpha + (la + lb);
        lp_run = lp_run * alpha + ((lp[0] + lp[1]) + (lp[2] + lp[3]));
        tmem_st_wait();
        tc_fence_before_sync();
        stamp(tr, t ? kEvSm1Done : kEvSm0Done, j);
        bool signal = true;
        if constexpr (kTrace) signal = !(t == 0 && j == p.fault_drop_block);
        if (signal) mbar_arrive(&p_full[t]);
        m_run = m_use;
      }
      if (!ok) break;
      const int sb = ((ntl & 1) * 2 + t) * kBlockM + r;  // row-stat slot [buffer][sub-tile][row]
      sRowSum[sb] = l_run;
      sRowSumP[sb] = lp_run;
      sRowMax[sb] = m_run;
      mbar_arrive(&fin[(ntl & 1) * 2 + t]);
      ++ntl;
    }
  } else if (wg == 2) {
    // ------------------------------------------------------------ correction + epilogue
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kRegsCorrection) : "memory");
    const int q4 = warp & 3;
    const int r = q4 * 32 + lane;
    const uint32_t lane_base = (uint32_t)(q4 * 32) << 16;
    uint32_t nst[2] = {0, 0};  // alpha phases consumed, per sub-tile (stats[t])
    uint32_t ntl[2] = {0, 0};  // tiles finished, per sub-tile (fin, pv_done)
    bool ok = true;
    // Advances k to the next tile with work and decodes it; a split tile
    // with no visible key on the way gets its empty partial result here
    // (weight 0 in the merge).  A half of a split tail tile is always
    // returned: even with no KV block it owes its partner a partial result.
    auto next_work = [&](int& k, Tile& tl) -> bool {
      for (;; ++k) {
        int pr = -1;
        const int ti = tile_of<kTail>(p, k, pr);
        if (ti < 0) return false;
        tl = decode_tile(p, ti, pr);
        if (tl.n_blocks > 0 || tl.pair >= 0) return true;
#pragma unroll 1
        for (int h = 0; h < 2; ++h) {
          const int rho = tl.m0 + h * kBlockM + r;
          if (rho < R) {
            const size_t row = (size_t)tl.split * p.total_rows + (size_t)tl.zkv * R + rho;
            p.lse_part[row] = -INFINITY;
            float4* dst = reinterpret_cast<float4*>(p.o_part + row * D);
            for (int c = 0; c < D / 4; ++c) dst[c] = make_float4(0.f, 0.f, 0.f, 0.f);
          }
        }
      }
    };
    int k = 0;
    Tile cur;
    bool have = next_work(k, cur);
    // block 0 of the first tile needs nothing from this warpgroup
    if (have) {
      mbar_arrive(&p_full[0]);
      if (cur.has_sub1) mbar_arrive(&p_full[1]);
    }
    while (have) {
      const int n_sub = cur.has_sub1 ? 2 : 1;
      const bool tr = trace_cta && k == 0 && lane == 0 && (warp & 3) == 0;
      // Block j >= 1: the softmax's alpha arrives on stats[t]; it is
      // published after the softmax saw S_t(j), whose commit follows
      // PV_t(j-1), so O_t already holds every earlier block.
      for (int j = 1; j < cur.n_blocks && ok; ++j) {
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (t >= n_sub) break;
          if (!warp_wait(&stats[t], nst[t] & 1, sAbort, budget)) { ok = false; break; }
          ++nst[t];
          const float alpha = sScale[t * kBlockM + r];
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
            if constexpr (C::kSumCol) {
              uint32_t o[16];
              tmem_ld_x16(tO + D, o);
              tmem_ld_wait();
              reg_after_wait(o);
#pragma unroll
              for (int i = 0; i < 16; ++i) o[i] = f2u(u2f(o[i]) * alpha);
              tmem_st_x16(tO + D, o);
            }
            tmem_st_wait();
          }
          tc_fence_before_sync();
          stamp(tr, t ? kEvCorr1 : kEvCorr0, j);
          mbar_arrive(&p_full[t]);
        }
      }
      if (!ok) break;
      int k_next = k + 1;
      Tile nxt;
      const bool have_next = next_work(k_next, nxt);
      // Split tail tile (the CTA's last): the two KV halves exchange
      // partial results.  With two sub-tiles each CTA writes one (the first
      // CTA sub-tile 0, the second sub-tile 1) and sends the other one's
      // partial to its partner; with one sub-tile the second CTA sends it and
      // the first writes it.  A partial is O_t normalised by its half's own
      // sum (fp32, [row][D], the 16-byte pieces of a row XOR-swizzled by
      // row % 8) and the half's base-2 log-sum-exp; it is staged at the
      // start of the sender's own idle K/V ring (and Q buffer) and lands at
      // C::kSplitIn into the receiver's (and at row 128 of its Q buffer), by
      // one bulk copy each, completing as transaction bytes on the
      // receiver's xfer_full.  A half with no KV block (not produced by the
      // launch's split rule, which needs long tiles, but handled) sends zeros
      // and a log-sum-exp of -inf (weight 0 in the merge).
      bool split_done = false;  // the exchange below took this tile's waits
      int t_write = -1;         // the sub-tile this CTA writes
      float sl[2] = {0.f, 0.f}, slp[2] = {0.f, 0.f}, sm[2] = {0.f, 0.f};
      if (cur.pair >= 0) {
        const uint32_t peer = cluster_ctarank() ^ 1u;
        const bool sym = cur.has_sub1;
        const int t_send = sym ? 1 - cur.pair : (cur.pair == 1 ? 0 : -1);
        t_write = sym ? cur.pair : (cur.pair == 0 ? 0 : -1);
        // every GEMM of the tile done: the ring and the Q buffer are idle,
        // and the row statistics final
        if (cur.n_blocks > 0) {
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (t >= n_sub) break;
            const int buf = (int)(ntl[t] & 1);
            if (!warp_wait(&fin[buf * 2 + t], (ntl[t] >> 1) & 1, sAbort, budget) ||
                !warp_wait(&pv_done[t], ntl[t] & 1, sAbort, budget)) {
              ok = false;
              break;
            }
            ++ntl[t];
            const int sb = (buf * 2 + t) * kBlockM + r;
            sl[t] = sRowSum[sb];
            slp[t] = sRowSumP[sb];
            sm[t] = sRowMax[sb];
          }
          tc_fence_after_sync();
          if constexpr (C::kSumCol) {
            // the sum of the bf16 probabilities, from O_t's sum columns
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              if (t < n_sub && ok) {
                uint32_t v = tmem_ld_x1(tmem + lane_base + (t ? C::kTmO1 : C::kTmO0) + D);
                tmem_ld_wait();
                asm volatile("" : "+r"(v));
                slp[t] = u2f(v);
              }
            }
          }
        }
        if (ok && t_send >= 0) {
          const bool empty = !(slp[t_send] > 0.f);
          const float inv_l = empty ? 0.f : 1.f / slp[t_send];
          reinterpret_cast<float*>(sQ)[r] = empty ? -INFINITY : sm[t_send] + log2f(sl[t_send]);
          const uint32_t row = smem_u32(sKV) + (uint32_t)(r * D * 4);
          const uint32_t tO = tmem + lane_base + (t_send ? C::kTmO1 : C::kTmO0);
#pragma unroll 1
          for (int ch = 0; ch < D / 16; ++ch) {
            uint32_t o[16];
            if (cur.n_blocks > 0) {
              tmem_ld_x16(tO + ch * 16, o);
              tmem_ld_wait();
              reg_after_wait(o);
            } else {
#pragma unroll
              for (int i = 0; i < 16; ++i) o[i] = 0u;
            }
#pragma unroll
            for (int qd = 0; qd < 4; ++qd) {
              const int cc = ch * 4 + qd;  // 16-byte piece of the row
              st_shared_v4(row + 16u * (uint32_t)(cc ^ (r & 7)), f2u(u2f(o[qd * 4 + 0]) * inv_l),
                           f2u(u2f(o[qd * 4 + 1]) * inv_l), f2u(u2f(o[qd * 4 + 2]) * inv_l),
                           f2u(u2f(o[qd * 4 + 3]) * inv_l));
            }
          }
          fence_proxy_async_smem();            // the staged rows before the bulk copy reads them
        }
        if (ok && t_write >= 0) {
          // this CTA's receiving region is idle: arm xfer_full with the bytes
          // to come and tell the partner
          if (threadIdx.x == 2 * 128)
            mbar_arrive_expect_tx(xfer_full, (uint32_t)(kBlockM * (D + 1) * 4));
          mbar_arrive_remote(mapa_shared(smem_u32(xfer_free), peer));
        }
        // every thread of the warpgroup has staged its row (and a wait that
        // ran out in any of them stops all)
        if (barrier_or(kBarCorrection, 128, !ok)) { ok = false; break; }
        if (t_send >= 0) {
          // the partner's receiving region is idle: the two copies (the test
          // of the hand-off's timeout path withholds them)
          if (!warp_wait_cluster(xfer_free, 0, sAbort, budget)) { ok = false; break; }
          if (threadIdx.x == 2 * 128 && !p.fault_drop_xfer) {
            const uint32_t bar = mapa_shared(smem_u32(xfer_full), peer);
            bulk_copy_to_cluster(mapa_shared(smem_u32(sKV) + C::kSplitIn, peer), smem_u32(sKV),
                                 (uint32_t)(kBlockM * D * 4), bar);
            bulk_copy_to_cluster(mapa_shared(smem_u32(sQ) + kBlockM * 4, peer), smem_u32(sQ),
                                 (uint32_t)(kBlockM * 4), bar);
          }
        }
        if (t_write < 0) break;  // the tail round is the last: no tile follows
        if (!warp_wait_cluster(xfer_full, 0, sAbort, budget)) { ok = false; break; }
        split_done = true;
      }
#pragma unroll
      for (int t = 0; t < 2; ++t) {
        if (t < n_sub) {
          // (a split tail tile: the partner writes the other sub-tile)
          if (split_done && t != t_write) continue;
          float l, m, lp;
          if (split_done) {
            l = sl[t];
            m = sm[t];
            lp = slp[t];
          } else {
            const int buf = (int)(ntl[t] & 1);
            if (!warp_wait(&fin[buf * 2 + t], (ntl[t] >> 1) & 1, sAbort, budget)) { ok = false; break; }
            if (!warp_wait(&pv_done[t], ntl[t] & 1, sAbort, budget)) { ok = false; break; }
            ++ntl[t];
            tc_fence_after_sync();
            const int sb = (buf * 2 + t) * kBlockM + r;
            l = sRowSum[sb];
            m = sRowMax[sb];
            lp = sRowSumP[sb];
            if constexpr (C::kSumCol) {
              // the sum of the bf16 probabilities, from O_t's sum columns
              uint32_t v = tmem_ld_x1(tmem + lane_base + (t ? C::kTmO1 : C::kTmO0) + D);
              tmem_ld_wait();
              asm volatile("" : "+r"(v));
              lp = u2f(v);
            }
          }
          stamp(tr, kEvEpilogue, t);
          // a row with no visible key (possible only within one KV split)
          // has l = 0: its partial result is O = 0, LSE = -inf
          const bool empty = !(lp > 0.f);
          const float inv_l = empty ? 0.f : 1.f / lp;
          const float lse_row = empty ? -INFINITY : (m + log2f(l)) * 0.69314718055994530942f;
          const uint32_t tO = tmem + lane_base + (t ? C::kTmO1 : C::kTmO0);
          const int rho = cur.m0 + t * kBlockM + r;
          // The tensor-memory loads are warp-wide; only the stores depend on
          // whether the row exists.
          //
          // A split tail tile's written sub-tile merges this half with the
          // partner's partial (received at C::kSplitIn) by the two halves'
          // log-sum-exps: O = w0 O_own + w1 O_partner.  Otherwise w0 = 1 / l,
          // w1 = 0.
          const bool merge = split_done;
          float w0 = inv_l, w1 = 0.f, lse_out = lse_row;
          uint32_t prow = 0;
          if (merge) {
            prow = smem_u32(sKV) + C::kSplitIn + (uint32_t)(r * D * 4);
            const float l1 = reinterpret_cast<const float*>(sQ)[kBlockM + r];
            const float l0 = empty ? -INFINITY : m + log2f(l);
            const float mx = fmaxf(l0, l1);
            w0 = 0.f;
            lse_out = -INFINITY;
            if (mx > -INFINITY) {
              const float e0 = ex2_approx(l0 - mx), e1 = ex2_approx(l1 - mx);
              const float inv = 1.f / (e0 + e1);
              w0 = e0 * inv * inv_l;  // this half's O is unnormalised in tensor memory
              w1 = e1 * inv;
              lse_out = (mx + log2f(e0 + e1)) * 0.69314718055994530942f;
            }
          }
          if (p.o_part != nullptr) {
            // split-KV partial: fp32 O normalised within the split, and its LSE
            const size_t row = (size_t)cur.split * p.total_rows + (size_t)cur.zkv * R + rho;
            float4* dst = reinterpret_cast<float4*>(p.o_part + row * D);
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) {
              uint32_t o[32];
              tmem_ld_x32(tO + ch * 32, o);
              tmem_ld_wait();
              reg_after_wait(o);
              if (rho < R) {
#pragma unroll
                for (int qd = 0; qd < 8; ++qd)
                  dst[ch * 8 + qd] =
                      make_float4(u2f(o[qd * 4 + 0]) * inv_l, u2f(o[qd * 4 + 1]) * inv_l,
                                  u2f(o[qd * 4 + 2]) * inv_l, u2f(o[qd * 4 + 3]) * inv_l);
              }
            }
            if (rho < R) p.lse_part[row] = lse_row;
          } else if constexpr (!kTrace) {
            // bf16 O through shared memory and TMA: per 64-column slab, each
            // warp writes its 32 rows into its own staging slab (128-byte
            // swizzle: 16-byte piece c of row r at piece c ^ (r % 8)), then
            // one lane stores the slab with one TMA copy (rows past R are
            // clipped by the tensor map).  The slab is reused once the
            // previous copy has read it.
            uint8_t* stage = smem + C::kOffStage + q4 * 4096;
            const uint32_t srow = smem_u32(stage) + (uint32_t)lane * 128u;
#pragma unroll 1
            for (int h = 0; h < D / 64; ++h) {
              if (lane == 0) tma_store_wait_read<0>();
              __syncwarp();
#pragma unroll 1
              for (int q16 = 0; q16 < 4; ++q16) {
                uint32_t o[16];
                tmem_ld_x16(tO + h * 64 + q16 * 16, o);
                tmem_ld_wait();
                reg_after_wait(o);
                if (merge) {
#pragma unroll
                  for (int qd = 0; qd < 4; ++qd) {
                    const int cc = h * 16 + q16 * 4 + qd;  // 16-byte fp32 piece of the partner's row
                    const float4 pv = ld_shared_v4f(prow + 16u * (uint32_t)(cc ^ (lane & 7)));
                    // w1 = 0 (an empty partner half) must not meet its unset values
                    const float a[4] = {pv.x, pv.y, pv.z, pv.w};
#pragma unroll
                    for (int e = 0; e < 4; ++e) {
                      // (w0 = 0: an empty own half, whose O was never written)
                      const float own = w0 != 0.f ? u2f(o[qd * 4 + e]) * w0 : 0.f;
                      o[qd * 4 + e] = f2u(w1 > 0.f ? fmaf(w1, a[e], own) : own);
                    }
                  }
                } else {
#pragma unroll
                  for (int i = 0; i < 16; ++i) o[i] = f2u(u2f(o[i]) * w0);
                }
#pragma unroll
                for (int qd = 0; qd < 2; ++qd) {
                  const int c = q16 * 2 + qd;  // 16-byte piece of the slab row
                  st_shared_v4(srow + 16u * (uint32_t)(c ^ (lane & 7)),
                               pack_bf16x2(u2f(o[qd * 8 + 0]), u2f(o[qd * 8 + 1])),
                               pack_bf16x2(u2f(o[qd * 8 + 2]), u2f(o[qd * 8 + 3])),
                               pack_bf16x2(u2f(o[qd * 8 + 4]), u2f(o[qd * 8 + 5])),
                               pack_bf16x2(u2f(o[qd * 8 + 6]), u2f(o[qd * 8 + 7])));
                }
              }
              fence_proxy_async_smem();
              __syncwarp();
              if (lane == 0) {
                tma_store_3d(&p.tm_o, stage, h * 64, cur.m0 + t * kBlockM + q4 * 32, cur.zkv);
                tma_store_commit();
              }
            }
            if (rho < R) p.lse[(size_t)cur.zkv * R + rho] = lse_out;
          } else {
            // (trace instantiation, whose timeline stamps use the staging
            // region, and which never splits a tail) bf16 O straight from
            // registers: each thread writes its own row in 16-byte pieces
            uint4* dst = reinterpret_cast<uint4*>(static_cast<uint16_t*>(p.o) +
                                                  ((size_t)cur.zkv * R + rho) * D);
#pragma unroll
            for (int ch = 0; ch < D / 32; ++ch) {
              uint32_t o[32];
              tmem_ld_x32(tO + ch * 32, o);
              tmem_ld_wait();
              reg_after_wait(o);
              if (rho < R) {
#pragma unroll
                for (int qd = 0; qd < 4; ++qd) {
                  uint4 val;
                  val.x = pack_bf16x2(u2f(o[qd * 8 + 0]) * inv_l, u2f(o[qd * 8 + 1]) * inv_l);
                  val.y = pack_bf16x2(u2f(o[qd * 8 + 2]) * inv_l, u2f(o[qd * 8 + 3]) * inv_l);
                  val.z = pack_bf16x2(u2f(o[qd * 8 + 4]) * inv_l, u2f(o[qd * 8 + 5]) * inv_l);
                  val.w = pack_bf16x2(u2f(o[qd * 8 + 6]) * inv_l, u2f(o[qd * 8 + 7]) * inv_l);
                  dst[ch * 4 + qd] = val;
                }
              }
            }
            if (rho < R) p.lse[(size_t)cur.zkv * R + rho] = lse_row;
          }
          tc_fence_before_sync();
        }
        // O_t has been read out and the row statistics are consumed: block 0
        // of the next tile may start on sub-tile t
        if (have_next && (t == 0 || nxt.has_sub1)) mbar_arrive(&p_full[t]);
      }
      if (!ok) break;
      stamp(tr, kEvEnd, 0);
      k = k_next;
      cur = nxt;
      have = have_next;
    }
  } else {
    // ------------------------------------------------------------ warpgroup 3
    asm volatile("setmaxnreg.dec.sync.aligned.u32 %0;\n" ::"n"(kRegsLoadMma) : "memory");
    if (warp == 12) {
      // tensor-core issuer: the whole warp runs the loop and its waits, with
      // all values warp-uniform; one elected lane issues every tcgen05.mma
      // and tcgen05.commit (they act for the issuing thread alone, and a
      // commit tracks the operations of the thread that executes it)
      const bool leader = elect_one();
      const uint64_t dq[2] = {kmajor_tile_desc(smem_u32(sQ)),
                              kmajor_tile_desc(smem_u32(sQ + C::kTileBytes))};
      const uint64_t dk0 = kmajor_tile_desc(smem_u32(sKV));
      const uint64_t dv0 = mnmajor_tile_desc<D>(smem_u32(sKV));
      constexpr uint64_t kSlotDesc = C::kTileBytes >> 4;  // start-address step per ring slot
      const uint32_t tS[2] = {tmem + C::kTmS0, tmem + C::kTmS1};
      // a negative scale: S = -Q K^T (the GEMM negates A), and the softmax
      // applies |scale|
      const bool neg_s = p.neg_scores != 0;
      const uint32_t tO[2] = {tmem + C::kTmO0, tmem + C::kTmO1};
      // The CTA's KV blocks form one stream over its tiles, b = 0, 1, ...
      // Ring entry 0 holds K of stream block 0; entry e >= 1 holds V of block
      // e - 1 and K of block e (if any), both used in the iteration of block
      // e - 1: one wait and one release per block.  The entry holding a
      // tile's first K is released once that tile's first S GEMMs are issued.
      uint32_t e_next = 0;       // next ring entry to wait for
      uint32_t nq[2] = {0, 0};   // tiles so far per sub-tile: the phase of q_full[t]
      uint32_t nb[2] = {0, 0};   // blocks so far per sub-tile: the phase of p_full[t]
      bool ok = true;
      for (int k = 0; ok; ++k) {
        int pr = -1;
        const int ti = tile_of<kTail>(p, k, pr);
        if (ti < 0) break;
        const Tile tl = decode_tile(p, ti, pr);
        const int n = tl.n_blocks;
        if (n <= 0) continue;
        const bool tr = trace_cta && k == 0;
        const int n_sub = tl.has_sub1 ? 2 : 1;
        // S_t(0) = Q_t K_0^T.  K_0 sits in entry e_next - 1, already waited
        // for in the previous tile's last iteration (entry 0 for the first).
        if (e_next == 0) {
          if (!warp_wait(&kv_full[0], 0, sAbort, budget)) { ok = false; break; }
          e_next = 1;
        }
        const uint32_t s_k0 = (e_next - 1) % C::kPairs;
        const uint64_t dk_first = dk0 + (uint64_t)(2 * s_k0) * kSlotDesc;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (t >= n_sub) break;
          if (!warp_wait(&q_full[t], nq[t] & 1, sAbort, budget)) { ok = false; break; }
          tc_fence_after_sync();
          if (leader) {
            issue_qk_gemm<D>(tS[t], dq[t], dk_first, neg_s);
            tc_commit(&s_full[t]);
            if (n == 1) tc_commit(&q_free[t]);  // the tile's last read of Q_t
          }
          stamp(tr && leader, t ? kEvMmaS1 : kEvMmaS0, 0);
        }
        if (!ok) break;
        if (leader) tc_commit(&kv_empty[s_k0]);
        for (int j = 0; j < n; ++j) {
          const bool more = (j + 1) < n;
          // entry e_next: V_j and the next K (K_{j+1}, or the next tile's
          // K_0).  Its loads were issued long before; waiting here, while the
          // softmax is still busy, keeps it off the path from "P ready" to
          // the GEMMs.
          const uint32_t st = e_next % C::kPairs;
          if (!warp_wait(&kv_full[st], (e_next / C::kPairs) & 1, sAbort, budget)) {
            ok = false;
            break;
          }
          ++e_next;
          const uint32_t vslot = (2 * st + C::kSlots - 1) % C::kSlots;
          uint64_t dv = dv0 + (uint64_t)vslot * kSlotDesc;
          if constexpr (C::kSumCol) {
            // [V | ones]: the ones atom sits at a fixed place above the ring,
            // so each V slot has its own leading offset to it
            const uint32_t va = smem_u32(sKV) + vslot * C::kTileBytes;
            dv = make_smem_desc_sw128(va, smem_u32(smem + C::kOffOnes) - va, 1024);
          }
          const uint64_t dk = dk0 + (uint64_t)(2 * st) * kSlotDesc;
          // per sub-tile: O_t += P_t V_j, then S_t = Q_t K_{j+1}^T
#pragma unroll
          for (int t = 0; t < 2; ++t) {
            if (t >= n_sub) break;
            if (!warp_wait(&p_full[t], (nb[t] + j) & 1, sAbort, budget)) { ok = false; break; }
            tc_fence_after_sync();
            stamp(tr && leader, t ? kEvMmaPV1Begin : kEvMmaPV0Begin, j);
            if (leader) {
              issue_pv_gemm<D, C::kOCols>(tO[t], tS[t], dv, j > 0);
              if (!more) tc_commit(&pv_done[t]);  // the epilogue waits for the last PV only
            }
            stamp(tr && leader, t ? kEvMmaPV1 : kEvMmaPV0, j);
            if (more) {
              stamp(tr && leader, t ? kEvMmaS1Begin : kEvMmaS0Begin, j + 1);
              if (leader) {
                issue_qk_gemm<D>(tS[t], dq[t], dk, neg_s);
                tc_commit(&s_full[t]);
                if (j + 2 == n) tc_commit(&q_free[t]);
              }
              stamp(tr && leader, t ? kEvMmaS1 : kEvMmaS0, j + 1);
            }
          }
          if (!ok) break;
          // release the entry last, off the critical path (after the last
          // block its K belongs to the next tile: released there)
          if (more && leader) tc_commit(&kv_empty[st]);
        }
        if (!ok) break;
#pragma unroll
        for (int t = 0; t < 2; ++t) {
          if (t >= n_sub) break;
          ++nq[t];
          nb[t] += n;
        }
      }
      // let every tensor-core op the leader issued finish before teardown
      if (leader) {
        tc_commit(drain);
        drain_wait(drain, 0, budget);
      }
      __syncwarp();
    } else if (warp == 13) {
      // TMA producer: the whole warp runs the loop and its waits; one
      // elected lane issues the copies and the expect-tx arrivals
      const bool leader = elect_one();
      const uint64_t pol_q = l2_policy_evict_first();
      const uint64_t pol_kv = l2_policy_evict_last();
      uint32_t e = 0;            // ring entries issued so far
      uint32_t nq[2] = {0, 0};   // Q_t loads issued so far
      // V tile owed to the next entry: row group (-1: none), first key, and
      // for the trace its block index and whether its tile is traced
      int v_zkv = -1, v_row = 0, v_j = 0;
      bool v_tr = false;
      // Issues ring entry e: the owed V tile, if any, and K rows k_row.. of
      // group k_zkv, if k_zkv >= 0 (see the tensor-core issuer for the layout).
      auto issue_entry = [&](int k_zkv, int k_row) -> bool {
        const uint32_t st = e % C::kPairs;
        const uint32_t round = e / C::kPairs;
        if (round > 0 && !warp_wait(&kv_empty[st], (round - 1) & 1, sAbort, budget)) return false;
        if (leader) {
          const uint32_t bytes =
              (v_zkv >= 0 ? C::kTileBytes : 0) + (k_zkv >= 0 ? C::kTileBytes : 0);
          mbar_arrive_expect_tx(&kv_full[st], bytes);
          if (v_zkv >= 0) {
            tma_load_tile<D>(sKV + ((2 * st + C::kSlots - 1) % C::kSlots) * C::kTileBytes,
                             &p.tm_v, &kv_full[st], v_row, v_zkv, pol_kv);
            stamp(v_tr, kEvLoadV, v_j);
          }
          if (k_zkv >= 0)
            tma_load_tile<D>(sKV + 2 * st * C::kTileBytes, &p.tm_k, &kv_full[st], k_row, k_zkv,
                             pol_kv);
        }
        ++e;
        return true;
      };
      bool ok = true;
      for (int k = 0; ok; ++k) {
        int pr = -1;
        const int ti = tile_of<kTail>(p, k, pr);
        if (ti < 0) break;
        const Tile tl = decode_tile(p, ti, pr);
        if (tl.n_blocks <= 0) continue;
        const bool tr = trace_cta && k == 0;
        for (int j = 0; j < tl.n_blocks; ++j) {
          const int row = (tl.jb + j) * kBlockN;
          if (!issue_entry(tl.zkv, row)) { ok = false; break; }
          stamp(tr && leader, kEvLoadK, j);
          v_zkv = tl.zkv;
          v_row = row;
          v_j = j;
          v_tr = tr;
          if (j == 0) {
            // Q of this tile, after the entry with its K_0 (which also holds
            // the previous tile's last V, needed first)
#pragma unroll
            for (int t = 0; t < 2; ++t) {
              if (t == 1 && !tl.has_sub1) break;
              // the previous tile's last S_t GEMM must be done reading Q_t
              if (nq[t] > 0 && !warp_wait(&q_free[t], (nq[t] - 1) & 1, sAbort, budget)) {
                ok = false;
                break;
              }
              if (leader) {
                mbar_arrive_expect_tx(&q_full[t], C::kTileBytes);
                tma_load_tile<D>(sQ + t * C::kTileBytes, &p.tm_q, &q_full[t],
                                 tl.m0 + t * kBlockM, tl.zkv, pol_q);
              }
              ++nq[t];
            }
            if (!ok) break;
          }
        }
      }
      // the last V closes the stream
      if (ok && v_zkv >= 0) issue_entry(-1, 0);
      // every copy issued must land before the CTA exits (on the normal path
      // these phases completed long ago)
      if (leader) {
#pragma unroll
        for (int t = 0; t < 2; ++t)
          if (nq[t] > 0) drain_wait(&q_full[t], (nq[t] - 1) & 1, budget);
        const uint32_t first = e > (uint32_t)C::kPairs ? e - C::kPairs : 0;
        for (uint32_t idx = first; idx < e; ++idx)
          drain_wait(&kv_full[idx % C::kPairs], (idx / C::kPairs) & 1, budget);
      }
    }
    __syncwarp();
  }

  // ------------------------------------------------------------ teardown
  // the epilogue's TMA stores are complete before the CTA exits
  if (!kTrace && wg == 2 && lane == 0) tma_store_wait_all();
  tc_fence_before_sync();
  __syncthreads();
  tc_fence_after_sync();
  // neither CTA of a pair exits while the other may still touch its shared
  // memory (every role of both reaches this point, all waits being bounded)
  if (kTail) cluster_sync_all();
  if (warp == 12) tmem_dealloc(tmem, C::kTmemCols);
  if (threadIdx.x == 0 && *sAbort) atomicCAS(&g_attn_status, 0, (int)ATTN_ERR_TIMEOUT);
  if constexpr (kTrace) {
    if (trace_cta) {
      for (int i = threadIdx.x; i < kNumTraceEvents * p.trace_blocks; i += kThreads) {
        const int ev = i / p.trace_blocks, j = i - ev * p.trace_blocks;
        const unsigned long long v = sTrace[ev * kMaxTraceBlocks + j];
        if (v != 0) p.trace[((size_t)blockIdx.x * kNumTraceEvents + ev) * p.trace_blocks + j] = v;
      }
    }
  }
}

namespace {

std::mutex g_launch_mu;
bool g_attr_set[2][2][2][64] = {};  // [D == 128][trace][split tail][device]
int g_sm_count[64] = {};
int g_tail_clusters[2][64] = {};    // [D == 128][device]: resident clusters of two, + 1 (0: unknown)

// The SM count of the current device and, once per instantiation and
// device, the kernel's shared-memory attribute.
template <int D, bool kTrace, bool kTail>
cudaError_t prepare(int* sms) {
  int dev = 0;
  cudaError_t err = cudaGetDevice(&dev);
  if (err != cudaSuccess) return err;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  std::lock_guard<std::mutex> lk(g_launch_mu);
  bool& attr_set = g_attr_set[D == 128][kTrace][kTail][dev];
  if (!attr_set) {
    err = cudaFuncSetAttribute(attn_fwd_kernel<D, kTrace, kTail>,
                               cudaFuncAttributeMaxDynamicSharedMemorySize, Cfg<D>::kSmemBytes);
    if (err != cudaSuccess) return err;
    attr_set = true;
  }
  if (g_sm_count[dev] == 0) {
    err = cudaDeviceGetAttribute(&g_sm_count[dev], cudaDevAttrMultiProcessorCount, dev);
    if (err != cudaSuccess) return err;
  }
  *sms = g_sm_count[dev];
  return cudaSuccess;
}

// Launch configuration of the split-tail instantiation: clusters of two.
template <int D>
cudaLaunchConfig_t tail_config(int grid, cudaStream_t stream, cudaLaunchAttribute* attr) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = Cfg<D>::kSmemBytes;
  cfg.stream = stream;
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cfg;
}

// How many clusters of two CTAs of the split-tail instantiation can be
// resident at once on the current device (queried once per device).
template <int D>
int resident_tail_clusters(int grid) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) return 0;
  int sms = 0;
  if (prepare<D, false, true>(&sms) != cudaSuccess) return 0;
  std::lock_guard<std::mutex> lk(g_launch_mu);
  int& cached = g_tail_clusters[D == 128][dev];
  if (cached == 0) {
    cudaLaunchAttribute attr[1];
    cudaLaunchConfig_t cfg = tail_config<D>(grid, nullptr, attr);
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, attn_fwd_kernel<D, false, true>, &cfg) != cudaSuccess) {
      cudaGetLastError();  // a failed query leaves a (non-sticky) error behind: clear it
      n = 0;
    }
    cached = n + 1;
  }
  return cached - 1;
}

// The split-tail plan of a launch of `grid` persistent CTAs: when the last
// round of whole tiles would leave more than half of the CTAs idle, each of
// its tiles goes to a pair of CTAs instead (half of its KV blocks each), so
// the round takes about half a tile.  Non-causal tiles only (with the causal
// mask the last round holds the shortest tiles), long ones, only when the
// tiles write O and LSE (a split-KV launch, even of one split, writes
// partials for its merge), and only when every cluster of two of the grid
// can be resident at once (else the extra clusters would wait for whole
// persistent CTAs to finish).  Sets tail_base / tail_pairs (0 = no split).
template <int D>
void plan_tail(AttnParams* q, int grid) {
  q->tail_base = 0;
  q->tail_pairs = 0;
  const int kv_blocks = (q->S_kv + kBlockN - 1) / kBlockN;
  if (q->kv_splits != 1 || q->o_part != nullptr || q->causal || kv_blocks < kSplitTailMinBlocks ||
      q->num_tiles <= grid || grid % 2 != 0)
    return;
  const int rounds = q->num_tiles / grid;
  const int tail = q->num_tiles - rounds * grid;
  if (tail <= 0 || tail > grid / 2) return;
  if (resident_tail_clusters<D>(grid) < grid / 2) return;
  q->tail_base = rounds * grid;
  q->tail_pairs = tail;
}

template <int D, bool kTrace>
cudaError_t launch_d(const AttnParams& p, cudaStream_t stream) {
  int sms = 0;
  cudaError_t err = prepare<D, kTrace, false>(&sms);
  if (err != cudaSuccess) return err;
  if (p.num_tiles <= 0 || sms <= 0) return cudaErrorInvalidValue;
  // persistent grid: one CTA per SM (the kernel's shared memory allows no
  // second), fewer when there are fewer tiles
  const int grid = p.num_tiles < sms ? p.num_tiles : sms;
  AttnParams q = p;
  q.tail_base = 0;
  q.tail_pairs = 0;
  if constexpr (!kTrace) {
    plan_tail<D>(&q, grid);
    if (q.tail_pairs > 0) {
      err = prepare<D, false, true>(&sms);
      if (err != cudaSuccess) return err;
      cudaLaunchAttribute attr[1];
      cudaLaunchConfig_t cfg = tail_config<D>(grid, stream, attr);
      return cudaLaunchKernelEx(&cfg, attn_fwd_kernel<D, false, true>, q);
    }
    // the hand-off test needs a split tail
    if (p.fault_drop_xfer) return cudaErrorInvalidValue;
  }
  attn_fwd_kernel<D, kTrace, false><<<grid, kThreads, Cfg<D>::kSmemBytes, stream>>>(q);
  return cudaGetLastError();
}

}  // namespace

int fwd_tail_pairs(const AttnParams& p, int D) {
  int sms = 0;
  AttnParams q = p;
  if (D == 128) {
    if (prepare<128, false, false>(&sms) != cudaSuccess || sms <= 0) return -1;
    plan_tail<128>(&q, p.num_tiles < sms ? p.num_tiles : sms);
  } else if (D == 64) {
    if (prepare<64, false, false>(&sms) != cudaSuccess || sms <= 0) return -1;
    plan_tail<64>(&q, p.num_tiles < sms ? p.num_tiles : sms);
  } else {
    return -1;
  }
  return q.tail_pairs;
}

cudaError_t launch_attn_fwd(const AttnParams& p, int D, cudaStream_t stream) {
  if (p.trace || p.fault_drop_block >= 0) {
    if (D == 128) return launch_d<128, true>(p, stream);
    if (D == 64) return launch_d<64, true>(p, stream);
    return cudaErrorInvalidValue;
  }
  if (D == 128) return launch_d<128, false>(p, stream);
  if (D == 64) return launch_d<64, false>(p, stream);
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
