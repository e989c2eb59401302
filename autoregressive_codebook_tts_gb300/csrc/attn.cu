// Single-query GQA decode attention for sm_103a, standalone and fused with the q/k
// norm + RoPE and the new-row KV write.
//
// Defines the operation of the "qwentts.cpp ... src/pipeline-tts.h" commit page
// (persistent-arenas section: window padded to a multiple of 256 with -inf over the
// padded tail; KV-cache section: decode appends one position and reads the
// [0, cur_len+1) window), batched over streams.
//
// Design (a bandwidth-bound GEMV, on CUDA cores with f32 accumulation):
//   * grid = (split, kv head, stream).  One CTA streams a contiguous range of one kv
//     head's positions and serves all Hq/Hkv q heads of the group from the same bytes,
//     so each K/V element is read from HBM once.
//   * Two producer warps feed a ring of shared-memory stages with 1-D bulk copies
//     (the TMA engine) of whole K and V tiles; the cache is head-major, so a tile of a
//     contiguous cache is one copy (a paged cache: one copy per page piece).  Copies
//     complete on per-stage mbarriers; consumer warps release stages on a second set.
//     One bulk copy costs about the same time whatever its size up to tens of KB and
//     copies issued by one thread run one after another, so tiles are 16 KB per copy
//     and K and V are issued by two producer warps side by side.
//   * A grid that fits the GPU at two CTAs per SM sizes each CTA's ring to hold its
//     whole split (the last, partial tile packed as K rows then V rows), so the split
//     streams in before the dependency wait ends.  Its producers keep one tile each in
//     flight: the whole layer's prefetch would otherwise queue in front of the
//     preceding launch's split merge, which is on the critical path.
//   * Consumer warps split each tile's rows.  A row is covered by LPR lanes with 16
//     bytes each (4 f32 or 8 bf16 elements); q.k is reduced across those lanes with
//     xor shuffles; each warp keeps its own online-softmax state (running max in log2
//     units, running sum, unnormalised output), merged at the end in shared memory.
//   * Rows at or past n_valid are never copied or read: the -inf of the padded tail
//     is realised as "not there", so poison in the tail cannot leak.
//   * Fused: one warp of the split holding the new position builds the new K/V row in
//     registers (norm + RoPE, conversion to the cache type), stores it to the cache and
//     starts its softmax state with it, so the row is never read back.
//   * Split-KV: every split writes (o, m, l) to the workspace and takes a ticket (one
//     acquire-release atomic per CTA); the last split of a (stream, kv head) merges all
//     partials with a log-sum-exp combine whose loads are all issued up front, and
//     resets the ticket.  No CTA ever waits for another.
//   * Launch configuration depends only on capacity; splits past the window exit early.
//   * Programmatic dependent launch: each launch lets the next one be scheduled as soon
//     as its own consumers pass their dependency wait.  With TTS_KV_PREFETCH_BEFORE_WAIT
//     the producers start streaming cache tiles (and the consumers read cur_len) before
//     the preceding kernel has finished.
//   * Every mbarrier wait is bounded (kWaitLimitCycles); on expiry TTS_EFLAG_TIMEOUT is
//     set, the copies already issued are waited for (bounded), and the CTA finishes.
#include <mutex>

#include "common.cuh"
#include "kernels.h"

// Tile geometry per (cache dtype, head_dim): rows per stage (T), ring stages (NS),
// consumer warps (NC).  Overridable at build time for tuning sweeps.
#ifndef TTS_F32_128_T
#define TTS_F32_128_T 32
#endif
#ifndef TTS_F32_128_NS
#define TTS_F32_128_NS 4
#endif
#ifndef TTS_F32_128_NC
#define TTS_F32_128_NC 4
#endif
#ifndef TTS_BF16_128_T
#define TTS_BF16_128_T 64
#endif
#ifndef TTS_BF16_128_NS
#define TTS_BF16_128_NS 4
#endif
#ifndef TTS_BF16_128_NC
#define TTS_BF16_128_NC 4
#endif
#ifndef TTS_F32_64_T
#define TTS_F32_64_T 64
#endif
#ifndef TTS_F32_64_NS
#define TTS_F32_64_NS 4
#endif
#ifndef TTS_F32_64_NC
#define TTS_F32_64_NC 4
#endif
#ifndef TTS_BF16_64_T
#define TTS_BF16_64_T 64
#endif
#ifndef TTS_BF16_64_NS
#define TTS_BF16_64_NS 4
#endif
// Ring sizes.  A grid that fits on the GPU at two CTAs per SM gives each CTA as many
// stages as fit in half an SM's shared memory, so a split of up to that many tiles is
// streamed in whole before the dependency wait ends.  A persistent grid (more work
// than fits at once) keeps TTS_RING_KB_STREAM per CTA; a cluster grid, which has
// fewer CTAs than SMs, TTS_RING_KB_CLUSTER.
#ifndef TTS_RING_KB_STREAM
#define TTS_RING_KB_STREAM 96
#endif
#ifndef TTS_RING_KB_CLUSTER
#define TTS_RING_KB_CLUSTER 128
#endif
#ifndef TTS_BF16_64_NC
#define TTS_BF16_64_NC 4
#endif
// Tiles a producer warp keeps in flight (0 = as many as the ring holds).  Once HBM is
// saturated a deeper queue streams no faster, but every other memory request of the
// GPU -- the preceding launch's split merge among them -- waits behind it.  A grid of
// single-item CTAs prefetches whole splits while the preceding launch finishes, so it
// is paced; a persistent grid streams item after item and is not.
#ifndef TTS_INFLIGHT_SINGLE
#define TTS_INFLIGHT_SINGLE 1
#endif
#ifndef TTS_INFLIGHT_STREAM
#define TTS_INFLIGHT_STREAM 0
#endif
// Persistent grids: the fixed cost of a work item (q load, merge, ticket), in cache
// rows' worth of streaming time, used to choose the split length of a launch.
#ifndef TTS_ITEM_COST_ROWS
#define TTS_ITEM_COST_ROWS 256
#endif
#ifndef TTS_ATTN_MIN_BLOCKS
#define TTS_ATTN_MIN_BLOCKS 2
#endif
// Lanes that share one K/V row (8: a quarter warp per row, 16 bytes per lane per
// vector, so a row reduction takes three shuffle levels).
#ifndef TTS_ATTN_LPR
#define TTS_ATTN_LPR 8
#endif

namespace tts {

#ifdef TTS_TRACE
// Optional timeline of the most recent attention launch (build with -DTTS_TRACE):
// per CTA, %globaltimer stamps at fixed points; read with tts_trace_read().
constexpr int kTraceSlots = 8;
constexpr int kTraceCtas = 8192;
__device__ unsigned long long g_trace[kTraceCtas][kTraceSlots];
__device__ __forceinline__ unsigned long long gtime() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
#define TTS_STAMP(slot)                                                                    \
  do {                                                                                     \
    const int cta_ = (blockIdx.z * gridDim.y + blockIdx.y) * gridDim.x + blockIdx.x;       \
    if (cta_ < kTraceCtas) g_trace[cta_][slot] = gtime();                                  \
  } while (0)
// per work item (persistent mode) rather than per CTA
#define TTS_STAMP_ITEM(slot, item)                                                         \
  do {                                                                                     \
    if ((item) < kTraceCtas) g_trace[(item)][slot] = gtime();                              \
  } while (0)
#define TTS_TRACE_SET(slot, item, value)                                                   \
  do {                                                                                     \
    if ((item) < kTraceCtas) g_trace[(item)][slot] = (value);                              \
  } while (0)
#else
#define TTS_TRACE_SET(slot, item, value) do {} while (0)
#define TTS_STAMP(slot) do {} while (0)
#define TTS_STAMP_ITEM(slot, item) do {} while (0)
#endif

namespace {

template <int T_, int NS_, int NC_>
struct TuneOf {
  static constexpr int T = T_, NS = NS_, NC = NC_;
};
template <typename KvT, int D> struct Tune;
template <> struct Tune<float, 128> : TuneOf<TTS_F32_128_T, TTS_F32_128_NS, TTS_F32_128_NC> {};
template <> struct Tune<__nv_bfloat16, 128> : TuneOf<TTS_BF16_128_T, TTS_BF16_128_NS, TTS_BF16_128_NC> {};
template <> struct Tune<float, 64> : TuneOf<TTS_F32_64_T, TTS_F32_64_NS, TTS_F32_64_NC> {};
template <> struct Tune<__nv_bfloat16, 64> : TuneOf<TTS_BF16_64_T, TTS_BF16_64_NS, TTS_BF16_64_NC> {};

template <typename KvT, int D_, int G_>
struct Cfg {
  static constexpr int D = D_;
  static constexpr int G = G_;
  static constexpr int kElem = sizeof(KvT);
  static constexpr int VE = 16 / kElem;       // elements per 16-byte vector
  // lanes per row: a quarter warp by default; half a warp for groups of four q heads
  // (whose per-lane q and output arrays would otherwise not fit in registers)
  static constexpr int LPR_WANT = (G_ >= 4 && TTS_ATTN_LPR < 16) ? 16 : TTS_ATTN_LPR;
  static constexpr int LPR = (LPR_WANT < D / VE) ? LPR_WANT : D / VE;
  static constexpr int EPL = D / LPR;         // elements per lane per row
  static constexpr int VEC = EPL / VE;        // 16-byte vectors per lane per row
  static constexpr int RPI = 32 / LPR;        // rows per warp step
  static constexpr int ROW_BYTES = D * kElem;
  static constexpr int T = Tune<KvT, D>::T;   // rows per stage
  static constexpr int NS = Tune<KvT, D>::NS; // maximum ring depth
  static constexpr int NC = Tune<KvT, D>::NC; // consumer warps
  static constexpr int NT = NC * 32;          // consumer threads
  static constexpr int RPW = T / NC;          // rows per warp per tile
  static constexpr int STEPS = RPW / RPI;
  static constexpr int TILE_BYTES = T * ROW_BYTES;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int THREADS = NT + 64;      // consumers + two producer warps
  static constexpr int Q4 = G * D / 4;        // float4 columns of one (stream, kv head) output
  static_assert(RPW % RPI == 0 && STEPS >= 1, "tile rows must split evenly over warp steps");
  static_assert(LPR >= 2 && LPR <= 32 && EPL % VE == 0, "row must span 2..32 lanes");
  static_assert(NT % Q4 == 0 || Q4 % NT == 0, "combine layout");

  // Shared memory: the ring of ns stages, its mbarriers (full[NS], empty[NS], the
  // cluster gather barrier, item-ready[4], item-free[4], q-ready[4]), then the areas
  // below.
  static constexpr int PART = G * (D + 2);    // floats of one split's partial (o, m, l per head)
  static constexpr size_t BAR_BYTES = ((2 * NS + 13) * sizeof(uint64_t) + 15) / 16 * 16;
  static constexpr size_t SCRATCH_BYTES = (static_cast<size_t>(NC) * PART * sizeof(float) + 15) / 16 * 16;
  static constexpr size_t FLAG_BYTES = 96;    // ticket flag, range length, item queue[4][4]
  // merge of up to kCombSplits partials (workspace path) or 16 (cluster path)
  static constexpr int kCombSplits = 256;
  static constexpr size_t comb_bytes(int n_splits) {
    return ((2 * G * static_cast<size_t>(n_splits) + G) * sizeof(float) + 15) / 16 * 16 + NT * 16;
  }
  static constexpr size_t COMB_BYTES = comb_bytes(kCombSplits);
  // Persistent mode: per item-queue slot the item's raw q rows (G heads) and its RoPE
  // row, copied in by the scheduler; and gamma_q, gamma_k staged once per CTA.
  static constexpr size_t QROW_BYTES = static_cast<size_t>(G) * D * sizeof(float);
  static constexpr size_t CSROW_BYTES = static_cast<size_t>(D / 2) * sizeof(float2);
  static constexpr size_t QSLOT_BYTES = QROW_BYTES + CSROW_BYTES;
  static constexpr size_t QBUF_BYTES = 4 * QSLOT_BYTES + 2 * D * sizeof(float);
  struct Layout {
    size_t bar, scratch, flag, comb, gather, list, qbuf, total;
  };
  // The merge scratch and the combine area are used only after the CTA's tiles are
  // consumed.  A CTA with a single item puts them over the ring (idle by then, every
  // copy it issued having landed) when the ring is large enough; a persistent CTA keeps
  // streaming its next item into the ring and gives them space of their own.
  static bool over_ring(size_t ring_bytes, bool persistent) {
    return !persistent && ring_bytes >= SCRATCH_BYTES + COMB_BYTES;
  }
  // ring_bytes: ns full stages, or (a split held whole) its full tiles' stages plus the
  // last, partial tile packed as K rows then V rows
  // n_splits: splits of the launch (a persistent CTA's combine area holds that many).
  static Layout layout(size_t ring_bytes, int cluster, bool persistent, int list_ints,
                       int n_splits = kCombSplits) {
    Layout L;
    L.bar = ring_bytes;
    size_t o = L.bar + BAR_BYTES;
    L.flag = o;
    o += FLAG_BYTES;
    if (over_ring(ring_bytes, persistent)) {
      L.scratch = 0;
      L.comb = SCRATCH_BYTES;
    } else {
      L.scratch = o;
      o += SCRATCH_BYTES;
      L.comb = o;
      o += persistent ? comb_bytes(n_splits < kCombSplits ? n_splits : kCombSplits) : COMB_BYTES;
    }
    L.gather = o;
    o += static_cast<size_t>(cluster > 1 ? cluster : 0) * PART * sizeof(float);
    L.qbuf = o;
    o += persistent ? QBUF_BYTES : 0;
    L.list = o;
    o += static_cast<size_t>(list_ints) * sizeof(int);
    L.total = o;
    return L;
  }
};

// The lane's elements of an f32 global row, in the lane layout of the cache rows:
// element e of vector j is row element (j * LPR + lr) * VE + e.
template <int VE, int VEC, int LPR>
__device__ __forceinline__ void load_row_f32(const float* row, int lr, float (&x)[VE * VEC]) {
#pragma unroll
  for (int j = 0; j < VEC; ++j)
#pragma unroll
    for (int e = 0; e < VE; e += 4) {
      const float4 v = __ldcg(reinterpret_cast<const float4*>(row + (j * LPR + lr) * VE + e));
      x[j * VE + e] = v.x; x[j * VE + e + 1] = v.y; x[j * VE + e + 2] = v.z; x[j * VE + e + 3] = v.w;
    }
}

__device__ __forceinline__ uint4 pack_vec(const float* x, float*) {
  return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                    __float_as_uint(x[3]));
}
__device__ __forceinline__ uint32_t pack2_bf16(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);  // .x = a (low half), round-to-nearest-even
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint4 pack_vec(const float* x, __nv_bfloat16*) {
  return make_uint4(pack2_bf16(x[0], x[1]), pack2_bf16(x[2], x[3]), pack2_bf16(x[4], x[5]),
                    pack2_bf16(x[6], x[7]));
}

// 2^x on the MUFU unit (ex2.approx, relative error about 2^-22; -inf gives +0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// The lane's elements of one staged K or V row as pairs of consecutive elements (zeros
// for rows at or past nrows).  A bf16 pair is one 32-bit word: the low half is the
// first element; widening to f32 puts the bf16 bits in the high half of each float.
__device__ __forceinline__ void unpack_pairs(const uint4 v, float2* f, float*) {
  f[0] = make_float2(__uint_as_float(v.x), __uint_as_float(v.y));
  f[1] = make_float2(__uint_as_float(v.z), __uint_as_float(v.w));
}
__device__ __forceinline__ void unpack_pairs(const uint4 v, float2* f, __nv_bfloat16*) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) f[i] = make_float2(__uint_as_float(w[i] << 16), __uint_as_float(w[i] & 0xffff0000u));
}

template <class C, typename KvT, bool PARTIAL>
__device__ __forceinline__ void load_smem_row(const unsigned char* __restrict__ tile, int row,
                                              int nrows, int lr, float2 (&f)[C::EPL / 2]) {
  constexpr int PV = C::VE / 2;  // pairs per 16-byte vector
  if (!PARTIAL || row < nrows) {
#pragma unroll
    for (int j = 0; j < C::VEC; ++j)
      unpack_pairs(lds128(tile + row * C::ROW_BYTES + (j * C::LPR + lr) * 16), f + j * PV,
                   static_cast<KvT*>(nullptr));
  } else {
#pragma unroll
    for (int i = 0; i < C::EPL / 2; ++i) f[i] = make_float2(0.f, 0.f);
  }
}

// Phase 1 of a tile for this warp: q.K scores of its rows (log2 units), reduced over
// the LPR lanes of each row; rows at or past nrows get -inf.  The lane's partial dot
// products run on pairs of elements (packed f32x2 multiply-adds).
template <class C, typename KvT, bool PARTIAL>
__device__ __forceinline__ void tile_scores(const unsigned char* __restrict__ kt, int nrows,
                                            int warp, int lane, const float2 (&q)[C::G][C::EPL / 2],
                                            float (&s)[C::STEPS][C::G]) {
  constexpr int G = C::G, NP = C::EPL / 2, LPR = C::LPR, STEPS = C::STEPS;
  const int lr = lane % LPR;
  const int row_base = warp * C::RPW + lane / LPR;
#pragma unroll
  for (int st = 0; st < STEPS; ++st) {
    const int row = row_base + st * C::RPI;
    float2 kf[NP];
    load_smem_row<C, KvT, PARTIAL>(kt, row, nrows, lr, kf);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float2 a = __fmul2_rn(q[h][0], kf[0]);
#pragma unroll
      for (int i = 1; i < NP; ++i) a = __ffma2_rn(q[h][i], kf[i], a);
      s[st][h] = a.x + a.y;
    }
  }
#pragma unroll
  for (int off = LPR / 2; off >= 1; off >>= 1)
#pragma unroll
    for (int st = 0; st < STEPS; ++st)
#pragma unroll
      for (int h = 0; h < G; ++h) s[st][h] += __shfl_xor_sync(kFull, s[st][h], off);
  if (PARTIAL) {
#pragma unroll
    for (int st = 0; st < STEPS; ++st)
      if (row_base + st * C::RPI >= nrows)
#pragma unroll
        for (int h = 0; h < G; ++h) s[st][h] = -INFINITY;
  }
}

// Phase 2 of a tile: online-softmax update with the tile's scores, then P.V on pairs.
template <class C, typename KvT, bool PARTIAL>
__device__ __forceinline__ void tile_softmax_pv(const unsigned char* __restrict__ vt, int nrows,
                                                int warp, int lane, float (&s)[C::STEPS][C::G],
                                                float (&m_run)[C::G], float (&l_run)[C::G],
                                                float2 (&o)[C::G][C::EPL / 2]) {
  constexpr int G = C::G, NP = C::EPL / 2, LPR = C::LPR, STEPS = C::STEPS;
  const int lr = lane % LPR;
  const int row_base = warp * C::RPW + lane / LPR;
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float mx = s[0][h];
#pragma unroll
    for (int st = 1; st < STEPS; ++st) mx = fmaxf(mx, s[st][h]);
#pragma unroll
    for (int off = LPR; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
    // Lazy rescaling: the reference maximum m_run moves only when the tile maximum
    // exceeds it by more than 8 (log2 units), so the o/l rescale is rare; until then the
    // weights 2^(s - m_run) stay below 2^8.  m_run and mx are warp-uniform, so is the
    // branch.  The result is exact up to rounding: o and l share the reference.
    if (mx > m_run[h] + 8.0f) {
      const float alpha = fast_exp2(m_run[h] - mx);  // 0 on the first tile (m_run = -inf)
      m_run[h] = mx;
      l_run[h] *= alpha;
      const float2 a2 = make_float2(alpha, alpha);
#pragma unroll
      for (int i = 0; i < NP; ++i) o[h][i] = __fmul2_rn(o[h][i], a2);
    }
    const float m_use = (m_run[h] == -INFINITY) ? 0.f : m_run[h];
#pragma unroll
    for (int st = 0; st < STEPS; ++st) {
      s[st][h] = fast_exp2(s[st][h] - m_use);
      l_run[h] += s[st][h];
    }
  }
#pragma unroll
  for (int st = 0; st < STEPS; ++st) {
    const int row = row_base + st * C::RPI;
    float2 vf[NP];
    load_smem_row<C, KvT, PARTIAL>(vt, row, nrows, lr, vf);
#pragma unroll
    for (int h = 0; h < G; ++h) {
      const float2 w2 = make_float2(s[st][h], s[st][h]);
#pragma unroll
      for (int i = 0; i < NP; ++i) o[h][i] = __ffma2_rn(w2, vf[i], o[h][i]);
    }
  }
}

// The packed projection input: column k of stream b at element (k / 8, b, k % 8) of
// [K / 8][slots][8] bf16 (round to nearest even, as the projection's own packing does).
__device__ __forceinline__ void store_packed1(__nv_bfloat16* xp, int slots, int b, int k, float v) {
  xp[(static_cast<int64_t>(k >> 3) * slots + b) * 8 + (k & 7)] = __float2bfloat16_rn(v);
}
__device__ __forceinline__ void store_packed4(__nv_bfloat16* xp, int slots, int b, int k, float4 v) {
  // k is a multiple of 4: the four values are half of one 16-byte group
  const __nv_bfloat162 lo = __floats2bfloat162_rn(v.x, v.y), hi = __floats2bfloat162_rn(v.z, v.w);
  uint2 u;
  u.x = *reinterpret_cast<const uint32_t*>(&lo);
  u.y = *reinterpret_cast<const uint32_t*>(&hi);
  *reinterpret_cast<uint2*>(xp + (static_cast<int64_t>(k >> 3) * slots + b) * 8 + (k & 7)) = u;
}

// Log-sum-exp merge of the n_act split partials of one (stream, kv head), run by the
// NT consumer threads of the CTA that took the last ticket.  The (m, l) pairs and the
// first batch of output partials are requested together; per-head maxima and sums use
// warp reductions.  `smem` is free shared memory (the ring).
template <class C>
__device__ __forceinline__ void combine_splits(const AttnParams& p, int b, int g, int n_act,
                                               int tid, unsigned char* smem) {
  constexpr int G = C::G, D = C::D, NT = C::NT, Q4 = C::Q4;
  constexpr int R = (NT >= Q4) ? NT / Q4 : 1;  // split groups working side by side
  constexpr int BATCH = 16;                    // partial rows in flight per thread
  const int Hq = p.n_q_heads;
  const int lane = tid & 31, warp = tid >> 5;
  float* sm_w = reinterpret_cast<float*>(smem);  // [G][n_act]: m, then the weights
  float* sm_l = sm_w + G * n_act;                // [G][n_act]
  float* sm_L = sm_l + G * n_act;                // [G]
  float4* sm_acc = reinterpret_cast<float4*>(smem + ((2 * G * n_act + G) * sizeof(float) + 15) / 16 * 16);
  const int64_t head0 = static_cast<int64_t>(b) * Hq + g * G;  // first q head of the group

  const int qi = tid % Q4;
  const int r = tid / Q4;
  const int h = qi / (D / 4);
  const int d4 = qi - h * (D / 4);
  const float4* op = reinterpret_cast<const float4*>(p.ws_o) + (head0 + h) * p.n_splits * (D / 4) + d4;
  // the (m, l) pairs gate the weights: requested first
  for (int i = tid; i < G * n_act; i += NT) {
    const int hh = i / n_act;
    const int s = i - hh * n_act;
    const float2 ml = __ldcg(reinterpret_cast<const float2*>(p.ws_ml) + (head0 + hh) * p.n_splits + s);
    sm_w[i] = ml.x;
    sm_l[i] = ml.y;
  }
  float4 v[BATCH];
#pragma unroll
  for (int k = 0; k < BATCH; ++k) {
    const int s = r + k * R;
    v[k] = (s < n_act) ? __ldcg(op + static_cast<int64_t>(s) * (D / 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
  }
  named_barrier(1, NT);
  // warp hh < G: M = max m, w_s = 2^(m_s - M), L = sum l_s w_s
  for (int hh = warp; hh < G; hh += C::NC) {
    float M = -INFINITY;
    for (int s = lane; s < n_act; s += 32) M = fmaxf(M, sm_w[hh * n_act + s]);
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
    float L = 0.f;
    for (int s = lane; s < n_act; s += 32) {
      const float w = fast_exp2(sm_w[hh * n_act + s] - M);
      sm_w[hh * n_act + s] = w;
      L = fmaf(sm_l[hh * n_act + s], w, L);
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) L += __shfl_xor_sync(kFull, L, off);
    if (lane == 0) sm_L[hh] = L;
  }
  named_barrier(1, NT);
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  const float* wh = sm_w + h * n_act;
#pragma unroll
  for (int k = 0; k < BATCH; ++k) {
    const int s = r + k * R;
    if (s < n_act) {
      const float w = wh[s];
      acc.x = fmaf(w, v[k].x, acc.x);
      acc.y = fmaf(w, v[k].y, acc.y);
      acc.z = fmaf(w, v[k].z, acc.z);
      acc.w = fmaf(w, v[k].w, acc.w);
    }
  }
  for (int s0 = r + BATCH * R; s0 < n_act; s0 += BATCH * R) {  // only for very many splits
#pragma unroll
    for (int k = 0; k < BATCH; ++k) {
      const int s = s0 + k * R;
      v[k] = (s < n_act) ? __ldcg(op + static_cast<int64_t>(s) * (D / 4)) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int k = 0; k < BATCH; ++k) {
      const int s = s0 + k * R;
      if (s < n_act) {
        const float w = wh[s];
        acc.x = fmaf(w, v[k].x, acc.x);
        acc.y = fmaf(w, v[k].y, acc.y);
        acc.z = fmaf(w, v[k].z, acc.z);
        acc.w = fmaf(w, v[k].w, acc.w);
      }
    }
  }
  if (R > 1) {
    sm_acc[r * Q4 + qi] = acc;
    named_barrier(1, NT);
  }
  if (tid < Q4) {
#pragma unroll 1
    for (int rr = 1; rr < R; ++rr) {
      const float4 a = sm_acc[rr * Q4 + qi];
      acc.x += a.x; acc.y += a.y; acc.z += a.z; acc.w += a.w;
    }
    const float L = sm_L[h];
    const float4 o4 = make_float4(acc.x / L, acc.y / L, acc.z / L, acc.w / L);
    if (p.out_packed == nullptr) {
      reinterpret_cast<float4*>(p.out + (head0 + h) * D)[d4] = o4;
    } else {
      const int k = (g * G + h) * D + d4 * 4;  // column of the stream's output row
      store_packed4(p.out_packed, p.out_slots, b, k, o4);
    }
  }
}

// One unit of work: the rows [r0, r0 + split_len) of one (query stream, kv head).
// Query stream b reads the cache of stream cb = b / q_per_stream (a prefill's
// q_per_stream queries share their stream's cache).
struct Item {
  int b, g, split;
  int cb;         // cache stream
  int nv;         // window length (clamped)
  int cur;        // fused: position of the new row
  bool fresh_ok;  // fused: cur is a valid position
  int r0, n_rows, ntiles;
  bool has_fresh;
  int n_act;      // splits of this stream that hold rows of the window
};

template <bool FUSED>
__device__ __forceinline__ Item make_item(const AttnParams& p, int T, int b, int g, int split, int raw,
                                          int split_len) {
  Item it;
  it.b = b;
  it.cb = b / p.q_per_stream;
  it.g = g;
  it.split = split;
  int cache_end;
  if (FUSED) {
    it.cur = raw;
    it.fresh_ok = raw >= 0 && raw < p.capacity;
    it.nv = min(max(raw + 1, 1), p.capacity);
    cache_end = it.fresh_ok ? raw : it.nv;
  } else {
    it.cur = 0;
    it.fresh_ok = false;
    it.nv = min(max(raw, 1), p.capacity);
    cache_end = it.nv;
  }
  it.r0 = split * split_len;
  it.n_rows = max(0, min(it.r0 + split_len, cache_end) - it.r0);
  it.has_fresh = FUSED && it.fresh_ok && it.cur >= it.r0 && it.cur < it.r0 + split_len;
  it.ntiles = (it.n_rows + T - 1) / T;
  it.n_act = min(p.n_splits, (it.nv + split_len - 1) / split_len);
  return it;
}

// A persistent item: rows [r0, r1) of the window of (query stream b, kv head g), the
// split-th of the n_act pieces the window is cut into.
template <bool FUSED>
__device__ __forceinline__ Item make_item_rows(const AttnParams& p, int T, int b, int g, int split,
                                               int raw, int r0, int r1, int n_act) {
  Item it;
  it.b = b;
  it.cb = b / p.q_per_stream;
  it.g = g;
  it.split = split;
  int cache_end;
  if (FUSED) {
    it.cur = raw;
    it.fresh_ok = raw >= 0 && raw < p.capacity;
    it.nv = min(max(raw + 1, 1), p.capacity);
    cache_end = it.fresh_ok ? raw : it.nv;
  } else {
    it.cur = 0;
    it.fresh_ok = false;
    it.nv = min(max(raw, 1), p.capacity);
    cache_end = it.nv;
  }
  it.r0 = r0;
  it.n_rows = max(0, min(r1, cache_end) - r0);
  it.has_fresh = FUSED && it.fresh_ok && it.cur >= r0 && it.cur < r1;
  it.ntiles = (it.n_rows + T - 1) / T;
  it.n_act = n_act;
  return it;
}

// The window input of query stream b: cur_len (fused) or n_valid, read from its cache
// stream's entry plus the query's offset within that stream (prefill queries).
__device__ __forceinline__ int raw_len(const AttnParams& p, int b) {
  const int cb = b / p.q_per_stream;
  return __ldcg(p.lens + cb) + (b - cb * p.q_per_stream) + p.lens_add;
}

__device__ __forceinline__ int window_len(const AttnParams& p, int raw, bool fused) {
  return fused ? min(max(raw + 1, 1), p.capacity) : min(max(raw, 1), p.capacity);
}

__device__ __forceinline__ int n_active(const AttnParams& p, int nv, int split_len) {
  return min(p.n_splits, (nv + split_len - 1) / split_len);
}

template <typename KvT, int D, int G, bool FUSED>
__global__ void __launch_bounds__(Cfg<KvT, D, G>::THREADS, (G >= 4 ? 2 : TTS_ATTN_MIN_BLOCKS))
decode_attn_kernel(const AttnParams p) {
  using C = Cfg<KvT, D, G>;
  constexpr int EPL = C::EPL, LPR = C::LPR, NC = C::NC, NT = C::NT, T = C::T;
  constexpr int VE = C::VE, VEC = C::VEC, STEPS = C::STEPS;
  extern __shared__ __align__(128) unsigned char smem[];

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ns = p.n_stages;
  const int Hq = p.n_q_heads, Hkv = p.n_kv_heads;

  unsigned char* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + p.sm_bar);
  uint64_t* empty = full + C::NS;
  uint64_t* gbar = empty + C::NS;
  uint64_t* ibar = gbar + 1;   // persistent: item published in queue slot j
  uint64_t* ifree = ibar + 4;  // persistent: queue slot j read by every reader
  uint64_t* qbar = ifree + 4;  // persistent: the q (and RoPE) rows of queue slot j landed
  // persistent: per queue slot the item's raw q rows then its RoPE row; then gamma_q,
  // gamma_k
  unsigned char* qbuf = smem + p.sm_qbuf;
  float* s_gamma = reinterpret_cast<float*>(qbuf + 4 * C::QSLOT_BYTES);
  float* scratch = reinterpret_cast<float*>(smem + p.sm_scratch);
  int* s_last = reinterpret_cast<int*>(smem + p.sm_flag);
  unsigned char* comb = smem + p.sm_comb;
  float* gather = reinterpret_cast<float*>(smem + p.sm_gather);
  // Cluster mode: the n_splits CTAs of one (stream, kv head) form a cluster and merge
  // their partials in rank 0's shared memory (rank == split).
  const bool clustered = p.cluster > 1;
  // Persistent mode: a fixed grid whose CTAs take the active items one after another:
  // item blockIdx.x first, then whatever an atomic work counter hands out.
  const bool persistent = p.persistent != 0;

  if (threadIdx.x == 0) {
    if (p.persistent == 0) TTS_STAMP(0);
    for (int s = 0; s < ns; ++s) {
      mbar_init(&full[s], 2);  // one arrival from each producer warp, plus the bytes
      mbar_init(&empty[s], NC);
    }
    if (clustered) mbar_init(gbar, p.cluster - 1);
    if (persistent) {
      for (int j = 0; j < 4; ++j) {
        mbar_init(&ibar[j], 1);        // the scheduler publishes
        mbar_init(&ifree[j], NC + 1);  // the V producer and every consumer warp read
        mbar_init(&qbar[j], 1);        // the scheduler's arrival (plus the q bytes)
      }
    }
    mbar_init_fence();
  }
  // every CTA's gather barrier is initialised before any peer can arrive on it
  if (clustered) cluster_sync_all();
  else __syncthreads();

  // With TTS_KV_PREFETCH_BEFORE_WAIT the caller has promised that the preceding kernel
  // writes neither this cache, its block table, cur_len, gamma nor the RoPE table, so
  // those may be read before the dependency wait.
  const bool early = FUSED && (p.flags & TTS_KV_PREFETCH_BEFORE_WAIT);
  if (!early) grid_wait();

  // Work list.  Persistent: a static partition of the launch's work into equal shares.
  // Every (stream b, kv head g) pair costs kItemCost + n_valid[b] units (a fixed cost
  // per piece, in cache rows' worth of streaming time, then one unit per window row);
  // the pairs are laid end to end in (b, g) order and CTA r takes the units
  // [r K, (r + 1) K), i.e. the window rows of the pairs that range covers, cut on
  // multiples of 16 rows.  K is the total over the grid, but at least enough that no
  // window is cut into more pieces than the workspace has split slots.  No CTA takes
  // work from another at run time, and every CTA computes the same partition from the
  // same windows.  Otherwise one item, the CTA's own (split, g, b).
  constexpr int kItemCost = TTS_ITEM_COST_ROWS;
  constexpr int kMinRangeRows = 64;
  const int split_len = p.split_len;
  long long* s_cost = reinterpret_cast<long long*>(smem + p.sm_list);  // [B + 1] prefix of Hkv (kItemCost + nv)
  int* s_nv = reinterpret_cast<int*>(smem + p.sm_list + (static_cast<size_t>(p.B) + 1) * sizeof(long long));
  int* s_raw = s_nv + p.B;  // persistent: the window input of every query stream (cur_len or n_valid)
  volatile long long* s_K = reinterpret_cast<volatile long long*>(smem + p.sm_flag + 8);
  long long K = 0, c_total = 0;
  if (persistent) {
    if (warp == 0) {
      long long carry = 0;
      int max_cost = 0;
      for (int b0 = 0; b0 < p.B; b0 += 32) {
        const int bb = b0 + lane;
        const int raw = bb < p.B ? raw_len(p, bb) : 0;
        const int nv = bb < p.B ? window_len(p, raw, FUSED) : 0;
        if (bb < p.B) {
          s_nv[bb] = nv;
          s_raw[bb] = raw;
        }
        long long v = bb < p.B ? static_cast<long long>(Hkv) * (kItemCost + nv) : 0;
        max_cost = max(max_cost, bb < p.B ? kItemCost + nv : 0);
#pragma unroll
        for (int off = 1; off < 32; off <<= 1) {
          const long long u = __shfl_up_sync(kFull, v, off);
          if (lane >= off) v += u;
        }
        if (bb < p.B) s_cost[bb + 1] = carry + v;
        carry += __shfl_sync(kFull, v, 31);
      }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) max_cost = max(max_cost, __shfl_xor_sync(kFull, max_cost, off));
      if (lane == 0) {
        s_cost[0] = 0;
        const long long R = gridDim.x;
        const long long even = (carry + R - 1) / R;
        // a window of n rows meets at most n / K + 2 ranges after the 16-row rounding
        // (boundaries move by at most 8 rows): K >= (max cost + 32) / (splits - 1)
        // keeps that within the workspace's n_splits slots
        const long long bound = (static_cast<long long>(max_cost) + 32 + p.n_splits - 2) / (p.n_splits - 1);
        *s_K = max(max(even, bound), static_cast<long long>(kMinRangeRows));
      }
    }
    __syncthreads();
    K = *s_K;
    c_total = s_cost[p.B];
  }
  // Window rows of pair (b, g) below the cost boundary min(r K, total), rounded to a
  // multiple of 16 and clamped to [0, nv]: non-decreasing in r, 0 at r = 0 and nv at
  // r = gridDim.x.  CTA r's piece of the pair is [row_at(r), row_at(r + 1)).
  auto row_at = [&](int b, int g, long long r) -> int {
    const int nv = s_nv[b];
    const long long start = s_cost[b] + static_cast<long long>(g) * (kItemCost + nv) + kItemCost;
    const long long x = min(r * K, c_total) - start;
    if (x <= 0) return 0;
    if (x >= nv) return nv;
    return min((static_cast<int>(x) + 8) & ~15, nv);
  };
  // Persistent: the queue entry of pair `pair` for this CTA: {pair, r0, r1, split | n_act << 16}
  // where the pieces of the pair belong to CTAs r_a..r_b (those with non-empty rows).
  auto piece_of = [&](int pair, int4& e) {
    const int b = pair / Hkv, g = pair - (pair / Hkv) * Hkv;
    const int R = gridDim.x;
    const int r = blockIdx.x;
    const int nv = s_nv[b];
    int lo = 0, hi = R;  // smallest r' with row_at(r') > 0
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (row_at(b, g, mid) > 0) hi = mid; else lo = mid;
    }
    const int ra = hi - 1;
    lo = 0;
    hi = R;              // smallest r' with row_at(r') >= nv
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (row_at(b, g, mid) >= nv) hi = mid; else lo = mid;
    }
    const int rb = hi - 1;
    e = make_int4(pair, row_at(b, g, r), row_at(b, g, r + 1), (r - ra) | ((rb - ra + 1) << 16));
  };
  // Persistent: the first pair at or after `from` in which this CTA has rows, or -1.
  auto next_pair = [&](int from) -> int {
    const long long hi_cost = min((static_cast<long long>(blockIdx.x) + 1) * K, c_total);
    for (int pr = from; pr < p.B * Hkv; ++pr) {
      const int b = pr / Hkv, g = pr - (pr / Hkv) * Hkv;
      if (s_cost[b] + static_cast<long long>(g) * (kItemCost + s_nv[b]) >= hi_cost) return -1;
      if (row_at(b, g, blockIdx.x) < row_at(b, g, static_cast<long long>(blockIdx.x) + 1)) return pr;
    }
    return -1;
  };
  // Persistent: the pair that holds the cost unit min(r K, total), where this CTA's
  // range starts.
  auto first_pair = [&]() -> int {
    const long long c0 = min(static_cast<long long>(blockIdx.x) * K, c_total);
    int lo = 0, hi = p.B;  // largest b with s_cost[b] <= c0
    while (hi - lo > 1) {
      const int mid = (lo + hi) >> 1;
      if (s_cost[mid] <= c0) lo = mid; else hi = mid;
    }
    const long long g = (c0 - s_cost[lo]) / (kItemCost + s_nv[lo]);
    return lo * Hkv + static_cast<int>(min(g, static_cast<long long>(Hkv - 1)));
  };
  volatile int4* s_item = reinterpret_cast<volatile int4*>(smem + p.sm_flag + 32);
  auto item_of = [&](const int4 e) -> Item {
    if (persistent) {
      const int b = e.x / Hkv;
      return make_item_rows<FUSED>(p, T, b, e.x - b * Hkv, e.w & 0xffff, s_raw[b], e.y, e.z,
                                   e.w >> 16);
    }
    return make_item<FUSED>(p, T, blockIdx.z, blockIdx.y, blockIdx.x, raw_len(p, blockIdx.z), split_len);
  };
  auto read_entry = [&](int j) -> int4 {
    const int4 e = make_int4(s_item[j].x, s_item[j].y, s_item[j].z, s_item[j].w);
    return e;
  };
  // Persistent mode: queue slot j = k % 4 carries this CTA's k-th entry (pair, rows,
  // split and piece count) from the scheduler (the K producer's lane 0) to the V
  // producer and the consumer warps; a negative pair ends the list.
  if (warp >= NC) {
    // ----------------------------------------------------------------- producers
    // Warp NC streams the K tiles, warp NC+1 the V tiles: bulk copies issued by
    // different warps proceed side by side, while one thread's copies run one after
    // another.  A paged tile's page pieces are issued by consecutive lanes.  The ring
    // runs on across items, so the next item's tiles stream in while this one drains.
    const int pw = warp - NC;
    const uint64_t pol = l2_evict_first_policy();
    const int inflight = (p.inflight > 0 && p.inflight < ns) ? p.inflight : 0;
    const unsigned char* src = static_cast<const unsigned char*>(pw == 0 ? p.k_cache : p.v_cache);
    int issued = 0;
    int stage = 0;
    uint32_t round = 0;
    bool ok = true;
    int k = 0;  // items taken so far
    int pair = (persistent && pw == 0) ? next_pair(first_pair()) : 0;
    int4 e = make_int4(-1, 0, 0, 0);
    for (;;) {
      if (persistent) {
        if (pw == 0) {
          // scheduler: publish item i in queue slot k % 4 once every reader is done with it
          const int j = k & 3;
          int w = 1;
          if (k >= 4 && lane == 0) w = mbar_wait(&ifree[j], static_cast<uint32_t>((k >> 2) - 1) & 1u) ? 1 : 0;
          if (__shfl_sync(kFull, w, 0) == 0) {
            if (lane == 0) set_err(p.err, TTS_EFLAG_TIMEOUT);
            break;
          }
          if (pair >= 0) piece_of(pair, e); else e = make_int4(-1, 0, 0, 0);
          if (lane == 0) {
            s_item[j].x = e.x;
            s_item[j].y = e.y;
            s_item[j].z = e.z;
            s_item[j].w = e.w;
            mbar_arrive(&ibar[j]);
            // From the second item on (the dependency wait is behind us: q is written by
            // the preceding kernel) the item's q rows, and in the fused form its RoPE
            // row, are copied into the slot, so the consumers find them in shared memory.
            if (k >= 1 && e.x >= 0) {
              const Item qi = item_of(e);
              const uint32_t bytes = static_cast<uint32_t>(C::QROW_BYTES + (FUSED ? C::CSROW_BYTES : 0));
              mbar_arrive_expect_tx(&qbar[j], bytes);
              bulk_g2s_plain(qbuf + j * C::QSLOT_BYTES,
                             p.q + static_cast<int64_t>(qi.b) * p.q_stride + static_cast<int64_t>(qi.g) * G * D,
                             static_cast<uint32_t>(C::QROW_BYTES), &qbar[j]);
              if (FUSED) {
                const int rope_pos = min(max(qi.cur, 0), p.max_pos - 1);
                bulk_g2s_plain(qbuf + j * C::QSLOT_BYTES + C::QROW_BYTES,
                               p.cs + static_cast<int64_t>(rope_pos) * (D / 2),
                               static_cast<uint32_t>(C::CSROW_BYTES), &qbar[j]);
              }
            } else {
              mbar_arrive(&qbar[j]);
            }
          }
          __syncwarp();
          ++k;
        } else {
          const int j = k & 3;
          if (!mbar_wait(&ibar[j], static_cast<uint32_t>(k >> 2) & 1u)) {
            if (lane == 0) set_err(p.err, TTS_EFLAG_TIMEOUT);
            break;
          }
          e = read_entry(j);
          __syncwarp();
          if (lane == 0) mbar_arrive(&ifree[j]);
          ++k;
        }
        if (e.x < 0) break;
      }
      const Item it = item_of(e);
      if (!persistent && it.split >= it.n_act) break;  // outside the window
      const int32_t* bt = p.paged ? p.block_table + static_cast<int64_t>(it.cb) * p.bt_stride : nullptr;
      // Paged: lane k issues piece k of a tile (the piece that starts the tile, then one
      // per page).  When every piece of a tile has its own lane, each lane's block-table
      // entry is loaded one tile ahead, so the load's latency overlaps the wait for a
      // free stage instead of delaying the copies.
      const bool ahead = p.paged && (T / p.page_size + 1 <= 32);
      auto piece_start = [&](int t) -> int {
        const int row0 = it.r0 + t * T;
        return lane == 0 ? row0 : (row0 & ~(p.page_size - 1)) + lane * p.page_size;
      };
      auto tile_end = [&](int t) -> int { return min(it.r0 + (t + 1) * T, it.r0 + it.n_rows); };
      int pg_next = -1;
      if (ahead && it.ntiles > 0) {
        const int st = piece_start(0);
        if (st < tile_end(0)) pg_next = __ldcg(bt + (st >> p.page_shift));
      }
      for (int t = 0; t < it.ntiles; ++t) {
        const int pg_cur = pg_next;
        if (ahead && t + 1 < it.ntiles) {
          const int st = piece_start(t + 1);
          pg_next = st < tile_end(t + 1) ? __ldcg(bt + (st >> p.page_shift)) : -1;
        }
        int w = 1;
        if (lane == 0) {
          // pace: the tile issued `inflight` tiles ago has landed (its stage is not
          // reused before this one is issued, since inflight <= ns)
          if (inflight > 0 && issued >= inflight) {
            const int k = issued - inflight;
            w = mbar_wait(&full[k % ns], static_cast<uint32_t>(k / ns) & 1u) ? 1 : 0;
          }
          if (w && issued >= ns) w = mbar_wait(&empty[stage], (round & 1u) ^ 1u) ? 1 : 0;
        }
        if (__shfl_sync(kFull, w, 0) == 0) {
          if (lane == 0) set_err(p.err, TTS_EFLAG_TIMEOUT);
          ok = false;
          break;
        }
        const int row0 = it.r0 + t * T;
        const int rows = min(T, it.r0 + it.n_rows - row0);
        // a stage holds the tile's K rows, then its V rows
        unsigned char* dst = ring + stage * C::STAGE_BYTES + pw * rows * C::ROW_BYTES;
        if (lane == 0) mbar_arrive_expect_tx(&full[stage], static_cast<uint32_t>(rows) * C::ROW_BYTES);
        __syncwarp();
        if (!p.paged) {
          if (lane == 0) {
            const size_t off =
                ((static_cast<size_t>(it.cb) * Hkv + it.g) * p.capacity + row0) * C::ROW_BYTES;
            bulk_g2s(dst, src + off, static_cast<uint32_t>(rows) * C::ROW_BYTES, &full[stage], pol);
          }
        } else if (ahead) {
          const int start = piece_start(t);
          if (start < row0 + rows) {
            int page = pg_cur;
            if (page < 0 || page >= p.n_pages) {
              set_err(p.err, TTS_EFLAG_PAGE);
              page = 0;
            }
            const int slot = start & (p.page_size - 1);
            const int n = min(p.page_size - slot, row0 + rows - start);
            const size_t off =
                ((static_cast<size_t>(page) * Hkv + it.g) * p.page_size + slot) * C::ROW_BYTES;
            bulk_g2s(dst + (start - row0) * C::ROW_BYTES, src + off,
                     static_cast<uint32_t>(n) * C::ROW_BYTES, &full[stage], pol);
          }
        } else {
          const int re = row0 + rows;
          const int page0 = row0 & ~(p.page_size - 1);
          for (int k = lane;; k += 32) {
            const int start = (k == 0) ? row0 : page0 + k * p.page_size;
            if (start >= re) break;
            int page = __ldcg(bt + (start >> p.page_shift));
            if (page < 0 || page >= p.n_pages) {
              set_err(p.err, TTS_EFLAG_PAGE);
              page = 0;
            }
            const int slot = start & (p.page_size - 1);
            const int n = min(p.page_size - slot, re - start);
            const size_t off =
                ((static_cast<size_t>(page) * Hkv + it.g) * p.page_size + slot) * C::ROW_BYTES;
            bulk_g2s(dst + (start - row0) * C::ROW_BYTES, src + off,
                     static_cast<uint32_t>(n) * C::ROW_BYTES, &full[stage], pol);
          }
        }
        ++issued;
        if (++stage == ns) {
          stage = 0;
          ++round;
        }
      }
      if (!ok || !persistent) break;
      if (pw == 0) {
        // the next item's q rows are copied after the dependency wait
        if (k == 1 && early) grid_wait();
        pair = next_pair(pair + 1);
      }
    }
    // Do not leave while copies into this CTA's shared memory may be in flight.
    if (lane == 0) {
      for (int t = max(0, issued - ns); t < issued; ++t)
        mbar_wait(&full[t % ns], static_cast<uint32_t>(t / ns) & 1u);
      if (persistent && pw == 0)
        for (int t = max(0, k - 4); t < k; ++t) mbar_wait(&qbar[t & 3], static_cast<uint32_t>(t >> 2) & 1u);
    }
    return;
  }

  // -------------------------------------------------------------------- consumers
  const int tid = threadIdx.x;  // < NT
  const int lr = lane % LPR;
  const int half = D / 2;
  // The new K/V row of the window (fused) is folded in by one warp, from registers.
  constexpr int kFreshWarp = 0;
  float gq[EPL], gk[EPL];
  float2 csr[EPL];
  auto load_consts = [&](const Item& it) {
    const int rope_pos = min(max(it.cur, 0), p.max_pos - 1);
    const float2* cs_row = p.cs + static_cast<int64_t>(rope_pos) * half;
    load_norm_consts<VE, VEC, LPR>(p.gamma_q, cs_row, lr, D, gq, csr);
    if (it.has_fresh && warp == kFreshWarp) load_norm_consts<VE, VEC, LPR>(p.gamma_k, cs_row, lr, D, gk, csr);
  };
  // A single-item CTA knows its item up front.  With the prefetch flag cur_len is not
  // written by the preceding launch, so the item is worked out before the dependency
  // wait, while that launch finishes.
  Item it0 = {};
  if (!persistent && early) it0 = item_of(make_int4(0, 0, 0, 0));
  if (persistent && FUSED) {
    // gamma_q and gamma_k, read once per CTA (constants of the layer)
    for (int e = tid; e < 2 * D; e += NT) s_gamma[e] = __ldcg((e < D ? p.gamma_q : p.gamma_k) + (e % D));
    named_barrier(1, NT);
  }
  if (early) grid_wait();
  grid_launch_dependents();
  if (tid == 0 && !persistent) TTS_STAMP(1);

  int sc = 0;          // ring stage of the next tile
  uint32_t pc = 0u;    // parity of its phase
  bool ok = true;
  int kq = 0;  // items taken from the queue so far (persistent)
  int jq = 0;  // queue slot of the current item (persistent)
  // persistent: the ticket of the previous item, issued at its end and resolved at the
  // end of the next one (thread 0 holds the atomic's result)
  int pend_b = -1, pend_g = 0, pend_nact = 0, pend_prev = 0;
  auto resolve_pending = [&]() {
    if (tid == 0) *s_last = (pend_prev == pend_nact - 1) ? 1 : 0;
    named_barrier(1, NT);
    if (*s_last != 0) {
      combine_splits<C>(p, pend_b, pend_g, pend_nact, tid, comb);
      if (tid == 0) p.ws_cnt[pend_b * Hkv + pend_g] = 0;
    }
    named_barrier(1, NT);
    pend_b = -1;
  };
  int4 ecur = make_int4(0, 0, 0, 0);
  for (int round_item = 0;; ++round_item) {
    int i = 0;
    if (persistent) {
      jq = kq & 3;
      if (!mbar_wait(&ibar[jq], static_cast<uint32_t>(kq >> 2) & 1u)) {
        set_err(p.err, TTS_EFLAG_TIMEOUT);
        break;
      }
      ecur = read_entry(jq);
      ++kq;
      i = static_cast<int>(blockIdx.x) * 8 + min(kq - 1, 7);  // trace slot of this item
      if (ecur.x < 0) {
        __syncwarp();
        if (lane == 0) mbar_arrive(&ifree[jq]);
        break;
      }
    } else if (round_item > 0) {
      break;
    }
    const Item it = (!persistent && early) ? it0 : item_of(ecur);
    const bool active = it.split < it.n_act;
    if (!persistent && !active) {
      // Outside the window: nothing to stream.  A cluster peer still reports in when
      // rank 0 waits for the cluster (more than one active split); when the window
      // fits in split 0, rank 0 writes the output alone and does not wait.
      if (clustered && it.n_act > 1) {
        named_barrier(1, NT);
        if (tid == 0) mbar_arrive_remote(map_shared_rank(gbar, 0));
      }
      return;
    }
    const int b = it.b, g = it.g, split = it.split;
    if (persistent && tid == 0) {
      TTS_STAMP_ITEM(0, i);
      unsigned smid;
      asm volatile("mov.u32 %0, %%smid;" : "=r"(smid));
      TTS_TRACE_SET(1, i, blockIdx.x | (static_cast<unsigned long long>(it.n_rows) << 16) |
                              (static_cast<unsigned long long>(kq) << 32) |
                              (static_cast<unsigned long long>(smid) << 40));
    }
    const bool reporter = (split == 0 && g == 0 && tid == 0);
    if (reporter) {
      if (FUSED) {
        if (!it.fresh_ok) set_err(p.err, TTS_EFLAG_POS_RANGE);
        if (it.cur < 0 || it.cur >= p.max_pos) set_err(p.err, TTS_EFLAG_POS_RANGE);
      } else {
        const int raw = raw_len(p, b);
        if (raw < 1 || raw > p.capacity) set_err(p.err, TTS_EFLAG_NVALID);
      }
    }

    // From a persistent CTA's second item on, the scheduler has copied the raw q rows
    // (and the RoPE row) into the item's queue slot; otherwise they come from global
    // memory.
    const bool q_in_smem = persistent && kq >= 2;
    const bool fresh_here = FUSED && it.has_fresh && warp == kFreshWarp;
    float q[G][EPL];
    if (q_in_smem) {
      if (!mbar_wait(&qbar[jq], static_cast<uint32_t>((kq - 1) >> 2) & 1u)) {
        set_err(p.err, TTS_EFLAG_TIMEOUT);
        ok = false;
      }
      const float* qs = reinterpret_cast<const float*>(qbuf + jq * C::QSLOT_BYTES);
      if (FUSED) {
        const float2* cs_row = reinterpret_cast<const float2*>(qbuf + jq * C::QSLOT_BYTES + C::QROW_BYTES);
        load_norm_consts_smem<VE, VEC, LPR>(s_gamma, cs_row, lr, D, gq, csr);
        if (fresh_here) load_norm_consts_smem<VE, VEC, LPR>(s_gamma + D, cs_row, lr, D, gk, csr);
      }
#pragma unroll
      for (int h = 0; h < G; ++h) load_row_smem<VE, VEC, LPR>(qs + h * D, lr, q[h]);
    } else {
      if (FUSED) load_consts(it);
#pragma unroll
      for (int h = 0; h < G; ++h)
        load_row_f32<VE, VEC, LPR>(
            p.q + static_cast<int64_t>(b) * p.q_stride + static_cast<int64_t>(g * G + h) * D, lr, q[h]);
    }
    // head_dim 64 (short rows, registers to spare): the new K/V row's loads go out with
    // q's, one round trip instead of two on a short window's critical path
    constexpr bool kFreshEarly = (D == 64);
    float kr[EPL], vr[EPL];
    if (kFreshEarly && fresh_here) {
      const int64_t roff = static_cast<int64_t>(b) * p.kv_new_stride + static_cast<int64_t>(g) * D;
      load_row_f32<VE, VEC, LPR>(p.k_new + roff, lr, kr);
      load_row_f32<VE, VEC, LPR>(p.v_new + roff, lr, vr);
    }
    if (persistent) {
      // every value of the slot this warp needs is in registers: release the slot
      __syncwarp();
      if (lane == 0) mbar_arrive(&ifree[jq]);
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      if (FUSED) norm_rope_regs<VE, VEC, LPR>(q[h], gq, csr, p.eps, lr, D);
#pragma unroll
      for (int k = 0; k < EPL; ++k) q[h][k] *= p.scale_log2;
    }
    float2 q2[G][EPL / 2];
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int i = 0; i < EPL / 2; ++i) q2[h][i] = make_float2(q[h][2 * i], q[h][2 * i + 1]);

    float m_run[G], l_run[G];
    float2 o[G][EPL / 2];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m_run[h] = -INFINITY;
      l_run[h] = 0.f;
#pragma unroll
      for (int k = 0; k < EPL / 2; ++k) o[h][k] = make_float2(0.f, 0.f);
    }

    // Fused: build the new K/V row (norm + RoPE on k, v as is), convert it to the cache
    // type and store it to the cache; then start this warp's softmax state with it.
    // Every row group of the warp holds the row, so the score and the running maximum
    // are warp-uniform; its weight 2^0 = 1 and its V row are counted by row group 0.
    if (fresh_here) {
      if (!kFreshEarly) {
        const int64_t roff = static_cast<int64_t>(b) * p.kv_new_stride + static_cast<int64_t>(g) * D;
        load_row_f32<VE, VEC, LPR>(p.k_new + roff, lr, kr);
        load_row_f32<VE, VEC, LPR>(p.v_new + roff, lr, vr);
      }
      norm_rope_regs<VE, VEC, LPR>(kr, gk, csr, p.eps, lr, D);
      uint4 kp[VEC], vp[VEC];
#pragma unroll
      for (int j = 0; j < VEC; ++j) {
        kp[j] = pack_vec(kr + j * VE, static_cast<KvT*>(nullptr));
        vp[j] = pack_vec(vr + j * VE, static_cast<KvT*>(nullptr));
      }
      if (lane < LPR) {
        size_t off;
        bool write = true;
        if (!p.paged) {
          off = ((static_cast<size_t>(b) * Hkv + g) * p.capacity + it.cur) * C::ROW_BYTES;
        } else {
          const int page = __ldcg(p.block_table + static_cast<int64_t>(b) * p.bt_stride + (it.cur >> p.page_shift));
          write = page >= 0 && page < p.n_pages;
          if (!write && lane == 0) set_err(p.err, TTS_EFLAG_PAGE);
          off = ((static_cast<size_t>(write ? page : 0) * Hkv + g) * p.page_size +
                 (it.cur & (p.page_size - 1))) * C::ROW_BYTES;
        }
        if (write) {
#pragma unroll
          for (int j = 0; j < VEC; ++j) {
            const size_t o16 = off + (j * LPR + lr) * 16;
            *reinterpret_cast<uint4*>(static_cast<unsigned char*>(p.k_cache_w) + o16) = kp[j];
            *reinterpret_cast<uint4*>(static_cast<unsigned char*>(p.v_cache_w) + o16) = vp[j];
          }
        }
      }
      // the row as the cache holds it (rounded to the cache type)
#pragma unroll
      for (int j = 0; j < VEC; ++j) {
        float kx[VE], vx[VE];
        KvVec<KvT>::unpack(kp[j], kx);
        KvVec<KvT>::unpack(vp[j], vx);
#pragma unroll
        for (int e = 0; e < VE; ++e) {
          kr[j * VE + e] = kx[e];
          vr[j * VE + e] = vx[e];
        }
      }
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float a0 = 0.f, a1 = 0.f;
#pragma unroll
        for (int k = 0; k < EPL; k += 2) {
          a0 = fmaf(q[h][k], kr[k], a0);
          a1 = fmaf(q[h][k + 1], kr[k + 1], a1);
        }
        float sc = a0 + a1;
#pragma unroll
        for (int off = LPR / 2; off >= 1; off >>= 1) sc += __shfl_xor_sync(kFull, sc, off);
        m_run[h] = sc;
        l_run[h] = lane < LPR ? 1.f : 0.f;
#pragma unroll
        for (int k = 0; k < EPL / 2; ++k)
          o[h][k] = lane < LPR ? make_float2(vr[2 * k], vr[2 * k + 1]) : make_float2(0.f, 0.f);
      }
    }

    if (tid == 0) { if (persistent) TTS_STAMP_ITEM(2, i); else TTS_STAMP(2); }
    // Tiles are consumed in a two-deep software pipeline: the scores of tile t+1 are
    // computed in the same basic block as the softmax and P.V of tile t, so the two
    // dependency chains overlap.  Only the last tile of an item may be partial.
    const int n_full = it.n_rows / T;
    const int tail = it.n_rows - n_full * T;
    float s_cur[STEPS][G], s_nxt[STEPS][G];
    if (ok && n_full > 0) {
      ok = mbar_wait(&full[sc], pc);
      if (tid == 0) { if (persistent) TTS_STAMP_ITEM(3, i); else TTS_STAMP(3); }
      if (ok) tile_scores<C, KvT, false>(ring + sc * C::STAGE_BYTES, T, warp, lane, q2, s_cur);
    }
    for (int t = 0; ok && t + 1 < n_full; ++t) {
      int sn = sc + 1;
      uint32_t pn = pc;
      if (sn == ns) {
        sn = 0;
        pn ^= 1u;
      }
      if (!mbar_wait(&full[sn], pn)) {
        ok = false;
        break;
      }
      tile_scores<C, KvT, false>(ring + sn * C::STAGE_BYTES, T, warp, lane, q2, s_nxt);
      tile_softmax_pv<C, KvT, false>(ring + sc * C::STAGE_BYTES + C::TILE_BYTES, T, warp, lane,
                                     s_cur, m_run, l_run, o);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[sc]);
#pragma unroll
      for (int st = 0; st < STEPS; ++st)
#pragma unroll
        for (int h = 0; h < G; ++h) s_cur[st][h] = s_nxt[st][h];
      sc = sn;
      pc = pn;
    }
    if (ok && n_full > 0) {
      tile_softmax_pv<C, KvT, false>(ring + sc * C::STAGE_BYTES + C::TILE_BYTES, T, warp, lane,
                                     s_cur, m_run, l_run, o);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[sc]);
      if (++sc == ns) {
        sc = 0;
        pc ^= 1u;
      }
    }
    if (ok && tail > 0) {
      if (mbar_wait(&full[sc], pc)) {
        if (n_full == 0 && tid == 0) { if (persistent) TTS_STAMP_ITEM(3, i); else TTS_STAMP(3); }
        tile_scores<C, KvT, true>(ring + sc * C::STAGE_BYTES, tail, warp, lane, q2, s_cur);
        tile_softmax_pv<C, KvT, true>(ring + sc * C::STAGE_BYTES + tail * C::ROW_BYTES, tail, warp,
                                      lane, s_cur, m_run, l_run, o);
        __syncwarp();
        if (lane == 0) mbar_arrive(&empty[sc]);
        if (++sc == ns) {
          sc = 0;
          pc ^= 1u;
        }
      } else {
        ok = false;
      }
    }
    if (!ok) set_err(p.err, TTS_EFLAG_TIMEOUT);
    if (tid == 0) { if (persistent) TTS_STAMP_ITEM(4, i); else TTS_STAMP(4); }

    // Merge the row groups of this warp, then the warps of this CTA.
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
      for (int off = LPR; off < 32; off <<= 1) {
        l_run[h] += __shfl_xor_sync(kFull, l_run[h], off);
#pragma unroll
        for (int k = 0; k < EPL / 2; ++k) {
          o[h][k].x += __shfl_xor_sync(kFull, o[h][k].x, off);
          o[h][k].y += __shfl_xor_sync(kFull, o[h][k].y, off);
        }
      }
    }
    // the scratch may lie over the ring, whose last tiles other warps may still read
    if (p.sm_scratch < p.sm_bar) named_barrier(1, NT);
    if (lane < LPR) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float* dst = scratch + (warp * G + h) * (D + 2);
#pragma unroll
        for (int j = 0; j < VEC; ++j)
#pragma unroll
          for (int e = 0; e < VE; e += 2) {
            dst[(j * LPR + lr) * VE + e] = o[h][(j * VE + e) / 2].x;
            dst[(j * LPR + lr) * VE + e + 1] = o[h][(j * VE + e) / 2].y;
          }
        if (lane == 0) {
          dst[D] = m_run[h];
          dst[D + 1] = l_run[h];
        }
      }
    }
    named_barrier(1, NT);

    const bool direct = it.n_act == 1;  // the window lies in one split: final output here
    for (int idx = tid; idx < G * D; idx += NT) {
      const int h = idx / D;
      const int d = idx - h * D;
      float mw[NC];
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NC; ++w) {
        mw[w] = scratch[(w * G + h) * (D + 2) + D];
        M = fmaxf(M, mw[w]);
      }
      float L = 0.f, O = 0.f;
#pragma unroll
      for (int w = 0; w < NC; ++w) {
        const float* srcp = scratch + (w * G + h) * (D + 2);
        // a warp without rows has m = -inf and l = o = 0; some warp always has rows
        const float f = (mw[w] == -INFINITY) ? 0.f : fast_exp2(mw[w] - M);
        L = fmaf(srcp[D + 1], f, L);
        O = fmaf(srcp[d], f, O);
      }
      const int hq = g * G + h;
      if (direct) {
        if (p.out_packed == nullptr) p.out[(static_cast<int64_t>(b) * Hq + hq) * D + d] = O / L;
        else store_packed1(p.out_packed, p.out_slots, b, hq * D + d, O / L);
      } else if (clustered) {
        float* slot = gather + (split * G + h) * (D + 2);
        if (split == 0) {
          slot[d] = O;
          if (d == 0) {
            slot[D] = M;
            slot[D + 1] = L;
          }
        } else {
          st_cluster_f32(map_shared_rank(slot + d, 0), O);
          if (d == 0) {
            st_cluster_f32(map_shared_rank(slot + D, 0), M);
            st_cluster_f32(map_shared_rank(slot + D + 1, 0), L);
          }
        }
      } else {
        const int64_t slot = (static_cast<int64_t>(b) * Hq + hq) * p.n_splits + split;
        p.ws_o[slot * D + d] = O;
        if (d == 0) reinterpret_cast<float2*>(p.ws_ml)[slot] = make_float2(M, L);
      }
    }
    if (tid == 0) { if (persistent) TTS_STAMP_ITEM(5, i); else TTS_STAMP(5); }

    if (clustered) {
      // Partials travel over distributed shared memory; rank 0 waits (bounded) for the
      // other ranks' arrivals, which release their stores, and merges from its own smem.
      named_barrier(1, NT);
      if (split != 0) {
        if (tid == 0) mbar_arrive_remote(map_shared_rank(gbar, 0));
        return;
      }
      if (!direct) {
        if (!mbar_wait_cluster(gbar, 0u, 8 * kWaitLimitCycles)) {
          if (tid == 0) set_err(p.err, TTS_EFLAG_TIMEOUT);
          return;
        }
        if (tid == 0) { if (persistent) TTS_STAMP_ITEM(6, i); else TTS_STAMP(6); }
        const int n_act = it.n_act;
        // per head: weights 2^(m_s - M) and the sum L, one warp per head (lanes over splits)
        float* sm_w = reinterpret_cast<float*>(comb);  // [G][16] weights, then [G] sums
        for (int h = warp; h < G; h += NC) {
          const float m = lane < n_act ? gather[(lane * G + h) * (D + 2) + D] : -INFINITY;
          float M = m;
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1) M = fmaxf(M, __shfl_xor_sync(kFull, M, off));
          const float w = lane < n_act ? fast_exp2(m - M) : 0.f;
          float L = lane < n_act ? w * gather[(lane * G + h) * (D + 2) + D + 1] : 0.f;
#pragma unroll
          for (int off = 16; off >= 1; off >>= 1) L += __shfl_xor_sync(kFull, L, off);
          if (lane < 16) sm_w[h * 16 + lane] = w;
          if (lane == 0) sm_w[G * 16 + h] = L;
        }
        named_barrier(1, NT);
        for (int idx = tid; idx < G * D; idx += NT) {
          const int h = idx / D;
          const int d = idx - h * D;
          float O = 0.f;
#pragma unroll 4
          for (int s2 = 0; s2 < n_act; ++s2) O = fmaf(gather[(s2 * G + h) * (D + 2) + d], sm_w[h * 16 + s2], O);
          if (p.out_packed == nullptr) p.out[(static_cast<int64_t>(b) * Hq + g * G + h) * D + d] = O / sm_w[G * 16 + h];
          else store_packed1(p.out_packed, p.out_slots, b, (g * G + h) * D + d, O / sm_w[G * 16 + h]);
        }
        if (tid == 0) { if (persistent) TTS_STAMP_ITEM(7, i); else TTS_STAMP(7); }
      }
      return;
    }

    if (persistent) {
      // The previous item's ticket has long returned: if it was the last of its
      // (stream, kv head), merge that pair's partials now.  Then take this item's
      // ticket without waiting for the atomic's result (resolved after the next item).
      if (pend_b >= 0) resolve_pending();
      if (!direct) {
        named_barrier(1, NT);  // every partial store of this item precedes the ticket
        if (tid == 0) pend_prev = atomic_add_acq_rel_gpu(p.ws_cnt + b * Hkv + g, 1);
        pend_b = b;
        pend_g = g;
        pend_nact = it.n_act;
        if (tid == 0) TTS_STAMP_ITEM(6, i);
      }
    } else if (!direct) {
      // Ticket: the last of this (stream, kv head)'s active splits merges all partials.
      named_barrier(1, NT);
      if (tid == 0) {
        const int prev = atomic_add_acq_rel_gpu(p.ws_cnt + b * Hkv + g, 1);
        *s_last = (prev == it.n_act - 1) ? 1 : 0;
      }
      named_barrier(1, NT);
      if (tid == 0) TTS_STAMP(6);
      if (*s_last != 0) {
        combine_splits<C>(p, b, g, it.n_act, tid, comb);
        if (tid == 0) {
          p.ws_cnt[b * Hkv + g] = 0;
          TTS_STAMP(7);
        }
      }
    }
    // the merge scratch and flag are reused by the next item
    named_barrier(1, NT);
    if (persistent && tid == 0) TTS_STAMP_ITEM(7, i);
  }
  if (persistent && pend_b >= 0) resolve_pending();
}

constexpr int kMaxCluster = 16;

constexpr int kMaxListStreams = 2048;  // persistent mode keeps per-stream costs in smem
// 32-bit words of the persistent work list: B + 1 64-bit cost prefix sums, B window
// lengths and B window inputs
constexpr int list_ints(int B) { return 2 * (B + 1) + 2 * B; }
constexpr int kMaxDevices = 64;

template <typename KvT, int D, int G, bool FUSED>
cudaError_t launch_one(const AttnParams& p_in, cudaStream_t s) {
  using C = Cfg<KvT, D, G>;
  auto kern = decode_attn_kernel<KvT, D, G, FUSED>;
  // Per device, computed once under a mutex and copied out (several host threads may
  // launch on several devices): the kernel attributes, the largest cluster of this
  // kernel the GPU can co-schedule (cluster mode is used only up to that size), the SM
  // count, how many CTAs of the persistent configuration fit on one SM, and the deepest
  // ring that still lets two single-item CTAs share an SM.
  struct DeviceInfo {
    bool ready;
    int max_cluster, n_sm, per_sm;
    size_t single_budget;
  };
  static std::mutex info_mutex;
  static DeviceInfo info[kMaxDevices] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= kMaxDevices) return cudaErrorInvalidDevice;
  auto ring_stages = [](int kb) {
    const int n = static_cast<int>((static_cast<size_t>(kb) << 10) / C::STAGE_BYTES);
    return n < 1 ? 1 : (n > C::NS ? C::NS : n);
  };
  DeviceInfo di;
  {
    std::lock_guard<std::mutex> lock(info_mutex);
    if (!info[dev].ready) {
      DeviceInfo nd = {};
      size_t max_smem = C::layout(static_cast<size_t>(C::NS) * C::STAGE_BYTES, kMaxCluster, true, list_ints(kMaxListStreams)).total;
      const size_t single = C::layout(static_cast<size_t>(C::NS) * C::STAGE_BYTES, 0, false, 0).total;
      if (single > max_smem) max_smem = single;
      // no launch can use more than a block may opt into; a layout above it fails to launch
      int optin = 0;
      if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) == cudaSuccess && optin > 0 &&
          max_smem > static_cast<size_t>(optin))
        max_smem = static_cast<size_t>(optin);
      cudaGetLastError();
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(max_smem));
      if (e != cudaSuccess) return e;
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeNonPortableClusterSizeAllowed, 1);
      if (e != cudaSuccess) return e;
      cudaLaunchConfig_t q = {};
      q.gridDim = dim3(kMaxCluster, 1, 1);
      q.blockDim = dim3(C::THREADS);
      q.dynamicSmemBytes =
          C::layout(static_cast<size_t>(ring_stages(TTS_RING_KB_CLUSTER)) * C::STAGE_BYTES, kMaxCluster, false, 0).total;
      cudaLaunchAttribute qa[1];
      qa[0].id = cudaLaunchAttributeClusterDimension;
      qa[0].val.clusterDim.x = kMaxCluster;
      qa[0].val.clusterDim.y = 1;
      qa[0].val.clusterDim.z = 1;
      q.attrs = qa;
      q.numAttrs = 1;
      int mc = 1;
      if (cudaOccupancyMaxPotentialClusterSize(&mc, kern, &q) != cudaSuccess) {
        cudaGetLastError();
        mc = 8;  // portable cluster size
      }
      nd.max_cluster = mc < 1 ? 1 : (mc > kMaxCluster ? kMaxCluster : mc);
      if (cudaDeviceGetAttribute(&nd.n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || nd.n_sm < 1) {
        cudaGetLastError();
        nd.n_sm = 1;
      }
      int occ = 0;
      const size_t stream_smem =
          C::layout(static_cast<size_t>(ring_stages(TTS_RING_KB_STREAM)) * C::STAGE_BYTES, 0, true, list_ints(64), 16).total;
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&occ, kern, C::THREADS, stream_smem) != cudaSuccess || occ < 1) {
        cudaGetLastError();
        occ = 1;
      }
      nd.per_sm = occ;
      int sm_bytes = 0, reserved = 0;
      if (cudaDeviceGetAttribute(&sm_bytes, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) != cudaSuccess ||
          cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) != cudaSuccess) {
        cudaGetLastError();
        sm_bytes = 0;
      }
      nd.single_budget = static_cast<size_t>(sm_bytes) / 2 - static_cast<size_t>(reserved);
      nd.ready = true;
      info[dev] = nd;
    }
    di = info[dev];
  }
  const int max_cluster = di.max_cluster, n_sm = di.n_sm, per_sm = di.per_sm;
  const size_t single_budget = di.single_budget;
  AttnParams p = p_in;
  // Clusters pay off when the whole grid is one wave of one CTA per SM (few streams).
  // A grid larger than what fits at once becomes persistent: as many CTAs as fit, each
  // walking the list of active (stream, kv head, split) items.
  const long long ctas = static_cast<long long>(p.n_splits) * p.n_kv_heads * p.B;
  const bool one_wave = ctas <= n_sm;
  p.cluster = (p.n_splits > 1 && p.n_splits <= max_cluster && p.ws_o != nullptr && one_wave) ? p.n_splits : 0;
  const long long resident = static_cast<long long>(n_sm) * per_sm;
  // (the work counters live in the workspace, which a one-split launch does not have;
  // such a grid runs as several plain waves)
  p.persistent = (p.cluster == 0 && ctas > resident && p.B <= kMaxListStreams && p.ws_sched != nullptr) ? 1 : 0;
  // Ring: a split held whole when it fits two CTAs to an SM, else as many full stages as
  // the mode allows (at most the split's tiles).
  const int ntiles = (p.split_len + C::T - 1) / C::T;
  size_t ring_bytes;
  if (p.persistent || p.cluster > 1) {
    int ns = ring_stages(p.persistent ? TTS_RING_KB_STREAM : TTS_RING_KB_CLUSTER);
    // a persistent launch picks its split length on the device (up to the capacity);
    // the consumers' two-deep pipeline needs two stages once an item has two tiles
    const int item_tiles = p.persistent ? (p.capacity + C::T - 1) / C::T : ntiles;
    if (ns > item_tiles) ns = item_tiles;
    if (ns < 2 && item_tiles >= 2) ns = 2;
    p.n_stages = ns;
    ring_bytes = static_cast<size_t>(ns) * C::STAGE_BYTES;
  } else {
    const int last = p.split_len - (ntiles - 1) * C::T;
    const size_t whole = static_cast<size_t>(ntiles - 1) * C::STAGE_BYTES + 2 * static_cast<size_t>(last) * C::ROW_BYTES;
    if (ntiles <= C::NS && C::layout(whole, 0, false, 0).total <= single_budget) {
      p.n_stages = ntiles;
      ring_bytes = whole;
    } else {
      int ns = ntiles < C::NS ? ntiles : C::NS;
      while (ns > 1 && C::layout(static_cast<size_t>(ns) * C::STAGE_BYTES, 0, false, 0).total > single_budget) --ns;
      p.n_stages = ns;
      ring_bytes = static_cast<size_t>(ns) * C::STAGE_BYTES;
    }
  }
  const typename C::Layout L =
      C::layout(ring_bytes, p.cluster, p.persistent != 0, p.persistent ? list_ints(p.B) : 0, p.n_splits);
  p.inflight = p.persistent ? TTS_INFLIGHT_STREAM : TTS_INFLIGHT_SINGLE;
  p.sm_bar = static_cast<uint32_t>(L.bar);
  p.sm_scratch = static_cast<uint32_t>(L.scratch);
  p.sm_flag = static_cast<uint32_t>(L.flag);
  p.sm_comb = static_cast<uint32_t>(L.comb);
  p.sm_gather = static_cast<uint32_t>(L.gather);
  p.sm_list = static_cast<uint32_t>(L.list);
  p.sm_qbuf = static_cast<uint32_t>(L.qbuf);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = p.persistent ? dim3(static_cast<unsigned>(resident), 1, 1) : dim3(p.n_splits, p.n_kv_heads, p.B);
  cfg.dynamicSmemBytes = L.total;
  cfg.blockDim = dim3(C::THREADS);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = p.cluster > 1 ? p.cluster : 1;
  attr[1].val.clusterDim.y = 1;
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = p.cluster > 1 ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <typename KvT, int D>
cudaError_t dispatch_group(const AttnParams& p, int group, bool fused, cudaStream_t s) {
  switch (group) {
    case 1: return fused ? launch_one<KvT, D, 1, true>(p, s) : launch_one<KvT, D, 1, false>(p, s);
    case 2: return fused ? launch_one<KvT, D, 2, true>(p, s) : launch_one<KvT, D, 2, false>(p, s);
    case 4: return fused ? launch_one<KvT, D, 4, true>(p, s) : launch_one<KvT, D, 4, false>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

template <typename KvT, int D>
AttnGeometry geometry_of() {
  using C = Cfg<KvT, D, 1>;
  return AttnGeometry{C::T, C::NS, C::STAGE_BYTES, C::THREADS};
}

}  // namespace

AttnGeometry attn_geometry(int kv_bf16, int head_dim) {
  if (kv_bf16) return head_dim == 64 ? geometry_of<__nv_bfloat16, 64>() : geometry_of<__nv_bfloat16, 128>();
  return head_dim == 64 ? geometry_of<float, 64>() : geometry_of<float, 128>();
}

cudaError_t launch_decode_attn(const AttnParams& p, int kv_bf16, int head_dim, int group,
                               bool fused, cudaStream_t s) {
  if (kv_bf16) {
    if (head_dim == 64) return dispatch_group<__nv_bfloat16, 64>(p, group, fused, s);
    if (head_dim == 128) return dispatch_group<__nv_bfloat16, 128>(p, group, fused, s);
  } else {
    if (head_dim == 64) return dispatch_group<float, 64>(p, group, fused, s);
    if (head_dim == 128) return dispatch_group<float, 128>(p, group, fused, s);
  }
  return cudaErrorInvalidValue;
}

#ifdef TTS_TRACE
// Copies the timeline of the last traced launch to host memory (n_ctas x 8 stamps).
extern "C" int tts_trace_read(unsigned long long* host, int n_ctas) {
  if (n_ctas > kTraceCtas) n_ctas = kTraceCtas;
  return static_cast<int>(cudaMemcpyFromSymbol(host, g_trace, sizeof(unsigned long long) * kTraceSlots * n_ctas));
}
extern "C" int tts_trace_clear(void) {
  static unsigned long long zeros[kTraceCtas][kTraceSlots];
  return static_cast<int>(cudaMemcpyToSymbol(g_trace, zeros, sizeof(zeros)));
}
#endif

}  // namespace tts
