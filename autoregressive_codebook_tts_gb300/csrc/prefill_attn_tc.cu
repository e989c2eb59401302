// Multi-query prefill attention on the 5th-generation tensor cores, for bf16 caches with
// head_dim 128 ("qwentts.cpp -- src/pipeline-tts.h" commit page, KV-cache section: the
// prefill writes the prompt's rows, query t of stream b sees positions
// [0, start[b] + t + 1)).  A work item is 128 query rows (128 / G queries of a stream
// times the G q heads of one kv head), the MMA's M; its window is cut on the device into
// n_ch chunks of whole tiles, one CTA per (item, chunk).  The chunks merge inside a
// thread-block cluster (2..8 chunks whose clusters the device keeps resident at once:
// distributed shared memory, chunk order) or in prefill_combine_kernel after the launch.
//
// Per 64-row tile of the chunk (N = 64 cache rows):
//   S = Q_hi K^T + Q_lo K^T          two K-major bf16 products (K = D = 128), the query
//                                    rows split once into a bf16 value and its bf16
//                                    remainder, so S carries about 16 bits of q; K is
//                                    exact in bf16;
//   online softmax in base 2 with the causal mask (the row's window end) and the chunk
//   end.  Two warpgroups share the work: query row r is TMEM lane r for both, the first
//   takes score columns 0-31 (and O columns 0-63), the second 32-63 (O 64-127); they
//   agree on the row maximum through shared memory at one named barrier a tile, whose
//   AND-reduction also makes every bounded wait's outcome common to both.  The running
//   maximum moves only when a row's maximum grows by more than 2^8, and then O is
//   rescaled in tensor memory (the result is the same: O and the row sum are both
//   relative to the maximum in use);
//   O += P_hi V + P_lo V             P split like q; V is the MN-major operand (stored
//                                    [row][d]); K = 64 rows.
// S has two tensor-memory buffers (the product of tile t+1 runs while tile t's softmax
// does), O one (128 columns); P has two shared-memory buffers, so tile t's softmax waits
// for O += P(t-2) V(t-2) only, and for O += P(t-1) V(t-1) only when it rescales O.  K
// and V have rings of their own (3 and 2 stages): a K stage frees when S is done, a V
// stage when its product with P is.  Warps 0-7 are the softmax warps, warp 8 streams K
// and V tiles with 3-D tensor-map loads (one per tile and operand), warp 9 allocates
// tensor memory and issues the products.  In the last tile, V rows past the chunk are
// zeroed before their product (a cache tail may hold anything).
// The K/V tiles below the prompt stream before the dependency wait (they were final
// before the rows launch let this one start); the producer waits before the first tile
// that holds prompt rows, the softmax warps before the query rows (both the rows
// launch's).  Every wait is bounded; on expiry TTS_EFLAG_TIMEOUT is set and the CTA
// winds down.
#include <cstdint>
#include <mutex>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace tts {
namespace {

constexpr int kD = 128;
constexpr int kM = 128;                   // query rows of an item
constexpr int kN = kPrefillTile;          // cache rows of a tile (64)
constexpr int kNK = 3, kNV = 2;           // K and V ring stages
constexpr int kSmxWarps = 8;              // two softmax warpgroups
constexpr int kProducerWarp = 8, kMmaWarp = 9;
constexpr int kThreads = 320;
constexpr int kQBytes = kM * kD * 2;      // 32 KB: two 64-column swizzled chunks
constexpr int kTileBytes = kN * kD * 2;   // 16 KB
constexpr int kPBytes = kM * kN * 2;      // 16 KB: one 64-column swizzled chunk
constexpr int kTmemCols = 256;            // S[2] (2 x 64) + O (128)
constexpr int kMaxClusterCh = 8;          // chunks merged in a cluster (portable size)

// smem: Q_hi | Q_lo | K ring x kNK | V ring x kNV | (P_hi | P_lo) x 2 | row maxima
// [2][2][128] | row sums [2][128] | barriers
constexpr int kOffQh = 0, kOffQl = kQBytes, kOffK = 2 * kQBytes, kOffV = kOffK + kNK * kTileBytes;
constexpr int kOffP = kOffV + kNV * kTileBytes;   // P buffer i: hi at kOffP + 2 i kPBytes, lo after it
constexpr int kOffMax = kOffP + 4 * kPBytes, kOffSum = kOffMax + 2 * 2 * kM * 4;
constexpr int kOffBar = kOffSum + 2 * kM * 4;
constexpr size_t kSmem = 1024 + kOffBar + 32 * sizeof(uint64_t);

__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo) {
  return static_cast<uint64_t>((addr & 0x3FFFF) >> 4) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(2) << 61);   // 128-byte swizzle
}

// Byte offset of bf16 element (r, col) of a tile of R rows stored as 64-column chunks of
// 128-byte rows with the 128-byte swizzle (16-byte unit u of row r at (u ^ r % 8)).
__device__ __forceinline__ uint32_t sw_off(int r, int col, int R) {
  const int c = col >> 6, o = (col & 63) * 2;
  return static_cast<uint32_t>(c * (R * 128) + r * 128 + ((((o >> 4) ^ (r & 7)) << 4) | (o & 15)));
}

__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c1, uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(0), "r"(c1), "r"(0), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

__device__ __forceinline__ void mma_f16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
      "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
      ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(acc) : "memory");
}
__device__ __forceinline__ void mma_commit(uint64_t* bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
               ::"r"(smem_u32(bar)) : "memory");
}

// 32 consecutive columns of this thread's TMEM lane (a row of its warp's 32 lanes).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]),
        "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]),
        "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const float (&v)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};"
      ::"r"(taddr), "r"(__float_as_uint(v[0])), "r"(__float_as_uint(v[1])), "r"(__float_as_uint(v[2])),
        "r"(__float_as_uint(v[3])), "r"(__float_as_uint(v[4])), "r"(__float_as_uint(v[5])),
        "r"(__float_as_uint(v[6])), "r"(__float_as_uint(v[7])), "r"(__float_as_uint(v[8])),
        "r"(__float_as_uint(v[9])), "r"(__float_as_uint(v[10])), "r"(__float_as_uint(v[11])),
        "r"(__float_as_uint(v[12])), "r"(__float_as_uint(v[13])), "r"(__float_as_uint(v[14])),
        "r"(__float_as_uint(v[15])), "r"(__float_as_uint(v[16])), "r"(__float_as_uint(v[17])),
        "r"(__float_as_uint(v[18])), "r"(__float_as_uint(v[19])), "r"(__float_as_uint(v[20])),
        "r"(__float_as_uint(v[21])), "r"(__float_as_uint(v[22])), "r"(__float_as_uint(v[23])),
        "r"(__float_as_uint(v[24])), "r"(__float_as_uint(v[25])), "r"(__float_as_uint(v[26])),
        "r"(__float_as_uint(v[27])), "r"(__float_as_uint(v[28])), "r"(__float_as_uint(v[29])),
        "r"(__float_as_uint(v[30])), "r"(__float_as_uint(v[31]))
      : "memory");
}

// 2 NP values as NP packed pairs of bf16 values (hi = bf16(x)) and of their bf16
// remainders (lo = bf16(x - hi); x - hi is exact, so the fused negate-add computes it
// without rounding); split_unit stores eight of them as one 16-byte unit of each at the
// swizzled unit position of row r.
template <int NP>
__device__ __forceinline__ void split_pairs(const float* x, uint32_t (&h)[NP], uint32_t (&l)[NP]) {
#pragma unroll
  for (int e = 0; e < NP; ++e) {
    const __nv_bfloat162 hb = __floats2bfloat162_rn(x[2 * e], x[2 * e + 1]);
    h[e] = *reinterpret_cast<const uint32_t*>(&hb);
    const float2 hf = make_float2(__uint_as_float(h[e] << 16), __uint_as_float(h[e] & 0xFFFF0000u));
    const float2 rem = __ffma2_rn(hf, make_float2(-1.f, -1.f), make_float2(x[2 * e], x[2 * e + 1]));
    const __nv_bfloat162 lb = __floats2bfloat162_rn(rem.x, rem.y);
    l[e] = *reinterpret_cast<const uint32_t*>(&lb);
  }
}
__device__ __forceinline__ void split_unit(const float* x, unsigned char* hi_row, unsigned char* lo_row, int u,
                                           int r) {
  uint32_t h[4], l[4];
  split_pairs(x, h, l);
  const uint32_t off = static_cast<uint32_t>((u ^ (r & 7)) << 4);
  *reinterpret_cast<uint4*>(hi_row + off) = make_uint4(h[0], h[1], h[2], h[3]);
  *reinterpret_cast<uint4*>(lo_row + off) = make_uint4(l[0], l[1], l[2], l[3]);
}

// 8 and 16 bytes of another CTA's shared memory (cluster-window addresses from mapa).
__device__ __forceinline__ float2 ld_cluster_f32x2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared::cluster.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ float4 ld_cluster_f32x4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
  return v;
}

// Named barrier 1 over the 256 softmax threads.
__device__ __forceinline__ void softmax_sync() { asm volatile("bar.sync 1, 256;" ::: "memory"); }
// The same barrier, returning the AND of every thread's v
// (warp-convergent: each warp reaches it with all lanes).
__device__ __forceinline__ bool softmax_sync_and(bool v) {
  uint32_t out;
  asm volatile(
      "{\n\t.reg .pred pi, po;\n\tsetp.ne.u32 pi, %1, 0;\n\t"
      "bar.red.and.pred po, 1, 256, pi;\n\tselp.u32 %0, 1, 0, po;\n\t}"
      : "=r"(out) : "r"(static_cast<uint32_t>(v)) : "memory");
  return out != 0;
}

// 2^x with the MUFU instruction (relative error about 2^-22; 2^-inf = 0, results below
// 2^-126 flush to 0, far below what a softmax weight can contribute).
__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

template <int G>
__global__ void __launch_bounds__(kThreads, 1) prefill_attn_tc_kernel(const __grid_constant__ CUtensorMap kmap,
                                                                       const __grid_constant__ CUtensorMap vmap,
                                                                       const PrefillAttnParams p) {
  constexpr int QB = kM / G;   // queries of an item
  constexpr int kSmx = kSmxWarps * 32;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  unsigned char* sQh = smem + kOffQh;
  unsigned char* sQl = smem + kOffQl;
  unsigned char* sK = smem + kOffK;
  unsigned char* sV = smem + kOffV;
  unsigned char* sP = smem + kOffP;
  float* s_max = reinterpret_cast<float*>(smem + kOffMax);       // [tile parity][half][row]
  float* s_sum = reinterpret_cast<float*>(smem + kOffSum);       // [half][row]
  float* so = reinterpret_cast<float*>(smem + kOffK);            // O staging [row][128] after the loop
  float2* s_ml = reinterpret_cast<float2*>(smem + kOffMax);      // (max, sum) per row after the loop
  uint64_t* fullK = reinterpret_cast<uint64_t*>(smem + kOffBar); // [kNK] K(t) landed
  uint64_t* emptyK = fullK + kNK;                                // [kNK] S(t) done
  uint64_t* fullV = emptyK + kNK;                                // [kNV] V(t) landed
  uint64_t* emptyV = fullV + kNV;                                // [kNV] O += P(t) V(t) done
  uint64_t* qready = emptyV + kNV;                               // the split query rows written
  uint64_t* sready = qready + 1;                                 // [2] S(t) in tensor memory
  uint64_t* sfree = sready + 2;                                  // [2] S(t) read by every thread
  uint64_t* pready = sfree + 2;                                  // [2] P(t) written (and O rescaled)
  uint64_t* pvdone = pready + 2;                                 // [2] O += P(t) V(t) done (P buffer t & 1)
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(pvdone + 2);

  const int item = blockIdx.x, ch = blockIdx.y;
  const int qb = item % p.n_qb, bg = item / p.n_qb;
  const int g = bg % p.n_kv_heads, b = bg / p.n_kv_heads;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = qb * QB;
  const int nq = min(QB, p.T - t0);

  if (tid == 0) {
    for (int s = 0; s < kNK; ++s) {
      mbar_init(&fullK[s], 1);
      mbar_init(&emptyK[s], 1);
    }
    for (int s = 0; s < kNV; ++s) {
      mbar_init(&fullV[s], 1);
      mbar_init(&emptyV[s], 1);
    }
    mbar_init(qready, kSmx);
    for (int i = 0; i < 2; ++i) {
      mbar_init(&sready[i], 1);
      mbar_init(&sfree[i], kSmx);
      mbar_init(&pready[i], kSmx);
      mbar_init(&pvdone[i], 1);
    }
    mbar_init_fence();
  }
  if (warp == kMmaWarp) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(s_tmem)), "n"(kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t tO = tmem + 2 * kN;   // S(t) at tmem + (t & 1) * kN
  grid_launch_dependents();
  // start[] and the cache rows below the prompt were final before the rows launch began
  // (it waits for its own predecessor before it lets this launch start), so they are
  // read before the dependency wait; the prompt's cache rows and the rotated q rows are
  // the rows launch's, read after it (the producer waits before the first tile that
  // holds a prompt row, the softmax warps before the query rows)
  const int st = __ldcg(p.start + b);
  const int nv_max = min(max(st + t0 + nq, 1), p.capacity);
  const int ch_len = prefill_chunk_len(nv_max, p.n_ch);
  const int c0 = ch * ch_len;
  const int c1 = min(c0 + ch_len, nv_max);
  const int ntiles = c0 < nv_max ? (c1 - c0 + kN - 1) / kN : 0;

  if (warp == kProducerWarp) {
    // ---------------------------------------------------------------- producer
    // K(t) goes into its stage once S(t - kNK) is done, V(t) once O += P(t - kNV) V(t - kNV) is
    if (lane == 0 && ntiles > 0) {
      int nk = 0, nvv = 0;   // K and V tiles issued
      bool ok = true, waited = false;
      for (int i = 0; i < ntiles; ++i) {
        const int r0 = c0 + i * kN;
        if (!waited && r0 + kN > st) {
          grid_wait();
          waited = true;
        }
        int row;
        if (!p.paged) {
          row = (b * p.n_kv_heads + g) * p.capacity + r0;
        } else {
          // pages of 64 rows or more: the tile (64 rows from a multiple of 64) lies in one page
          int page = __ldcg(p.block_table + static_cast<int64_t>(b) * p.bt_stride + r0 / p.page_size);
          if (page < 0 || page >= p.n_pages) {
            set_err(p.err, TTS_EFLAG_PAGE);
            page = 0;
          }
          row = (page * p.n_kv_heads + g) * p.page_size + (r0 & (p.page_size - 1));
        }
        const int ks = i % kNK, vs = i % kNV;
        if (i >= kNK && !mbar_wait(&emptyK[ks], static_cast<uint32_t>((i / kNK) - 1) & 1u)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&fullK[ks], kTileBytes);
        tma_load_3d(sK + ks * kTileBytes, &kmap, row, &fullK[ks]);
        nk = i + 1;
        if (i >= kNV && !mbar_wait(&emptyV[vs], static_cast<uint32_t>((i / kNV) - 1) & 1u)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&fullV[vs], kTileBytes);
        tma_load_3d(sV + vs * kTileBytes, &vmap, row, &fullV[vs]);
        nvv = i + 1;
      }
      if (!ok) set_err(p.err, TTS_EFLAG_TIMEOUT);
      // every copy still in flight lands before the CTA ends (earlier ones were consumed)
      for (int t = max(0, nk - kNK); t < nk; ++t) mbar_wait(&fullK[t % kNK], static_cast<uint32_t>(t / kNK) & 1u);
      for (int t = max(0, nvv - kNV); t < nvv; ++t) mbar_wait(&fullV[t % kNV], static_cast<uint32_t>(t / kNV) & 1u);
    }
  } else if (warp == kMmaWarp) {
    // -------------------------------------------------------------- MMA issuer
    // Barriers with one phase per tile come in pairs (tile parity) wherever a waiter could
    // otherwise see a later tile's phase: each wait below is for a phase that cannot be
    // overtaken before the waiter has passed it.
    if (lane == 0 && ntiles > 0) {
      // kind::f16, f32 accumulator, bf16 A and B; S: N = 64, both K-major; O: N = 128,
      // B (V) MN-major (bit 16)
      const uint32_t idS = (1u << 4) | (1u << 7) | (1u << 10) | ((kN >> 3) << 17) | ((kM >> 4) << 24);
      const uint32_t idO =
          (1u << 4) | (1u << 7) | (1u << 10) | (1u << 16) | ((kD >> 3) << 17) | ((kM >> 4) << 24);
      const uint32_t qh = smem_u32(sQh), ql = smem_u32(sQl), pb = smem_u32(sP);
      auto issue_s = [&](int t) {
        const uint32_t kb = smem_u32(sK + (t % kNK) * kTileBytes);
        const uint32_t d = tmem + (t & 1) * kN;
        // K = 128 in steps of 16: 64-column chunk j / 4, 32 bytes a step within it
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t qo = (j >> 2) * (kM * 128) + (j & 3) * 32, ko = (j >> 2) * (kN * 128) + (j & 3) * 32;
          mma_f16(d, smem_desc(qh + qo, 16, 1024), smem_desc(kb + ko, 16, 1024), idS, j > 0 ? 1u : 0u);
        }
#pragma unroll
        for (int j = 0; j < 8; ++j) {
          const uint32_t qo = (j >> 2) * (kM * 128) + (j & 3) * 32, ko = (j >> 2) * (kN * 128) + (j & 3) * 32;
          mma_f16(d, smem_desc(ql + qo, 16, 1024), smem_desc(kb + ko, 16, 1024), idS, 1u);
        }
        mma_commit(&sready[t & 1]);
        mma_commit(&emptyK[t % kNK]);
      };
      auto issue_pv = [&](int t) {
        const uint32_t vb = smem_u32(sV + (t % kNV) * kTileBytes);
        const uint32_t ph = pb + (t & 1) * 2 * kPBytes, pl = ph + kPBytes;
        // K = 64 cache rows in steps of 16: P 32 bytes a step; V (MN-major) 16 rows =
        // 2048 bytes a step, its 64-column chunks 8192 bytes apart
#pragma unroll
        for (int j = 0; j < 4; ++j)
          mma_f16(tO, smem_desc(ph + j * 32, 16, 1024), smem_desc(vb + j * 2048, 8192, 1024), idO,
                  (t > 0 || j > 0) ? 1u : 0u);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          mma_f16(tO, smem_desc(pl + j * 32, 16, 1024), smem_desc(vb + j * 2048, 8192, 1024), idO, 1u);
        mma_commit(&emptyV[t % kNV]);
        mma_commit(&pvdone[t & 1]);
      };
      auto wait_pv_inputs = [&](int t) {
        return mbar_wait(&pready[t & 1], static_cast<uint32_t>(t >> 1) & 1u) &&
               mbar_wait(&fullV[t % kNV], static_cast<uint32_t>(t / kNV) & 1u);
      };
      bool ok = mbar_wait(qready, 0);
      int t = 0;
      for (; ok && t < ntiles; ++t) {
        if (!mbar_wait(&fullK[t % kNK], static_cast<uint32_t>(t / kNK) & 1u)) ok = false;
        if (ok && t >= 2 && !mbar_wait(&sfree[t & 1], static_cast<uint32_t>((t - 2) >> 1) & 1u)) ok = false;
        if (!ok) break;
        tc_fence_after();
        issue_s(t);
        if (t >= 1) {
          if (!wait_pv_inputs(t - 1)) {
            ok = false;
            break;
          }
          tc_fence_after();
          issue_pv(t - 1);
        }
      }
      if (ok) {
        if (wait_pv_inputs(ntiles - 1)) {
          tc_fence_after();
          issue_pv(ntiles - 1);
        } else {
          ok = false;
        }
      }
      if (!ok) set_err(p.err, TTS_EFLAG_TIMEOUT);
    }
  } else {
    // ---------------------------------------------------------- softmax warps
    const int w = warp >> 2;                    // column half: S 32 w.., O 64 w..
    const int r = (warp & 3) * 32 + lane;       // query row = TMEM lane
    const int tl = r / G, h = r - tl * G;
    const int raw = st + t0 + tl + 1;
    // the row's window end within the chunk; rows past the prompt run on zero query rows
    // and store nothing
    const int lim = tl < nq ? min(min(max(raw, 1), p.capacity), c1) : c1;
    if (w == 0 && ch == 0 && g == 0 && h == 0 && tl < nq && (raw < 1 || raw > p.capacity))
      set_err(p.err, TTS_EFLAG_NVALID);
    // the query rows (normed and rotated by the rows launch: read after the dependency
    // wait), split into bf16 value and remainder in the swizzled A layout: warp k takes
    // rows 16k..16k+15, one coalesced 512-byte row per load (lane j holds columns
    // 4j..4j+3: 64-column chunk j / 16, 16-byte unit (j % 16) / 2, half j % 2)
    {
      grid_wait();
      float4 v[16];
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int rr = warp * 16 + i, tr = rr / G, hr = rr - tr * G;
        v[i] = tr < nq ? __ldcg(reinterpret_cast<const float4*>(p.q + static_cast<int64_t>(b * p.T + t0 + tr) * p.q_stride +
                                                                (g * G + hr) * kD) + lane)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const int rr = warp * 16 + i;
        const uint32_t off = static_cast<uint32_t>((lane >> 4) * (kM * 128) + rr * 128 +
                                                   ((((lane & 15) >> 1) ^ (rr & 7)) << 4) + ((lane & 1) << 3));
        const float x[4] = {v[i].x, v[i].y, v[i].z, v[i].w};
        uint32_t hq[2], lq[2];
        split_pairs(x, hq, lq);
        *reinterpret_cast<uint2*>(sQh + off) = make_uint2(hq[0], hq[1]);
        *reinterpret_cast<uint2*>(sQl + off) = make_uint2(lq[0], lq[1]);
      }
    }
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_arrive(qready);
    const uint32_t lane_base = static_cast<uint32_t>((warp & 3) * 32) << 16;
    const float c = p.scale_log2;
    float m_used = -INFINITY, l = 0.f;
    bool ok = ntiles > 0, bad = false;
    for (int t = 0; ok && t < ntiles; ++t) {
      const int r0 = c0 + t * kN, base = r0 + 32 * w;   // cache row of this thread's first score
      float sv[32];
      float mx = -INFINITY;
      // wait results are made warp-uniform (the tensor-memory loads are warp-wide) and
      // then common to both warpgroups at the barrier below
      bool good = __all_sync(kFull, mbar_wait(&sready[t & 1], static_cast<uint32_t>(t >> 1) & 1u));
      if (good) {
        tc_fence_after();
        tmem_ld32(tmem + (t & 1) * kN + lane_base + 32 * w, sv);
        tc_fence_before();
        mbar_arrive(&sfree[t & 1]);
        if (!__all_sync(kFull, base + 32 <= lim)) {
#pragma unroll
          for (int j = 0; j < 32; ++j) sv[j] = base + j < lim ? sv[j] : -INFINITY;
        }
        float m16[16];
#pragma unroll
        for (int j = 0; j < 16; ++j) m16[j] = fmaxf(sv[j], sv[j + 16]);
#pragma unroll
        for (int s = 8; s >= 1; s >>= 1)
#pragma unroll
          for (int j = 0; j < s; ++j) m16[j] = fmaxf(m16[j], m16[j + s]);
        mx = m16[0];
        // P buffer t & 1 is the product's until O += P(t-2) V(t-2) is done
        if (t >= 2) good = __all_sync(kFull, mbar_wait(&pvdone[t & 1], static_cast<uint32_t>((t - 2) >> 1) & 1u));
        // the last tile's V rows past the chunk are zeroed below: the tile must have landed
        if (good && t == ntiles - 1 && c1 - r0 < kN)
          good = __all_sync(kFull, mbar_wait(&fullV[t % kNV], static_cast<uint32_t>(t / kNV) & 1u));
      }
      float* mrow = s_max + (t & 1) * 2 * kM;
      mrow[w * kM + r] = mx;
      if (!softmax_sync_and(good && !bad)) {
        ok = false;
        break;
      }
      const float mxs = fmaxf(mx, mrow[(1 - w) * kM + r]) * c;   // the row's maximum, base 2
      // a row moves its maximum in use only when it grew by more than 2^8; rows whose
      // O holds earlier tiles rescale their half of it (every lane of the warp takes part
      // in the tensor-memory round trip, a row that keeps its maximum with factor 1)
      const bool move = mxs > m_used + 8.0f;
      const bool rescale = move && m_used > -INFINITY;
      const float alpha = rescale ? ex2(m_used - mxs) : 1.0f;
      if (__any_sync(kFull, rescale)) {
        // O holds tiles up to t-1 once O += P(t-1) V(t-1) is done (t >= 1 here: the
        // maximum in use is finite); an expired wait skips the rescale and ends the loop
        // at the next barrier
        if (__all_sync(kFull, mbar_wait(&pvdone[(t - 1) & 1], static_cast<uint32_t>((t - 1) >> 1) & 1u))) {
          tc_fence_after();
#pragma unroll
          for (int cc = 0; cc < 2; ++cc) {
            float o[32];
            tmem_ld32(tO + lane_base + 64 * w + 32 * cc, o);
#pragma unroll
            for (int e = 0; e < 32; ++e) o[e] *= alpha;
            tmem_st32(tO + lane_base + 64 * w + 32 * cc, o);
          }
          asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory");
        } else {
          bad = true;
        }
      }
      if (move) {
        l *= alpha;
        m_used = mxs;
      }
      const float msub = m_used == -INFINITY ? 0.f : m_used;
      float2 acc[4] = {make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f), make_float2(0.f, 0.f)};
#pragma unroll
      for (int i = 0; i < 16; ++i) {
        const float2 z = __ffma2_rn(make_float2(sv[2 * i], sv[2 * i + 1]), make_float2(c, c), make_float2(-msub, -msub));
        sv[2 * i] = ex2(z.x);
        sv[2 * i + 1] = ex2(z.y);
        acc[i & 3] = __fadd2_rn(acc[i & 3], make_float2(sv[2 * i], sv[2 * i + 1]));
      }
      const float2 a01 = __fadd2_rn(acc[0], acc[1]), a23 = __fadd2_rn(acc[2], acc[3]);
      const float2 a = __fadd2_rn(a01, a23);
      l += a.x + a.y;
      if (t == ntiles - 1 && c1 - r0 < kN) {
        // V rows past the chunk take part in the product with weight 0: make them 0
        const int nrow = c1 - r0;
        unsigned char* vt = sV + (t % kNV) * kTileBytes;
        for (int idx = tid; idx < (kN - nrow) * 16; idx += kSmx) {
          const int row = nrow + idx / 16, u = idx % 16;
          *reinterpret_cast<uint4*>(vt + sw_off(row, u * 8, kN)) = make_uint4(0, 0, 0, 0);
        }
      }
      unsigned char* ph = sP + (t & 1) * 2 * kPBytes + r * 128;
#pragma unroll
      for (int u = 0; u < 4; ++u) split_unit(sv + 8 * u, ph, ph + kPBytes, 4 * w + u, r);
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      tc_fence_before();
      mbar_arrive(&pready[t & 1]);
    }
    bool staged = false;
    if (ok) {
      const int tlast = ntiles - 1;
      const bool done = __all_sync(kFull, mbar_wait(&pvdone[tlast & 1], static_cast<uint32_t>(tlast >> 1) & 1u));
      s_sum[w * kM + r] = l;
      ok = softmax_sync_and(done && !bad);
      if (ok) {
        tc_fence_after();
        const float lt = l + s_sum[(1 - w) * kM + r];
        const float inv = p.n_ch == 1 ? (lt > 0.f ? 1.f / lt : 0.f) : 1.f;
        // O staged in the K and V rings (every product is done, every load consumed):
        // row r's 16-byte unit u at (u ^ r % 32), so that both the row-per-lane writes
        // here and the unit-per-lane reads below are conflict-free
#pragma unroll
        for (int cc = 0; cc < 2; ++cc) {
          float o[32];
          tmem_ld32(tO + lane_base + 64 * w + 32 * cc, o);
#pragma unroll
          for (int e = 0; e < 8; ++e) {
            const int u = 16 * w + 8 * cc + e;
            *reinterpret_cast<float4*>(so + r * kD + ((u ^ (r & 31)) << 2)) =
                make_float4(o[4 * e] * inv, o[4 * e + 1] * inv, o[4 * e + 2] * inv, o[4 * e + 3] * inv);
          }
        }
        staged = true;
        if (p.merge_in_cluster) {
          if (w == 0) s_ml[r] = make_float2(m_used, lt);   // the loop's maxima are all read
        } else {
          if (w == 0 && tl < nq && p.n_ch > 1)
            reinterpret_cast<float2*>(p.ml)[(static_cast<int64_t>(item) * p.n_ch + ch) * kM + r] =
                make_float2(m_used, lt);
          softmax_sync();
          // coalesced stores: warp k writes rows 16k..16k+15, lane j the row's unit j;
          // rows past the prompt store nothing
#pragma unroll 4
          for (int i = 0; i < 16; ++i) {
            const int rr = warp * 16 + i, tr = rr / G, hr = rr - tr * G;
            if (tr < nq) {
              const int64_t orow = p.n_ch == 1 ? static_cast<int64_t>(b * p.T + t0 + tr) * p.n_q_heads + g * G + hr
                                               : (static_cast<int64_t>(item) * p.n_ch + ch) * kM + rr;
              float* dst = (p.n_ch == 1 ? p.out : p.part) + orow * kD;
              reinterpret_cast<float4*>(dst)[lane] =
                  *reinterpret_cast<const float4*>(so + rr * kD + ((lane ^ (rr & 31)) << 2));
            }
          }
        }
      }
    }
    // a chunk with no rows (or whose waits ran out) adds nothing to the cluster's merge
    if (p.merge_in_cluster && !staged && w == 0) s_ml[r] = make_float2(-INFINITY, 0.f);
    if (!ok && ntiles > 0 && lane == 0) set_err(p.err, TTS_EFLAG_TIMEOUT);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == kMmaWarp) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols) : "memory");
  }
  if (p.merge_in_cluster) {
    // Every CTA of the cluster (the item's n_ch chunks, rank = chunk) has staged its rows
    // and their (max, sum).  Rank k merges rows [128 k / n_ch, 128 (k + 1) / n_ch) in
    // chunk order, reading the other CTAs' shared memory: M = max m_c,
    // L = sum l_c 2^(m_c - M), out = sum O_c 2^(m_c - M) / L; warp k of 8 takes rows
    // k, k + 8, ... of the range, lane j the row's 16-byte unit j.  Every thread of every
    // CTA reaches both cluster barriers.
    cluster_sync_all();
    const int S = p.n_ch, rank = static_cast<int>(cluster_rank());
    if (warp < kSmxWarps) {
      uint32_t o_peer[kMaxClusterCh], ml_peer[kMaxClusterCh];
#pragma unroll
      for (int c = 0; c < kMaxClusterCh; ++c) {
        o_peer[c] = c < S ? map_shared_rank(so, static_cast<uint32_t>(c)) : 0u;
        ml_peer[c] = c < S ? map_shared_rank(s_ml, static_cast<uint32_t>(c)) : 0u;
      }
      const int r_hi = (rank + 1) * kM / S;
      for (int rr = rank * kM / S + warp; rr < r_hi; rr += kSmxWarps) {
        const int tr = rr / G, hr = rr - tr * G;
        if (tr >= nq) continue;
        float2 mlc[kMaxClusterCh];
        float M = -INFINITY;
#pragma unroll
        for (int c = 0; c < kMaxClusterCh; ++c) {
          mlc[c] = c < S ? ld_cluster_f32x2(ml_peer[c] + rr * 8) : make_float2(-INFINITY, 0.f);
          M = fmaxf(M, mlc[c].x);
        }
        const uint32_t uoff = static_cast<uint32_t>(rr * kD + ((lane ^ (rr & 31)) << 2)) * 4u;
        float4 x[kMaxClusterCh];
#pragma unroll
        for (int c = 0; c < kMaxClusterCh; ++c)
          x[c] = mlc[c].x > -INFINITY ? ld_cluster_f32x4(o_peer[c] + uoff) : make_float4(0.f, 0.f, 0.f, 0.f);
        float L = 0.f;
        float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int c = 0; c < kMaxClusterCh; ++c) {
          const float wc = mlc[c].x > -INFINITY ? exp2f(mlc[c].x - M) : 0.f;
          L = fmaf(mlc[c].y, wc, L);
          acc.x = fmaf(x[c].x, wc, acc.x);
          acc.y = fmaf(x[c].y, wc, acc.y);
          acc.z = fmaf(x[c].z, wc, acc.z);
          acc.w = fmaf(x[c].w, wc, acc.w);
        }
        const float inv = L > 0.f ? 1.f / L : 0.f;
        reinterpret_cast<float4*>(p.out + (static_cast<int64_t>(b * p.T + t0 + tr) * p.n_q_heads + g * G + hr) * kD)[lane] =
            make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
      }
    }
    __syncwarp();
    // no CTA leaves while a peer still reads its rows (the reads are complete once their
    // sums are stored, so the arrival needs no release)
    asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
  }
}


PFN_cuTensorMapEncodeTiled_v12000 tc_encoder() {
  static std::mutex mtx;
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  std::lock_guard<std::mutex> lock(mtx);
  if (fn == nullptr) {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) == cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
    else
      cudaGetLastError();
  }
  return fn;
}

// Sets the kernel's shared-memory attribute once per device.
template <int G>
cudaError_t configure_tc(int dev) {
  static std::mutex mtx;
  static bool configured[64] = {};
  std::lock_guard<std::mutex> lock(mtx);
  if (!configured[dev]) {
    const cudaError_t e =
        cudaFuncSetAttribute(prefill_attn_tc_kernel<G>, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kSmem));
    if (e != cudaSuccess) return e;
    configured[dev] = true;
  }
  return cudaSuccess;
}

// Clusters of S CTAs of this kernel the device keeps resident at once (cached per device
// and S; 0 when they cannot be launched).
template <int G>
int active_clusters(int dev, int S) {
  static std::mutex mtx;
  static int known[64][kMaxClusterCh + 1];
  static bool have[64][kMaxClusterCh + 1] = {};
  if (configure_tc<G>(dev) != cudaSuccess) {
    cudaGetLastError();
    return 0;
  }
  std::lock_guard<std::mutex> lock(mtx);
  if (!have[dev][S]) {
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(1, S);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmem;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = 1;
    attr[0].val.clusterDim.y = static_cast<unsigned>(S);
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    if (cudaOccupancyMaxActiveClusters(&n, prefill_attn_tc_kernel<G>, &cfg) != cudaSuccess) {
      cudaGetLastError();
      n = 0;
    }
    known[dev][S] = n;
    have[dev][S] = true;
  }
  return known[dev][S];
}

template <int G>
cudaError_t launch_tc_t(const PrefillAttnParams& p, const void* kc, const void* vc, cudaStream_t s, bool* merged) {
  auto kern = prefill_attn_tc_kernel<G>;
  PFN_cuTensorMapEncodeTiled_v12000 enc = tc_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  // the cache as [2 chunks of 64 columns][rows][64 bf16], a box of 64 rows (a whole tile)
  const uint64_t rows = p.paged ? static_cast<uint64_t>(p.n_pages) * p.n_kv_heads * p.page_size
                                : static_cast<uint64_t>(p.B) * p.n_kv_heads * p.capacity;
  cuuint64_t dims[3] = {64, rows, kD / 64};
  cuuint64_t strides[2] = {kD * 2, 128};
  cuuint32_t box[3] = {64, kN, kD / 64};
  cuuint32_t estr[3] = {1, 1, 1};
  CUtensorMap kmap, vmap;
  if (enc(&kmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(kc), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS ||
      enc(&vmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(vc), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  e = configure_tc<G>(dev);
  if (e != cudaSuccess) return e;
  const int items = p.B * p.n_kv_heads * p.n_qb;
  // 2..8 chunks whose clusters (one per item) are all resident at once: merged in the
  // launch; otherwise one chunk (rows normalised in place) or the combine launch after
  // this one
  const bool merge = prefill_tc_merges(items, G, p.n_ch);
  PrefillAttnParams q = p;
  q.merge_in_cluster = merge ? 1 : 0;
  *merged = merge;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(items, p.n_ch);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = static_cast<unsigned>(p.n_ch);
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = merge ? 2 : 1;
  return cudaLaunchKernelEx(&cfg, kern, kmap, vmap, q);
}

}  // namespace

int prefill_tc_active_clusters(int group, int S) {
  int dev = 0;
  if (S < 2 || S > kMaxClusterCh || cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= 64) {
    cudaGetLastError();
    return 0;
  }
  if (group == 1) return active_clusters<1>(dev, S);
  if (group == 2) return active_clusters<2>(dev, S);
  if (group == 4) return active_clusters<4>(dev, S);
  return 0;
}

bool prefill_tc_merges(int items, int group, int n_ch) {
  return n_ch > 1 && n_ch <= kMaxClusterCh && items <= prefill_tc_active_clusters(group, n_ch);
}

bool prefill_attn_tc_supported(int kv_bf16, int head_dim, int paged, int page_size) {
  return kv_bf16 && head_dim == kD && (!paged || page_size >= kN);
}

cudaError_t launch_prefill_attn_tc(const PrefillAttnParams& p, const void* k_cache, const void* v_cache, int group,
                                   cudaStream_t s, bool* merged) {
  if (p.rows != kM) return cudaErrorInvalidValue;
  *merged = false;
  if (group == 1) return launch_tc_t<1>(p, k_cache, v_cache, s, merged);
  if (group == 2) return launch_tc_t<2>(p, k_cache, v_cache, s, merged);
  if (group == 4) return launch_tc_t<4>(p, k_cache, v_cache, s, merged);
  return cudaErrorInvalidValue;
}

}  // namespace tts
