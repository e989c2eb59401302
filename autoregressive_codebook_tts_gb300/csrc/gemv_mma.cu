// Decode-layer GEMVs for 1 to 32 streams on the 5th-generation tensor cores (tcgen05):
// y[b][n] = sum_k x[b][k] W[n][k] for B streams, bf16 weights and activations, f32
// accumulation ("minicpm-o-4.5 ... optimizations.md", core table: fused residual add +
// RMSNorm and SiLU-multiply around the projections, integer round-to-nearest-even).
//
// With B streams a weight element feeds B multiply-adds: at 32 streams the four
// projections of a layer are 3.2 GFLOP, more than the CUDA cores issue while the 100 MB
// of weights stream from HBM, so the contraction runs on the tensor cores.  The weights
// are the only large operand, so the design keeps every CTA's chain of dependent memory
// round trips short:
//   * the activations are packed once per projection (pack_x_kernel: f32 rows, or the
//     RMS norm of the f32 residual stream times gamma, rounded to bf16) into the
//     K-major core-matrix layout the MMA reads, P[k / 8][slot][k % 8] for NB = 16 or 32
//     stream slots (slots >= B zero); the SiLU-multiply epilogue writes its output in
//     that layout directly, ready for the down projection;
//   * one CTA per (tile of 128 weight rows, range of columns); for the SiLU-multiply
//     a tile is 64 gate rows and their 64 up rows.  The tile is the MMA's M = 128
//     operand, the streams its N and K steps of 16.  The column ranges of a tile form
//     one thread-block cluster;
//   * warp 4 streams stages of 256 columns through a shared-memory ring: the weights
//     (64 KB: four 128-row x 64-column sub-tiles in the 128-byte swizzled K-major layout)
//     by ONE 3-D (SiLU-multiply: 4-D) TMA tensor load, and the matching NB x 256
//     activation chunk (contiguous in the packed layout) by one 1-D bulk copy, both on
//     the stage's mbarrier.  An SM keeps only a few bulk copies in flight, so its
//     streaming rate grows with the bytes per copy: 16 KB copies stop near 50 GB/s an SM,
//     far below HBM's share.  Weights are constants, so the first stages' weight loads
//     start before the dependency wait;
//   * lane 0 of warp 5 issues tcgen05.mma (f32 accumulator in tensor memory, 32 columns
//     allocated by warp 5), sixteen per stage, and commits each stage back to the
//     producer, then the whole tile to the epilogue;
//   * warps 0..3 read the accumulator back (tcgen05.ld, one row a thread, one column a
//     stream) into shared memory; after a cluster barrier CTA r of the cluster sums the
//     ranges' partials of its 128 / S rows from every CTA's shared memory, in rank order
//     (so the sum does not depend on timing), and applies the epilogue: store f32, add
//     into the residual stream, or SiLU-multiply and round to bf16.
// Every mbarrier wait is bounded; on expiry TTS_EFLAG_TIMEOUT is set and the CTA winds
// down (it still reaches both cluster barriers, so its peers never wait on it).
#include <cstdint>
#include <map>
#include <mutex>
#include <tuple>

#include <cuda.h>
#include <cudaTypedefs.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace tts {

#ifdef TTS_TRACE
// Optional timeline of the projections (build with -DTTS_TRACE): one row per CTA of
// every launch, appended in start order: a tag (kind, grid, block, SM) and %globaltimer
// stamps at entry, after the dependency wait, when the accumulator is complete and at
// exit; read with tts_gtrace_read().
constexpr int kGTraceRows = 65536;
__device__ unsigned long long g_gtrace[kGTraceRows][8];
__device__ unsigned int g_gtrace_n;
__device__ __forceinline__ unsigned long long gtrace_time() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ unsigned int gtrace_smid() {
  unsigned int r;
  asm volatile("mov.u32 %0, %%smid;" : "=r"(r));
  return r;
}
#define TTS_GTRACE_BEGIN(kind, row_var)                                                             \
  __shared__ unsigned int row_var;                                                                 \
  if (threadIdx.x == 0) {                                                                          \
    const unsigned long long t_ = gtrace_time();                                                   \
    row_var = atomicAdd(&g_gtrace_n, 1u);                                                          \
    if (row_var < kGTraceRows) {                                                                   \
      g_gtrace[row_var][0] = (static_cast<unsigned long long>(kind)) |                             \
                             (static_cast<unsigned long long>(gridDim.x) << 8) |                   \
                             (static_cast<unsigned long long>(gridDim.y) << 20) |                  \
                             (static_cast<unsigned long long>(blockIdx.x) << 28) |                 \
                             (static_cast<unsigned long long>(blockIdx.y) << 40) |                 \
                             (static_cast<unsigned long long>(gtrace_smid()) << 48);               \
      g_gtrace[row_var][1] = t_;                                                                   \
    }                                                                                              \
  }
#define TTS_GTRACE(row_var, slot)                                                                   \
  do {                                                                                             \
    if ((row_var) < kGTraceRows) g_gtrace[(row_var)][slot] = gtrace_time();                        \
  } while (0)
#else
#define TTS_GTRACE_BEGIN(kind, row_var)
#define TTS_GTRACE(row_var, slot) do {} while (0)
#endif

namespace {

enum Epilogue { EPI_STORE = 0, EPI_RESIDUAL = 1, EPI_SILU_MUL = 2 };
enum XMode { X_PACKED = 0, X_F32 = 1, X_RMSNORM = 2 };

constexpr int kMmaM = 128;            // weight rows a tile
constexpr int kChunkCols = 64;        // columns of one swizzled sub-tile (128 bytes of bf16)
#ifndef TTS_GEMV_CHUNKS
#define TTS_GEMV_CHUNKS 4
#endif
constexpr int kChunks = TTS_GEMV_CHUNKS;  // sub-tiles a stage (K is a multiple of 256)
static_assert(kChunks == 1 || kChunks == 2 || kChunks == 4, "sub-tiles a stage");
constexpr int kStageCols = kChunkCols * kChunks;
constexpr int kChunkBytes = kMmaM * kChunkCols * 2;
constexpr int kWBytes = kChunkBytes * kChunks;
constexpr int kMaxStages = 8;
constexpr int kMaxCluster = 8;        // column ranges of a tile (portable cluster size)
constexpr int kThreads = 192;         // warps 0-3 epilogue, 4 producer, 5 MMA
constexpr int kTmemCols = 32;
constexpr int kRedLd = kMmaM + 16;    // floats between the streams' rows of the partial

struct MmaGemvParams {
  GemvParams g;         // x: the packed activations
  int stages;           // ring depth
};

constexpr int stage_bytes(int nb) { return kWBytes + nb * kStageCols * 2; }

__device__ __forceinline__ uint16_t bf16_rne_bits(float x) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<const uint16_t*>(&h);
}

__device__ __forceinline__ uint32_t pack2_bf16(float lo, float hi) {
  return static_cast<uint32_t>(bf16_rne_bits(lo)) | (static_cast<uint32_t>(bf16_rne_bits(hi)) << 16);
}

// Shared-memory matrix descriptor of tcgen05.mma: start address, leading- and
// stride-dimension byte offsets (all in 16-byte units), the descriptor version (bit 46)
// and the swizzle mode (bits 61..63: 0 none, 2 128-byte).
__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint32_t swizzle) {
  return static_cast<uint64_t>((addr & 0x3FFFF) >> 4) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFF) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFF) << 32) | (static_cast<uint64_t>(1) << 46) |
         (static_cast<uint64_t>(swizzle & 7) << 61);
}

// One tensor-map load of the stage's weights: every sub-tile of 64 columns x 128 rows in
// the 128-byte swizzled layout, one after the other (3-D box {64, 128, chunks}; for the
// SiLU-multiply a 4-D box {64, 64, gate/up, chunks}, so each sub-tile holds its 64 gate
// rows then their 64 up rows).
__device__ __forceinline__ void tma_load_3d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar)),
        "l"(policy)
      : "memory");
}
__device__ __forceinline__ void tma_load_4d(void* dst, const CUtensorMap* map, int c0, int c1, int c2, int c3,
                                            uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.4d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4, %5}], [%6], %7;"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(c3),
        "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() { asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory"); }
__device__ __forceinline__ void tc_fence_after() { asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory"); }

// 16 bytes of another CTA's shared memory (a cluster-window address from mapa).
__device__ __forceinline__ float4 ld_cluster_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared::cluster.v4.f32 {%0, %1, %2, %3}, [%4];"
               : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr) : "memory");
  return v;
}

__device__ __forceinline__ void add4(float4& a, const float4 b) {
  a.x += b.x;
  a.y += b.y;
  a.z += b.z;
  a.w += b.w;
}

// Accumulator row of this thread (TMEM lane 32 w + lane of warp w < 4), NB columns.
template <int NB>
__device__ __forceinline__ void tmem_row(uint32_t taddr, float (&v)[NB]);
template <>
__device__ __forceinline__ void tmem_row<16>(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}
template <>
__device__ __forceinline__ void tmem_row<32>(uint32_t taddr, float (&v)[32]) {
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

// Activations of a projection, packed for the MMA: P[k / 8][b][k % 8] (bf16, 16 bytes
// per (group of 8 columns, stream slot)), one CTA per stream slot.  f32 rows are rounded
// to nearest even; in the RMS-norm mode each element is first scaled by the row's
// 1 / sqrt(mean(x^2) + eps) (statistics in f32) and by gamma.  Slots b >= B are zero.
// Every thread keeps its (at most 4) groups in registers, so the row is read once.
constexpr int kPackThreads = 256;
constexpr int kPackGroups = kGemvMaxK / 8 / kPackThreads;
template <int XM>
__global__ void __launch_bounds__(kPackThreads) pack_x_kernel(const float* x, int64_t stride, const float* gamma,
                                                              float eps, int K, int B, int NB, uint4* xp) {
  __shared__ float red[kPackThreads / 32];
  TTS_GTRACE_BEGIN(0x10 | XM, trow);
  grid_wait();
  grid_launch_dependents();
  const int b = blockIdx.x, tid = threadIdx.x;
#ifdef TTS_TRACE
  __syncthreads();
  if (tid == 0) TTS_GTRACE(trow, 2);
#endif
  const int groups = K / 8;
  if (b >= B) {
    for (int c = tid; c < groups; c += kPackThreads) xp[static_cast<int64_t>(c) * NB + b] = make_uint4(0, 0, 0, 0);
#ifdef TTS_TRACE
    if (tid == 0) TTS_GTRACE(trow, 4);
#endif
    return;
  }
  const float4* row = reinterpret_cast<const float4*>(x + static_cast<int64_t>(b) * stride);
  float4 v[kPackGroups][2];
#pragma unroll
  for (int j = 0; j < kPackGroups; ++j) {
    const int c = tid + j * kPackThreads;
    if (c < groups) {
      v[j][0] = __ldcg(row + 2 * c);
      v[j][1] = __ldcg(row + 2 * c + 1);
    } else {
      v[j][0] = v[j][1] = make_float4(0.f, 0.f, 0.f, 0.f);
    }
  }
  float sc = 1.f;
  if (XM == X_RMSNORM) {
    float ss = 0.f;
#pragma unroll
    for (int j = 0; j < kPackGroups; ++j)
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        ss = fmaf(v[j][h].x, v[j][h].x, ss);
        ss = fmaf(v[j][h].y, v[j][h].y, ss);
        ss = fmaf(v[j][h].z, v[j][h].z, ss);
        ss = fmaf(v[j][h].w, v[j][h].w, ss);
      }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(kFull, ss, off);
    if ((tid & 31) == 0) red[tid >> 5] = ss;
    __syncthreads();
    float t = 0.f;
#pragma unroll
    for (int w = 0; w < kPackThreads / 32; ++w) t += red[w];
    sc = 1.0f / sqrtf(t / static_cast<float>(K) + eps);
  }
#pragma unroll
  for (int j = 0; j < kPackGroups; ++j) {
    const int c = tid + j * kPackThreads;
    if (c < groups) {
      float f[8] = {v[j][0].x, v[j][0].y, v[j][0].z, v[j][0].w, v[j][1].x, v[j][1].y, v[j][1].z, v[j][1].w};
      if (XM == X_RMSNORM) {
        const float4 g0 = __ldg(reinterpret_cast<const float4*>(gamma) + 2 * c);
        const float4 g1 = __ldg(reinterpret_cast<const float4*>(gamma) + 2 * c + 1);
        const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
        for (int e = 0; e < 8; ++e) f[e] = f[e] * sc * g[e];
      }
      xp[static_cast<int64_t>(c) * NB + b] =
          make_uint4(pack2_bf16(f[0], f[1]), pack2_bf16(f[2], f[3]), pack2_bf16(f[4], f[5]), pack2_bf16(f[6], f[7]));
    }
  }
#ifdef TTS_TRACE
  if (tid == 0) TTS_GTRACE(trow, 4);
#endif
}

template <int EPI, int NB>
__global__ void __launch_bounds__(kThreads, 1) gemv_mma_kernel(const __grid_constant__ CUtensorMap wmap,
                                                                const MmaGemvParams mp) {
  constexpr int kXBytes = NB * kStageCols * 2;   // activation chunk of a stage
  constexpr int kStage = kWBytes + kXBytes;      // a multiple of 1024 (the swizzle period)
  static_assert(kStage % 1024 == 0, "stage size");
  const GemvParams& p = mp.g;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // the 128-byte swizzle repeats every 1024 bytes: the stages start on such a boundary
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int NS = mp.stages;
  unsigned char* ring = smem;                                          // NS stages: weights | x
  // the partial sums, [NB][kRedLd] f32, over the ring once every MMA has read it
  float* red = reinterpret_cast<float*>(ring);
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + NS * kStage);    // [NS]
  uint64_t* empty = full + kMaxStages;                                 // [NS]
  uint64_t* done = empty + kMaxStages;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(done + 1);
  TTS_GTRACE_BEGIN(EPI | (NB == 32 ? 4 : 0), trow);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x;
  // epilogue of a store / residual tile: rows in groups of 4, rank r of the cluster
  // taking groups [32 r / S, 32 (r + 1) / S) of every stream, unit u = (stream, group)
  // handled by thread u % 128 (at most kUnits each)
  constexpr int kUnits = NB / 4;
  float4 old[kUnits];
  // the tile's column ranges = the cluster; range r holds stages [r n / S, (r + 1) n / S)
  // of the n = K / 64 stages of a row
  const int S = gridDim.y, rank = blockIdx.y;
  const int n_all = p.K / kStageCols;
  const int st0 = rank * n_all / S, nst = (rank + 1) * n_all / S - st0;
  const int k0 = st0 * kStageCols;
  const int q0 = 32 * rank / S, qpr = 32 * (rank + 1) / S - q0;

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(done, 1);
    mbar_init_fence();
  }
  if (warp == 5) {
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;"
                 ::"r"(smem_u32(s_tmem)), "n"(kTmemCols) : "memory");
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  grid_launch_dependents();

  if (warp == 4) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      const uint64_t pol = l2_evict_first_policy();
      const unsigned char* xsrc = static_cast<const unsigned char*>(p.x) + static_cast<int64_t>(k0) * NB * 2;
      auto load_w = [&](int i) {
        const int s = i % NS;
        const int chunk = (k0 + i * kStageCols) / kChunkCols;
        mbar_arrive_expect_tx(&full[s], kStage);
        if (EPI == EPI_SILU_MUL) tma_load_4d(ring + s * kStage, &wmap, 0, tile * 64, 0, chunk, &full[s], pol);
        else tma_load_3d(ring + s * kStage, &wmap, 0, tile * kMmaM, chunk, &full[s], pol);
      };
      auto load_x = [&](int i) {
        const int s = i % NS;
        bulk_g2s_plain(ring + s * kStage + kWBytes, xsrc + static_cast<int64_t>(i) * kXBytes, kXBytes, &full[s]);
      };
      // the first stages' weights before the wait (constants), their activations after
      const int pre = nst < NS ? nst : NS;
      for (int i = 0; i < pre; ++i) load_w(i);
      grid_wait();
      TTS_GTRACE(trow, 2);
      for (int i = 0; i < pre; ++i) load_x(i);
      int issued = pre;
      bool ok = true;
      for (; issued < nst; ++issued) {
        const int s = issued % NS;
        if (!mbar_wait(&empty[s], static_cast<uint32_t>((issued / NS) - 1) & 1u)) {
          ok = false;
          break;
        }
        load_w(issued);
        load_x(issued);
      }
      if (!ok) set_err(p.err, TTS_EFLAG_TIMEOUT);
      // no copy may still be landing when the CTA leaves
      for (int t = max(0, issued - NS); t < issued; ++t) mbar_wait(&full[t % NS], static_cast<uint32_t>(t / NS) & 1u);
    }
  } else if (warp == 5) {
    // -------------------------------------------------------------- MMA issuer
    if (lane == 0) {
      // kind::f16: f32 accumulator (bits 4-5 = 1), bf16 A and B (bits 7-9, 10-12 = 1),
      // both K-major, N >> 3 at bit 17, M >> 4 at bit 24
      const uint32_t idesc = (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(NB >> 3) << 17) |
                             (static_cast<uint32_t>(kMmaM >> 4) << 24);
      bool ok = true;
      for (int i = 0; i < nst; ++i) {
        const int s = i % NS;
        if (!mbar_wait(&full[s], static_cast<uint32_t>(i / NS) & 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
        const uint32_t base = smem_u32(ring + s * kStage);
#pragma unroll
        for (int j = 0; j < kStageCols / 16; ++j) {
          // A: sub-tile j / 4 of the weights, 128-byte swizzled rows of 64 columns, 8-row
          // groups 1024 bytes apart, advanced 32 bytes a K step; B: the activation chunk,
          // core matrices of 8 streams x 8 columns, 8-column groups NB * 16 bytes apart
          const uint64_t ad = smem_desc(base + (j >> 2) * kChunkBytes + (j & 3) * 32, 16, 1024, 2);
          const uint64_t bd = smem_desc(base + kWBytes + 2 * j * (NB * 16), NB * 16, 128, 0);
          const uint32_t acc = (i > 0 || j > 0) ? 1u : 0u;
          asm volatile(
              "{\n\t.reg .pred p;\n\tsetp.ne.b32 p, %4, 0;\n\t"
              "tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n\t}"
              ::"r"(tmem), "l"(ad), "l"(bd), "r"(idesc), "r"(acc) : "memory");
        }
        // the stage is free once these MMAs have read it
        asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                     ::"r"(smem_u32(&empty[s])) : "memory");
      }
      if (!ok) set_err(p.err, TTS_EFLAG_TIMEOUT);
      // the accumulator is complete once every MMA issued above has finished
      asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];"
                   ::"r"(smem_u32(done)) : "memory");
    }
  } else {
    // ---------------------------------------- the partial of this column range
    grid_wait();   // the residual stream and the outputs belong to earlier kernels too
    if (EPI == EPI_RESIDUAL) {
      // this thread's old residual values, loaded while the weights stream
#pragma unroll
      for (int k = 0; k < kUnits; ++k) {
        const int u = tid + 128 * k;
        old[k] = make_float4(0.f, 0.f, 0.f, 0.f);
        if (u < qpr * NB) {
          const int b = u / qpr, row = tile * kMmaM + (q0 + u - b * qpr) * 4;
          if (b < p.B && row < p.n_out)
            old[k] = __ldcg(reinterpret_cast<const float4*>(static_cast<const float*>(p.y) +
                                                            static_cast<int64_t>(b) * p.y_stride + row));
        }
      }
    }
    const int m = warp * 32 + lane;
    float v[NB];
    const bool got = mbar_wait(done, 0);
    if (tid == 0) TTS_GTRACE(trow, 3);
    if (!got && lane == 0) set_err(p.err, TTS_EFLAG_TIMEOUT);
    tc_fence_after();
    if (got) tmem_row<NB>(tmem + (static_cast<uint32_t>(warp * 32) << 16), v);
    else
#pragma unroll
      for (int b = 0; b < NB; ++b) v[b] = 0.f;
    // transposed, so that 4 rows of a stream are 16 contiguous bytes
#pragma unroll
    for (int b = 0; b < NB; ++b) red[b * kRedLd + m] = v[b];
  }
  __syncwarp();   // the producer and MMA lanes rejoin their warps before the aligned barrier
  if (tid == 0) TTS_GTRACE(trow, 5);
  tc_fence_before();
  cluster_sync_all();   // every range's partial is in its CTA's shared memory
  if (tid == 0) TTS_GTRACE(trow, 6);
  if (warp < 4) {
    uint32_t peer[kMaxCluster];
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r) peer[r] = r < S ? map_shared_rank(red, r) : 0u;
    if (EPI == EPI_SILU_MUL) {
      // items (gate row i, up row 64 + i) in groups of 8: rank r takes groups
      // [8 r / S, 8 (r + 1) / S) of every stream
      const int g0 = 8 * rank / S, gpr = 8 * (rank + 1) / S - g0;
      for (int u = tid; u < gpr * NB; u += 128) {
        const int b = u / gpr, il = (g0 + u - b * gpr) * 8;
        const int item = tile * 64 + il;
        float4 ga = make_float4(0.f, 0.f, 0.f, 0.f), gb = ga, ua = ga, ub = ga;
        const uint32_t off = static_cast<uint32_t>((b * kRedLd + il) * 4);
        // two ranks' loads in flight at a time, summed in rank order
#pragma unroll
        for (int r = 0; r < kMaxCluster; r += 2) {
          if (r < S) {
            float4 q[2][4];
#pragma unroll
            for (int h = 0; h < 2; ++h) {
              const uint32_t a = peer[r + h] + off;
              q[h][0] = q[h][1] = q[h][2] = q[h][3] = make_float4(0.f, 0.f, 0.f, 0.f);
              if (r + h < S) {
                q[h][0] = ld_cluster_f4(a);
                q[h][1] = ld_cluster_f4(a + 16);
                q[h][2] = ld_cluster_f4(a + 256);
                q[h][3] = ld_cluster_f4(a + 272);
              }
            }
#pragma unroll
            for (int h = 0; h < 2; ++h)
              if (r + h < S) {
                add4(ga, q[h][0]);
                add4(gb, q[h][1]);
                add4(ua, q[h][2]);
                add4(ub, q[h][3]);
              }
          }
        }
        if (item < p.n_out) {
          const float gt[8] = {ga.x, ga.y, ga.z, ga.w, gb.x, gb.y, gb.z, gb.w};
          const float up[8] = {ua.x, ua.y, ua.z, ua.w, ub.x, ub.y, ub.z, ub.w};
          float o[8];
#pragma unroll
          // silu(g) = g / (1 + e^-g) with the fast exponential and division (a few ulp;
          // for g below about -88 the denominator is inf and the quotient 0, the limit)
          for (int e = 0; e < 8; ++e) o[e] = b < p.B ? __fdividef(gt[e], 1.0f + __expf(-gt[e])) * up[e] : 0.f;
          static_cast<uint4*>(p.y)[static_cast<int64_t>(item / 8) * NB + b] =
              make_uint4(pack2_bf16(o[0], o[1]), pack2_bf16(o[2], o[3]), pack2_bf16(o[4], o[5]), pack2_bf16(o[6], o[7]));
        }
      }
    } else {
#pragma unroll
      for (int k = 0; k < kUnits; ++k) {
        const int u = tid + 128 * k;
        if (u >= qpr * NB) break;
        const int b = u / qpr, rl = (q0 + u - b * qpr) * 4;
        const int row = tile * kMmaM + rl;
        if (b >= p.B) continue;
        const uint32_t off = static_cast<uint32_t>((b * kRedLd + rl) * 4);
        float4 q[kMaxCluster];
#pragma unroll
        for (int r = 0; r < kMaxCluster; ++r) q[r] = r < S ? ld_cluster_f4(peer[r] + off) : make_float4(0.f, 0.f, 0.f, 0.f);
        float4 acc = q[0];
#pragma unroll
        for (int r = 1; r < kMaxCluster; ++r)
          if (r < S) add4(acc, q[r]);
        if (row < p.n_out) {
          float4* yp = reinterpret_cast<float4*>(static_cast<float*>(p.y) + static_cast<int64_t>(b) * p.y_stride + row);
          if (EPI == EPI_RESIDUAL)
            acc = make_float4(__fadd_rn(old[k].x, acc.x), __fadd_rn(old[k].y, acc.y), __fadd_rn(old[k].z, acc.z),
                              __fadd_rn(old[k].w, acc.w));
          *yp = acc;
        }
      }
    }
  }
  if (tid == 0) TTS_GTRACE(trow, 7);
  // no CTA leaves while a peer still reads its partial (the reads are complete once
  // their sums are stored, so the arrival needs no release)
  asm volatile("barrier.cluster.arrive.relaxed.aligned;\n\tbarrier.cluster.wait.aligned;" ::: "memory");
  if (tid == 0) TTS_GTRACE(trow, 4);
  if (warp == 5) {
    tc_fence_after();
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(tmem), "n"(kTmemCols) : "memory");
  }
}

// cuTensorMapEncodeTiled, looked up once through the runtime (no link against the driver)
PFN_cuTensorMapEncodeTiled_v12000 tensor_map_encoder() {
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

size_t smem_bytes(int NB, int stages) {
  return 1024 + static_cast<size_t>(stages) * stage_bytes(NB) + (2 * kMaxStages + 1) * sizeof(uint64_t) + 16;
}

// One CTA per SM: a kernel that allocates tensor memory is given at most one block per
// SM, so a launch is planned as a single wave.  Tiles of 128 rows, split into S column
// ranges (the cluster size), S as large as keeps every tile's cluster resident at once
// (the largest S with tiles <= the device's maximum of active S-CTA clusters); the ring
// as deep as one CTA's shared memory allows.

struct OccKey {
  int dev, epi, nb, s, stages;
  bool operator<(const OccKey& o) const {
    return std::tie(dev, epi, nb, s, stages) < std::tie(o.dev, o.epi, o.nb, o.s, o.stages);
  }
};

// The dynamic shared memory one CTA of the kernel may take on device `dev` (the opt-in
// maximum less the kernel's static shared memory), set as the kernel's limit once per
// device; 0 on failure.
template <int EPI, int NB>
size_t configure(int dev) {
  static std::mutex mtx;
  static size_t budget[64] = {};
  std::lock_guard<std::mutex> lock(mtx);
  if (budget[dev] != 0) return budget[dev];
  int optin = 0;
  cudaFuncAttributes fa;
  if (cudaDeviceGetAttribute(&optin, cudaDevAttrMaxSharedMemoryPerBlockOptin, dev) != cudaSuccess ||
      cudaFuncGetAttributes(&fa, gemv_mma_kernel<EPI, NB>) != cudaSuccess ||
      static_cast<size_t>(optin) <= fa.sharedSizeBytes)
    return 0;
  const size_t b = static_cast<size_t>(optin) - fa.sharedSizeBytes;
  if (cudaFuncSetAttribute(gemv_mma_kernel<EPI, NB>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                           static_cast<int>(b)) != cudaSuccess)
    return 0;
  budget[dev] = b;
  return b;
}

// Clusters of S CTAs of this kernel the device keeps resident at once (cached).
template <int EPI, int NB>
int max_active_clusters(int dev, int S, int stages) {
  static std::mutex mtx;
  static std::map<OccKey, int> cache;
  const OccKey key = {dev, EPI, NB, S, stages};
  {
    std::lock_guard<std::mutex> lock(mtx);
    const auto it = cache.find(key);
    if (it != cache.end()) return it->second;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(1, S);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes(NB, stages);
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 1;
  attr[0].val.clusterDim.y = static_cast<unsigned>(S);
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  int n = 0;
  if (cudaOccupancyMaxActiveClusters(&n, gemv_mma_kernel<EPI, NB>, &cfg) != cudaSuccess) {
    cudaGetLastError();
    n = 0;
  }
  std::lock_guard<std::mutex> lock(mtx);
  cache[key] = n;
  return n;
}

template <int EPI, int NB>
cudaError_t launch_mma_t(const GemvParams& p, cudaStream_t s) {
  auto kern = gemv_mma_kernel<EPI, NB>;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  const size_t budget = configure<EPI, NB>(dev);
  if (budget == 0) {
    const cudaError_t le = cudaGetLastError();
    return le != cudaSuccess ? le : cudaErrorInvalidValue;
  }
  // the plan
  const int n_all = p.K / kStageCols;
  const int tiles = EPI == EPI_SILU_MUL ? (p.n_out + 63) / 64 : (p.n_out + kMmaM - 1) / kMmaM;
  int S = 0, stages = 0;
  for (int c = n_all < kMaxCluster ? n_all : kMaxCluster; c >= 1 && S == 0; --c) {
    const int longest = (n_all + c - 1) / c;
    int ns = longest < kMaxStages ? longest : kMaxStages;
    while (ns > 1 && smem_bytes(NB, ns) > budget) --ns;
    if (c == 1 || tiles <= max_active_clusters<EPI, NB>(dev, c, ns)) {
      S = c;
      stages = ns;
    }
  }
  MmaGemvParams mp = {};
  mp.g = p;
  mp.stages = stages;
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  // the weight matrix, rows of K bf16, seen as [K / 64 sub-tile columns][rows][64]
  // (strides: a row K * 2 bytes, a sub-tile column 128 bytes); a box of 4 sub-tile
  // columns x 128 rows x 64, 128-byte swizzle.  SiLU-multiply: [K / 64][gate / up][inter
  // rows][64], a box of 4 x 2 x 64 x 64 (the up half inter * K * 2 bytes on).
  const cuuint64_t K = static_cast<cuuint64_t>(p.K);
  CUtensorMap map;
  CUresult r;
  if (EPI == EPI_SILU_MUL) {
    cuuint64_t dims[4] = {kChunkCols, static_cast<cuuint64_t>(p.inter), 2, K / kChunkCols};
    cuuint64_t strides[3] = {K * 2, static_cast<cuuint64_t>(p.inter) * K * 2, kChunkCols * 2};
    cuuint32_t box[4] = {kChunkCols, 64, 2, kChunks};
    cuuint32_t estr[4] = {1, 1, 1, 1};
    r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 4, const_cast<void*>(p.w), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  } else {
    cuuint64_t dims[3] = {kChunkCols, static_cast<cuuint64_t>(p.n_out), K / kChunkCols};
    cuuint64_t strides[2] = {K * 2, kChunkCols * 2};
    cuuint32_t box[3] = {kChunkCols, static_cast<cuuint32_t>(kMmaM), kChunks};
    cuuint32_t estr[3] = {1, 1, 1};
    r = enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 3, const_cast<void*>(p.w), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  }
  if (r != CUDA_SUCCESS) return cudaErrorInvalidValue;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles, S);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem_bytes(NB, stages);
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = static_cast<unsigned>(S);
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, map, mp);
}

}  // namespace

#ifdef TTS_TRACE
extern "C" int tts_gtrace_read(unsigned long long* host, int n_rows) {
  return static_cast<int>(cudaMemcpyFromSymbol(host, g_gtrace, static_cast<size_t>(n_rows) * 8 * sizeof(unsigned long long)));
}
extern "C" int tts_gtrace_clear(void) {
  static unsigned long long zeros[1024][8];
  unsigned int z = 0;
  for (int r = 0; r < kGTraceRows; r += 1024)
    if (cudaMemcpyToSymbol(g_gtrace, zeros, sizeof(zeros), static_cast<size_t>(r) * 8 * sizeof(unsigned long long)) != cudaSuccess)
      return 1;
  return static_cast<int>(cudaMemcpyToSymbol(g_gtrace_n, &z, sizeof(z)));
}
#endif

int gemv_mma_slots(int B) { return B <= 16 ? 16 : 32; }

cudaError_t launch_gemv_mma(const GemvParams& p, int x_mode, int epilogue, void* xpack, cudaStream_t s) {
  if (p.B < 1 || p.B > kGemvMmaMaxB || p.K % kStageCols != 0 || p.K > kGemvMaxK || p.n_out % 8 != 0)
    return cudaErrorInvalidValue;
  const int nb = gemv_mma_slots(p.B);
  const uintptr_t align = reinterpret_cast<uintptr_t>(p.y) | reinterpret_cast<uintptr_t>(xpack) |
                          reinterpret_cast<uintptr_t>(p.x);
  if ((align & 15u) != 0 || (epilogue != EPI_SILU_MUL && p.y_stride % 4 != 0)) return cudaErrorInvalidValue;
  GemvParams g = p;
  if (x_mode != X_PACKED) {
    if (xpack == nullptr || (x_mode == X_RMSNORM && p.gamma == nullptr) || p.x_stride % 4 != 0)
      return cudaErrorInvalidValue;
    const float* x = static_cast<const float*>(p.x);
    const cudaError_t e =
        x_mode == X_RMSNORM
            ? launch_pdl(pack_x_kernel<X_RMSNORM>, dim3(nb), dim3(kPackThreads), 0, s, x, p.x_stride, p.gamma,
                         p.eps, p.K, p.B, nb, static_cast<uint4*>(xpack))
            : launch_pdl(pack_x_kernel<X_F32>, dim3(nb), dim3(kPackThreads), 0, s, x, p.x_stride, p.gamma, p.eps,
                         p.K, p.B, nb, static_cast<uint4*>(xpack));
    if (e != cudaSuccess) return e;
    g.x = xpack;
  }
  if (epilogue == EPI_STORE) return nb == 16 ? launch_mma_t<EPI_STORE, 16>(g, s) : launch_mma_t<EPI_STORE, 32>(g, s);
  if (epilogue == EPI_RESIDUAL)
    return nb == 16 ? launch_mma_t<EPI_RESIDUAL, 16>(g, s) : launch_mma_t<EPI_RESIDUAL, 32>(g, s);
  if (epilogue == EPI_SILU_MUL)
    return nb == 16 ? launch_mma_t<EPI_SILU_MUL, 16>(g, s) : launch_mma_t<EPI_SILU_MUL, 32>(g, s);
  return cudaErrorInvalidValue;
}

}  // namespace tts
