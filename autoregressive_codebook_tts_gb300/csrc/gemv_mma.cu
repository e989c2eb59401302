// Decode-layer GEMVs for 4 to 32 streams on the 5th-generation tensor cores (tcgen05):
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
//   * one CTA per (tile of 128 weight rows, range of kc columns); for the SiLU-multiply
//     a tile is 64 gate rows and their 64 up rows.  The tile is the MMA's M = 128
//     operand, the streams its N and K steps of 16.  The column ranges of a tile form
//     one thread-block cluster;
//   * warp 4 streams stages of 64 columns through a shared-memory ring: the weight tile
//     (16 KB) by a 2-D TMA tensor load in the 128-byte swizzled K-major layout, and the
//     matching NB x 64 activation chunk (contiguous in the packed layout) by a 1-D bulk
//     copy, both on the stage's mbarrier.  Weights are constants, so the first stages'
//     weight loads start before the dependency wait;
//   * lane 0 of warp 5 issues tcgen05.mma (f32 accumulator in tensor memory, 32 columns
//     allocated by warp 5), four per stage, and commits each stage back to the producer,
//     then the whole tile to the epilogue;
//   * warps 0..3 read the accumulator back (tcgen05.ld, one row a thread, one column a
//     stream) into shared memory; after a cluster barrier CTA r of the cluster sums the
//     ranges' partials of its 128 / S rows from every CTA's shared memory, in rank order
//     (so the sum does not depend on timing), and applies the epilogue: store f32, add
//     into the residual stream, or SiLU-multiply and round to bf16.
// Every mbarrier wait is bounded; on expiry TTS_EFLAG_TIMEOUT is set and the CTA winds
// down (it still reaches both cluster barriers, so its peers never wait on it).
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

enum Epilogue { EPI_STORE = 0, EPI_RESIDUAL = 1, EPI_SILU_MUL = 2 };
enum XMode { X_PACKED = 0, X_F32 = 1, X_RMSNORM = 2 };

constexpr int kMmaM = 128;            // weight rows a tile
constexpr int kStageCols = 64;        // columns a stage (128 bytes of bf16: one swizzle row)
constexpr int kWBytes = kMmaM * kStageCols * 2;
constexpr int kMaxStages = 8;
constexpr int kMaxCluster = 8;        // column ranges of a tile (portable cluster size)
constexpr int kThreads = 192;         // warps 0-3 epilogue, 4 producer, 5 MMA
constexpr int kTmemCols = 32;
constexpr int kRedLd = kMmaM + 16;    // floats between the streams' rows of the partial

struct MmaGemvParams {
  GemvParams g;         // x: the packed activations
  int kc, stages;
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

__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* map, int c0, int c1, uint64_t* bar,
                                            uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3}], [%4], %5;"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(smem_u32(bar)), "l"(policy)
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
  grid_wait();
  grid_launch_dependents();
  const int b = blockIdx.x, tid = threadIdx.x;
  const int groups = K / 8;
  if (b >= B) {
    for (int c = tid; c < groups; c += kPackThreads) xp[static_cast<int64_t>(c) * NB + b] = make_uint4(0, 0, 0, 0);
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
  const int NS = mp.stages, kc = mp.kc;
  unsigned char* ring = smem;                                          // NS stages: weights | x
  // the partial sums, [NB][kRedLd] f32, over the ring once every MMA has read it
  float* red = reinterpret_cast<float*>(ring);
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + NS * kStage);    // [NS]
  uint64_t* empty = full + kMaxStages;                                 // [NS]
  uint64_t* done = empty + kMaxStages;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(done + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x;
  const int S = gridDim.y, rank = blockIdx.y;   // the tile's column ranges = the cluster
  const int k0 = rank * kc;
  const int nst = kc / kStageCols;

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
        const int col = k0 + i * kStageCols;
        mbar_arrive_expect_tx(&full[s], kStage);
        if (EPI == EPI_SILU_MUL) {
          tma_load_2d(ring + s * kStage, &wmap, col, tile * 64, &full[s], pol);
          tma_load_2d(ring + s * kStage + kWBytes / 2, &wmap, col, p.inter + tile * 64, &full[s], pol);
        } else {
          tma_load_2d(ring + s * kStage, &wmap, col, tile * kMmaM, &full[s], pol);
        }
      };
      auto load_x = [&](int i) {
        const int s = i % NS;
        bulk_g2s_plain(ring + s * kStage + kWBytes, xsrc + static_cast<int64_t>(i) * kXBytes, kXBytes, &full[s]);
      };
      // the first stages' weights before the wait (constants), their activations after
      const int pre = nst < NS ? nst : NS;
      for (int i = 0; i < pre; ++i) load_w(i);
      grid_wait();
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
          // A: the weight tile, 128-byte swizzled rows of 64 columns, 8-row groups 1024
          // bytes apart, advanced 32 bytes a K step; B: the activation chunk, core
          // matrices of 8 streams x 8 columns, 8-column groups NB * 16 bytes apart
          const uint64_t ad = smem_desc(base + j * 32, 16, 1024, 2);
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
    const int m = warp * 32 + lane;
    float v[NB];
    const bool got = mbar_wait(done, 0);
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
  tc_fence_before();
  cluster_sync_all();   // every range's partial is in its CTA's shared memory
  if (warp < 4) {
    grid_wait();   // the residual stream and the outputs belong to earlier kernels too
    uint32_t peer[kMaxCluster];
#pragma unroll
    for (int r = 0; r < kMaxCluster; ++r) peer[r] = r < S ? map_shared_rank(red, r) : 0u;
    if (EPI == EPI_SILU_MUL) {
      // items (gate row i, up row 64 + i) of this rank: 64 / S, in groups of 8 per stream
      const int per = 64 / S, gpr = per / 8;
      for (int u = tid; u < gpr * NB; u += 128) {
        const int b = u / gpr, il = rank * per + (u - b * gpr) * 8;
        const int item = tile * 64 + il;
        float4 g0 = make_float4(0.f, 0.f, 0.f, 0.f), g1 = g0, u0 = g0, u1 = g0;
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
                add4(g0, q[h][0]);
                add4(g1, q[h][1]);
                add4(u0, q[h][2]);
                add4(u1, q[h][3]);
              }
          }
        }
        if (item < p.n_out) {
          const float gt[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
          const float up[8] = {u0.x, u0.y, u0.z, u0.w, u1.x, u1.y, u1.z, u1.w};
          float o[8];
#pragma unroll
          for (int e = 0; e < 8; ++e) o[e] = b < p.B ? gt[e] / (1.0f + expf(-gt[e])) * up[e] : 0.f;
          static_cast<uint4*>(p.y)[static_cast<int64_t>(item / 8) * NB + b] =
              make_uint4(pack2_bf16(o[0], o[1]), pack2_bf16(o[2], o[3]), pack2_bf16(o[4], o[5]), pack2_bf16(o[6], o[7]));
        }
      }
    } else {
      // rows of this rank: 128 / S, in groups of 4 per stream
      const int per = kMmaM / S, qpr = per / 4;
      for (int u = tid; u < qpr * NB; u += 128) {
        const int b = u / qpr, rl = rank * per + (u - b * qpr) * 4;
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
          if (EPI == EPI_RESIDUAL) {
            const float4 old = __ldcg(yp);
            acc = make_float4(__fadd_rn(old.x, acc.x), __fadd_rn(old.y, acc.y), __fadd_rn(old.z, acc.z),
                              __fadd_rn(old.w, acc.w));
          }
          *yp = acc;
        }
      }
    }
  }
  cluster_sync_all();   // no CTA leaves while a peer still reads its partial
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

// Launch plan: tiles, column ranges per tile (the cluster size) and ring depth.  Ranges
// are a power-of-two share of K (a multiple of 64 columns), as many as keep the grid
// within one wave at two CTAs per SM (at most kMaxCluster); the ring as deep as lets two
// CTAs share an SM when the grid needs that, else as deep as one CTA may be.
constexpr size_t kTwoPerSmBytes = 113 * 1024;
constexpr size_t kOnePerSmBytes = 227 * 1024;
void gemv_mma_plan(int K, int n_out, int epilogue, int n_sm, int nb, int& tiles, int& splits, int& kc,
                   int& stages) {
  tiles = epilogue == EPI_SILU_MUL ? (n_out + 63) / 64 : (n_out + kMmaM - 1) / kMmaM;
  int s = 1;
  while (s < kMaxCluster && tiles * s * 2 <= 2 * n_sm && K % (2 * s * kStageCols) == 0) s *= 2;
  splits = s;
  kc = K / s;
  const int nst = kc / kStageCols;
  const size_t budget = tiles * s <= n_sm ? kOnePerSmBytes : kTwoPerSmBytes;
  int ns = nst < kMaxStages ? nst : kMaxStages;
  while (ns > 2 && smem_bytes(nb, ns) > budget) --ns;
  stages = ns;
}

template <int EPI, int NB>
cudaError_t launch_mma_t(const MmaGemvParams& mp, int splits, int tiles, cudaStream_t s) {
  auto kern = gemv_mma_kernel<EPI, NB>;
  const GemvParams& p = mp.g;
  PFN_cuTensorMapEncodeTiled_v12000 enc = tensor_map_encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  // the weight matrix: rows of K bf16, a box of 64 columns x 128 rows (64 for the gate
  // and up halves of a SiLU-multiply tile), 128-byte swizzle
  const int rows = EPI == EPI_SILU_MUL ? 2 * p.inter : p.n_out;
  CUtensorMap map;
  cuuint64_t dims[2] = {static_cast<cuuint64_t>(p.K), static_cast<cuuint64_t>(rows)};
  cuuint64_t strides[1] = {static_cast<cuuint64_t>(p.K) * 2};
  cuuint32_t box[2] = {kStageCols, EPI == EPI_SILU_MUL ? 64u : static_cast<cuuint32_t>(kMmaM)};
  cuuint32_t estr[2] = {1, 1};
  if (enc(&map, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(p.w), dims, strides, box, estr,
          CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
          CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) != CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const size_t smem = smem_bytes(NB, mp.stages);
  static std::mutex mtx;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mtx);
    if (!configured[dev]) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kOnePerSmBytes));
      if (e != cudaSuccess) return e;
      configured[dev] = true;
    }
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(tiles, splits);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  attr[1].id = cudaLaunchAttributeClusterDimension;
  attr[1].val.clusterDim.x = 1;
  attr[1].val.clusterDim.y = static_cast<unsigned>(splits);
  attr[1].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  return cudaLaunchKernelEx(&cfg, kern, map, mp);
}

}  // namespace

int gemv_mma_slots(int B) { return B <= 16 ? 16 : 32; }

cudaError_t launch_gemv_mma(const GemvParams& p, int x_mode, int epilogue, void* xpack, int n_sm, cudaStream_t s) {
  if (p.B < 1 || p.B > kGemvMmaMaxB || p.K % kStageCols != 0 || p.K > kGemvMaxK || p.n_out % 8 != 0)
    return cudaErrorInvalidValue;
  const int nb = gemv_mma_slots(p.B);
  const uintptr_t align = reinterpret_cast<uintptr_t>(p.y) | reinterpret_cast<uintptr_t>(xpack) |
                          reinterpret_cast<uintptr_t>(p.x);
  if ((align & 15u) != 0 || (epilogue != EPI_SILU_MUL && p.y_stride % 4 != 0)) return cudaErrorInvalidValue;
  MmaGemvParams mp = {};
  mp.g = p;
  int tiles, splits;
  gemv_mma_plan(p.K, p.n_out, epilogue, n_sm, nb, tiles, splits, mp.kc, mp.stages);
  if (smem_bytes(nb, mp.stages) > kOnePerSmBytes) return cudaErrorInvalidValue;
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
    mp.g.x = xpack;
  }
  if (epilogue == EPI_STORE) return nb == 16 ? launch_mma_t<EPI_STORE, 16>(mp, splits, tiles, s)
                                             : launch_mma_t<EPI_STORE, 32>(mp, splits, tiles, s);
  if (epilogue == EPI_RESIDUAL) return nb == 16 ? launch_mma_t<EPI_RESIDUAL, 16>(mp, splits, tiles, s)
                                                : launch_mma_t<EPI_RESIDUAL, 32>(mp, splits, tiles, s);
  if (epilogue == EPI_SILU_MUL) return nb == 16 ? launch_mma_t<EPI_SILU_MUL, 16>(mp, splits, tiles, s)
                                                : launch_mma_t<EPI_SILU_MUL, 32>(mp, splits, tiles, s);
  return cudaErrorInvalidValue;
}

}  // namespace tts
