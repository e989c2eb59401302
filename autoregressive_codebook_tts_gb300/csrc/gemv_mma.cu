// Decode-layer GEMVs for 4 to 32 streams on the 5th-generation tensor cores (tcgen05):
// y[b][n] = sum_k x[b][k] W[n][k] for B streams, bf16 weights and activations, f32
// accumulation ("minicpm-o-4.5 ... optimizations.md", core table: fused residual add +
// RMSNorm and SiLU-multiply around the projections, integer round-to-nearest-even).
//
// With B streams a weight element feeds B multiply-adds: at 32 streams the four
// projections of a layer are 3.2 GFLOP, more than the CUDA cores issue while the 100 MB
// of weights stream from HBM, so the contraction runs on the tensor cores:
//   * one CTA per (tile of 128 weight rows, range of kc columns); for the SiLU-multiply a
//     tile is 64 gate rows and their 64 up rows.  The tile is the MMA's M = 128 operand,
//     the streams its N (16 or 32, zero-padded) and K steps of 16;
//   * warp 4 streams the weight tile through a ring of shared-memory stages (64 columns,
//     16 KB each) with 2-D TMA tensor loads in the 128-byte swizzled K-major layout the
//     MMA reads; the weights are constants, so it starts before the dependency wait;
//   * warps 0..3 stage the activations once as bf16 in the K-major core-matrix layout
//     (8 rows x 16 bytes): a bf16 input as is, an f32 input rounded, or the RMS norm of
//     the f32 residual stream (statistics over the whole row, in f32) times gamma;
//   * lane 0 of warp 5 issues tcgen05.mma (f32 accumulator in tensor memory, 32
//     columns allocated by warp 5) four per stage and commits each stage back to the
//     producer, then the whole tile to the epilogue;
//   * warps 0..3 read the accumulator rows back (tcgen05.ld, one row a thread, one
//     column a stream).  With several column ranges each CTA writes its partial to the
//     workspace and takes a ticket; the last CTA of a tile sums the partials in range
//     order (so the result does not depend on which CTA finishes last) and applies the
//     epilogue: store f32, add into the residual stream, or SiLU-multiply and round to
//     bf16.
// Every wait is bounded; on expiry TTS_EFLAG_TIMEOUT is set and the CTA winds down.
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
enum XMode { X_BF16 = 0, X_F32 = 1, X_RMSNORM = 2 };

constexpr int kMmaM = 128;            // weight rows a tile
constexpr int kStageCols = 64;        // columns a stage (128 bytes of bf16: one swizzle row)
constexpr int kStageBytes = kMmaM * kStageCols * 2;
constexpr int kMaxStages = 6;
constexpr int kThreads = 192;         // warps 0-3 activations/epilogue, 4 producer, 5 MMA
constexpr int kTmemCols = 32;

struct MmaGemvParams {
  GemvParams g;
  float* part;       // [splits][tiles][128][NB] partial sums (splits > 1)
  int* tickets;      // [tiles], zero between launches
  int tiles, splits, kc, stages;
};

__device__ __forceinline__ uint16_t bf16_rne_bits(float x) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<const uint16_t*>(&h);
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

template <int XM, int EPI, int NB>
__global__ void __launch_bounds__(kThreads, 1) gemv_mma_kernel(const __grid_constant__ CUtensorMap wmap,
                                                                const MmaGemvParams mp) {
  const GemvParams& p = mp.g;
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  // the 128-byte swizzle repeats every 1024 bytes: the stages start on such a boundary
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  const int NS = mp.stages, kc = mp.kc;
  unsigned char* ring = smem;                                          // NS stages
  unsigned char* xs = smem + NS * kStageBytes;                         // NB x kc bf16, core matrices
  float* s_scale = reinterpret_cast<float*>(xs + NB * kc * 2);         // [NB]
  float* s_up = s_scale + NB;                                          // [64][NB] SiLU up sums
  uint64_t* full = reinterpret_cast<uint64_t*>(s_up + 64 * NB);        // [NS]
  uint64_t* empty = full + kMaxStages;                                 // [NS]
  uint64_t* xready = empty + kMaxStages;
  uint64_t* done = xready + 1;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(done + 1);
  int* s_last = reinterpret_cast<int*>(s_tmem + 1);

  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int tile = blockIdx.x, split = blockIdx.y;
  const int k0 = split * kc;
  const int nst = kc / kStageCols;
  const int B = p.B;

  if (tid == 0) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], 1);
    }
    mbar_init(xready, 128);
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
      int issued = 0;
      bool ok = true;
      for (; issued < nst; ++issued) {
        const int s = issued % NS;
        if (issued >= NS && !mbar_wait(&empty[s], static_cast<uint32_t>((issued / NS) - 1) & 1u)) {
          ok = false;
          break;
        }
        mbar_arrive_expect_tx(&full[s], kStageBytes);
        const int col = k0 + issued * kStageCols;
        if (EPI == EPI_SILU_MUL) {
          tma_load_2d(ring + s * kStageBytes, &wmap, col, tile * 64, &full[s], pol);
          tma_load_2d(ring + s * kStageBytes + kStageBytes / 2, &wmap, col, p.inter + tile * 64, &full[s], pol);
        } else {
          tma_load_2d(ring + s * kStageBytes, &wmap, col, tile * kMmaM, &full[s], pol);
        }
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
      bool ok = mbar_wait(xready, 0);
      for (int i = 0; ok && i < nst; ++i) {
        const int s = i % NS;
        if (!mbar_wait(&full[s], static_cast<uint32_t>(i / NS) & 1u)) {
          ok = false;
          break;
        }
        tc_fence_after();
#pragma unroll
        for (int j = 0; j < kStageCols / 16; ++j) {
          // A: the stage, 128-byte swizzled rows of 64 columns, 8-row groups 1024 bytes
          // apart, advanced 32 bytes a K step; B: the activations, core matrices of 8
          // streams x 8 columns, 8-column groups NB * 16 bytes apart
          const uint64_t ad = smem_desc(smem_u32(ring + s * kStageBytes) + j * 32, 16, 1024, 2);
          const uint64_t bd = smem_desc(smem_u32(xs) + (i * 8 + 2 * j) * (NB * 16), NB * 16, 128, 0);
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
    // ------------------------------------------------ activations and epilogue
    constexpr int kCT = 128;
    grid_wait();
    // element (b, k) of the chunk at byte (k / 8) * NB * 16 + (b / 8) * 128 + (b % 8) * 16
    // + (k % 8) * 2: one 16-byte store per (stream, group of 8 columns)
    auto put8 = [&](int b, int kg, const uint4 v) {
      *reinterpret_cast<uint4*>(xs + kg * (NB * 16) + (b >> 3) * 128 + (b & 7) * 16) = v;
    };
    const int groups = kc / 8;
    if (XM == X_RMSNORM) {
      const float* h = static_cast<const float*>(p.x);
      // 1 / rms of every stream over the whole row: warp w takes streams w, w + 4, ...,
      // all of them at once, so their loads are in flight together
      constexpr int PW = NB / 4;
      float ss[PW];
#pragma unroll
      for (int j = 0; j < PW; ++j) ss[j] = 0.f;
      for (int k4 = lane; k4 < p.K / 4; k4 += 32) {
        float4 v[PW];
#pragma unroll
        for (int j = 0; j < PW; ++j) {
          const int b = warp + 4 * j;
          v[j] = b < B ? __ldcg(reinterpret_cast<const float4*>(h + static_cast<int64_t>(b) * p.x_stride) + k4)
                       : make_float4(0.f, 0.f, 0.f, 0.f);
        }
#pragma unroll
        for (int j = 0; j < PW; ++j) {
          ss[j] = fmaf(v[j].x, v[j].x, ss[j]);
          ss[j] = fmaf(v[j].y, v[j].y, ss[j]);
          ss[j] = fmaf(v[j].z, v[j].z, ss[j]);
          ss[j] = fmaf(v[j].w, v[j].w, ss[j]);
        }
      }
#pragma unroll
      for (int j = 0; j < PW; ++j) {
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) ss[j] += __shfl_xor_sync(kFull, ss[j], off);
        if (lane == 0) s_scale[warp + 4 * j] = 1.0f / sqrtf(ss[j] / static_cast<float>(p.K) + p.eps);
      }
      named_barrier(1, kCT);
    }
    for (int u = tid; u < NB * groups; u += kCT) {
      const int b = u / groups, kg = u - b * groups;
      const int k = k0 + kg * 8;
      uint4 out = make_uint4(0, 0, 0, 0);
      if (b < B) {
        if (XM == X_BF16) {
          out = __ldcg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.x) +
                                                      static_cast<int64_t>(b) * p.x_stride + k));
        } else {
          const float* row = static_cast<const float*>(p.x) + static_cast<int64_t>(b) * p.x_stride + k;
          const float4 a = __ldcg(reinterpret_cast<const float4*>(row));
          const float4 c = __ldcg(reinterpret_cast<const float4*>(row) + 1);
          float f[8] = {a.x, a.y, a.z, a.w, c.x, c.y, c.z, c.w};
          if (XM == X_RMSNORM) {
            const float sc = s_scale[b];
            const float4 g0 = __ldg(reinterpret_cast<const float4*>(p.gamma + k));
            const float4 g1 = __ldg(reinterpret_cast<const float4*>(p.gamma + k) + 1);
            const float g[8] = {g0.x, g0.y, g0.z, g0.w, g1.x, g1.y, g1.z, g1.w};
#pragma unroll
            for (int e = 0; e < 8; ++e) f[e] = f[e] * sc * g[e];
          }
          out = make_uint4(bf16_rne_bits(f[0]) | (static_cast<uint32_t>(bf16_rne_bits(f[1])) << 16),
                           bf16_rne_bits(f[2]) | (static_cast<uint32_t>(bf16_rne_bits(f[3])) << 16),
                           bf16_rne_bits(f[4]) | (static_cast<uint32_t>(bf16_rne_bits(f[5])) << 16),
                           bf16_rne_bits(f[6]) | (static_cast<uint32_t>(bf16_rne_bits(f[7])) << 16));
        }
      }
      put8(b, kg, out);
    }
    // the MMA reads the activations through the async proxy
    asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
    mbar_arrive(xready);

    // accumulator row m of this tile
    const int m = warp * 32 + lane;
    float v[NB];
    const bool got = mbar_wait(done, 0);
    if (!got && lane == 0) set_err(p.err, TTS_EFLAG_TIMEOUT);
    tc_fence_after();
    if (got) tmem_row<NB>(tmem + (static_cast<uint32_t>(warp * 32) << 16), v);
    else
#pragma unroll
      for (int b = 0; b < NB; ++b) v[b] = 0.f;
    bool write = got;
    if (mp.splits > 1) {
      // the partial of this column range; the last range of the tile sums them in order
      float4* dst = reinterpret_cast<float4*>(mp.part + ((static_cast<int64_t>(split) * mp.tiles + tile) * kMmaM + m) * NB);
#pragma unroll
      for (int b = 0; b < NB; b += 4) dst[b / 4] = make_float4(v[b], v[b + 1], v[b + 2], v[b + 3]);
      named_barrier(1, kCT);
      if (tid == 0) *s_last = (atomic_add_acq_rel_gpu(mp.tickets + tile, 1) == mp.splits - 1) ? 1 : 0;
      named_barrier(1, kCT);
      write = got && *s_last != 0;
      if (*s_last != 0) {
#pragma unroll
        for (int b = 0; b < NB; ++b) v[b] = 0.f;
        // ranges in order, two at a time so that twice the loads are in flight
        for (int s2 = 0; s2 < mp.splits; s2 += 2) {
          const float4* src0 =
              reinterpret_cast<const float4*>(mp.part + ((static_cast<int64_t>(s2) * mp.tiles + tile) * kMmaM + m) * NB);
          const float4* src1 = src0 + static_cast<int64_t>(mp.tiles) * kMmaM * (NB / 4);
          const bool two = s2 + 1 < mp.splits;
          float4 q0[NB / 4], q1[NB / 4];
#pragma unroll
          for (int c = 0; c < NB / 4; ++c) {
            q0[c] = __ldcg(src0 + c);
            q1[c] = two ? __ldcg(src1 + c) : make_float4(0.f, 0.f, 0.f, 0.f);
          }
#pragma unroll
          for (int c = 0; c < NB / 4; ++c) {
            v[4 * c] += q0[c].x;
            v[4 * c + 1] += q0[c].y;
            v[4 * c + 2] += q0[c].z;
            v[4 * c + 3] += q0[c].w;
          }
          if (two) {
#pragma unroll
            for (int c = 0; c < NB / 4; ++c) {
              v[4 * c] += q1[c].x;
              v[4 * c + 1] += q1[c].y;
              v[4 * c + 2] += q1[c].z;
              v[4 * c + 3] += q1[c].w;
            }
          }
        }
        if (tid == 0) mp.tickets[tile] = 0;
      }
    }
    if (EPI == EPI_SILU_MUL) {
      // rows 64..127 are the up rows of the items of rows 0..63
      if (write && m >= 64)
#pragma unroll
        for (int b = 0; b < NB; ++b) s_up[(m - 64) * NB + b] = v[b];
      named_barrier(1, kCT);
      if (write && m < 64) {
        const int item = tile * 64 + m;
        if (item < p.n_out)
#pragma unroll
          for (int b = 0; b < NB; ++b)
            if (b < B) {
              const float gt = v[b], up = s_up[m * NB + b];
              const float a = gt / (1.0f + expf(-gt)) * up;
              static_cast<uint16_t*>(p.y)[static_cast<int64_t>(b) * p.y_stride + item] = bf16_rne_bits(a);
            }
      }
    } else if (write) {
      const int row = tile * kMmaM + m;
      if (row < p.n_out) {
        float* yp = static_cast<float*>(p.y) + row;
        if (EPI == EPI_RESIDUAL) {
          // every stream's old value first (loads in flight together), then the sums
          float old[NB];
#pragma unroll
          for (int b = 0; b < NB; ++b) old[b] = b < B ? __ldcg(yp + static_cast<int64_t>(b) * p.y_stride) : 0.f;
#pragma unroll
          for (int b = 0; b < NB; ++b)
            if (b < B) yp[static_cast<int64_t>(b) * p.y_stride] = __fadd_rn(old[b], v[b]);
        } else {
#pragma unroll
          for (int b = 0; b < NB; ++b)
            if (b < B) yp[static_cast<int64_t>(b) * p.y_stride] = v[b];
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
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

size_t smem_bytes(int NB, int kc, int stages) {
  return 1024 + static_cast<size_t>(stages) * kStageBytes + static_cast<size_t>(NB) * kc * 2 +
         (static_cast<size_t>(NB) + 64 * NB) * sizeof(float) + (2 * kMaxStages + 2) * sizeof(uint64_t) + 16;
}

template <int XM, int EPI, int NB>
cudaError_t launch_mma_t(const MmaGemvParams& mp, cudaStream_t s) {
  auto kern = gemv_mma_kernel<XM, EPI, NB>;
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
  const size_t smem = smem_bytes(NB, mp.kc, mp.stages);
  static std::mutex mtx;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mtx);
    if (!configured[dev]) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, 227 * 1024);
      if (e != cudaSuccess) return e;
      configured[dev] = true;
    }
  }
  return launch_pdl(kern, dim3(mp.tiles, mp.splits), dim3(kThreads), smem, s, map, mp);
}

}  // namespace

// Column ranges per tile: enough CTAs to cover the GPU, ranges a multiple of 64 columns
// that divide K; the RMS-norm input reads every stream's whole row in every CTA, so it
// keeps to at most four ranges.
void gemv_mma_plan(int K, int n_out, int epilogue, int x_mode, int n_sm, int& tiles, int& splits, int& kc) {
  tiles = epilogue == EPI_SILU_MUL ? (n_out + 63) / 64 : (n_out + kMmaM - 1) / kMmaM;
  int s = (n_sm + tiles - 1) / tiles;
  if (s < 1) s = 1;
  const int max_s = x_mode == X_RMSNORM ? 4 : 16;
  if (s > max_s) s = max_s;
  while (s > 1 && K % (s * kStageCols) != 0) --s;
  splits = s;
  kc = K / s;
}

// Workspace of one launch: the tickets (at a fixed place, so that launches with other
// plans sharing the workspace find them at zero), then the partials.
constexpr size_t kTicketBytes = 4096;

size_t gemv_mma_workspace(int K, int n_out, int epilogue, int x_mode, int n_sm, int nb) {
  int tiles, splits, kc;
  gemv_mma_plan(K, n_out, epilogue, x_mode, n_sm, tiles, splits, kc);
  const size_t part = splits > 1 ? static_cast<size_t>(splits) * tiles * kMmaM * nb * sizeof(float) : 0;
  return kTicketBytes + part;
}

cudaError_t launch_gemv_mma(const GemvParams& p, int x_mode, int epilogue, void* workspace, size_t ws_bytes,
                            int n_sm, cudaStream_t s) {
  if (p.B < 1 || p.B > kGemvMmaMaxB || p.K % kStageCols != 0) return cudaErrorInvalidValue;
  const int nb = p.B <= 16 ? 16 : 32;
  MmaGemvParams mp = {};
  mp.g = p;
  gemv_mma_plan(p.K, p.n_out, epilogue, x_mode, n_sm, mp.tiles, mp.splits, mp.kc);
  const int nst = mp.kc / kStageCols;
  mp.stages = nst < kMaxStages ? nst : kMaxStages;
  const size_t part = mp.splits > 1 ? static_cast<size_t>(mp.splits) * mp.tiles * kMmaM * nb * sizeof(float) : 0;
  if (workspace == nullptr || ws_bytes < kTicketBytes + part ||
      static_cast<size_t>(mp.tiles) * sizeof(int) > kTicketBytes)
    return cudaErrorInvalidValue;
  mp.tickets = static_cast<int*>(workspace);
  mp.part = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) + kTicketBytes);
  if (smem_bytes(nb, mp.kc, mp.stages) > 227 * 1024) return cudaErrorInvalidValue;
#define TTS_MMA_CASE(XM, EPI)                                                          \
  if (x_mode == XM && epilogue == EPI)                                                 \
    return nb == 16 ? launch_mma_t<XM, EPI, 16>(mp, s) : launch_mma_t<XM, EPI, 32>(mp, s);
  TTS_MMA_CASE(X_RMSNORM, EPI_STORE)
  TTS_MMA_CASE(X_F32, EPI_RESIDUAL)
  TTS_MMA_CASE(X_RMSNORM, EPI_SILU_MUL)
  TTS_MMA_CASE(X_BF16, EPI_RESIDUAL)
#undef TTS_MMA_CASE
  return cudaErrorInvalidValue;
}

}  // namespace tts
