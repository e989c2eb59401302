// One whole talker decode layer with bf16 weights ("minicpm-o-4.5 ... optimizations.md",
// core table: fused residual add + RMSNorm, q/k norm + RoPE, SiLU-multiply, with the
// reference rounding reproduced by integer round-to-nearest-even; "Lean Talker frame":
// q/k/v as strided views of one projection).
//
//   qkv = bf16(rmsnorm(h)) W_qkv^T (f32)      GEMV <X_RMSNORM, EPI_STORE>
//   attn = decode step (q, k, v)              decode_attn_kernel (fused), unchanged
//   h += bf16(attn) W_o^T                     GEMV <X_F32, EPI_RESIDUAL>
//   a = bf16(silu(x W_g^T) * x W_u^T), x = bf16(rmsnorm(h))
//                                             GEMV <X_RMSNORM, EPI_SILU_MUL>
//   h += a W_down^T                           GEMV <X_BF16, EPI_RESIDUAL>
//
// At the batch sizes of a decode step (B <= 8 here) every product is a GEMV bound by
// streaming the weights from HBM.  For one stream the weights are streamed into a
// shared-memory ring by bulk copies (gemv_bf16_kernel), for two to eight through
// registers (gemv_regs_kernel); both start loading before the dependency wait (the weights
// are constants), stage the activations once per CTA as bf16 (the RMS norm computed there,
// so it needs no launch of its own), accumulate each row in f32 and apply a fused
// epilogue: store, add into the residual stream, or SiLU-multiply.  The norm is computed in f32 by every
// CTA, and so is the SiLU.  A bf16 rounding of an intermediate can therefore land one
// step from the exact value's.
#include <cstdint>
#include <mutex>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace tts {
namespace {

__device__ __forceinline__ uint16_t bf16_bits_rne(float x) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<const uint16_t*>(&h);
}

enum Epilogue { EPI_STORE = 0, EPI_RESIDUAL = 1, EPI_SILU_MUL = 2 };
enum XMode { X_BF16 = 0, X_F32 = 1, X_RMSNORM = 2 };

constexpr int kRowWarps = 8;                         // consumer warps: one weight row each
constexpr int kGemvThreads = (kRowWarps + 1) * 32;   // + one producer warp
constexpr int kSegMax = 2048;                        // elements of a row segment (4 KB)
constexpr int kGemvMaxStages = 4;
constexpr size_t kCoResidentSmem = 110 * 1024;       // two CTAs of this size share an SM
constexpr size_t kGemvMaxSmem = 220 * 1024;

// y[b][n] = sum_k x[b][k] W[n][k], one CTA per SM, CTA c owning the output rows (gate/up
// pairs for the SiLU-multiply) [c n_out / grid, (c+1) n_out / grid).  Rows are split into
// segments of `seg` elements (<= 2048, 4 KB of bf16); a stage of the shared-memory ring
// holds one segment of each of eight weight rows (a group: eight output rows, or four
// gate rows and their four up rows), and consumer warp w always takes slot w, so a warp
// keeps its row across the segments of a group.  A producer warp streams the stages with
// 1-D bulk copies (complete_tx on a per-stage "full" mbarrier; the consumers release a
// stage on its "empty" mbarrier).  The weights are constants of the model, so the
// producer never waits for the preceding kernel: the ring fills while that kernel runs,
// and with at most ~110 KB of shared memory and few registers (56 a thread for one
// stream) the CTA fits on an SM beside a CTA of the neighbouring kernel, so consecutive
// launches overlap their weight streams.  The code handles up to MAXB streams; the
// launcher uses it for one.  The consumers wait for the preceding kernel, stage the activations once as
// bf16 (a bf16 input as is, an f32 input rounded, or the RMS norm of the f32 residual
// stream times gamma, in f32), and accumulate in f32.
template <int XM, int EPI, int MAXB>
__global__ void __maxnreg__(MAXB <= 2 ? 56 : 96) gemv_bf16_kernel(const GemvParams p) {
  extern __shared__ __align__(128) unsigned char smem[];
  __shared__ float s_red[kRowWarps][MAXB];
  __shared__ float s_pair[2][kRowWarps][MAXB];
  __shared__ __align__(8) uint64_t s_full[kGemvMaxStages];
  __shared__ __align__(8) uint64_t s_empty[kGemvMaxStages];
  constexpr int RPI = EPI == EPI_SILU_MUL ? 2 : 1;  // weight rows per output item
  constexpr int IPG = kRowWarps / RPI;             // output items per group
  const int B = p.B, K = p.K, seg = p.seg, NS = p.stages;
  const int S = K / seg;  // segments per row (stages per group)
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int i0 = static_cast<int>(static_cast<int64_t>(blockIdx.x) * p.n_out / gridDim.x);
  const int i1 = static_cast<int>(static_cast<int64_t>(blockIdx.x + 1) * p.n_out / gridDim.x);
  const int T = (i1 - i0 + IPG - 1) / IPG * S;  // stages of this CTA
  const uint32_t seg_bytes = static_cast<uint32_t>(seg) * 2u;
  unsigned char* ring = smem;
  uint16_t* s_x = reinterpret_cast<uint16_t*>(smem + p.x_off);  // after the ring
  if (tid == kRowWarps * 32) {
    for (int i = 0; i < NS; ++i) {
      mbar_init(&s_full[i], 1);
      mbar_init(&s_empty[i], kRowWarps);
    }
    mbar_init_fence();
  }
  __syncthreads();
  grid_launch_dependents();

  if (warp == kRowWarps) {  // producer
    const uint64_t pol = l2_evict_first_policy();
    const uint16_t* W = static_cast<const uint16_t*>(p.w);
    bool ok = true;
    int issued = 0;
    for (; issued < T; ++issued) {
      const int t = issued, slot = t % NS;
      if (t >= NS) {
        if (lane == 0) ok = mbar_wait(&s_empty[slot], ((t / NS) - 1) & 1);
        ok = __shfl_sync(kFull, ok, 0);
        if (!ok) break;
      }
      const int g = t / S, sgi = t - g * S;
      const int first = i0 + g * IPG;
      const int nval = min(IPG, i1 - first);
      if (lane == 0) mbar_arrive_expect_tx(&s_full[slot], static_cast<uint32_t>(nval * RPI) * seg_bytes);
      __syncwarp();
      if (lane < kRowWarps && lane % IPG < nval) {
        const int64_t row = first + lane % IPG + (lane / IPG ? p.inter : 0);
        bulk_g2s(ring + (static_cast<size_t>(slot) * kRowWarps + lane) * seg_bytes,
                 W + row * K + static_cast<int64_t>(sgi) * seg, seg_bytes, &s_full[slot], pol);
      }
    }
    if (!ok) set_err(p.err, TTS_EFLAG_TIMEOUT);
    // leave no copy in flight: wait (bounded) for the last stages issued
    if (lane == 0)
      for (int t = max(0, issued - NS); t < issued; ++t)
        if (!mbar_wait(&s_full[t % NS], (t / NS) & 1)) set_err(p.err, TTS_EFLAG_TIMEOUT);
    return;
  }

  // ---- consumers (warps 0..7, 256 threads) ----
  constexpr int kCT = kRowWarps * 32;
  // residual elements a thread keeps in registers per stream (the rest are read twice)
  constexpr int kNormRegs = MAXB <= 2 ? 8 : 16 / MAXB;
  float gam[kNormRegs];
  if (XM == X_RMSNORM) {
#pragma unroll
    for (int j = 0; j < kNormRegs; ++j) {
      const int k = tid + kCT * j;
      gam[j] = k < K ? __ldg(p.gamma + k) : 0.f;
    }
  }
  grid_wait();
  // residual epilogue: lane b's h[b][n] of this warp's rows, two groups ahead
  auto resid = [&](int g) -> float {
    const int it = i0 + g * IPG + warp % IPG;
    return (it < i1 && lane < B) ? __ldcg(static_cast<const float*>(p.y) + static_cast<int64_t>(lane) * p.y_stride + it)
                                 : 0.f;
  };
  float old0 = 0.f, old1 = 0.f;
  if (EPI == EPI_RESIDUAL) {
    old0 = resid(0);
    old1 = resid(1);
  }
  if (XM == X_RMSNORM) {
    const float* h = static_cast<const float*>(p.x);
    float hv[MAXB][kNormRegs];
    float ss[MAXB];
#pragma unroll
    for (int b = 0; b < MAXB; ++b) {
      ss[b] = 0.f;
#pragma unroll
      for (int j = 0; j < kNormRegs; ++j) {
        const int k = tid + kCT * j;
        hv[b][j] = (b < B && k < K) ? __ldcg(h + static_cast<int64_t>(b) * p.x_stride + k) : 0.f;
      }
    }
#pragma unroll
    for (int b = 0; b < MAXB; ++b) {
#pragma unroll
      for (int j = 0; j < kNormRegs; ++j) ss[b] = fmaf(hv[b][j], hv[b][j], ss[b]);
      if (b < B)
        for (int k = tid + kCT * kNormRegs; k < K; k += kCT) {
          const float v = __ldcg(h + static_cast<int64_t>(b) * p.x_stride + k);
          ss[b] = fmaf(v, v, ss[b]);
        }
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) ss[b] += __shfl_xor_sync(kFull, ss[b], off);
      if (lane == 0) s_red[warp][b] = ss[b];
    }
    named_barrier(1, kCT);
#pragma unroll
    for (int b = 0; b < MAXB; ++b) {
      if (b >= B) break;
      float t = 0.f;
#pragma unroll
      for (int w = 0; w < kRowWarps; ++w) t += s_red[w][b];
      const float scale = 1.0f / sqrtf(t / static_cast<float>(K) + p.eps);
#pragma unroll
      for (int j = 0; j < kNormRegs; ++j) {
        const int k = tid + kCT * j;
        if (k < K) s_x[b * K + k] = bf16_bits_rne(hv[b][j] * scale * gam[j]);
      }
      for (int k = tid + kCT * kNormRegs; k < K; k += kCT)
        s_x[b * K + k] = bf16_bits_rne(__ldcg(h + static_cast<int64_t>(b) * p.x_stride + k) * scale *
                                       __ldg(p.gamma + k));
    }
  } else if (XM == X_F32) {
    const int per = K / 4;  // float4 units a stream
    for (int u0 = tid; u0 < B * per; u0 += 4 * kCT) {
      float4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int u = u0 + j * kCT;
        if (u < B * per) {
          const int b = u / per, k4 = u - b * per;
          v[j] = __ldcg(reinterpret_cast<const float4*>(static_cast<const float*>(p.x) +
                                                        static_cast<int64_t>(b) * p.x_stride) + k4);
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int u = u0 + j * kCT;
        if (u < B * per) {
          const uint32_t lo = bf16_bits_rne(v[j].x) | (static_cast<uint32_t>(bf16_bits_rne(v[j].y)) << 16);
          const uint32_t hi = bf16_bits_rne(v[j].z) | (static_cast<uint32_t>(bf16_bits_rne(v[j].w)) << 16);
          reinterpret_cast<uint2*>(s_x)[u] = make_uint2(lo, hi);  // u = b * per + k4
        }
      }
    }
  } else {
    const int per = K / 8;  // 16-byte units a stream
    for (int u0 = tid; u0 < B * per; u0 += 4 * kCT) {
      uint4 v[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int u = u0 + j * kCT;
        if (u < B * per) {
          const int b = u / per, k8 = u - b * per;
          v[j] = __ldcg(reinterpret_cast<const uint4*>(static_cast<const uint16_t*>(p.x) +
                                                       static_cast<int64_t>(b) * p.x_stride) + k8);
        }
      }
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int u = u0 + j * kCT;
        if (u < B * per) reinterpret_cast<uint4*>(s_x)[u] = v[j];
      }
    }
  }
  named_barrier(1, kCT);

  float acc[MAXB];
#pragma unroll
  for (int b = 0; b < MAXB; ++b) acc[b] = 0.f;
  bool failed = false;
  const int chunks = seg / 256;  // at most kSegMax / 256
  for (int t = 0; t < T; ++t) {
    const int slot = t % NS;
    const int g = t / S, sgi = t - g * S;
    const int item = i0 + g * IPG + warp % IPG;
    const bool valid = item < i1;
    if (!failed) {
      const bool ok = __all_sync(kFull, mbar_wait(&s_full[slot], (t / NS) & 1));
      if (!ok) {
        failed = true;
        if (lane == 0) set_err(p.err, TTS_EFLAG_TIMEOUT);
      }
    }
    if (valid && !failed) {
      const unsigned char* wrow = ring + (static_cast<size_t>(slot) * kRowWarps + warp) * seg_bytes;
      const uint16_t* xs = s_x + sgi * seg + lane * 8;
      for (int c = 0; c < chunks; ++c) {
        float wf[8];
        unpack_bf16x8(lds128(wrow + (c * 256 + lane * 8) * 2), wf);
#pragma unroll
        for (int b = 0; b < MAXB; ++b) {
          if (b >= B) break;
          float xf[8];
          unpack_bf16x8(lds128(xs + b * K + c * 256), xf);
#pragma unroll
          for (int e = 0; e < 8; ++e) acc[b] = fmaf(wf[e], xf[e], acc[b]);
        }
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&s_empty[slot]);
    if (sgi != S - 1) continue;
    // the group's rows are complete: reduce, epilogue
#pragma unroll
    for (int b = 0; b < MAXB; ++b)
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) acc[b] += __shfl_xor_sync(kFull, acc[b], off);
    float mine = acc[0];  // lane b keeps stream b's sum
#pragma unroll
    for (int b = 1; b < MAXB; ++b)
      if (lane == b) mine = acc[b];
#pragma unroll
    for (int b = 0; b < MAXB; ++b) acc[b] = 0.f;
    if (EPI == EPI_STORE) {
      if (valid && lane < B && !failed)
        static_cast<float*>(p.y)[static_cast<int64_t>(lane) * p.y_stride + item] = mine;
    } else if (EPI == EPI_RESIDUAL) {
      if (valid && lane < B && !failed)
        static_cast<float*>(p.y)[static_cast<int64_t>(lane) * p.y_stride + item] = __fadd_rn(old0, mine);
      old0 = old1;
      old1 = resid(g + 2);
    } else {
      // warp w < IPG holds gate row of item w, warp w + IPG its up row
      if (lane < MAXB) s_pair[g & 1][warp][lane] = mine;
      named_barrier(1, kCT);
      if (warp < IPG && valid && lane < B && !failed) {
        const float gt = s_pair[g & 1][warp][lane], up = s_pair[g & 1][warp + IPG][lane];
        const float a = gt / (1.0f + expf(-gt)) * up;
        static_cast<uint16_t*>(p.y)[static_cast<int64_t>(lane) * p.y_stride + item] = bf16_bits_rne(a);
      }
    }
  }
}

// Two to eight streams: B FMAs per weight element make the ring's eight consumer warps
// the bottleneck, so this kernel streams the weights through registers instead,
// over up to two CTAs of eight warps per SM: warp w of CTA c takes output rows w + 8c,
// w + 8c + 8 * gridDim.x, ... (gate/up row pairs for the SiLU-multiply), each row in
// 256-element chunks, kDepth chunks in flight (about 4 KB a warp), the first issued
// before the dependency wait.  Activations are staged and epilogues applied as in the
// ring kernel.
constexpr int kRegWarps = 8;
constexpr int kRegDepth = 8;

template <int XM, int EPI>
__global__ void __launch_bounds__(kRegWarps * 32) gemv_regs_kernel(const GemvParams p) {
  constexpr int MAXB = kGemvMaxB;
  extern __shared__ __align__(16) uint16_t s_x[];  // [B][K] bf16
  __shared__ float s_red[kRegWarps][MAXB];
  __shared__ float s_scale[MAXB];
  constexpr int RPW = EPI == EPI_SILU_MUL ? 2 : 1;
  // 256-element chunks of each row in flight per warp (about 4 KB a warp)
  constexpr int kDepth = kRegDepth / RPW;
  const int B = p.B, K = p.K;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int chunks = K / 256;  // K is a multiple of 256
  const int stride_rows = kRegWarps * gridDim.x;
  int n = blockIdx.x * kRegWarps + warp;  // this warp's first output row (or pair)
  const uint16_t* W = static_cast<const uint16_t*>(p.w);
  auto row_ptr = [&](int row, int r) {
    return W + (static_cast<int64_t>(row) + (r ? p.inter : 0)) * K;
  };
  // first weight chunks, before the wait
  uint4 wv[kDepth][RPW];
  if (n < p.n_out) {
#pragma unroll
    for (int d = 0; d < kDepth; ++d)
#pragma unroll
      for (int r = 0; r < RPW; ++r)
        if (d < chunks) wv[d][r] = __ldcs(reinterpret_cast<const uint4*>(row_ptr(n, r) + d * 256) + lane);
  }
  grid_wait();
  grid_launch_dependents();
  // stage the activations
  if (XM == X_RMSNORM) {
    float ss[MAXB];
#pragma unroll
    for (int b = 0; b < MAXB; ++b) ss[b] = 0.f;
    const float* h = static_cast<const float*>(p.x);
    for (int k = tid; k < K; k += kRegWarps * 32)
#pragma unroll
      for (int b = 0; b < MAXB; ++b)
        if (b < B) {
          const float v = __ldcg(h + static_cast<int64_t>(b) * p.x_stride + k);
          ss[b] = fmaf(v, v, ss[b]);
        }
#pragma unroll
    for (int b = 0; b < MAXB; ++b) {
#pragma unroll
      for (int off = 16; off >= 1; off >>= 1) ss[b] += __shfl_xor_sync(kFull, ss[b], off);
      if (lane == 0) s_red[warp][b] = ss[b];
    }
    __syncthreads();
    if (tid < MAXB) {
      float t = 0.f;
      for (int w = 0; w < kRegWarps; ++w) t += s_red[w][tid];
      s_scale[tid] = 1.0f / sqrtf(t / static_cast<float>(K) + p.eps);
    }
    __syncthreads();
    for (int i = tid; i < B * K; i += kRegWarps * 32) {
      const int b = i / K, k = i - b * K;
      const float v = __ldcg(h + static_cast<int64_t>(b) * p.x_stride + k);
      s_x[i] = bf16_bits_rne(v * s_scale[b] * __ldg(p.gamma + k));
    }
  } else {
    for (int i = tid; i < B * K; i += kRegWarps * 32) {
      const int b = i / K, k = i - b * K;
      if (XM == X_F32)
        s_x[i] = bf16_bits_rne(__ldcg(static_cast<const float*>(p.x) + static_cast<int64_t>(b) * p.x_stride + k));
      else
        s_x[i] = __ldcg(static_cast<const uint16_t*>(p.x) + static_cast<int64_t>(b) * p.x_stride + k);
    }
  }
  __syncthreads();
  for (; n < p.n_out; n += stride_rows) {
    float acc[RPW][MAXB];
#pragma unroll
    for (int r = 0; r < RPW; ++r)
#pragma unroll
      for (int b = 0; b < MAXB; ++b) acc[r][b] = 0.f;
    for (int c0 = 0; c0 < chunks; c0 += kDepth) {
      uint4 cur[kDepth][RPW];
#pragma unroll
      for (int d = 0; d < kDepth; ++d)
#pragma unroll
        for (int r = 0; r < RPW; ++r) cur[d][r] = wv[d][r];
      // the next group: later chunks of this row, or the first of the next row
      const int c1 = c0 + kDepth;
      const int nn = c1 < chunks ? n : n + stride_rows;
      const int cc = c1 < chunks ? c1 : 0;
      if (nn < p.n_out) {
#pragma unroll
        for (int d = 0; d < kDepth; ++d)
#pragma unroll
          for (int r = 0; r < RPW; ++r)
            if (cc + d < chunks) wv[d][r] = __ldcs(reinterpret_cast<const uint4*>(row_ptr(nn, r) + (cc + d) * 256) + lane);
      }
#pragma unroll
      for (int d = 0; d < kDepth; ++d) {
        if (c0 + d >= chunks) break;
        float wf[RPW][8];
#pragma unroll
        for (int r = 0; r < RPW; ++r) unpack_bf16x8(cur[d][r], wf[r]);
        const int k0 = (c0 + d) * 256 + lane * 8;
#pragma unroll
        for (int b = 0; b < MAXB; ++b) {
          if (b >= B) break;
          float xf[8];
          unpack_bf16x8(*reinterpret_cast<const uint4*>(s_x + b * K + k0), xf);
#pragma unroll
          for (int r = 0; r < RPW; ++r)
#pragma unroll
            for (int e = 0; e < 8; ++e) acc[r][b] = fmaf(wf[r][e], xf[e], acc[r][b]);
        }
      }
    }
#pragma unroll
    for (int r = 0; r < RPW; ++r)
#pragma unroll
      for (int b = 0; b < MAXB; ++b)
#pragma unroll
        for (int off = 16; off >= 1; off >>= 1) acc[r][b] += __shfl_xor_sync(kFull, acc[r][b], off);
    if (lane < B) {
      // lane b writes stream b's result (every lane holds every sum after the reduction)
      float mine[RPW];
#pragma unroll
      for (int r = 0; r < RPW; ++r) {
        mine[r] = acc[r][0];
#pragma unroll
        for (int b = 1; b < MAXB; ++b)
          if (lane == b) mine[r] = acc[r][b];
      }
      const int b = lane;
      if (EPI == EPI_STORE) {
        static_cast<float*>(p.y)[static_cast<int64_t>(b) * p.y_stride + n] = mine[0];
      } else if (EPI == EPI_RESIDUAL) {
        float* hp = static_cast<float*>(p.y) + static_cast<int64_t>(b) * p.y_stride + n;
        *hp = __fadd_rn(*hp, mine[0]);
      } else {
        const float g = mine[0], u = mine[RPW - 1];
        const float a = g / (1.0f + expf(-g)) * u;
        static_cast<uint16_t*>(p.y)[static_cast<int64_t>(b) * p.y_stride + n] = bf16_bits_rne(a);
      }
    }
  }
}

template <int XM, int EPI>
cudaError_t launch_gemv_regs(const GemvParams& p, cudaStream_t s) {
  auto kern = gemv_regs_kernel<XM, EPI>;
  const size_t smem = static_cast<size_t>(p.B) * p.K * sizeof(uint16_t);
  // computed once per device under a lock, copied out before use
  static std::mutex cfg_mutex;
  static int configured_for = -1;
  static int cfg_n_sm = 1;
  static int cfg_per_sm = 1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int n_sm, per_sm;
  {
    std::lock_guard<std::mutex> cfg_lock(cfg_mutex);
    if (configured_for != dev) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(kGemvMaxB * kGemvMaxK * sizeof(uint16_t)));
      if (e != cudaSuccess) return e;
      if (cudaDeviceGetAttribute(&cfg_n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || cfg_n_sm < 1) {
        cudaGetLastError();
        cfg_n_sm = 1;
      }
      // CTAs that fit on an SM with the activation block of 8 streams x 2048
      if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&cfg_per_sm, kern, kRegWarps * 32,
                                                        kGemvMaxB * 2048 * sizeof(uint16_t)) != cudaSuccess ||
          cfg_per_sm < 1) {
        cudaGetLastError();
        cfg_per_sm = 1;
      }
      configured_for = dev;
    }
    n_sm = cfg_n_sm;
    per_sm = cfg_per_sm;
  }
  int ctas = (p.n_out + kRegWarps - 1) / kRegWarps;
  if (ctas > per_sm * n_sm) ctas = per_sm * n_sm;
  return launch_pdl(kern, dim3(ctas), dim3(kRegWarps * 32), smem, s, p);
}

template <int XM, int EPI, int MAXB>
cudaError_t launch_gemv_t(const GemvParams& p0, cudaStream_t s) {
  auto kern = gemv_bf16_kernel<XM, EPI, MAXB>;
  GemvParams p = p0;
  // segment: the longest multiple of 256 elements that divides K and is at most 2048
  int nseg = (p.K + kSegMax - 1) / kSegMax;
  while (p.K % nseg != 0 || (p.K / nseg) % 256 != 0) ++nseg;
  p.seg = p.K / nseg;
  // computed once per device under a lock, copied out before use
  static std::mutex cfg_mutex;
  static int configured_for = -1;
  static int cfg_n_sm = 1;
  static size_t cfg_co_budget = kCoResidentSmem;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  int n_sm;
  size_t co_budget;
  {
  std::lock_guard<std::mutex> cfg_lock(cfg_mutex);
  if (configured_for != dev) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(kGemvMaxSmem));
    if (e != cudaSuccess) return e;
    e = cudaFuncSetAttribute(kern, cudaFuncAttributePreferredSharedMemoryCarveout, cudaSharedmemCarveoutMaxShared);
    if (e != cudaSuccess) return e;
    if (cudaDeviceGetAttribute(&cfg_n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || cfg_n_sm < 1) {
      cudaGetLastError();
      cfg_n_sm = 1;
    }
    // dynamic shared memory that still lets two CTAs (of this or a neighbouring GEMV)
    // share an SM: half the SM's shared memory less the per-CTA reservation and the
    // kernel's static shared memory
    int per_sm = 0, reserved = 0;
    cudaFuncAttributes fa = {};
    if (cudaDeviceGetAttribute(&per_sm, cudaDevAttrMaxSharedMemoryPerMultiprocessor, dev) == cudaSuccess &&
        cudaDeviceGetAttribute(&reserved, cudaDevAttrReservedSharedMemoryPerBlock, dev) == cudaSuccess &&
        cudaFuncGetAttributes(&fa, kern) == cudaSuccess && per_sm > 0) {
      const long long b = per_sm / 2 - reserved - static_cast<long long>(fa.sharedSizeBytes);
      cfg_co_budget = b > 0 ? static_cast<size_t>(b) & ~static_cast<size_t>(127) : kCoResidentSmem;
    } else {
      cudaGetLastError();
    }
    configured_for = dev;
  }
  n_sm = cfg_n_sm;
  co_budget = cfg_co_budget;
  }
  const int ctas = p.n_out < n_sm ? p.n_out : n_sm;
  const size_t stage = static_cast<size_t>(kRowWarps) * p.seg * 2;
  const size_t x_bytes = static_cast<size_t>(p.B) * p.K * 2;
  // the deepest ring that leaves room for a neighbouring GEMV CTA on the SM, else the
  // deepest that fits at all
  int ns = kGemvMaxStages;
  while (ns > 2 && ns * stage + x_bytes > co_budget) --ns;
  if (ns * stage + x_bytes > co_budget) {
    ns = kGemvMaxStages;
    while (ns > 2 && ns * stage + x_bytes > kGemvMaxSmem) --ns;
  }
  p.stages = ns;
  p.x_off = static_cast<uint32_t>(ns * stage);
  const size_t smem = ns * stage + x_bytes;
  if (smem > kGemvMaxSmem) return cudaErrorInvalidValue;
  return launch_pdl(kern, dim3(ctas), dim3(kGemvThreads), smem, s, p);
}

}  // namespace

cudaError_t launch_gemv_bf16(const GemvParams& p, int x_mode, int epilogue, cudaStream_t s) {
  if (p.B < 1 || p.B > kGemvMaxB) return cudaErrorInvalidValue;
  // one stream: the ring kernel; two to eight: the register kernel (faster from two
  // streams on, where B FMAs per weight element keep the ring's consumers busy)
#define TTS_GEMV_CASE(XM, EPI)                                                                 \
  if (x_mode == XM && epilogue == EPI) {                                                       \
    if (p.B == 1) return launch_gemv_t<XM, EPI, 1>(p, s);                                      \
    return launch_gemv_regs<XM, EPI>(p, s);                                                    \
  }
  TTS_GEMV_CASE(X_RMSNORM, EPI_STORE)     // qkv
  TTS_GEMV_CASE(X_F32, EPI_RESIDUAL)      // o
  TTS_GEMV_CASE(X_RMSNORM, EPI_SILU_MUL)  // gate/up
  TTS_GEMV_CASE(X_BF16, EPI_RESIDUAL)     // down
#undef TTS_GEMV_CASE
  return cudaErrorInvalidValue;
}

}  // namespace tts
