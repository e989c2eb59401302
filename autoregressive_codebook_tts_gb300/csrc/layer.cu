// One whole talker decode layer with bf16 weights ("minicpm-o-4.5 ... optimizations.md",
// core table: fused residual add + RMSNorm, q/k norm + RoPE, SiLU-multiply, with the
// reference rounding reproduced by integer round-to-nearest-even; "Lean Talker frame":
// q/k/v as strided views of one projection).
//
//   qkv = bf16(rmsnorm(h)) W_qkv^T (f32)      gemv_bf16_kernel<X_RMSNORM, EPI_STORE>
//   attn = decode step (q, k, v)              decode_attn_kernel (fused), unchanged
//   h += bf16(attn) W_o^T                     gemv_bf16_kernel<X_F32, EPI_RESIDUAL>
//   a = bf16(silu(x W_g^T) * x W_u^T), x = bf16(rmsnorm(h))
//                                             gemv_bf16_kernel<X_RMSNORM, EPI_SILU_MUL>
//   h += a W_down^T                           gemv_bf16_kernel<X_BF16, EPI_RESIDUAL>
//
// At the batch sizes of a decode step (B <= 8 here) every product is a GEMV bound by
// streaming the weights from HBM: one warp per output row (a gate/up pair for the MLP),
// 16-byte coalesced weight loads four chunks deep, started before the dependency wait,
// the activations staged once per CTA in shared memory as bf16 (the RMS norm computed
// there, so it needs no launch of its own), f32 accumulation, a warp reduction and a
// fused epilogue.  The norm is computed in f32 by every CTA (double arithmetic there
// cost more than the weight stream); the SiLU, one value per output, in double.  A bf16
// rounding of an intermediate can therefore land one step from the exact value's.
#include <cstdint>

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

constexpr int kGemvWarps = 8;
#ifndef TTS_GEMV_DEPTH
#define TTS_GEMV_DEPTH 8
#endif

__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// y[b][n] = sum_k x[b][k] W[n][k] over a grid of at most two CTAs per SM: warp w of
// CTA c takes output rows w + 8c, w + 8c + 8 * gridDim.x, ... (gate/up row pairs for
// the SiLU-multiply), streaming each row in 256-element chunks, kGemvDepth chunks in
// flight.  The weights are constants of the model, so the first loads are issued before
// the dependency wait and overlap the preceding kernel.  The activations are staged
// once per CTA as bf16: a bf16 input as is, an f32 input rounded, or (X_RMSNORM) the
// RMS norm of the f32 residual stream times gamma, in f32.
#ifndef TTS_GEMV_MIN_BLOCKS
#define TTS_GEMV_MIN_BLOCKS 1
#endif

template <int XM, int EPI, int MAXB>
__global__ void __launch_bounds__(kGemvWarps * 32, TTS_GEMV_MIN_BLOCKS) gemv_bf16_kernel(const GemvParams p) {
  extern __shared__ __align__(16) uint16_t s_x[];  // [B][K] bf16
  __shared__ float s_red[kGemvWarps][MAXB];
  __shared__ float s_scale[MAXB];
  constexpr int RPW = EPI == EPI_SILU_MUL ? 2 : 1;
  // 256-element chunks of each row in flight per warp (about 4 KB a warp)
  constexpr int kGemvDepth = TTS_GEMV_DEPTH / RPW;
  const int B = p.B, K = p.K;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int chunks = K / 256;  // K is a multiple of 256
  const int stride_rows = kGemvWarps * gridDim.x;
  int n = blockIdx.x * kGemvWarps + warp;  // this warp's first output row (or pair)
  const uint16_t* W = static_cast<const uint16_t*>(p.w);
  auto row_ptr = [&](int row, int r) {
    return W + (static_cast<int64_t>(row) + (r ? p.inter : 0)) * K;
  };
  // first weight chunks, before the wait
  uint4 wv[kGemvDepth][RPW];
  if (n < p.n_out) {
#pragma unroll
    for (int d = 0; d < kGemvDepth; ++d)
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
    for (int k = tid; k < K; k += kGemvWarps * 32)
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
      for (int w = 0; w < kGemvWarps; ++w) t += s_red[w][tid];
      s_scale[tid] = 1.0f / sqrtf(t / static_cast<float>(K) + p.eps);
    }
    __syncthreads();
    for (int i = tid; i < B * K; i += kGemvWarps * 32) {
      const int b = i / K, k = i - b * K;
      const float v = __ldcg(h + static_cast<int64_t>(b) * p.x_stride + k);
      s_x[i] = bf16_bits_rne(v * s_scale[b] * __ldg(p.gamma + k));
    }
  } else {
    for (int i = tid; i < B * K; i += kGemvWarps * 32) {
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
    for (int c0 = 0; c0 < chunks; c0 += kGemvDepth) {
      uint4 cur[kGemvDepth][RPW];
#pragma unroll
      for (int d = 0; d < kGemvDepth; ++d)
#pragma unroll
        for (int r = 0; r < RPW; ++r) cur[d][r] = wv[d][r];
      // the next group: later chunks of this row, or the first of the next row
      const int c1 = c0 + kGemvDepth;
      const int nn = c1 < chunks ? n : n + stride_rows;
      const int cc = c1 < chunks ? c1 : 0;
      if (nn < p.n_out) {
#pragma unroll
        for (int d = 0; d < kGemvDepth; ++d)
#pragma unroll
          for (int r = 0; r < RPW; ++r)
            if (cc + d < chunks) wv[d][r] = __ldcs(reinterpret_cast<const uint4*>(row_ptr(nn, r) + (cc + d) * 256) + lane);
      }
#pragma unroll
      for (int d = 0; d < kGemvDepth; ++d) {
        if (c0 + d >= chunks) break;
        float wf[RPW][8];
#pragma unroll
        for (int r = 0; r < RPW; ++r) bf16x8_to_f32(cur[d][r], wf[r]);
        const int k0 = (c0 + d) * 256 + lane * 8;
#pragma unroll
        for (int b = 0; b < MAXB; ++b) {
          if (b >= B) break;
          float xf[8];
          bf16x8_to_f32(*reinterpret_cast<const uint4*>(s_x + b * K + k0), xf);
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
        const double g = mine[0], u = mine[RPW - 1];
        const float a = static_cast<float>(g / (1.0 + exp(-g)) * u);
        static_cast<uint16_t*>(p.y)[static_cast<int64_t>(b) * p.y_stride + n] = bf16_bits_rne(a);
      }
    }
  }
}

template <int XM, int EPI>
cudaError_t launch_gemv_t(const GemvParams& p, cudaStream_t s) {
  auto kern = gemv_bf16_kernel<XM, EPI, kGemvMaxB>;
  const size_t smem = static_cast<size_t>(p.B) * p.K * sizeof(uint16_t);
  static int configured_for = -1;
  static int n_sm = 1;
  static int per_sm = 1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_for != dev) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kGemvMaxB * kGemvMaxK * sizeof(uint16_t)));
    if (e != cudaSuccess) return e;
    if (cudaDeviceGetAttribute(&n_sm, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n_sm < 1) {
      cudaGetLastError();
      n_sm = 1;
    }
    // CTAs that fit on an SM with the largest activation block (8 streams x 8192)
    if (cudaOccupancyMaxActiveBlocksPerMultiprocessor(&per_sm, kern, kGemvWarps * 32,
                                                      kGemvMaxB * 2048 * sizeof(uint16_t)) != cudaSuccess ||
        per_sm < 1) {
      cudaGetLastError();
      per_sm = 1;
    }
    configured_for = dev;
  }
  int ctas = (p.n_out + kGemvWarps - 1) / kGemvWarps;
  if (ctas > per_sm * n_sm) ctas = per_sm * n_sm;
  return launch_pdl(kern, dim3(ctas), dim3(kGemvWarps * 32), smem, s, p);
}

}  // namespace

cudaError_t launch_gemv_bf16(const GemvParams& p, int x_mode, int epilogue, cudaStream_t s) {
#define TTS_GEMV_CASE(XM)                                                                      \
  if (x_mode == XM) {                                                                          \
    if (epilogue == EPI_STORE) return launch_gemv_t<XM, EPI_STORE>(p, s);                      \
    if (epilogue == EPI_RESIDUAL) return launch_gemv_t<XM, EPI_RESIDUAL>(p, s);                \
    if (epilogue == EPI_SILU_MUL) return launch_gemv_t<XM, EPI_SILU_MUL>(p, s);                \
  }
  TTS_GEMV_CASE(X_BF16)
  TTS_GEMV_CASE(X_F32)
  TTS_GEMV_CASE(X_RMSNORM)
#undef TTS_GEMV_CASE
  return cudaErrorInvalidValue;
}

}  // namespace tts
