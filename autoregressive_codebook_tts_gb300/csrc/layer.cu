// One whole talker decode layer with bf16 weights ("minicpm-o-4.5 ... optimizations.md",
// core table: fused residual add + RMSNorm, q/k norm + RoPE, SiLU-multiply, with the
// reference rounding reproduced by integer round-to-nearest-even; "Lean Talker frame":
// q/k/v as strided views of one projection).
//
//   x = rmsnorm(h) -> bf16            rmsnorm_bf16_kernel
//   qkv = x W_qkv^T (f32)             gemv_bf16_kernel<EPI_STORE>
//   attn = decode step (q, k, v)      decode_attn_kernel (fused), unchanged
//   h += bf16(attn) W_o^T             gemv_bf16_kernel<EPI_RESIDUAL>
//   x = rmsnorm(h) -> bf16            rmsnorm_bf16_kernel
//   a = silu(x W_g^T) * x W_u^T -> bf16   gemv_bf16_kernel<EPI_SILU_MUL>
//   h += a W_down^T                   gemv_bf16_kernel<EPI_RESIDUAL>
//
// At the batch sizes of a decode step (B <= 8 here) every product is a GEMV bound by
// streaming the weights from HBM: one warp per output row (a gate/up pair for the MLP),
// 16-byte coalesced weight loads four chunks deep, the activations staged once per CTA
// in shared memory as bf16, f32 accumulation, a warp reduction and a fused epilogue.
// Norm statistics and the SiLU are evaluated in double (a few thousand values a step),
// so the bf16 roundings follow the exact values.
#include <cstdint>

#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace tts {
namespace {

constexpr int kNormThreads = 256;

__device__ __forceinline__ uint16_t bf16_bits_rne(float x) {
  const __nv_bfloat16 h = __float2bfloat16_rn(x);
  return *reinterpret_cast<const uint16_t*>(&h);
}

// x[b] = bf16(h[b] * (mean(h[b]^2) + eps)^-1/2 * gamma): one CTA per stream, the sum of
// squares and the scaling in double, one rounding to f32, then RNE to bf16.
__global__ void __launch_bounds__(kNormThreads) rmsnorm_bf16_kernel(const float* h, const float* gamma,
                                                                    float eps, int H, uint16_t* x) {
  grid_wait();
  grid_launch_dependents();
  const int b = blockIdx.x;
  const float* row = h + static_cast<int64_t>(b) * H;
  __shared__ double s_part[kNormThreads / 32];
  __shared__ double s_r;
  double ss = 0.0;
  for (int i = threadIdx.x; i < H; i += kNormThreads) {
    const double v = __ldcg(row + i);
    ss = fma(v, v, ss);
  }
#pragma unroll
  for (int off = 16; off >= 1; off >>= 1) ss += __shfl_xor_sync(kFull, ss, off);
  if ((threadIdx.x & 31) == 0) s_part[threadIdx.x >> 5] = ss;
  __syncthreads();
  if (threadIdx.x == 0) {
    double t = 0.0;
    for (int w = 0; w < kNormThreads / 32; ++w) t += s_part[w];
    s_r = 1.0 / sqrt(t / H + static_cast<double>(eps));
  }
  __syncthreads();
  const double r = s_r;
  for (int i = threadIdx.x; i < H; i += kNormThreads) {
    const float y = static_cast<float>(static_cast<double>(__ldcg(row + i)) * r * static_cast<double>(gamma[i]));
    x[static_cast<int64_t>(b) * H + i] = bf16_bits_rne(y);
  }
}

enum Epilogue { EPI_STORE = 0, EPI_RESIDUAL = 1, EPI_SILU_MUL = 2 };

constexpr int kGemvWarps = 8;
constexpr int kGemvDepth = 4;  // 256-element chunks of a row in flight per warp

__device__ __forceinline__ void bf16x8_to_f32(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

// y[b][n] = sum_k x[b][k] W[n][k].  XT: the activations' type in global memory (f32 is
// rounded to bf16 when staged; bf16 is staged as is).  RPW output rows per warp: one,
// or (SILU_MUL) gate row n and up row n + inter.
template <typename XT, int EPI, int MAXB>
__global__ void __launch_bounds__(kGemvWarps * 32) gemv_bf16_kernel(const GemvParams p) {
  extern __shared__ __align__(16) uint16_t s_x[];  // [B][K] bf16
  constexpr int RPW = EPI == EPI_SILU_MUL ? 2 : 1;
  grid_wait();
  grid_launch_dependents();
  const int B = p.B, K = p.K;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  // stage the activations (every row of every stream) as bf16
  for (int i = tid; i < B * K; i += kGemvWarps * 32) {
    const int b = i / K, k = i - b * K;
    const XT v = static_cast<const XT*>(p.x)[static_cast<int64_t>(b) * p.x_stride + k];
    if constexpr (sizeof(XT) == 4) s_x[i] = bf16_bits_rne(v);
    else s_x[i] = *reinterpret_cast<const uint16_t*>(&v);
  }
  __syncthreads();
  const int n = blockIdx.x * kGemvWarps + warp;  // output row (SILU_MUL: pair index)
  if (n >= p.n_out) return;
  const uint16_t* wrow[RPW];
  wrow[0] = static_cast<const uint16_t*>(p.w) + static_cast<int64_t>(n) * K;
  if (RPW == 2) wrow[RPW - 1] = static_cast<const uint16_t*>(p.w) + static_cast<int64_t>(n + p.inter) * K;
  float acc[RPW][MAXB];
#pragma unroll
  for (int r = 0; r < RPW; ++r)
#pragma unroll
    for (int b = 0; b < MAXB; ++b) acc[r][b] = 0.f;
  const int chunks = K / 256;  // K is a multiple of 256
  for (int c0 = 0; c0 < chunks; c0 += kGemvDepth) {
    uint4 wv[kGemvDepth][RPW];
#pragma unroll
    for (int d = 0; d < kGemvDepth; ++d)
#pragma unroll
      for (int r = 0; r < RPW; ++r)
        if (c0 + d < chunks)
          wv[d][r] = __ldcs(reinterpret_cast<const uint4*>(wrow[r] + (c0 + d) * 256) + lane);
#pragma unroll
    for (int d = 0; d < kGemvDepth; ++d) {
      if (c0 + d >= chunks) break;
      float wf[RPW][8];
#pragma unroll
      for (int r = 0; r < RPW; ++r) bf16x8_to_f32(wv[d][r], wf[r]);
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
  if (lane >= B) return;
  // lane b writes stream b's result (acc values are warp-uniform after the reduction)
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

template <typename XT, int EPI>
cudaError_t launch_gemv_t(const GemvParams& p, cudaStream_t s) {
  auto kern = gemv_bf16_kernel<XT, EPI, kGemvMaxB>;
  const size_t smem = static_cast<size_t>(p.B) * p.K * sizeof(uint16_t);
  static int configured_for = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_for != dev) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(kGemvMaxB * kGemvMaxK * sizeof(uint16_t)));
    if (e != cudaSuccess) return e;
    configured_for = dev;
  }
  const dim3 grid((p.n_out + kGemvWarps - 1) / kGemvWarps);
  return launch_pdl(kern, grid, dim3(kGemvWarps * 32), smem, s, p);
}

}  // namespace

cudaError_t launch_rmsnorm_bf16(const float* h, const float* gamma, float eps, int B, int H, void* x,
                                cudaStream_t s) {
  return launch_pdl(rmsnorm_bf16_kernel, dim3(B), dim3(kNormThreads), 0, s, h, gamma, eps, H,
                    static_cast<uint16_t*>(x));
}

cudaError_t launch_gemv_bf16(const GemvParams& p, int x_f32, int epilogue, cudaStream_t s) {
  if (epilogue == EPI_STORE) return x_f32 ? launch_gemv_t<float, EPI_STORE>(p, s) : launch_gemv_t<__nv_bfloat16, EPI_STORE>(p, s);
  if (epilogue == EPI_RESIDUAL) return x_f32 ? launch_gemv_t<float, EPI_RESIDUAL>(p, s) : launch_gemv_t<__nv_bfloat16, EPI_RESIDUAL>(p, s);
  if (epilogue == EPI_SILU_MUL) return x_f32 ? launch_gemv_t<float, EPI_SILU_MUL>(p, s) : launch_gemv_t<__nv_bfloat16, EPI_SILU_MUL>(p, s);
  return cudaErrorInvalidValue;
}

}  // namespace tts
