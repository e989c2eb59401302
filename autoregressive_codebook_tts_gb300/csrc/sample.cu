// In-graph token sampler with a counter RNG ("qwentts.cpp" pages: the code-predictor
// frame unroll keeps its in-graph sampler; "minicpm-o-4.5 ... optimizations.md",
// options table, "Lean Talker frame": one-kernel counter RNG).
//
// One CTA per stream.  The logits row is staged in shared memory; the top_k candidates
// (larger logit first, lower index first on a tie) are taken by top_k rounds of a
// block-wide arg-max that skips the candidates already taken.  Thread 0 then turns them
// into weights 2^((l_i - l_0) * log2(e) / T) and walks the running sum against
// u * sum, u from Philox4x64-10 at counter words (counter, stream) and key (seed, 0).
// Every value that decides the token is computed in f32 in a fixed order with explicit
// round-to-nearest operations (no contraction into fused multiply-adds); the
// exponential is this file's own (a degree-9 Taylor polynomial of 2^f, f in [0, 1),
// scaled by 2^floor(x)), not the math library's.
#include <cstdint>

#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"

namespace tts {
namespace {

constexpr int kSampleThreads = 256;
constexpr int kSampleWarps = kSampleThreads / 32;

// Philox4x64 with 10 rounds (Salmon, Moraes, Dror, Shaw, SC 2011).
__device__ __forceinline__ void philox4x64_10(uint64_t (&c)[4], uint64_t k0, uint64_t k1) {
  constexpr uint64_t kM0 = 0xD2E7470EE14C6C93ull, kM1 = 0xCA5A826395121157ull;
  constexpr uint64_t kW0 = 0x9E3779B97F4A7C15ull, kW1 = 0xBB67AE8584CAA73Bull;
#pragma unroll
  for (int r = 0; r < 10; ++r) {
    if (r > 0) {
      k0 += kW0;
      k1 += kW1;
    }
    const uint64_t hi0 = __umul64hi(kM0, c[0]), lo0 = kM0 * c[0];
    const uint64_t hi1 = __umul64hi(kM1, c[2]), lo1 = kM1 * c[2];
    const uint64_t n0 = hi1 ^ c[1] ^ k0, n2 = hi0 ^ c[3] ^ k1;
    c[0] = n0;
    c[1] = lo1;
    c[2] = n2;
    c[3] = lo0;
  }
}

// 2^x for x <= 0 in f32: 0 below -126, else Horner over the Taylor coefficients
// (ln 2)^j / j! (j = 0..9, rounded to f32) at f = x - floor(x), times 2^floor(x).
__device__ __forceinline__ float exp2_f32(float x) {
  if (!(x >= -126.0f)) return 0.0f;
  const float nf = floorf(x);
  const float f = __fsub_rn(x, nf);
  const float c[10] = {0x1.000000p+0f,  0x1.62e430p-1f,  0x1.ebfbe0p-3f,  0x1.c6b08ep-5f,
                       0x1.3b2ab6p-7f,  0x1.5d87fep-10f, 0x1.430912p-13f, 0x1.ffcbfcp-17f,
                       0x1.62c022p-20f, 0x1.b5253ep-24f};
  float p = c[9];
#pragma unroll
  for (int j = 8; j >= 0; --j) p = __fadd_rn(__fmul_rn(p, f), c[j]);
  const int n = static_cast<int>(nf);  // -126 <= n <= 0
  return __fmul_rn(p, __int_as_float((n + 127) << 23));
}

// Is (va, ia) ahead of (vb, ib): larger value first, lower index first on a tie.
__device__ __forceinline__ bool ahead(float va, int ia, float vb, int ib) {
  return ib < 0 || (ia >= 0 && (va > vb || (va == vb && ia < ib)));
}

__global__ void __launch_bounds__(kSampleThreads) sample_kernel(const SampleParams p) {
  extern __shared__ float s_val[];  // the row; NaN marks a taken candidate
  __shared__ float s_wv[kSampleWarps];
  __shared__ int s_wi[kSampleWarps];
  __shared__ float s_cv[TTS_MAX_TOP_K];
  __shared__ int s_ci[TTS_MAX_TOP_K];
  grid_wait();
  grid_launch_dependents();
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const float* row = p.logits + static_cast<int64_t>(b) * p.stride;
  for (int i = tid; i < p.V; i += kSampleThreads) {
    const float v = __ldcg(row + i);
    s_val[i] = (v != v) ? -INFINITY : v;  // a NaN logit counts as -inf
  }
  __syncthreads();
  const int rounds = p.top_k > 1 ? p.top_k : 1;
  for (int j = 0; j < rounds; ++j) {
    float bv = -INFINITY;
    int bi = -1;
    for (int i = tid; i < p.V; i += kSampleThreads) {
      const float v = s_val[i];
      if (v == v && ahead(v, i, bv, bi)) {
        bv = v;
        bi = i;
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const float ov = __shfl_xor_sync(kFull, bv, off);
      const int oi = __shfl_xor_sync(kFull, bi, off);
      if (ahead(ov, oi, bv, bi)) {
        bv = ov;
        bi = oi;
      }
    }
    if (lane == 0) {
      s_wv[warp] = bv;
      s_wi[warp] = bi;
    }
    __syncthreads();
    if (tid == 0) {
      for (int w = 1; w < kSampleWarps; ++w)
        if (ahead(s_wv[w], s_wi[w], bv, bi)) {
          bv = s_wv[w];
          bi = s_wi[w];
        }
      s_cv[j] = bv;
      s_ci[j] = bi;
      s_val[bi] = __int_as_float(0x7fc00000);  // taken
    }
    __syncthreads();
  }
  if (tid != 0) return;
  int pick = 0;
  const float m = s_cv[0];
  if (p.top_k > 1 && m > -INFINITY && m < INFINITY) {
    float w[TTS_MAX_TOP_K];
    float S = 0.0f;
    for (int j = 0; j < p.top_k; ++j) {
      w[j] = exp2_f32(__fmul_rn(__fsub_rn(s_cv[j], m), p.c));
      S = __fadd_rn(S, w[j]);
    }
    uint64_t ctr[4] = {__ldcg(p.counter), static_cast<uint64_t>(b), 0ull, 0ull};
    philox4x64_10(ctr, p.seed, 0ull);
    const float u = static_cast<float>(ctr[0] >> 40) * 0x1.0p-24f;  // exact
    const float r = __fmul_rn(u, S);
    float acc = 0.0f;
    pick = p.top_k - 1;
    for (int j = 0; j < p.top_k; ++j) {
      acc = __fadd_rn(acc, w[j]);
      if (acc > r) {
        pick = j;
        break;
      }
    }
  }
  p.out[static_cast<int64_t>(b) * p.out_stride] = s_ci[pick];
}

__global__ void counter_advance_kernel(uint64_t* counter, uint64_t by) {
  grid_wait();
  grid_launch_dependents();
  *counter += by;
}

}  // namespace

cudaError_t launch_sample(const SampleParams& p, cudaStream_t s) {
  const size_t smem = static_cast<size_t>(p.V) * sizeof(float);
  static int configured_for = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_for != dev) {
    e = cudaFuncSetAttribute(sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(TTS_MAX_SAMPLE_VOCAB * sizeof(float)));
    if (e != cudaSuccess) return e;
    configured_for = dev;
  }
  return launch_pdl(sample_kernel, dim3(p.B), dim3(kSampleThreads), smem, s, p);
}

cudaError_t launch_counter_advance(uint64_t* counter, uint64_t by, cudaStream_t s) {
  return launch_pdl(counter_advance_kernel, dim3(1), dim3(1), 0, s, counter, by);
}

}  // namespace tts
