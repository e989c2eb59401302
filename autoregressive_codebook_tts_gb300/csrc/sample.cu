// In-graph token sampler with a counter RNG ("qwentts.cpp" pages: the code-predictor
// frame unroll keeps its in-graph sampler; "minicpm-o-4.5 ... optimizations.md",
// options table, "Lean Talker frame": one-kernel counter RNG).
//
// One CTA per stream.  The logits row is staged in shared memory as order-preserving
// integer keys; the k-th largest is found by a radix selection (four 8-bit passes, each
// counting into one shared-memory histogram per warp; three barriers a pass).  After the first pass one scan of
// the row takes every key whose top byte is above the selected digit as a candidate and
// lists the indices of those with the selected top byte; the other three passes and the
// rest of the gather run over that list only.  Ties at the threshold go to the lowest
// indices (the last pass's count of keys equal to the threshold says whether there is a
// tie to break at all).  The candidates are ordered by rank (larger logit first, lower
// index first).  Each candidate's weight 2^((l_i - l_0) * log2(e) / T)
// is computed by its own thread; thread 0 forms the running sums in order while thread
// 32 draws u from Philox4x64-10 at counter words (counter, stream, draw, 0) and key
// (seed, 0); the token is the first candidate whose running sum exceeds u * sum (the
// running sums do not decrease, so every thread can test its own).
// Every value that decides the token is computed in f32 in a fixed order with explicit
// round-to-nearest operations (no contraction into fused multiply-adds); the
// exponential is this file's own (a degree-9 Taylor polynomial of 2^f, f in [0, 1),
// scaled by 2^floor(x)), not the math library's.
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "common.cuh"
#include "kernels.h"
#include "table_rows.cuh"

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

// Order-preserving 32-bit key of a float (a larger float has a larger key); the
// caller maps NaN to -inf and -0 to +0 first, so equal floats have equal keys.
__device__ __forceinline__ uint32_t float_key(float v) {
  const uint32_t u = __float_as_uint(v);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float key_float(uint32_t k) {
  return __uint_as_float((k & 0x80000000u) ? (k & 0x7fffffffu) : ~k);
}

// Is (ka, ia) ahead of (kb, ib): larger key first, lower index first on a tie.
__device__ __forceinline__ bool key_ahead(uint32_t ka, int ia, uint32_t kb, int ib) {
  return ka > kb || (ka == kb && ia < ib);
}

constexpr int kChunk = TTS_MAX_SAMPLE_VOCAB / kSampleThreads;  // indices per thread, at most
static_assert(TTS_MAX_TOP_K % 16 == 0 && TTS_MAX_TOP_K <= kSampleThreads, "running sums are formed 16 at a time");

// Inclusive sum of v over threads 0..tid of the block (kSampleThreads threads, all of
// them calling); s_part holds kSampleWarps ints of scratch.
__device__ __forceinline__ int block_inclusive_sum(int v, int* s_part) {
  const int lane = threadIdx.x & 31, warp = threadIdx.x >> 5;
#pragma unroll
  for (int off = 1; off < 32; off <<= 1) {
    const int o = __shfl_up_sync(kFull, v, off);
    if (lane >= off) v += o;
  }
  if (lane == 31) s_part[warp] = v;
  __syncthreads();
  int before = 0;
#pragma unroll
  for (int w = 0; w < kSampleWarps; ++w) before += w < warp ? s_part[w] : 0;
  __syncthreads();  // s_part may be reused by the caller's next scan
  return v + before;
}

// The drawn token's table row into emb_out[b] (the frame-input composition of one table
// without an overlay: the row itself, entries widened or dequantised exactly).  Every
// thread of the CTA calls this; `pick` is read after a barrier.
template <typename TabT>
__device__ __forceinline__ void gather_row_t(const SampleParams& p, int b, int id) {
  const TabT* row = table_row<TabT>(p.emb_tab, id, p.emb_hidden);
  float4* dst = reinterpret_cast<float4*>(p.emb_out + static_cast<int64_t>(b) * p.emb_hidden);
  for (int c4 = threadIdx.x; c4 < p.emb_hidden / 4; c4 += kSampleThreads) dst[c4] = load_row4(row, c4);
}
__device__ __forceinline__ void gather_row(const SampleParams& p, int b, volatile int& pick) {
  if (p.emb_out == nullptr) return;
  __syncthreads();
  const int id = pick;
  if (p.emb_dtype == TTS_BF16) gather_row_t<__nv_bfloat16>(p, b, id);
  else if (p.emb_dtype == TTS_Q8_0) gather_row_t<Q8Block>(p, b, id);
  else gather_row_t<float>(p, b, id);
}

__global__ void __launch_bounds__(kSampleThreads) sample_kernel(const SampleParams p) {
  extern __shared__ uint32_t s_key[];  // the row as keys, then (top_k >= 2) V ints of index list
  __shared__ int s_hist[kSampleWarps][256];  // per-warp digit counts of a pass
  __shared__ int s_sel[2][3];          // per pass parity: digit, keys still to take, bin count
  __shared__ int s_part[kSampleWarps];
  __shared__ int s_n, s_m;
  __shared__ uint2 s_cand[TTS_MAX_TOP_K];    // (key, index), in any order
  __shared__ uint2 s_sorted[TTS_MAX_TOP_K];  // the same, by rank
  __shared__ __align__(16) float s_w[TTS_MAX_TOP_K];
  __shared__ __align__(16) float s_acc[TTS_MAX_TOP_K];  // running sums of the weights, in order
  __shared__ int s_wc[2][kSampleWarps];      // per-warp counts of a two-phase compaction
  __shared__ float s_u;
  __shared__ int s_first;
  __shared__ uint32_t s_wk[kSampleWarps];
  __shared__ int s_wi[kSampleWarps];
  __shared__ int s_pick;
  grid_wait();
  grid_launch_dependents();
  const int b = blockIdx.x;
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int V = p.V;
  const float* row = p.logits + static_cast<int64_t>(b) * p.stride;
  for (int i = tid; i < V; i += kSampleThreads) {
    float v = __ldcg(row + i);
    if (v != v) v = -INFINITY;  // a NaN logit counts as -inf
    if (v == 0.0f) v = 0.0f;    // -0 and +0 are the same logit
    s_key[i] = float_key(v);
  }
#pragma unroll
  for (int w = 0; w < kSampleWarps; ++w) s_hist[w][255 - tid] = 0;  // thread t owns bin 255 - t
  if (tid == 0) {
    s_n = 0;
    s_m = 0;
  }
  // the draw's counter value, read early (its latency hides under the selection)
  const uint64_t ctr0 = (tid == 32 && p.top_k > 1) ? __ldcg(p.counter) : 0ull;
  __syncthreads();

  if (p.top_k <= 1) {
    // greedy: the largest logit, the lowest index on a tie
    uint32_t bk = 0;
    int bi = -1;
    for (int i = tid; i < V; i += kSampleThreads) {
      const uint32_t k = s_key[i];
      if (bi < 0 || key_ahead(k, i, bk, bi)) {
        bk = k;
        bi = i;
      }
    }
#pragma unroll
    for (int off = 16; off >= 1; off >>= 1) {
      const uint32_t ok = __shfl_xor_sync(kFull, bk, off);
      const int oi = __shfl_xor_sync(kFull, bi, off);
      if (oi >= 0 && (bi < 0 || key_ahead(ok, oi, bk, bi))) {
        bk = ok;
        bi = oi;
      }
    }
    if (lane == 0) {
      s_wk[warp] = bk;
      s_wi[warp] = bi;
    }
    __syncthreads();
    if (tid == 0) {
      for (int w = 1; w < kSampleWarps; ++w)
        if (s_wi[w] >= 0 && (bi < 0 || key_ahead(s_wk[w], s_wi[w], bk, bi))) {
          bk = s_wk[w];
          bi = s_wi[w];
        }
      p.out[static_cast<int64_t>(b) * p.out_stride] = bi;
      s_pick = bi;
    }
    gather_row(p, b, s_pick);
    return;
  }

  // The k-th largest key by radix selection, 8 bits a pass from the top: `prefix`
  // holds the digits fixed so far, `need` how many keys with that prefix are still to
  // take.  After the last pass, `prefix` is the threshold key, `need` how many of the
  // keys equal to it belong to the top k (the lowest-index ones) and `n_eq` how many
  // keys equal it.
  const int k = p.top_k;
  int* s_list = reinterpret_cast<int*>(s_key + V);  // indices whose keys share the fixed digits
  uint32_t prefix = 0, mask = 0;
  int need = k, n_eq = 0, n_list = V;
  for (int pass = 0; pass < 4; ++pass) {
    const int shift = 24 - 8 * pass;
    // keys that match the digits fixed so far (pass 0: the whole row; later: the list),
    // counted per next digit in the warp's own histogram
    int* hw = s_hist[warp];
    for (int base = 0; base < n_list; base += kSampleThreads) {
      const int j = base + tid;
      if (j < n_list) {
        const uint32_t key = s_key[pass == 0 ? j : s_list[j]];
        if ((key & mask) == prefix) atomicAdd(&hw[(key >> shift) & 255u], 1);
      }
    }
    __syncthreads();
    // the digit d with (keys in bins above d) < need <= (keys in bins from d up):
    // thread t holds bin 255 - t (summed over the warps' histograms, which it then
    // clears for the next pass: no other thread reads them), so its inclusive sum
    // counts the bins from it upward
    int c = 0;
#pragma unroll
    for (int w = 0; w < kSampleWarps; ++w) {
      c += s_hist[w][255 - tid];
      s_hist[w][255 - tid] = 0;
    }
    int incl = c;
#pragma unroll
    for (int off = 1; off < 32; off <<= 1) {
      const int o = __shfl_up_sync(kFull, incl, off);
      if (lane >= off) incl += o;
    }
    if (lane == 31) s_part[warp] = incl;
    __syncthreads();
#pragma unroll
    for (int w = 0; w < kSampleWarps; ++w) incl += w < warp ? s_part[w] : 0;
    const int excl = incl - c;
    if (excl < need && incl >= need) {
      s_sel[pass & 1][0] = 255 - tid;
      s_sel[pass & 1][1] = need - excl;
      s_sel[pass & 1][2] = c;
    }
    __syncthreads();
    prefix |= static_cast<uint32_t>(s_sel[pass & 1][0]) << shift;
    mask |= 255u << shift;
    need = s_sel[pass & 1][1];
    n_eq = s_sel[pass & 1][2];
    if (pass == 0) {
      // one scan of the row: keys whose top byte is above the digit are candidates
      // already; the indices of those with the digit form the list of the next passes.
      // Two phases without atomics: each warp counts its keys of either kind, then
      // writes them from its offset (warps in order, lanes in order within a ballot).
      const uint32_t d0 = prefix >> 24;
      int na = 0, ns = 0;
      for (int base = 0; base < V; base += kSampleThreads) {
        const int i = base + tid;
        const uint32_t top = i < V ? s_key[i] >> 24 : 0u;
        na += __popc(__ballot_sync(kFull, i < V && top > d0));
        ns += __popc(__ballot_sync(kFull, i < V && top == d0));
      }
      if (lane == 0) {
        s_wc[0][warp] = na;
        s_wc[1][warp] = ns;
      }
      __syncthreads();
      int oa = 0, os = 0;
#pragma unroll
      for (int w = 0; w < kSampleWarps; ++w) {
        oa += w < warp ? s_wc[0][w] : 0;
        os += w < warp ? s_wc[1][w] : 0;
      }
      const unsigned below = (1u << lane) - 1u;
      for (int base = 0; base < V; base += kSampleThreads) {
        const int i = base + tid;
        const uint32_t key = i < V ? s_key[i] : 0u;
        const uint32_t top = key >> 24;
        const bool above = i < V && top > d0, same = i < V && top == d0;
        const unsigned ba = __ballot_sync(kFull, above), bs = __ballot_sync(kFull, same);
        if (above) s_cand[oa + __popc(ba & below)] = make_uint2(key, static_cast<uint32_t>(i));
        if (same) s_list[os + __popc(bs & below)] = i;
        oa += __popc(ba);
        os += __popc(bs);
      }
      if (tid == 0) {
        int ta = 0, ts = 0;
        for (int w = 0; w < kSampleWarps; ++w) {
          ta += s_wc[0][w];
          ts += s_wc[1][w];
        }
        s_n = ta;
        s_m = ts;
      }
      __syncthreads();
      n_list = s_m;
    }
  }
  // The rest of the candidates: every listed key above the threshold and the `need`
  // lowest indices of those equal to it.
  if (n_eq == need) {
    // no tie to break: the listed keys at or above the threshold
    for (int base = 0; base < n_list; base += kSampleThreads) {
      const int j = base + tid;
      const int i = j < n_list ? s_list[j] : 0;
      const uint32_t key = j < n_list ? s_key[i] : 0u;
      const bool take = j < n_list && key >= prefix;
      const unsigned bal = __ballot_sync(kFull, take);
      int slot0 = 0;
      if (lane == 0 && bal != 0u) slot0 = atomicAdd(&s_n, __popc(bal));
      slot0 = __shfl_sync(kFull, slot0, 0);
      if (take) s_cand[slot0 + __popc(bal & ((1u << lane) - 1u))] = make_uint2(key, static_cast<uint32_t>(i));
    }
  } else {
    // ties at the threshold (rare): start over on the whole row; each thread owns a
    // contiguous index range, so an exclusive scan of the per-thread counts ranks the
    // equal keys by index
    __syncthreads();
    if (tid == 0) s_n = 0;
    const int i0 = tid * kChunk;
    const int i1 = min(i0 + kChunk, V);
    int eq = 0;
    for (int i = i0; i < i1; ++i) eq += s_key[i] == prefix;
    int rank = block_inclusive_sum(eq, s_part) - eq;  // equal keys at lower indices (also a barrier)
    for (int i = i0; i < i1; ++i) {
      const uint32_t key = s_key[i];
      bool take = key > prefix;
      if (key == prefix) take = rank++ < need;
      if (take) s_cand[atomicAdd(&s_n, 1)] = make_uint2(key, static_cast<uint32_t>(i));
    }
  }
  __syncthreads();
  // Order them (larger key first, lower index first) by rank, and weigh them.
  if (tid < TTS_MAX_TOP_K) {
    // a candidate's rank: how many others are ahead of it (entries past k are not read
    // as candidates: their comparisons are masked)
    const uint2 me = tid < k ? s_cand[tid] : make_uint2(0u, 0u);
    int r = 0;
#pragma unroll 16
    for (int j = 0; j < TTS_MAX_TOP_K; ++j) {
      const uint2 o = s_cand[j];
      const bool ahead = (o.x > me.x) | ((o.x == me.x) & (o.y < me.y));
      r += static_cast<int>((j < k) & ahead);
    }
    if (tid < k) s_sorted[r] = me;
  }
  __syncthreads();
  const float m = key_float(s_sorted[0].x);
  const bool finite_top = m > -INFINITY && m < INFINITY;
  if (tid < k && finite_top) s_w[tid] = exp2_f32(__fmul_rn(__fsub_rn(key_float(s_sorted[tid].x), m), p.c));
  if (tid == 0) s_first = k - 1;
  __syncthreads();
  if (finite_top) {
    if (tid == 0) {
      // the running sums in candidate order (the weights read into registers first);
      // the last is the total
      float acc = 0.0f;
      for (int j0 = 0; j0 < k; j0 += 16) {
        float w[16];
#pragma unroll
        for (int j = 0; j < 16; j += 4) {
          const float4 v = *reinterpret_cast<const float4*>(s_w + j0 + j);
          w[j] = v.x;
          w[j + 1] = v.y;
          w[j + 2] = v.z;
          w[j + 3] = v.w;
        }
#pragma unroll
        for (int j = 0; j < 16; ++j) {
          if (j0 + j < k) acc = __fadd_rn(acc, w[j]);
          w[j] = acc;
        }
#pragma unroll
        for (int j = 0; j < 16; j += 4)
          *reinterpret_cast<float4*>(s_acc + j0 + j) = make_float4(w[j], w[j + 1], w[j + 2], w[j + 3]);
      }
    } else if (tid == 32) {
      uint64_t ctr[4] = {ctr0, static_cast<uint64_t>(b), static_cast<uint64_t>(p.draw), 0ull};
      philox4x64_10(ctr, p.seed, 0ull);
      s_u = static_cast<float>(ctr[0] >> 40) * 0x1.0p-24f;  // exact
    }
    __syncthreads();
    // the first candidate whose running sum exceeds u * total (the last if none does)
    const float r = __fmul_rn(s_u, s_acc[k - 1]);
    if (tid < k && s_acc[tid] > r && (tid == 0 || !(s_acc[tid - 1] > r))) s_first = tid;
    __syncthreads();
  }
  if (tid == 0) {
    const int pick = finite_top ? s_first : 0;
    const int id = static_cast<int>(s_sorted[pick].y);
    p.out[static_cast<int64_t>(b) * p.out_stride] = id;
    s_pick = id;
  }
  gather_row(p, b, s_pick);
}

__global__ void counter_advance_kernel(uint64_t* counter, uint64_t by) {
  grid_wait();
  grid_launch_dependents();
  *counter += by;
}

}  // namespace

cudaError_t launch_sample(const SampleParams& p, cudaStream_t s) {
  // the keys, and for top_k >= 2 the index list after them
  const size_t smem = static_cast<size_t>(p.V) * sizeof(uint32_t) * (p.top_k > 1 ? 2 : 1);
  static std::mutex cfg_mutex;  // launches may come from several host threads
  static int configured_for = -1;
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  {
    std::lock_guard<std::mutex> cfg_lock(cfg_mutex);
    if (configured_for != dev) {
      e = cudaFuncSetAttribute(sample_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                               static_cast<int>(2 * TTS_MAX_SAMPLE_VOCAB * sizeof(uint32_t)));
      if (e != cudaSuccess) return e;
      configured_for = dev;
    }
  }
  return launch_pdl(sample_kernel, dim3(p.B), dim3(kSampleThreads), smem, s, p);
}

cudaError_t launch_counter_advance(uint64_t* counter, uint64_t by, cudaStream_t s) {
  return launch_pdl(counter_advance_kernel, dim3(1), dim3(1), 0, s, counter, by);
}

}  // namespace tts
