// Per-frame kernels around the attention: frame-input composition, RoPE table,
// standalone q/k norm + RoPE, set_rows KV write, workspace clear.
#include <cuda_fp16.h>

#include "common.cuh"
#include "kernels.h"
#include "table_rows.cuh"

namespace tts {
namespace {

// ---------------------------------------------------------------------------
// Frame-input composition ("qwentts.cpp ... src/pipeline-tts.h", on-device AR input
// assembly): out[b] = ((E_0[c0] + E_1[c1]) + ...) + overlay[b].  One thread per four
// columns; the (up to 16) row loads are issued together, then added strictly left to
// right with single f32 additions, the overlay last, so the result is bit-identical to
// that sequence of additions.
// ---------------------------------------------------------------------------
constexpr int kEmbedThreads = 128;

template <typename TabT>
__global__ void __launch_bounds__(kEmbedThreads) frame_embed_kernel(const EmbedParams p) {
  grid_wait();
  grid_launch_dependents();
  const int b = blockIdx.y;
  const int c4 = blockIdx.x * kEmbedThreads + threadIdx.x;  // float4 column
  if (c4 * 4 >= p.hidden) return;
  const int n = p.n_tables;
  float4 rows[TTS_MAX_TABLES];
  bool bad = false;
#pragma unroll
  for (int t = 0; t < TTS_MAX_TABLES; ++t) {
    if (t < n) {
      int id = __ldcg(p.ids + static_cast<int64_t>(b) * p.ids_stride + t);
      if (id < 0 || id >= p.vocab) {
        bad = true;
        id = min(max(id, 0), p.vocab - 1);
      }
      rows[t] = load_row4(table_row<TabT>(p.tab[t], id, p.hidden), c4);
    }
  }
  float4 acc = rows[0];
#pragma unroll
  for (int t = 1; t < TTS_MAX_TABLES; ++t) {
    if (t < n) {
      acc.x = __fadd_rn(acc.x, rows[t].x);
      acc.y = __fadd_rn(acc.y, rows[t].y);
      acc.z = __fadd_rn(acc.z, rows[t].z);
      acc.w = __fadd_rn(acc.w, rows[t].w);
    }
  }
  if (p.overlay != nullptr) {
    const float4 ov = __ldcg(reinterpret_cast<const float4*>(p.overlay + static_cast<int64_t>(b) * p.overlay_stride) + c4);
    acc.x = __fadd_rn(acc.x, ov.x);
    acc.y = __fadd_rn(acc.y, ov.y);
    acc.z = __fadd_rn(acc.z, ov.z);
    acc.w = __fadd_rn(acc.w, ov.w);
  }
  reinterpret_cast<float4*>(p.out + static_cast<int64_t>(b) * p.hidden)[c4] = acc;
  if (bad && c4 == 0) set_err(p.err, TTS_EFLAG_ID_RANGE);
}

// ---------------------------------------------------------------------------
// RoPE table: cs[pos][i] = (cos, sin)(pos * base^(-2i/D)), angle and cos/sin in double.
// ---------------------------------------------------------------------------
__global__ void rope_table_kernel(float2* cs, int max_pos, int head_dim, double base) {
  grid_wait();
  grid_launch_dependents();
  const int half = head_dim / 2;
  const int64_t idx = static_cast<int64_t>(blockIdx.x) * blockDim.x + threadIdx.x;
  if (idx >= static_cast<int64_t>(max_pos) * half) return;
  const int pos = static_cast<int>(idx / half);
  const int i = static_cast<int>(idx - static_cast<int64_t>(pos) * half);
  const double theta = static_cast<double>(pos) * pow(base, -2.0 * i / head_dim);
  double sn, cn;
  sincos(theta, &sn, &cn);
  cs[idx] = make_float2(static_cast<float>(cn), static_cast<float>(sn));
}

// ---------------------------------------------------------------------------
// Standalone q/k RMSNorm + RoPE, in place ("minicpm-o-4.5 ... optimizations.md",
// core table, fused q/k norm + RoPE).  One group of D/4 lanes per head row.
// ---------------------------------------------------------------------------
constexpr int kNormWarps = 4;

template <int D>
__global__ void __launch_bounds__(kNormWarps * 32) qk_norm_rope_kernel(const NormRopeParams p) {
  constexpr int EPL = 4, LPR = D / EPL, RPW = 32 / LPR;
  grid_wait();
  grid_launch_dependents();
  const int b = blockIdx.y;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int n_rows = p.n_q_heads + p.n_kv_heads;
  const int row = (blockIdx.x * kNormWarps + warp) * RPW + lane / LPR;
  const bool live = row < n_rows;  // whole row groups are live or not; shuffles stay in group
  int pos = __ldcg(p.pos + b);
  if (pos < 0 || pos >= p.max_pos) {
    if (live && (lane % LPR) == 0 && row == 0) set_err(p.err, TTS_EFLAG_POS_RANGE);
    pos = min(max(pos, 0), p.max_pos - 1);
  }
  const int e0 = (lane % LPR) * EPL;
  const bool is_q = row < p.n_q_heads;
  float* ptr = is_q ? p.q + static_cast<int64_t>(b) * p.q_stride + static_cast<int64_t>(row) * D
                    : p.k + static_cast<int64_t>(b) * p.k_stride + static_cast<int64_t>(row - p.n_q_heads) * D;
  const float* gamma = is_q ? p.gamma_q : p.gamma_k;
  float x[EPL] = {0.f, 0.f, 0.f, 0.f};
  if (live) {
    const float4 v = __ldcg(reinterpret_cast<const float4*>(ptr + e0));
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
  }
  // Dead row groups run the same shuffles on zeros (gamma/cs reads stay in bounds).
  float gam[EPL];
  float2 cs[EPL];
  load_norm_consts<EPL, 1, LPR>(live ? gamma : p.gamma_q, p.cs + static_cast<int64_t>(pos) * (D / 2),
                                lane % LPR, D, gam, cs);
  norm_rope_regs<EPL, 1, LPR>(x, gam, cs, p.eps, lane % LPR, D);
  if (live) *reinterpret_cast<float4*>(ptr + e0) = make_float4(x[0], x[1], x[2], x[3]);
}

// ---------------------------------------------------------------------------
// set_rows KV write ("qwentts.cpp ... src/pipeline-tts.h", fixed-topology section):
// the destination position is device data.  One thread per four elements of the
// stream's Hkv*D row; bf16 conversion rounds to nearest even.
// ---------------------------------------------------------------------------
constexpr int kSetRowsThreads = 128;

__device__ __forceinline__ void store4(float* dst, float4 v) { *reinterpret_cast<float4*>(dst) = v; }
__device__ __forceinline__ void store4(__nv_bfloat16* dst, float4 v) {
  const __nv_bfloat162 a = __floats2bfloat162_rn(v.x, v.y);
  const __nv_bfloat162 c = __floats2bfloat162_rn(v.z, v.w);
  uint2 w;
  w.x = *reinterpret_cast<const uint32_t*>(&a);
  w.y = *reinterpret_cast<const uint32_t*>(&c);
  *reinterpret_cast<uint2*>(dst) = w;
}

template <typename KvT>
__global__ void __launch_bounds__(kSetRowsThreads) set_rows_kernel(const SetRowsParams p) {
  grid_wait();
  grid_launch_dependents();
  const int b = blockIdx.y;
  const int D = p.head_dim;
  const int idx4 = blockIdx.x * kSetRowsThreads + threadIdx.x;  // float4 index in the row
  if (idx4 * 4 >= p.n_kv_heads * D) return;
  const int pos = __ldcg(p.pos + b);
  if (pos < 0 || pos >= p.capacity) {
    if (idx4 == 0) set_err(p.err, TTS_EFLAG_POS_RANGE);
    return;
  }
  const int g = (idx4 * 4) / D;
  const int d = idx4 * 4 - g * D;
  size_t row;
  if (!p.paged) {
    row = (static_cast<size_t>(b) * p.n_kv_heads + g) * p.capacity + pos;
  } else {
    const int page = __ldcg(p.block_table + static_cast<int64_t>(b) * p.bt_stride + pos / p.page_size);
    if (page < 0 || page >= p.n_pages) {
      if (idx4 == 0) set_err(p.err, TTS_EFLAG_PAGE);
      return;
    }
    row = (static_cast<size_t>(page) * p.n_kv_heads + g) * p.page_size + pos % p.page_size;
  }
  const float4 kv = __ldcg(reinterpret_cast<const float4*>(p.k + static_cast<int64_t>(b) * p.row_stride) + idx4);
  const float4 vv = __ldcg(reinterpret_cast<const float4*>(p.v + static_cast<int64_t>(b) * p.row_stride) + idx4);
  store4(static_cast<KvT*>(p.k_cache) + row * D + d, kv);
  store4(static_cast<KvT*>(p.v_cache) + row * D + d, vv);
}

// ---------------------------------------------------------------------------
// Prefill rows ("qwentts.cpp ... src/pipeline-tts.h", KV cache section: the prefill
// writes the prompt's positions into the cache).  Row r = b * T + t sits at position
// start[b] + t: its q heads are RMS-normed and rotated into q_out (the attention reads
// them there; the caller's q rows are left as they are), its k heads normed, rotated and
// written into the cache, its v heads written as they are.  One group of D/4 lanes per head row, as in the standalone norm.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void store4(float* dst, const float (&x)[4]) {
  *reinterpret_cast<float4*>(dst) = make_float4(x[0], x[1], x[2], x[3]);
}
__device__ __forceinline__ void store4(__nv_bfloat16* dst, const float (&x)[4]) {
  store4(dst, make_float4(x[0], x[1], x[2], x[3]));
}

template <int D, typename KvT>
__global__ void __launch_bounds__(kNormWarps * 32) prefill_rows_kernel(const PrefillRowsParams p) {
  constexpr int EPL = 4, LPR = D / EPL, RPW = 32 / LPR;
  grid_wait();
  grid_launch_dependents();
  const int r = blockIdx.y;  // b * T + t
  const int b = r / p.T;
  const int t = r - b * p.T;
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int Hq = p.n_q_heads, Hkv = p.n_kv_heads;
  const int row = (blockIdx.x * kNormWarps + warp) * RPW + lane / LPR;  // head row
  const bool live = row < Hq + 2 * Hkv;  // whole row groups are live or not
  const int pos = __ldcg(p.start + b) + t;
  const bool pos_ok = pos >= 0 && pos < p.capacity && pos < p.max_pos;
  if (!pos_ok && row == 0 && (lane % LPR) == 0) set_err(p.err, TTS_EFLAG_POS_RANGE);
  const int rpos = min(max(pos, 0), p.max_pos - 1);
  const int kind = row < Hq ? 0 : (row < Hq + Hkv ? 1 : 2);  // q, k, v
  // q rows nobody reads from here are skipped: a warp whose rows are all such leaves;
  // otherwise they run the norm's shuffles on zeros and store nothing
  const bool skip = kind == 0 && p.q_out == nullptr;
  if (__all_sync(kFull, skip)) return;
  const int e0 = (lane % LPR) * EPL;
  const int64_t base = static_cast<int64_t>(r) * p.row_stride;
  const float* src = kind == 0 ? p.q + base + static_cast<int64_t>(row) * D
                   : kind == 1 ? p.k + base + static_cast<int64_t>(row - Hq) * D
                               : p.v + base + static_cast<int64_t>(row - Hq - Hkv) * D;
  float x[EPL] = {0.f, 0.f, 0.f, 0.f};
  if (live && !skip) {
    const float4 v = __ldcg(reinterpret_cast<const float4*>(src + e0));
    x[0] = v.x; x[1] = v.y; x[2] = v.z; x[3] = v.w;
  }
  // Every group runs the norm's shuffles (v and dead rows on their own values or zeros,
  // results discarded), so the full-warp shuffles stay convergent.
  float y[EPL] = {x[0], x[1], x[2], x[3]};
  float gam[EPL];
  float2 cs[EPL];
  load_norm_consts<EPL, 1, LPR>(kind == 1 ? p.gamma_k : p.gamma_q, p.cs + static_cast<int64_t>(rpos) * (D / 2),
                                lane % LPR, D, gam, cs);
  norm_rope_regs<EPL, 1, LPR>(y, gam, cs, p.eps, lane % LPR, D);
  if (!live) return;
  if (kind == 0) {
    if (!skip)
      *reinterpret_cast<float4*>(p.q_out + static_cast<int64_t>(r) * Hq * D + static_cast<int64_t>(row) * D + e0) =
          make_float4(y[0], y[1], y[2], y[3]);
    return;
  }
  if (!pos_ok) return;
  const int g = kind == 1 ? row - Hq : row - Hq - Hkv;
  size_t crow;
  if (!p.paged) {
    crow = (static_cast<size_t>(b) * Hkv + g) * p.capacity + pos;
  } else {
    const int page = __ldcg(p.block_table + static_cast<int64_t>(b) * p.bt_stride + pos / p.page_size);
    if (page < 0 || page >= p.n_pages) {
      if ((lane % LPR) == 0) set_err(p.err, TTS_EFLAG_PAGE);
      return;
    }
    crow = (static_cast<size_t>(page) * Hkv + g) * p.page_size + pos % p.page_size;
  }
  KvT* dst = static_cast<KvT*>(kind == 1 ? p.k_cache : p.v_cache) + crow * D + e0;
  if (kind == 1) store4(dst, y);
  else store4(dst, x);
}

__global__ void zero_kernel(uint4* p, size_t n16) {
  grid_wait();
  grid_launch_dependents();
  for (size_t i = static_cast<size_t>(blockIdx.x) * blockDim.x + threadIdx.x; i < n16;
       i += static_cast<size_t>(gridDim.x) * blockDim.x)
    p[i] = make_uint4(0, 0, 0, 0);
}

}  // namespace

cudaError_t launch_frame_embed(const EmbedParams& p, cudaStream_t s) {
  const int cols4 = p.hidden / 4;
  dim3 grid((cols4 + kEmbedThreads - 1) / kEmbedThreads, p.B);
  if (p.tab_dtype == TTS_BF16) return launch_pdl(frame_embed_kernel<__nv_bfloat16>, grid, dim3(kEmbedThreads), 0, s, p);
  if (p.tab_dtype == TTS_Q8_0) return launch_pdl(frame_embed_kernel<Q8Block>, grid, dim3(kEmbedThreads), 0, s, p);
  return launch_pdl(frame_embed_kernel<float>, grid, dim3(kEmbedThreads), 0, s, p);
}

cudaError_t launch_rope_table(float* cs, int max_pos, int head_dim, double base, cudaStream_t s) {
  const int64_t n = static_cast<int64_t>(max_pos) * (head_dim / 2);
  const int threads = 256;
  dim3 grid(static_cast<unsigned>((n + threads - 1) / threads));
  return launch_pdl(rope_table_kernel, grid, dim3(threads), 0, s, reinterpret_cast<float2*>(cs),
                    max_pos, head_dim, base);
}

cudaError_t launch_qk_norm_rope(const NormRopeParams& p, cudaStream_t s) {
  const int rows = p.n_q_heads + p.n_kv_heads;
  const int rows_per_block = kNormWarps * (32 / (p.head_dim / 4));
  dim3 grid((rows + rows_per_block - 1) / rows_per_block, p.B);
  if (p.head_dim == 64) return launch_pdl(qk_norm_rope_kernel<64>, grid, dim3(kNormWarps * 32), 0, s, p);
  if (p.head_dim == 128) return launch_pdl(qk_norm_rope_kernel<128>, grid, dim3(kNormWarps * 32), 0, s, p);
  return cudaErrorInvalidValue;
}

cudaError_t launch_set_rows(const SetRowsParams& p, cudaStream_t s) {
  const int n4 = p.n_kv_heads * p.head_dim / 4;
  dim3 grid((n4 + kSetRowsThreads - 1) / kSetRowsThreads, p.B);
  if (p.kv_bf16) return launch_pdl(set_rows_kernel<__nv_bfloat16>, grid, dim3(kSetRowsThreads), 0, s, p);
  return launch_pdl(set_rows_kernel<float>, grid, dim3(kSetRowsThreads), 0, s, p);
}

cudaError_t launch_prefill_rows(const PrefillRowsParams& p, cudaStream_t s) {
  const int rows = p.n_q_heads + 2 * p.n_kv_heads;
  const int rows_per_block = kNormWarps * (32 / (p.head_dim / 4));
  dim3 grid((rows + rows_per_block - 1) / rows_per_block, p.B * p.T);
  if (p.head_dim == 64)
    return p.kv_bf16 ? launch_pdl(prefill_rows_kernel<64, __nv_bfloat16>, grid, dim3(kNormWarps * 32), 0, s, p)
                     : launch_pdl(prefill_rows_kernel<64, float>, grid, dim3(kNormWarps * 32), 0, s, p);
  if (p.head_dim == 128)
    return p.kv_bf16 ? launch_pdl(prefill_rows_kernel<128, __nv_bfloat16>, grid, dim3(kNormWarps * 32), 0, s, p)
                     : launch_pdl(prefill_rows_kernel<128, float>, grid, dim3(kNormWarps * 32), 0, s, p);
  return cudaErrorInvalidValue;
}

// Self-test of the bounded wait: one thread waits for phase 0 of an mbarrier that nothing
// arrives on, through the same mbar_wait every kernel uses; when the wait limit runs out it
// sets TTS_EFLAG_TIMEOUT and returns.
__global__ void wait_timeout_probe_kernel(int32_t* err) {
  __shared__ uint64_t bar;
  mbar_init(&bar, 1);
  mbar_init_fence();
  if (!mbar_wait(&bar, 0u)) set_err(err, TTS_EFLAG_TIMEOUT);
}

cudaError_t launch_wait_timeout_probe(int32_t* err, cudaStream_t s) {
  wait_timeout_probe_kernel<<<1, 1, 0, s>>>(err);
  return cudaGetLastError();
}

cudaError_t launch_zero(void* ptr, size_t bytes, cudaStream_t s) {
  const size_t n16 = bytes / 16;
  if (n16 == 0) return cudaSuccess;
  const int threads = 256;
  const size_t blocks = (n16 + threads - 1) / threads;
  dim3 grid(static_cast<unsigned>(blocks < 1024 ? blocks : 1024));
  return launch_pdl(zero_kernel, grid, dim3(threads), 0, s, static_cast<uint4*>(ptr), n16);
}

}  // namespace tts
