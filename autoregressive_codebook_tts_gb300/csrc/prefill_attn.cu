// Multi-query prefill attention: the T new positions of a stream attend to the cache
// causally ("qwentts.cpp -- src/pipeline-tts.h" commit page, KV-cache section: the
// prefill writes the prompt's rows from the reset position; query t of stream b sees
// positions [0, start[b] + t + 1)).  The decode-step kernel would stream each query's
// whole window once per query; here a block of query rows shares every K/V tile:
//
//   * work item = (stream b, kv head g, block of QB = 64 / G queries), i.e. 64 query
//     rows (query t_local, q head h of the group, row t_local * G + h); its window
//     [0, start + t_last + 1) is cut on the device into n_ch chunks of whole tiles
//     (prefill_chunk_len), one CTA per (chunk, item);
//   * warp 8 (one lane) streams the chunk's 64-row K and V tiles into a 2-stage ring
//     with 3-D tensor-map loads in the 128-byte swizzled layout (f32: boxes of 32
//     floats x rows x D/32; bf16: 64 x rows x D/64), one load per tile and operand
//     (paged: one per page of the tile);
//   * warps 0..7 own 8 query rows each.  Scores S = Q K^T (f32, q rows broadcast from
//     shared memory, lane l takes key rows l and l + 32); an online softmax per row in
//     base 2 (scale folded into log2 e) with the causal mask as each row's window end;
//     the probabilities go to a warp-private patch of shared memory and O += P V with
//     lane l owning D/32 consecutive columns of its 8 rows;
//   * a chunk's result is written unnormalised with its row max and sum, and a second
//     kernel merges the chunks of every row in chunk order (max, rescale, sum, divide);
//     with one chunk per item the first kernel writes the normalised rows itself.
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

constexpr int kRows = 64;          // query rows of an item
constexpr int kTile = 64;          // cache rows of a tile
constexpr int kWarps = 8;          // compute warps, 8 query rows each
constexpr int kThreads = (kWarps + 1) * 32;
constexpr int kStages = 2;

template <typename KvT> struct KvTraits;
template <> struct KvTraits<float> {
  static constexpr int kPerUnit = 4;       // elements of a 16-byte unit
  static constexpr int kPerChunk = 32;     // elements of a 128-byte swizzle row
};
template <> struct KvTraits<__nv_bfloat16> {
  static constexpr int kPerUnit = 8;
  static constexpr int kPerChunk = 64;
};

// Default L2 policy: the items of the other query blocks of a (stream, kv head) read the
// same tiles soon after.
__device__ __forceinline__ void tma_load_3d_pf(void* dst, const CUtensorMap* map, int c0, int c1, int c2,
                                               uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(smem_u32(dst)), "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(c2), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ float4 lds_f4(uint32_t addr) {
  float4 v;
  asm volatile("ld.shared.v4.f32 {%0, %1, %2, %3}, [%4];" : "=f"(v.x), "=f"(v.y), "=f"(v.z), "=f"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint2 lds_u2(uint32_t addr) {
  uint2 v;
  asm volatile("ld.shared.v2.u32 {%0, %1}, [%2];" : "=r"(v.x), "=r"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ float2 lds_f2(uint32_t addr) {
  float2 v;
  asm volatile("ld.shared.v2.f32 {%0, %1}, [%2];" : "=f"(v.x), "=f"(v.y) : "r"(addr));
  return v;
}
__device__ __forceinline__ uint4 lds128_addr(uint32_t addr) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];" : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(addr));
  return v;
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }


// Placement of a tile in shared memory: boxes of br = 2^br_shift rows, each box
// [128-byte chunk c][row][128 bytes], so row j's chunk c starts at
//   row_base(j) + c * br * 128,  row_base(j) = ((j >> br_shift) * chunks * br + (j & (br - 1))) * 128,
// and its 16-byte unit uc sits at ((uc ^ (j & 7)) << 4) within the chunk.
template <typename KvT, int D>
__device__ __forceinline__ uint32_t row_base(int j, int br_shift) {
  constexpr int kChunks = D / KvTraits<KvT>::kPerChunk;
  return static_cast<uint32_t>((((j >> br_shift) * kChunks << br_shift) + (j & ((1 << br_shift) - 1))) * 128);
}

// Scores of the warp's 8 query rows against tile rows `lane` and `lane + 32` (the same
// row % 8, so one swizzle serves both), as pairs of partial sums over the even and odd
// columns of D (packed f32 multiply-adds on adjacent elements); the caller adds the
// halves.
template <typename KvT, int D>
__device__ __forceinline__ void tile_scores(uint32_t kb, uint32_t qw, int lane, int br_shift, float2 (&sc)[8][2]) {
  using Tr = KvTraits<KvT>;
  constexpr int kChunks = D / Tr::kPerChunk;
  const uint32_t b0 = kb + row_base<KvT, D>(lane, br_shift);
  const uint32_t b1 = kb + row_base<KvT, D>(lane + 32, br_shift);
  const uint32_t cstride = 128u << br_shift;
  const int j7 = lane & 7;
#pragma unroll
  for (int i = 0; i < 8; ++i) sc[i][0] = sc[i][1] = make_float2(0.f, 0.f);
#pragma unroll
  for (int c = 0; c < kChunks; ++c) {
#pragma unroll 4
    for (int uc = 0; uc < 8; ++uc) {
      const uint32_t off = c * cstride + ((uc ^ j7) << 4);
      const int u = c * 8 + uc;
      if constexpr (Tr::kPerUnit == 4) {
        const float4 k0 = lds_f4(b0 + off), k1 = lds_f4(b1 + off);
        const float2 k0a = make_float2(k0.x, k0.y), k0b = make_float2(k0.z, k0.w);
        const float2 k1a = make_float2(k1.x, k1.y), k1b = make_float2(k1.z, k1.w);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 q = lds_f4(qw + (i * D + u * 4) * 4);
          const float2 qa = make_float2(q.x, q.y), qb = make_float2(q.z, q.w);
          sc[i][0] = __ffma2_rn(qa, k0a, sc[i][0]);
          sc[i][1] = __ffma2_rn(qa, k1a, sc[i][1]);
          sc[i][0] = __ffma2_rn(qb, k0b, sc[i][0]);
          sc[i][1] = __ffma2_rn(qb, k1b, sc[i][1]);
        }
      } else {
        const uint4 w0 = lds128_addr(b0 + off), w1 = lds128_addr(b1 + off);
        const float2 k0[4] = {make_float2(bf16_lo(w0.x), bf16_hi(w0.x)), make_float2(bf16_lo(w0.y), bf16_hi(w0.y)),
                              make_float2(bf16_lo(w0.z), bf16_hi(w0.z)), make_float2(bf16_lo(w0.w), bf16_hi(w0.w))};
        const float2 k1[4] = {make_float2(bf16_lo(w1.x), bf16_hi(w1.x)), make_float2(bf16_lo(w1.y), bf16_hi(w1.y)),
                              make_float2(bf16_lo(w1.z), bf16_hi(w1.z)), make_float2(bf16_lo(w1.w), bf16_hi(w1.w))};
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float4 qa = lds_f4(qw + (i * D + u * 8) * 4);
          const float4 qc = lds_f4(qw + (i * D + u * 8 + 4) * 4);
          const float2 q[4] = {make_float2(qa.x, qa.y), make_float2(qa.z, qa.w), make_float2(qc.x, qc.y),
                               make_float2(qc.z, qc.w)};
#pragma unroll
          for (int e = 0; e < 4; ++e) {
            sc[i][0] = __ffma2_rn(q[e], k0[e], sc[i][0]);
            sc[i][1] = __ffma2_rn(q[e], k1[e], sc[i][1]);
          }
        }
      }
    }
  }
}

// Columns [lane * DPL, lane * DPL + DPL) of V tile row j, widened to f32.
template <typename KvT, int D>
__device__ __forceinline__ void v_cols(uint32_t vb, int j, int lane, int br_shift, float (&v)[D / 32]) {
  using Tr = KvTraits<KvT>;
  constexpr int DPL = D / 32;
  constexpr int kLanesPerUnit = Tr::kPerUnit / DPL;
  const int u = lane / kLanesPerUnit, part = lane % kLanesPerUnit;
  const uint32_t a = vb + row_base<KvT, D>(j, br_shift) + (u >> 3) * (128u << br_shift) + (((u & 7) ^ (j & 7)) << 4) +
                     part * DPL * static_cast<int>(sizeof(KvT));
  if constexpr (sizeof(KvT) == 4 && DPL == 4) {
    const float4 x = lds_f4(a);
    v[0] = x.x; v[1] = x.y; v[2] = x.z; v[3] = x.w;
  } else if constexpr (sizeof(KvT) == 4 && DPL == 2) {
    const float2 x = lds_f2(a);
    v[0] = x.x; v[1] = x.y;
  } else if constexpr (DPL == 4) {
    const uint2 w = lds_u2(a);
    v[0] = bf16_lo(w.x); v[1] = bf16_hi(w.x); v[2] = bf16_lo(w.y); v[3] = bf16_hi(w.y);
  } else {
    uint32_t w;
    asm volatile("ld.shared.u32 %0, [%1];" : "=r"(w) : "r"(a));
    v[0] = bf16_lo(w); v[1] = bf16_hi(w);
  }
}

__device__ __forceinline__ float warp_max(float x) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) x = fmaxf(x, __shfl_xor_sync(kFull, x, o));
  return x;
}
__device__ __forceinline__ float warp_sum(float x) {
#pragma unroll
  for (int o = 16; o >= 1; o >>= 1) x += __shfl_xor_sync(kFull, x, o);
  return x;
}

template <typename KvT, int D, int G>
__global__ void __launch_bounds__(kThreads, 1) prefill_attn_kernel(const __grid_constant__ CUtensorMap kmap,
                                                                    const __grid_constant__ CUtensorMap vmap,
                                                                    const PrefillAttnParams p) {
  constexpr int kTileBytes = kTile * D * static_cast<int>(sizeof(KvT));
  constexpr int QB = kRows / G;   // queries of an item
  constexpr int DPL = D / 32;     // output columns of a lane
  extern __shared__ __align__(1024) unsigned char smem_raw[];
  unsigned char* smem = smem_raw + ((1024u - (smem_u32(smem_raw) & 1023u)) & 1023u);
  unsigned char* ring = smem;                                                     // kStages x (K | V)
  float* sq = reinterpret_cast<float*>(ring + kStages * 2 * kTileBytes);          // [64][D]
  float* sp = sq + kRows * D;                                                     // [8][64][8]
  uint64_t* full = reinterpret_cast<uint64_t*>(sp + kWarps * kTile * 8);
  uint64_t* empty = full + kStages;

  const int item = blockIdx.x, ch = blockIdx.y;
  const int qb = item % p.n_qb, bg = item / p.n_qb;
  const int g = bg % p.n_kv_heads, b = bg / p.n_kv_heads;
  const int tid = threadIdx.x, warp = tid >> 5, lane = tid & 31;
  const int t0 = qb * QB;
  const int nq = min(QB, p.T - t0);

  if (tid == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], kWarps);
    }
    mbar_init_fence();
  }
  __syncthreads();
  grid_launch_dependents();
  // start[] and the cache rows below the prompt were final before the rows launch began
  // (it waits for its own predecessor before it lets this launch start), so they are
  // read before the dependency wait; the prompt's cache rows and the rotated q rows are
  // the rows launch's, read after it (the producer waits before the first tile that
  // holds a prompt row, the consumers before the query rows)
  const int st = __ldcg(p.start + b);
  // the item's window ends with its last query's: [0, start + t0 + nq)
  const int nv_max = min(max(st + t0 + nq, 1), p.capacity);
  const int ch_len = prefill_chunk_len(nv_max, p.n_ch);
  const int c0 = ch * ch_len;
  if (c0 >= nv_max) return;   // the chunk holds no row of any window of the item
  const int c1 = min(c0 + ch_len, nv_max);
  const int ntiles = (c1 - c0 + kTile - 1) / kTile;
  const int br = p.paged ? min(kTile, p.page_size) : kTile;
  const int br_shift = 31 - __clz(br);

  if (warp == kWarps) {
    // ---------------------------------------------------------------- producer
    if (lane == 0) {
      int issued = 0;
      bool ok = true, waited = false;
      const int box_bytes = br * D * static_cast<int>(sizeof(KvT));
      for (; issued < ntiles; ++issued) {
        if (!waited && c0 + (issued + 1) * kTile > st) {
          grid_wait();
          waited = true;
        }
        const int s = issued % kStages;
        if (issued >= kStages && !mbar_wait(&empty[s], static_cast<uint32_t>((issued / kStages) - 1) & 1u)) {
          ok = false;
          break;
        }
        unsigned char* kd = ring + s * 2 * kTileBytes;
        unsigned char* vd = kd + kTileBytes;
        const int r0 = c0 + issued * kTile;
        if (!p.paged) {
          mbar_arrive_expect_tx(&full[s], 2 * kTileBytes);
          const int row = (b * p.n_kv_heads + g) * p.capacity + r0;
          tma_load_3d_pf(kd, &kmap, 0, row, 0, &full[s]);
          tma_load_3d_pf(vd, &vmap, 0, row, 0, &full[s]);
        } else {
          // the boxes (pages, or 64-row parts of a page) that hold rows of the chunk
          const int rend = min(r0 + kTile, c1);
          const int nbox = (rend - r0 + br - 1) / br;
          mbar_arrive_expect_tx(&full[s], 2 * nbox * box_bytes);
          for (int k = 0; k < nbox; ++k) {
            const int pos = r0 + k * br;
            int page = __ldcg(p.block_table + static_cast<int64_t>(b) * p.bt_stride + pos / p.page_size);
            if (page < 0 || page >= p.n_pages) {
              set_err(p.err, TTS_EFLAG_PAGE);
              page = 0;
            }
            const int row = (page * p.n_kv_heads + g) * p.page_size + (pos & (p.page_size - 1));
            tma_load_3d_pf(kd + k * box_bytes, &kmap, 0, row, 0, &full[s]);
            tma_load_3d_pf(vd + k * box_bytes, &vmap, 0, row, 0, &full[s]);
          }
        }
      }
      if (!ok) set_err(p.err, TTS_EFLAG_TIMEOUT);
      // no copy may still be landing when the CTA leaves
      for (int t = max(0, issued - kStages); t < issued; ++t)
        mbar_wait(&full[t % kStages], static_cast<uint32_t>(t / kStages) & 1u);
    }
    return;
  }

  // ------------------------------------------------------------------ consumers
  grid_wait();   // the rows launch normed and rotated the query rows
  // the warp's 8 query rows (row r = t_local * G + h), zero past the prompt
  float* sqw = sq + warp * 8 * D;
  for (int e = lane; e < 8 * D / 4; e += 32) {
    const int i = e / (D / 4), d4 = e - i * (D / 4);
    const int r = warp * 8 + i, tl = r / G, h = r - tl * G;
    float4 v = make_float4(0.f, 0.f, 0.f, 0.f);
    if (tl < nq)
      v = __ldcg(reinterpret_cast<const float4*>(p.q + static_cast<int64_t>(b * p.T + t0 + tl) * p.q_stride +
                                                 (g * G + h) * D) + d4);
    reinterpret_cast<float4*>(sqw)[e] = v;
  }
  __syncwarp();
  int nv[8];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = warp * 8 + i, tl = r / G;
    const int raw = st + t0 + tl + 1;
    nv[i] = tl < nq ? min(max(raw, 1), p.capacity) : 0;
    if (ch == 0 && lane == 0 && tl < nq && (r - tl * G) == 0 && g == 0 && (raw < 1 || raw > p.capacity))
      set_err(p.err, TTS_EFLAG_NVALID);
  }
  // o2[ip][c]: columns lane * DPL + c of rows 2 ip and 2 ip + 1 (packed multiply-adds)
  float m[8], l[8];
  float2 o2[4][DPL];
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    m[i] = -INFINITY;
    l[i] = 0.f;
  }
#pragma unroll
  for (int ip = 0; ip < 4; ++ip)
#pragma unroll
    for (int c = 0; c < DPL; ++c) o2[ip][c] = make_float2(0.f, 0.f);
  const uint32_t qw = smem_u32(sqw);
  float* spw = sp + warp * kTile * 8;
  const uint32_t pw = smem_u32(spw);
  bool ok = true;
  for (int it = 0; it < ntiles; ++it) {
    const int s = it % kStages;
    if (!mbar_wait(&full[s], static_cast<uint32_t>(it / kStages) & 1u)) {
      ok = false;
      break;
    }
    const uint32_t kb = smem_u32(ring + s * 2 * kTileBytes), vb = kb + kTileBytes;
    const int r0 = c0 + it * kTile, nrow = min(kTile, c1 - r0);
    float2 sc2[8][2];
    tile_scores<KvT, D>(kb, qw, lane, br_shift, sc2);
    // online softmax in base 2; a row past a query's window (or past the chunk) gets -inf
    float p0[8], p1[8], al[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const float s0 = sc2[i][0].x + sc2[i][0].y, s1 = sc2[i][1].x + sc2[i][1].y;
      const float a0 = (lane < nrow && r0 + lane < nv[i]) ? s0 * p.scale_log2 : -INFINITY;
      const float a1 = (lane + 32 < nrow && r0 + lane + 32 < nv[i]) ? s1 * p.scale_log2 : -INFINITY;
      const float mn = fmaxf(m[i], warp_max(fmaxf(a0, a1)));
      float alpha = 1.f;
      if (mn == -INFINITY) {
        p0[i] = p1[i] = 0.f;
      } else {
        alpha = exp2f(m[i] - mn);
        p0[i] = exp2f(a0 - mn);
        p1[i] = exp2f(a1 - mn);
      }
      l[i] = fmaf(l[i], alpha, warp_sum(p0[i] + p1[i]));
      m[i] = mn;
      al[i] = alpha;
    }
#pragma unroll
    for (int ip = 0; ip < 4; ++ip) {
      const float2 a2 = make_float2(al[2 * ip], al[2 * ip + 1]);
#pragma unroll
      for (int c = 0; c < DPL; ++c) o2[ip][c] = __fmul2_rn(o2[ip][c], a2);
    }
    // the warp's probabilities: [tile row][8 query rows]
    reinterpret_cast<float4*>(spw + lane * 8)[0] = make_float4(p0[0], p0[1], p0[2], p0[3]);
    reinterpret_cast<float4*>(spw + lane * 8)[1] = make_float4(p0[4], p0[5], p0[6], p0[7]);
    reinterpret_cast<float4*>(spw + (lane + 32) * 8)[0] = make_float4(p1[0], p1[1], p1[2], p1[3]);
    reinterpret_cast<float4*>(spw + (lane + 32) * 8)[1] = make_float4(p1[4], p1[5], p1[6], p1[7]);
    __syncwarp();
#pragma unroll 4
    for (int j = 0; j < nrow; ++j) {
      const float4 pa = lds_f4(pw + j * 32), pb = lds_f4(pw + j * 32 + 16);
      const float2 pr[4] = {make_float2(pa.x, pa.y), make_float2(pa.z, pa.w), make_float2(pb.x, pb.y),
                            make_float2(pb.z, pb.w)};
      float v[DPL];
      v_cols<KvT, D>(vb, j, lane, br_shift, v);
#pragma unroll
      for (int c = 0; c < DPL; ++c) {
        const float2 v2 = make_float2(v[c], v[c]);
#pragma unroll
        for (int ip = 0; ip < 4; ++ip) o2[ip][c] = __ffma2_rn(pr[ip], v2, o2[ip][c]);
      }
    }
    __syncwarp();
    if (lane == 0) mbar_arrive(&empty[s]);
  }
  if (!ok && lane == 0) set_err(p.err, TTS_EFLAG_TIMEOUT);

  // the chunk's rows: normalised when it is the only chunk, else with their max and sum
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const int r = warp * 8 + i, tl = r / G, h = r - tl * G;
    if (tl >= nq) continue;
    float o[DPL];
#pragma unroll
    for (int c = 0; c < DPL; ++c) o[c] = (i & 1) ? o2[i >> 1][c].y : o2[i >> 1][c].x;
    if (p.n_ch == 1) {
      const float inv = l[i] > 0.f ? 1.f / l[i] : 0.f;
      float* dst = p.out + (static_cast<int64_t>(b * p.T + t0 + tl) * p.n_q_heads + g * G + h) * D + lane * DPL;
#pragma unroll
      for (int c = 0; c < DPL; ++c) dst[c] = o[c] * inv;
    } else {
      const int64_t row = (static_cast<int64_t>(item) * p.n_ch + ch) * kRows + r;
      float* dst = p.part + row * D + lane * DPL;
#pragma unroll
      for (int c = 0; c < DPL; ++c) dst[c] = o[c];
      if (lane == 0) reinterpret_cast<float2*>(p.ml)[row] = make_float2(m[i], l[i]);
    }
  }
}


// The chunks of every query row merged in chunk order: M = max m_c, L = sum l_c 2^(m_c - M),
// out = sum O_c 2^(m_c - M) / L.  One CTA per (item, 8 query rows), a thread per (row,
// 4 columns).  The chunks are taken 8 at a time, all 16 loads of a batch issued before
// any is used, with the running sums moved to each batch's maximum (the same merge as
// one pass over all chunks, up to rounding); chunk 0 holds a row of every window, so M
// is finite from the first batch on.
constexpr int kCombineRows = 8;
constexpr int kMaxCombineChunks = 64;
constexpr int kCombineBatch = 8;
__global__ void __launch_bounds__(256) prefill_combine_kernel(const PrefillAttnParams p, int G, int D) {
  grid_wait();
  grid_launch_dependents();
  const int item = blockIdx.x;
  const int QB = p.rows / G;
  const int qb = item % p.n_qb, bg = item / p.n_qb;
  const int g = bg % p.n_kv_heads, b = bg / p.n_kv_heads;
  const int t0 = qb * QB, nq = min(QB, p.T - t0);
  const int st = __ldcg(p.start + b);
  const int nv_max = min(max(st + t0 + nq, 1), p.capacity);
  const int ch_len = prefill_chunk_len(nv_max, p.n_ch);
  const int n_act = min(min(p.n_ch, kMaxCombineChunks), (nv_max + ch_len - 1) / ch_len);
  const int D4 = D / 4;
  const int e = threadIdx.x;
  if (e >= kCombineRows * D4) return;
  const int r = blockIdx.y * kCombineRows + e / D4, d4 = e % D4, tl = r / G, h = r - tl * G;
  if (tl >= nq) return;
  const int64_t row0 = static_cast<int64_t>(item) * p.n_ch * p.rows + r;
  const float2* ml = reinterpret_cast<const float2*>(p.ml) + row0;
  const float4* part = reinterpret_cast<const float4*>(p.part + row0 * D) + d4;
  const int64_t cstride4 = static_cast<int64_t>(p.rows) * D4;   // float4s between chunks of a row
  float M = -INFINITY, L = 0.f;
  float4 acc = make_float4(0.f, 0.f, 0.f, 0.f);
  for (int c0 = 0; c0 < n_act; c0 += kCombineBatch) {
    float2 mlc[kCombineBatch];
    float4 x[kCombineBatch];
#pragma unroll
    for (int i = 0; i < kCombineBatch; ++i) {
      if (c0 + i < n_act) {
        mlc[i] = __ldcg(ml + static_cast<int64_t>(c0 + i) * p.rows);
        x[i] = __ldcg(part + (c0 + i) * cstride4);
      } else {
        mlc[i] = make_float2(-INFINITY, 0.f);
        x[i] = make_float4(0.f, 0.f, 0.f, 0.f);
      }
    }
    float Mb = M;
#pragma unroll
    for (int i = 0; i < kCombineBatch; ++i) Mb = fmaxf(Mb, mlc[i].x);
    const float s = M == -INFINITY ? 0.f : exp2f(M - Mb);
    L *= s;
    acc = make_float4(acc.x * s, acc.y * s, acc.z * s, acc.w * s);
    M = Mb;
#pragma unroll
    for (int i = 0; i < kCombineBatch; ++i) {
      const float w = mlc[i].x == -INFINITY ? 0.f : exp2f(mlc[i].x - M);
      L = fmaf(mlc[i].y, w, L);
      acc.x = fmaf(x[i].x, w, acc.x);
      acc.y = fmaf(x[i].y, w, acc.y);
      acc.z = fmaf(x[i].z, w, acc.z);
      acc.w = fmaf(x[i].w, w, acc.w);
    }
  }
  const float inv = L > 0.f ? 1.f / L : 0.f;
  reinterpret_cast<float4*>(p.out + (static_cast<int64_t>(b * p.T + t0 + tl) * p.n_q_heads + g * G + h) * D)[d4] =
      make_float4(acc.x * inv, acc.y * inv, acc.z * inv, acc.w * inv);
}

PFN_cuTensorMapEncodeTiled_v12000 encoder() {
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

template <typename KvT, int D>
size_t prefill_smem() {
  return 1024 + static_cast<size_t>(kStages) * 2 * kTile * D * sizeof(KvT) + static_cast<size_t>(kRows) * D * 4 +
         static_cast<size_t>(kWarps) * kTile * 8 * 4 + 2 * kStages * sizeof(uint64_t);
}

template <typename KvT, int D, int G>
cudaError_t launch_t(const PrefillAttnParams& p, const void* kc, const void* vc, cudaStream_t s) {
  using Tr = KvTraits<KvT>;
  auto kern = prefill_attn_kernel<KvT, D, G>;
  PFN_cuTensorMapEncodeTiled_v12000 enc = encoder();
  if (enc == nullptr) return cudaErrorNotSupported;
  // the cache as [D / chunk][rows][chunk elements]: rows of D elements (stride D x size),
  // 128-byte chunks of a row 128 bytes apart; boxes of br rows
  const uint64_t rows = p.paged ? static_cast<uint64_t>(p.n_pages) * p.n_kv_heads * p.page_size
                                : static_cast<uint64_t>(p.B) * p.n_kv_heads * p.capacity;
  const int br = p.paged ? (p.page_size < kTile ? p.page_size : kTile) : kTile;
  cuuint64_t dims[3] = {static_cast<cuuint64_t>(Tr::kPerChunk), rows, static_cast<cuuint64_t>(D / Tr::kPerChunk)};
  cuuint64_t strides[2] = {static_cast<cuuint64_t>(D) * sizeof(KvT), 128};
  cuuint32_t box[3] = {static_cast<cuuint32_t>(Tr::kPerChunk), static_cast<cuuint32_t>(br),
                       static_cast<cuuint32_t>(D / Tr::kPerChunk)};
  cuuint32_t estr[3] = {1, 1, 1};
  const CUtensorMapDataType dt = sizeof(KvT) == 4 ? CU_TENSOR_MAP_DATA_TYPE_FLOAT32 : CU_TENSOR_MAP_DATA_TYPE_BFLOAT16;
  CUtensorMap kmap, vmap;
  if (enc(&kmap, dt, 3, const_cast<void*>(kc), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
          CUDA_SUCCESS ||
      enc(&vmap, dt, 3, const_cast<void*>(vc), dims, strides, box, estr, CU_TENSOR_MAP_INTERLEAVE_NONE,
          CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B, CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) !=
          CUDA_SUCCESS)
    return cudaErrorInvalidValue;
  const size_t smem = prefill_smem<KvT, D>();
  static std::mutex mtx;
  static bool configured[64] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mtx);
    if (!configured[dev]) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(smem));
      if (e != cudaSuccess) return e;
      configured[dev] = true;
    }
  }
  const int items = p.B * p.n_kv_heads * p.n_qb;
  e = launch_pdl(kern, dim3(items, p.n_ch), dim3(kThreads), smem, s, kmap, vmap, p);
  if (e != cudaSuccess || p.n_ch == 1) return e;
  return launch_pdl(prefill_combine_kernel, dim3(items, kRows / kCombineRows), dim3(256), 0, s, p, G, D);
}

cudaError_t launch_combine(const PrefillAttnParams& p, int G, int D, cudaStream_t s) {
  const int items = p.B * p.n_kv_heads * p.n_qb;
  return launch_pdl(prefill_combine_kernel, dim3(items, p.rows / kCombineRows), dim3(256), 0, s, p, G, D);
}

}  // namespace

bool prefill_attn_supported(int head_dim, int group, int paged, int page_size, int T) {
  return (head_dim == 64 || head_dim == 128) && (group == 1 || group == 2 || group == 4) &&
         (!paged || page_size >= 8) && T >= kPrefillMinT;
}

int prefill_rows_per_item(int kv_bf16, int head_dim, int paged, int page_size) {
  return prefill_attn_tc_supported(kv_bf16, head_dim, paged, page_size) ? 2 * kRows : kRows;
}

void prefill_attn_plan(int B, int T, int n_kv_heads, int group, int capacity, int n_splits, int n_sm, int rows,
                       int& n_qb, int& n_ch) {
  const int QB = rows / group;
  n_qb = (T + QB - 1) / QB;
  const int items = B * n_kv_heads * n_qb;
  // Both kernels hold one CTA per SM.  Each item's window is cut into n_ch parts on the
  // device (prefill_chunk_len).
  //   Tensor cores (a CTA's fixed costs are a third of it): as many chunks as fill one
  //   wave.  An item's 2..8 chunks can form a cluster and merge there, saving the combine
  //   launch and the partial rows' round trip (worth about two tiles of the loop): the
  //   largest cluster size whose clusters are all resident at once is taken when it
  //   keeps at least 0.4 of the chunks of the one-wave cut (measured: 8 items of the
  //   talker shapes run 8 clusters of 8 in 9.2 / 16.0 us a layer against 19 chunks and
  //   the combine in 11.1 / 16.9 us, windows of 132 / 3032 rows).
  //   CUDA cores: about four CTAs per SM over the items, chunks of at least 256 rows, so
  //   that SMs that finish short windows early take more (measured against one wave:
  //   122.5 -> 115.9 us a layer for 128 rows after 3000, 80.2 -> 65-68 us for 512 from 0).
  int c = n_splits;
  if (n_splits <= 0 && rows == 2 * kRows) {
    c = n_sm / items;
    int sc = 0;
    for (int s = 8; s >= 2 && sc == 0; --s)
      if (items <= prefill_tc_active_clusters(group, s)) sc = s;
    if (sc >= 2 && 5 * sc >= 2 * c) c = sc;
  } else if (n_splits <= 0) {
    c = (4 * n_sm + items - 1) / items;
    const int max_c = (capacity + 4 * kTile - 1) / (4 * kTile);
    if (c > max_c) c = max_c;
  }
  const int max_ch = (capacity + kTile - 1) / kTile;
  if (c > max_ch) c = max_ch;
  if (c > kMaxCombineChunks) c = kMaxCombineChunks;
  if (c < 1) c = 1;
  n_ch = c;
}

size_t prefill_attn_workspace(int B, int T, int n_kv_heads, int group, int head_dim, int capacity, int n_splits,
                              int n_sm, int rows_per_item) {
  int n_qb, n_ch;
  prefill_attn_plan(B, T, n_kv_heads, group, capacity, n_splits, n_sm, rows_per_item, n_qb, n_ch);
  if (n_ch == 1) return 0;
  const size_t rows = static_cast<size_t>(B) * n_kv_heads * n_qb * n_ch * rows_per_item;
  return rows * (static_cast<size_t>(head_dim) + 2) * sizeof(float);
}

cudaError_t launch_prefill_attn(const PrefillAttnParams& p, const void* k_cache, const void* v_cache, bool kv_bf16,
                                int head_dim, int group, cudaStream_t s) {
  if (p.rows == 2 * kRows) {
    bool merged = false;
    const cudaError_t e = launch_prefill_attn_tc(p, k_cache, v_cache, group, s, &merged);
    if (e != cudaSuccess || p.n_ch == 1 || merged) return e;
    return launch_combine(p, group, head_dim, s);
  }
  if (p.rows != kRows) return cudaErrorInvalidValue;
#define TTS_PF_CASE(KT, DD, GG) \
  if (head_dim == DD && group == GG) return launch_t<KT, DD, GG>(p, k_cache, v_cache, s);
  if (kv_bf16) {
    TTS_PF_CASE(__nv_bfloat16, 128, 1) TTS_PF_CASE(__nv_bfloat16, 128, 2) TTS_PF_CASE(__nv_bfloat16, 128, 4)
    TTS_PF_CASE(__nv_bfloat16, 64, 1) TTS_PF_CASE(__nv_bfloat16, 64, 2) TTS_PF_CASE(__nv_bfloat16, 64, 4)
  } else {
    TTS_PF_CASE(float, 128, 1) TTS_PF_CASE(float, 128, 2) TTS_PF_CASE(float, 128, 4)
    TTS_PF_CASE(float, 64, 1) TTS_PF_CASE(float, 64, 2) TTS_PF_CASE(float, 64, 4)
  }
#undef TTS_PF_CASE
  return cudaErrorInvalidValue;
}

}  // namespace tts
