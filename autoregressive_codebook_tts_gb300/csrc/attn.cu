// Single-query GQA decode attention for sm_103a, standalone and fused with the q/k
// norm + RoPE and the new-row KV write.
//
// Defines the operation of the "qwentts.cpp ... src/pipeline-tts.h" commit page
// (persistent-arenas section: window padded to a multiple of 256 with -inf over the
// padded tail; KV-cache section: decode appends one position and reads the
// [0, cur_len+1) window), batched over streams.
//
// Design (a bandwidth-bound GEMV, on CUDA cores with f32 accumulation):
//   * grid = (split, kv head, stream).  One CTA streams a contiguous range of one kv
//     head's positions and serves all Hq/Hkv q heads of the group from the same bytes,
//     so each K/V element is read from HBM once.
//   * One producer warp feeds a ring of shared-memory stages with 1-D bulk copies
//     (the TMA engine) of whole K and V tiles; the cache is head-major, so a tile of a
//     contiguous cache is one copy (a paged cache: one copy per page piece).  Copies
//     complete on per-stage mbarriers; consumer warps release stages on a second set.
//   * Four consumer warps split each tile's rows.  A row is covered by LPR lanes with
//     16 bytes each (4 f32 or 8 bf16 elements); q.k is reduced across those lanes with
//     xor shuffles; each warp keeps its own online-softmax state (running max in
//     log2 units, running sum, unnormalised output), merged at the end through
//     shared memory.
//   * Rows at or past n_valid are never copied or read: the -inf of the padded tail
//     is realised as "not there", so poison in the tail cannot leak.
//   * Split-KV: every split writes (o, m, l) to the workspace and takes a ticket; the
//     last split of a (stream, kv head) merges all partials with a log-sum-exp combine
//     and resets the ticket.  No CTA ever waits for another.
//   * Launch configuration depends only on capacity; splits past the window exit early.
//   * Every mbarrier wait is bounded (kWaitLimitCycles); on expiry TTS_EFLAG_TIMEOUT is
//     set, the copies already issued are waited for (bounded), and the CTA finishes.
#include "common.cuh"
#include "kernels.h"

namespace tts {
namespace {

template <typename KvT, int D_, int G_>
struct Cfg {
  static constexpr int D = D_;
  static constexpr int G = G_;
  static constexpr int kElem = sizeof(KvT);
  static constexpr int EPL = 16 / kElem;      // elements per lane per 16-byte vector
  static constexpr int LPR = D / EPL;         // lanes per row
  static constexpr int RPI = 32 / LPR;        // rows per warp step
  static constexpr int ROW_BYTES = D * kElem;
  static constexpr int NC = 4;                // consumer warps
  static constexpr int T = (ROW_BYTES >= 512) ? 32 : 64;  // rows per stage
  static constexpr int NS = 3;                // maximum ring depth
  static constexpr int RPW = T / NC;          // rows per warp per tile
  static constexpr int STEPS = RPW / RPI;
  static constexpr int TILE_BYTES = T * ROW_BYTES;
  static constexpr int STAGE_BYTES = 2 * TILE_BYTES;
  static constexpr int THREADS = (NC + 1) * 32;
  static_assert(RPW % RPI == 0, "tile rows must split evenly over warp steps");
  static_assert(LPR >= 2 && LPR <= 32, "row must span 2..32 lanes");

  static constexpr size_t bar_off(int ns) { return static_cast<size_t>(ns) * STAGE_BYTES; }
  static constexpr size_t fresh_off(int ns) { return bar_off(ns) + 2 * NS * sizeof(uint64_t); }
  static constexpr size_t scratch_off(int ns) { return fresh_off(ns) + 2 * ROW_BYTES; }
  static constexpr size_t flag_off(int ns) {
    return scratch_off(ns) + static_cast<size_t>(NC) * G * (D + 2) * sizeof(float);
  }
  static constexpr size_t smem_bytes(int ns) { return flag_off(ns) + 16; }
};

// 16 bytes of f32 row data starting at element e0 of a global row.
template <int EPL>
__device__ __forceinline__ void load_row_f32(const float* row, int e0, float (&x)[EPL]) {
#pragma unroll
  for (int i = 0; i < EPL; i += 4) {
    const float4 v = __ldcg(reinterpret_cast<const float4*>(row + e0 + i));
    x[i] = v.x; x[i + 1] = v.y; x[i + 2] = v.z; x[i + 3] = v.w;
  }
}

__device__ __forceinline__ uint4 pack_row(const float (&x)[4], float*) {
  return make_uint4(__float_as_uint(x[0]), __float_as_uint(x[1]), __float_as_uint(x[2]),
                    __float_as_uint(x[3]));
}
__device__ __forceinline__ uint32_t pack2_bf16(float a, float b) {
  const __nv_bfloat162 h = __floats2bfloat162_rn(a, b);  // .x = a (low half), round-to-nearest-even
  return *reinterpret_cast<const uint32_t*>(&h);
}
__device__ __forceinline__ uint4 pack_row(const float (&x)[8], __nv_bfloat16*) {
  return make_uint4(pack2_bf16(x[0], x[1]), pack2_bf16(x[2], x[3]), pack2_bf16(x[4], x[5]),
                    pack2_bf16(x[6], x[7]));
}

// Consume one tile (nrows valid rows) for this warp: scores, online softmax, P.V.
template <class C, typename KvT, bool PARTIAL>
__device__ __forceinline__ void consume_tile(const unsigned char* __restrict__ kt,
                                             const unsigned char* __restrict__ vt, int nrows,
                                             int warp, int lane, const float (&q)[C::G][C::EPL],
                                             float (&m_run)[C::G], float (&l_run)[C::G],
                                             float (&o)[C::G][C::EPL]) {
  constexpr int G = C::G, EPL = C::EPL, LPR = C::LPR, STEPS = C::STEPS;
  const int lr = lane % LPR;
  const int rg = lane / LPR;
  const int row_base = warp * C::RPW + rg;
  float s[STEPS][G];
#pragma unroll
  for (int st = 0; st < STEPS; ++st) {
    const int row = row_base + st * C::RPI;
    float kf[EPL];
    if (!PARTIAL || row < nrows) {
      KvVec<KvT>::unpack(lds128(kt + row * C::ROW_BYTES + lr * 16), kf);
    } else {
#pragma unroll
      for (int i = 0; i < EPL; ++i) kf[i] = 0.f;
    }
#pragma unroll
    for (int h = 0; h < G; ++h) {
      float a = 0.f;
#pragma unroll
      for (int i = 0; i < EPL; ++i) a = fmaf(q[h][i], kf[i], a);
      s[st][h] = a;
    }
  }
#pragma unroll
  for (int st = 0; st < STEPS; ++st)
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int off = LPR / 2; off >= 1; off >>= 1) s[st][h] += __shfl_xor_sync(kFull, s[st][h], off);
  if (PARTIAL) {
#pragma unroll
    for (int st = 0; st < STEPS; ++st)
      if (row_base + st * C::RPI >= nrows)
#pragma unroll
        for (int h = 0; h < G; ++h) s[st][h] = -INFINITY;
  }
#pragma unroll
  for (int h = 0; h < G; ++h) {
    float mx = s[0][h];
#pragma unroll
    for (int st = 1; st < STEPS; ++st) mx = fmaxf(mx, s[st][h]);
#pragma unroll
    for (int off = LPR; off < 32; off <<= 1) mx = fmaxf(mx, __shfl_xor_sync(kFull, mx, off));
    const float m_new = fmaxf(m_run[h], mx);
    const float m_use = (m_new == -INFINITY) ? 0.f : m_new;
    const float alpha = exp2f(m_run[h] - m_use);
    m_run[h] = m_new;
    l_run[h] *= alpha;
#pragma unroll
    for (int i = 0; i < EPL; ++i) o[h][i] *= alpha;
#pragma unroll
    for (int st = 0; st < STEPS; ++st) {
      s[st][h] = exp2f(s[st][h] - m_use);
      l_run[h] += s[st][h];
    }
  }
#pragma unroll
  for (int st = 0; st < STEPS; ++st) {
    const int row = row_base + st * C::RPI;
    float vf[EPL];
    if (!PARTIAL || row < nrows) {
      KvVec<KvT>::unpack(lds128(vt + row * C::ROW_BYTES + lr * 16), vf);
    } else {
#pragma unroll
      for (int i = 0; i < EPL; ++i) vf[i] = 0.f;
    }
#pragma unroll
    for (int h = 0; h < G; ++h)
#pragma unroll
      for (int i = 0; i < EPL; ++i) o[h][i] = fmaf(s[st][h], vf[i], o[h][i]);
  }
}

template <typename KvT, int D, int G, bool FUSED>
__global__ void __launch_bounds__(Cfg<KvT, D, G>::THREADS, 2)
decode_attn_kernel(const AttnParams p) {
  using C = Cfg<KvT, D, G>;
  constexpr int EPL = C::EPL, LPR = C::LPR, NC = C::NC, T = C::T;
  extern __shared__ __align__(128) unsigned char smem[];

  const int split = blockIdx.x;
  const int g = blockIdx.y;
  const int b = blockIdx.z;
  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const int ns = p.n_stages;
  const int Hq = p.n_q_heads, Hkv = p.n_kv_heads;

  unsigned char* ring = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + C::bar_off(ns));
  uint64_t* empty = full + C::NS;
  unsigned char* fresh_k = smem + C::fresh_off(ns);
  unsigned char* fresh_v = fresh_k + C::ROW_BYTES;
  float* scratch = reinterpret_cast<float*>(smem + C::scratch_off(ns));
  int* s_last = reinterpret_cast<int*>(smem + C::flag_off(ns));

  if (threadIdx.x == 0) {
    for (int s = 0; s < ns; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], NC);
    }
    mbar_init_fence();
  }
  __syncthreads();

  // The producer may stream cache rows before the preceding kernel finishes only when
  // the caller has promised that kernel does not write them (TTS_KV_PREFETCH_BEFORE_WAIT).
  const bool early = FUSED && (p.flags & TTS_KV_PREFETCH_BEFORE_WAIT);
  if (!early || warp < NC) grid_wait();
  if (warp < NC) grid_launch_dependents();

  const bool reporter = (split == 0 && g == 0 && threadIdx.x == 0);
  int nv, cache_end;
  bool fresh_ok = false;
  int cur = 0;
  if (FUSED) {
    cur = __ldcg(p.lens + b);
    fresh_ok = (cur >= 0 && cur < p.capacity);
    if (!fresh_ok && reporter) set_err(p.err, TTS_EFLAG_POS_RANGE);
    nv = min(max(cur + 1, 1), p.capacity);
    cache_end = fresh_ok ? cur : nv;
  } else {
    nv = __ldcg(p.lens + b);
    if ((nv < 1 || nv > p.capacity) && reporter) set_err(p.err, TTS_EFLAG_NVALID);
    nv = min(max(nv, 1), p.capacity);
    cache_end = nv;
  }
  const int r0 = split * p.split_len;
  const int n_rows = max(0, min(r0 + p.split_len, cache_end) - r0);
  const bool has_fresh = FUSED && fresh_ok && cur >= r0 && cur < r0 + p.split_len;
  const bool active = r0 < nv;
  const int ntiles = (n_rows + T - 1) / T;

  if (warp == NC) {
    // ------------------------------------------------------------------ producer
    if (lane == 0 && ntiles > 0) {
      const uint64_t pol = l2_evict_first_policy();
      const unsigned char* kc = static_cast<const unsigned char*>(p.k_cache);
      const unsigned char* vc = static_cast<const unsigned char*>(p.v_cache);
      const int32_t* bt = p.paged ? p.block_table + static_cast<int64_t>(b) * p.bt_stride : nullptr;
      int issued = 0;
      int stage = 0;
      uint32_t round = 0;
      for (int t = 0; t < ntiles; ++t) {
        if (t >= ns && !mbar_wait(&empty[stage], (round & 1u) ^ 1u)) {
          set_err(p.err, TTS_EFLAG_TIMEOUT);
          break;
        }
        const int row0 = r0 + t * T;
        const int rows = min(T, r0 + n_rows - row0);
        const uint32_t bytes = static_cast<uint32_t>(rows) * C::ROW_BYTES;
        unsigned char* kd = ring + stage * C::STAGE_BYTES;
        unsigned char* vd = kd + C::TILE_BYTES;
        mbar_arrive_expect_tx(&full[stage], 2u * bytes);
        if (!p.paged) {
          const size_t off =
              ((static_cast<size_t>(b) * Hkv + g) * p.capacity + row0) * C::ROW_BYTES;
          bulk_g2s(kd, kc + off, bytes, &full[stage], pol);
          bulk_g2s(vd, vc + off, bytes, &full[stage], pol);
        } else {
          int r = row0;
          const int re = row0 + rows;
          while (r < re) {
            int page = __ldcg(bt + (r >> p.page_shift));
            if (page < 0 || page >= p.n_pages) {
              set_err(p.err, TTS_EFLAG_PAGE);
              page = 0;
            }
            const int slot = r & (p.page_size - 1);
            const int n = min(p.page_size - slot, re - r);
            const size_t off =
                ((static_cast<size_t>(page) * Hkv + g) * p.page_size + slot) * C::ROW_BYTES;
            const uint32_t nb = static_cast<uint32_t>(n) * C::ROW_BYTES;
            bulk_g2s(kd + (r - row0) * C::ROW_BYTES, kc + off, nb, &full[stage], pol);
            bulk_g2s(vd + (r - row0) * C::ROW_BYTES, vc + off, nb, &full[stage], pol);
            r += n;
          }
        }
        ++issued;
        if (++stage == ns) {
          stage = 0;
          ++round;
        }
      }
      // Do not leave while copies into this CTA's shared memory may be in flight.
      for (int t = max(0, issued - ns); t < issued; ++t)
        mbar_wait(&full[t % ns], static_cast<uint32_t>(t / ns) & 1u);
    }
    return;
  }

  // -------------------------------------------------------------------- consumers
  const int tid = threadIdx.x;  // < NC * 32
  const int lr = lane % LPR;
  const int e0 = lr * EPL;
  const int half = D / 2;

  if (active) {
    int rope_pos = 0;
    if (FUSED) {
      rope_pos = min(max(cur, 0), p.max_pos - 1);
      if ((cur < 0 || cur >= p.max_pos) && reporter) set_err(p.err, TTS_EFLAG_POS_RANGE);
    }
    const float2* cs_row = p.cs + static_cast<int64_t>(rope_pos) * half;

    float q[G][EPL];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      load_row_f32<EPL>(p.q + static_cast<int64_t>(b) * p.q_stride + static_cast<int64_t>(g * G + h) * D,
                        e0, q[h]);
      if (FUSED) norm_rope_lanes<EPL, LPR>(q[h], p.gamma_q, cs_row, p.eps, e0, D);
#pragma unroll
      for (int i = 0; i < EPL; ++i) q[h][i] *= p.scale_log2;
    }

    // Fused: build the new K/V row (norm + RoPE on k, v as is), convert it to the cache
    // type, store it to the cache and keep a copy in shared memory for this CTA.
    if (FUSED && has_fresh && warp == 0) {
      float kr[EPL], vr[EPL];
      const int64_t roff = static_cast<int64_t>(b) * p.kv_new_stride + static_cast<int64_t>(g) * D;
      load_row_f32<EPL>(p.k_new + roff, e0, kr);
      load_row_f32<EPL>(p.v_new + roff, e0, vr);
      norm_rope_lanes<EPL, LPR>(kr, p.gamma_k, cs_row, p.eps, e0, D);
      if (lane < LPR) {
        const uint4 kp = pack_row(kr, static_cast<KvT*>(nullptr));
        const uint4 vp = pack_row(vr, static_cast<KvT*>(nullptr));
        *reinterpret_cast<uint4*>(fresh_k + lr * 16) = kp;
        *reinterpret_cast<uint4*>(fresh_v + lr * 16) = vp;
        size_t off;
        bool write = true;
        if (!p.paged) {
          off = ((static_cast<size_t>(b) * Hkv + g) * p.capacity + cur) * C::ROW_BYTES;
        } else {
          const int page = __ldcg(p.block_table + static_cast<int64_t>(b) * p.bt_stride + (cur >> p.page_shift));
          write = page >= 0 && page < p.n_pages;
          if (!write && lane == 0) set_err(p.err, TTS_EFLAG_PAGE);
          off = ((static_cast<size_t>(write ? page : 0) * Hkv + g) * p.page_size +
                 (cur & (p.page_size - 1))) * C::ROW_BYTES;
        }
        if (write) {
          *reinterpret_cast<uint4*>(static_cast<unsigned char*>(p.k_cache_w) + off + lr * 16) = kp;
          *reinterpret_cast<uint4*>(static_cast<unsigned char*>(p.v_cache_w) + off + lr * 16) = vp;
        }
      }
      __syncwarp();
    }

    float m_run[G], l_run[G], o[G][EPL];
#pragma unroll
    for (int h = 0; h < G; ++h) {
      m_run[h] = -INFINITY;
      l_run[h] = 0.f;
#pragma unroll
      for (int i = 0; i < EPL; ++i) o[h][i] = 0.f;
    }

    bool ok = true;
    int stage = 0;
    uint32_t round = 0;
    for (int t = 0; t < ntiles; ++t) {
      if (!mbar_wait(&full[stage], round & 1u)) {
        set_err(p.err, TTS_EFLAG_TIMEOUT);
        ok = false;
        break;
      }
      const unsigned char* kt = ring + stage * C::STAGE_BYTES;
      const unsigned char* vt = kt + C::TILE_BYTES;
      const int rows = min(T, n_rows - t * T);
      if (rows == T)
        consume_tile<C, KvT, false>(kt, vt, T, warp, lane, q, m_run, l_run, o);
      else
        consume_tile<C, KvT, true>(kt, vt, rows, warp, lane, q, m_run, l_run, o);
      __syncwarp();
      if (lane == 0) mbar_arrive(&empty[stage]);
      if (++stage == ns) {
        stage = 0;
        ++round;
      }
    }
    if (FUSED && has_fresh && ok)
      consume_tile<C, KvT, true>(fresh_k, fresh_v, 1, warp, lane, q, m_run, l_run, o);

    // Merge the row groups of this warp, then the warps of this CTA.
#pragma unroll
    for (int h = 0; h < G; ++h) {
#pragma unroll
      for (int off = LPR; off < 32; off <<= 1) {
        l_run[h] += __shfl_xor_sync(kFull, l_run[h], off);
#pragma unroll
        for (int i = 0; i < EPL; ++i) o[h][i] += __shfl_xor_sync(kFull, o[h][i], off);
      }
    }
    if (lane < LPR) {
#pragma unroll
      for (int h = 0; h < G; ++h) {
        float* dst = scratch + (warp * G + h) * (D + 2);
#pragma unroll
        for (int i = 0; i < EPL; ++i) dst[e0 + i] = o[h][i];
        if (lane == 0) {
          dst[D] = m_run[h];
          dst[D + 1] = l_run[h];
        }
      }
    }
    named_barrier(1, NC * 32);

    for (int idx = tid; idx < G * D; idx += NC * 32) {
      const int h = idx / D;
      const int d = idx - h * D;
      float M = -INFINITY;
#pragma unroll
      for (int w = 0; w < NC; ++w) M = fmaxf(M, scratch[(w * G + h) * (D + 2) + D]);
      float L = 0.f, O = 0.f;
#pragma unroll
      for (int w = 0; w < NC; ++w) {
        const float* src = scratch + (w * G + h) * (D + 2);
        const float f = (src[D] == -INFINITY) ? 0.f : exp2f(src[D] - M);
        L = fmaf(src[D + 1], f, L);
        O = fmaf(src[d], f, O);
      }
      const int hq = g * G + h;
      if (p.n_splits == 1) {
        p.out[(static_cast<int64_t>(b) * Hq + hq) * D + d] = O / L;
      } else {
        const int64_t slot = (static_cast<int64_t>(b) * Hq + hq) * p.n_splits + split;
        p.ws_o[slot * D + d] = O;
        if (d == 0) {
          p.ws_ml[slot * 2] = M;
          p.ws_ml[slot * 2 + 1] = L;
        }
      }
    }
  }

  if (p.n_splits == 1) return;

  // Ticket: the last split of this (stream, kv head) to finish merges all partials.
  __threadfence();
  named_barrier(1, NC * 32);
  if (tid == 0) {
    const int prev = atomicAdd(p.ws_cnt + b * Hkv + g, 1);
    *s_last = (prev == p.n_splits - 1) ? 1 : 0;
  }
  named_barrier(1, NC * 32);
  if (*s_last == 0) return;
  __threadfence();
  const int n_act = min(p.n_splits, (nv + p.split_len - 1) / p.split_len);
  for (int idx = tid; idx < G * D; idx += NC * 32) {
    const int h = idx / D;
    const int d = idx - h * D;
    const int hq = g * G + h;
    const int64_t base = (static_cast<int64_t>(b) * Hq + hq) * p.n_splits;
    float M = -INFINITY;
    for (int s = 0; s < n_act; ++s) M = fmaxf(M, __ldcg(p.ws_ml + (base + s) * 2));
    float L = 0.f, O = 0.f;
    for (int s = 0; s < n_act; ++s) {
      const float f = exp2f(__ldcg(p.ws_ml + (base + s) * 2) - M);
      L = fmaf(__ldcg(p.ws_ml + (base + s) * 2 + 1), f, L);
      O = fmaf(__ldcg(p.ws_o + (base + s) * D + d), f, O);
    }
    p.out[(static_cast<int64_t>(b) * Hq + hq) * D + d] = O / L;
  }
  if (tid == 0) p.ws_cnt[b * Hkv + g] = 0;
}

template <typename KvT, int D, int G, bool FUSED>
cudaError_t launch_one(const AttnParams& p, cudaStream_t s) {
  using C = Cfg<KvT, D, G>;
  auto kern = decode_attn_kernel<KvT, D, G, FUSED>;
  const size_t smem = C::smem_bytes(p.n_stages);
  static int configured_for = -1;  // device whose max-dynamic-smem attribute is set
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (configured_for != dev) {
    e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize,
                             static_cast<int>(C::smem_bytes(C::NS)));
    if (e != cudaSuccess) return e;
    configured_for = dev;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(p.n_splits, p.n_kv_heads, p.B);
  cfg.blockDim = dim3(C::THREADS);
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, p);
}

template <typename KvT, int D>
cudaError_t dispatch_group(const AttnParams& p, int group, bool fused, cudaStream_t s) {
  switch (group) {
    case 1: return fused ? launch_one<KvT, D, 1, true>(p, s) : launch_one<KvT, D, 1, false>(p, s);
    case 2: return fused ? launch_one<KvT, D, 2, true>(p, s) : launch_one<KvT, D, 2, false>(p, s);
    case 4: return fused ? launch_one<KvT, D, 4, true>(p, s) : launch_one<KvT, D, 4, false>(p, s);
    default: return cudaErrorInvalidValue;
  }
}

template <typename KvT, int D>
AttnGeometry geometry_of() {
  using C = Cfg<KvT, D, 1>;
  return AttnGeometry{C::T, C::NS, C::STAGE_BYTES, C::THREADS};
}

template <typename KvT, int D>
size_t smem_of(int group, int ns) {
  switch (group) {
    case 1: return Cfg<KvT, D, 1>::smem_bytes(ns);
    case 2: return Cfg<KvT, D, 2>::smem_bytes(ns);
    case 4: return Cfg<KvT, D, 4>::smem_bytes(ns);
    default: return 0;
  }
}

}  // namespace

AttnGeometry attn_geometry(int kv_bf16, int head_dim) {
  if (kv_bf16) return head_dim == 64 ? geometry_of<__nv_bfloat16, 64>() : geometry_of<__nv_bfloat16, 128>();
  return head_dim == 64 ? geometry_of<float, 64>() : geometry_of<float, 128>();
}

size_t attn_smem_bytes(int kv_bf16, int head_dim, int group, int n_stages) {
  if (kv_bf16)
    return head_dim == 64 ? smem_of<__nv_bfloat16, 64>(group, n_stages)
                          : smem_of<__nv_bfloat16, 128>(group, n_stages);
  return head_dim == 64 ? smem_of<float, 64>(group, n_stages) : smem_of<float, 128>(group, n_stages);
}

cudaError_t launch_decode_attn(const AttnParams& p, int kv_bf16, int head_dim, int group,
                               bool fused, cudaStream_t s) {
  if (kv_bf16) {
    if (head_dim == 64) return dispatch_group<__nv_bfloat16, 64>(p, group, fused, s);
    if (head_dim == 128) return dispatch_group<__nv_bfloat16, 128>(p, group, fused, s);
  } else {
    if (head_dim == 64) return dispatch_group<float, 64>(p, group, fused, s);
    if (head_dim == 128) return dispatch_group<float, 128>(p, group, fused, s);
  }
  return cudaErrorInvalidValue;
}

}  // namespace tts
