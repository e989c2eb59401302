// Device helpers shared by the decode-path kernels (sm_103a): error flag, bounded
// mbarrier waits, 1-D bulk (TMA) copies global -> shared, programmatic dependent
// launch controls, 16-byte vector loads and bf16 unpacking.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/tts_decode.h"

namespace tts {

constexpr unsigned kFull = 0xffffffffu;

// Upper bound on any in-kernel wait, in SM clock cycles (about a second at the
// GB300's clocks).  A wait that runs out sets TTS_EFLAG_TIMEOUT and the kernel winds
// down instead of hanging.
constexpr long long kWaitLimitCycles = 2000000000LL;

__device__ __forceinline__ void set_err(int32_t* flag, int bits) {
  if (flag != nullptr) atomicOr(flag, bits);
}

// ---------------------------------------------------------------------------
// Programmatic dependent launch.  `grid_wait` blocks until the preceding kernel on
// the stream has completed and its writes are visible (a no-op when the kernel was
// launched without the programmatic-serialisation attribute); `grid_launch_dependents`
// lets the next kernel be scheduled early.
// ---------------------------------------------------------------------------
__device__ __forceinline__ void grid_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------------------
// Shared-memory mbarriers
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}

// Makes barrier initialisation visible to the async (bulk-copy) proxy.
__device__ __forceinline__ void mbar_init_fence() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}

__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes) {
  uint64_t state;
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 %0, [%1], %2;"
               : "=l"(state) : "r"(smem_u32(bar)), "r"(bytes) : "memory");
  (void)state;
}

__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  uint64_t state;
  asm volatile("mbarrier.arrive.shared::cta.b64 %0, [%1];" : "=l"(state) : "r"(smem_u32(bar)) : "memory");
  (void)state;
}

__device__ __forceinline__ bool mbar_try_wait(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}

// Waits until the phase with the given parity has completed.  Bounded: returns false
// after kWaitLimitCycles.
__device__ __forceinline__ bool mbar_wait(uint64_t* bar, uint32_t parity) {
  if (mbar_try_wait(bar, parity)) return true;
  const long long start = clock64();
  while (!mbar_try_wait(bar, parity)) {
    if (clock64() - start > kWaitLimitCycles) return false;
  }
  return true;
}

// ---------------------------------------------------------------------------
// 1-D bulk copy global -> shared (TMA engine), completion counted in bytes on an
// mbarrier.  Addresses 16-byte aligned, size a multiple of 16.  The L2 policy marks
// the streamed KV lines evict-first: each is read once per step.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint64_t l2_evict_first_policy() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

__device__ __forceinline__ void bulk_g2s(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                         uint64_t* bar, uint64_t policy) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1], %2, [%3], %4;"
      ::"r"(smem_u32(smem_dst)), "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar)), "l"(policy)
      : "memory");
}

// The same copy with the default L2 policy (for small rows read again soon).
__device__ __forceinline__ void bulk_g2s_plain(void* smem_dst, const void* gmem_src, uint32_t bytes,
                                               uint64_t* bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
      ::"r"(smem_u32(smem_dst)), "l"(gmem_src), "r"(bytes), "r"(smem_u32(bar))
      : "memory");
}

// Named barrier over a subset of the CTA's warps (id 0 is __syncthreads).
__device__ __forceinline__ void named_barrier(int id, int threads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(threads) : "memory");
}

// ---------------------------------------------------------------------------
// Vector loads and bf16 unpacking
// ---------------------------------------------------------------------------
// 16 bytes from shared memory (an explicit shared-window load, never a generic one).
__device__ __forceinline__ uint4 lds128(const void* p) {
  uint4 v;
  asm volatile("ld.shared.v4.u32 {%0, %1, %2, %3}, [%4];"
               : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w) : "r"(smem_u32(p)));
  return v;
}

// Eight bf16 packed in a uint4 (element 0 in the low half of .x) -> eight floats.
// Widening bf16 -> f32 is exact: the bf16 bits become the high half of the f32.
__device__ __forceinline__ void unpack_bf16x8(const uint4 v, float (&f)[8]) {
  const uint32_t w[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    f[2 * i] = __uint_as_float(w[i] << 16);
    f[2 * i + 1] = __uint_as_float(w[i] & 0xffff0000u);
  }
}

__device__ __forceinline__ void unpack_f32x4(const uint4 v, float (&f)[4]) {
  f[0] = __uint_as_float(v.x);
  f[1] = __uint_as_float(v.y);
  f[2] = __uint_as_float(v.z);
  f[3] = __uint_as_float(v.w);
}

template <typename KvT> struct KvVec;
template <> struct KvVec<float> {
  static constexpr int kElems = 4;
  static __device__ __forceinline__ void unpack(const uint4 v, float (&f)[4]) { unpack_f32x4(v, f); }
};
template <> struct KvVec<__nv_bfloat16> {
  static constexpr int kElems = 8;
  static __device__ __forceinline__ void unpack(const uint4 v, float (&f)[8]) { unpack_bf16x8(v, f); }
};

// f32 -> cache element, round-to-nearest-even for bf16.
__device__ __forceinline__ float to_cache(float x, float*) { return x; }
__device__ __forceinline__ __nv_bfloat16 to_cache(float x, __nv_bfloat16*) { return __float2bfloat16_rn(x); }

// ---------------------------------------------------------------------------
// Per-head RMSNorm + rotate-half RoPE on a row of D elements held by a group of LPR
// lanes.  Lane lr of the group holds VEC vectors of VE elements; element e of vector
// j is row element (j * LPR + lr) * VE + e, so D = VEC * LPR * VE.  All lanes of the
// warp must call it (the sum of squares is reduced over the group with shuffles).
//   t = x * (mean(x^2) + eps)^(-1/2) * gamma
//   (t_i, t_{i+D/2}) -> (t_i c - t_{i+D/2} s, t_i s + t_{i+D/2} c),  (c, s) of theta_i
// With VEC >= 2 the partner i + D/2 of element i sits in the same lane (vector
// j + VEC/2); with VEC == 1 it sits in lane lr ^ (LPR/2).
// gam[k] = gamma of the lane's element k; cs[k] = (cos, sin) of frequency
// (row index of element k) mod D/2.
// ---------------------------------------------------------------------------
template <int VE, int VEC, int LPR>
__device__ __forceinline__ void load_norm_consts(const float* gamma, const float2* cs_row, int lr,
                                                 int D, float (&gam)[VE * VEC],
                                                 float2 (&cs)[VE * VEC]) {
  const int half = D / 2;
#pragma unroll
  for (int j = 0; j < VEC; ++j) {
    const int idx = (j * LPR + lr) * VE;
    const int f = idx < half ? idx : idx - half;
#pragma unroll
    for (int e = 0; e < VE; e += 4) {
      const float4 gv = __ldcg(reinterpret_cast<const float4*>(gamma + idx + e));
      gam[j * VE + e] = gv.x; gam[j * VE + e + 1] = gv.y;
      gam[j * VE + e + 2] = gv.z; gam[j * VE + e + 3] = gv.w;
      const float4 c0 = __ldcg(reinterpret_cast<const float4*>(cs_row + f + e));
      const float4 c1 = __ldcg(reinterpret_cast<const float4*>(cs_row + f + e + 2));
      cs[j * VE + e] = make_float2(c0.x, c0.y); cs[j * VE + e + 1] = make_float2(c0.z, c0.w);
      cs[j * VE + e + 2] = make_float2(c1.x, c1.y); cs[j * VE + e + 3] = make_float2(c1.z, c1.w);
    }
  }
}

// load_norm_consts from shared-memory copies of gamma and of the RoPE row.
template <int VE, int VEC, int LPR>
__device__ __forceinline__ void load_norm_consts_smem(const float* gamma, const float2* cs_row, int lr,
                                                      int D, float (&gam)[VE * VEC],
                                                      float2 (&cs)[VE * VEC]) {
  const int half = D / 2;
#pragma unroll
  for (int j = 0; j < VEC; ++j) {
    const int idx = (j * LPR + lr) * VE;
    const int f = idx < half ? idx : idx - half;
#pragma unroll
    for (int e = 0; e < VE; e += 4) {
      const uint4 gv = lds128(gamma + idx + e);
      gam[j * VE + e] = __uint_as_float(gv.x); gam[j * VE + e + 1] = __uint_as_float(gv.y);
      gam[j * VE + e + 2] = __uint_as_float(gv.z); gam[j * VE + e + 3] = __uint_as_float(gv.w);
      const uint4 c0 = lds128(cs_row + f + e);
      const uint4 c1 = lds128(cs_row + f + e + 2);
      cs[j * VE + e] = make_float2(__uint_as_float(c0.x), __uint_as_float(c0.y));
      cs[j * VE + e + 1] = make_float2(__uint_as_float(c0.z), __uint_as_float(c0.w));
      cs[j * VE + e + 2] = make_float2(__uint_as_float(c1.x), __uint_as_float(c1.y));
      cs[j * VE + e + 3] = make_float2(__uint_as_float(c1.z), __uint_as_float(c1.w));
    }
  }
}

// The lane's elements of an f32 row held in shared memory, in the lane layout of the
// cache rows: element e of vector j is row element (j * LPR + lr) * VE + e.
template <int VE, int VEC, int LPR>
__device__ __forceinline__ void load_row_smem(const float* row, int lr, float (&x)[VE * VEC]) {
#pragma unroll
  for (int j = 0; j < VEC; ++j)
#pragma unroll
    for (int e = 0; e < VE; e += 4) {
      const uint4 v = lds128(row + (j * LPR + lr) * VE + e);
      x[j * VE + e] = __uint_as_float(v.x); x[j * VE + e + 1] = __uint_as_float(v.y);
      x[j * VE + e + 2] = __uint_as_float(v.z); x[j * VE + e + 3] = __uint_as_float(v.w);
    }
}

template <int VE, int VEC, int LPR>
__device__ __forceinline__ void norm_rope_regs(float (&x)[VE * VEC], const float (&gam)[VE * VEC],
                                               const float2 (&cs)[VE * VEC], float eps, int lr,
                                               int D) {
  constexpr int EPL = VE * VEC;
  float ss = 0.f;
#pragma unroll
  for (int i = 0; i < EPL; ++i) ss = fmaf(x[i], x[i], ss);
#pragma unroll
  for (int o = LPR / 2; o >= 1; o >>= 1) ss += __shfl_xor_sync(kFull, ss, o);
  const float r = 1.0f / sqrtf(ss / static_cast<float>(D) + eps);
  float t[EPL];
#pragma unroll
  for (int i = 0; i < EPL; ++i) t[i] = x[i] * r * gam[i];
  if (VEC >= 2) {
#pragma unroll
    for (int j = 0; j < VEC / 2; ++j)
#pragma unroll
      for (int e = 0; e < VE; ++e) {
        const int a = j * VE + e, c = (j + VEC / 2) * VE + e;
        x[a] = fmaf(t[a], cs[a].x, -t[c] * cs[a].y);
        x[c] = fmaf(t[a], cs[a].y, t[c] * cs[a].x);
      }
  } else {
    const bool lo = lr < LPR / 2;
#pragma unroll
    for (int i = 0; i < EPL; ++i) {
      const float pt = __shfl_xor_sync(kFull, t[i], LPR / 2);
      // lower half: t*c - partner*s ; upper half: partner*s + t*c
      x[i] = lo ? fmaf(t[i], cs[i].x, -pt * cs[i].y) : fmaf(pt, cs[i].y, t[i] * cs[i].x);
    }
  }
}

// ---------------------------------------------------------------------------
// Thread-block clusters: rank, cluster-wide barrier, distributed shared memory.
// ---------------------------------------------------------------------------
__device__ __forceinline__ uint32_t cluster_rank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}

// All threads of all CTAs of the cluster; also a barrier for this CTA.
__device__ __forceinline__ void cluster_sync_all() {
  asm volatile("barrier.cluster.arrive.release.aligned;\n\tbarrier.cluster.wait.acquire.aligned;" ::: "memory");
}

// Address of the same shared-memory location in CTA `rank` of the cluster.
__device__ __forceinline__ uint32_t map_shared_rank(const void* local, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(local)), "r"(rank));
  return r;
}

__device__ __forceinline__ void st_cluster_f32(uint32_t addr, float v) {
  asm volatile("st.shared::cluster.f32 [%0], %1;" ::"r"(addr), "f"(v) : "memory");
}

// Arrive on an mbarrier of another CTA of the cluster, releasing this CTA's prior
// shared-memory writes (ordered before this call by a CTA barrier) at cluster scope.
__device__ __forceinline__ void mbar_arrive_remote(uint32_t cluster_addr) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(cluster_addr) : "memory");
}

__device__ __forceinline__ bool mbar_try_wait_cluster(uint64_t* bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.acquire.cluster.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok) : "r"(smem_u32(bar)), "r"(parity) : "memory");
  return ok != 0;
}

// Bounded wait for a phase completed by other CTAs of the cluster (acquire).
__device__ __forceinline__ bool mbar_wait_cluster(uint64_t* bar, uint32_t parity, long long limit) {
  if (mbar_try_wait_cluster(bar, parity)) return true;
  const long long start = clock64();
  while (!mbar_try_wait_cluster(bar, parity)) {
    if (clock64() - start > limit) return false;
  }
  return true;
}

// Ticket counter with acquire-release semantics at GPU scope.  Called by one thread
// after a CTA barrier, it publishes every store the CTA made before the barrier.
__device__ __forceinline__ int atomic_add_acq_rel_gpu(int* p, int v) {
  int old;
  asm volatile("atom.add.acq_rel.gpu.global.s32 %0, [%1], %2;" : "=r"(old) : "l"(p), "r"(v) : "memory");
  return old;
}

// Launch with programmatic stream serialisation (the kernel itself calls grid_wait
// before it touches its inputs and grid_launch_dependents to let the next one start).
template <typename Kernel, typename... Args>
cudaError_t launch_pdl(Kernel kern, dim3 grid, dim3 block, size_t smem, cudaStream_t s,
                       Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kern, args...);
}

}  // namespace tts
