// Codebook-table rows as f32, shared by the frame-input composition and the sampler's
// gather: f32 rows, bf16 rows widened exactly, or Q8_0 blocks dequantised exactly.
#pragma once

#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_runtime.h>

namespace tts {

// Four consecutive table entries as f32: a 16-byte load of f32, an 8-byte load of bf16
// widened exactly (the bf16 bits are the high half of the f32), or four Q8_0 quants
// times their block's scale.
__device__ __forceinline__ float4 load_row4(const float* row, int c4) {
  return __ldg(reinterpret_cast<const float4*>(row) + c4);
}
__device__ __forceinline__ float4 load_row4(const __nv_bfloat16* row, int c4) {
  const uint2 w = __ldg(reinterpret_cast<const uint2*>(row) + c4);
  return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xffff0000u),
                     __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xffff0000u));
}

// Q8_0 blocks: 32 table entries in 34 bytes, a binary16 scale d then 32 int8 quants q,
// entry = d * q.  The product of an 11-bit and an 8-bit significand is exact in f32.
struct Q8Block {};
constexpr int kQ8Block = 32;
constexpr int kQ8Bytes = 34;
__device__ __forceinline__ float4 load_row4(const Q8Block* row, int c4) {
  const unsigned char* blk = reinterpret_cast<const unsigned char*>(row) + ((4 * c4) / kQ8Block) * kQ8Bytes;
  const float d = __half2float(__ushort_as_half(__ldg(reinterpret_cast<const unsigned short*>(blk))));
  // the block and its quants start on even bytes: two 2-byte loads
  const unsigned short* qs = reinterpret_cast<const unsigned short*>(blk + 2 + (4 * c4) % kQ8Block);
  const unsigned short lo = __ldg(qs), hi = __ldg(qs + 1);
  const float q0 = static_cast<float>(static_cast<signed char>(lo & 0xff));
  const float q1 = static_cast<float>(static_cast<signed char>(lo >> 8));
  const float q2 = static_cast<float>(static_cast<signed char>(hi & 0xff));
  const float q3 = static_cast<float>(static_cast<signed char>(hi >> 8));
  return make_float4(__fmul_rn(d, q0), __fmul_rn(d, q1), __fmul_rn(d, q2), __fmul_rn(d, q3));
}

// Address of row `id` of a table of `hidden` entries per row.
template <typename TabT>
__device__ __forceinline__ const TabT* table_row(const void* tab, int id, int hidden) {
  return static_cast<const TabT*>(tab) + static_cast<int64_t>(id) * hidden;
}
template <>
__device__ __forceinline__ const Q8Block* table_row<Q8Block>(const void* tab, int id, int hidden) {
  return reinterpret_cast<const Q8Block*>(static_cast<const unsigned char*>(tab) +
                                          static_cast<int64_t>(id) * (hidden / kQ8Block) * kQ8Bytes);
}

}  // namespace tts
