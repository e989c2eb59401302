// tts_decode_step_noalloc: the fused decode step with its split-KV scratch taken from
// a fixed, library-owned device array instead of a caller-supplied workspace.
//
// Who needs this: some callers cannot allocate device memory at the point where they
// run a decode step -- for example a real-time audio callback that must not enter an
// allocator (unbounded latency, locks), a host framework that hands out only the
// tensors it owns and exposes no allocation hook, or code that runs while allocation is
// forbidden (inside a region that records work for later replay without a memory pool).
// They still own and pass every input and output; only the scratch comes from here.
//
// The scratch is a file-scope device array of kNoAllocScratchBytes.  Every GPU that
// loads the library holds it until the process exits.  In host code the array's name
// is only a stand-in for the device symbol, so the launch path uses the device address
// obtained once per device with cudaGetSymbolAddress.
#include <cstddef>
#include <cstdint>
#include <mutex>

#include <cuda_runtime.h>

#include "../../include/tts_decode.h"

namespace {

constexpr size_t kNoAllocScratchBytes = size_t(4) << 20;  // 4 MiB
constexpr int kMaxDevices = 64;

__device__ __align__(256) unsigned char g_noalloc_scratch[kNoAllocScratchBytes];

std::mutex g_setup_mutex;
void* g_scratch_ptr[kMaxDevices] = {};

// Once per device, with that device current: look up the array's device address.
// Synchronous, so the first call on a device must not be inside a stream capture.
tts_status scratch_for_current_device(void** out) {
  int dev = 0;
  if (cudaGetDevice(&dev) != cudaSuccess || dev < 0 || dev >= kMaxDevices) return TTS_ERR_CUDA;
  std::lock_guard<std::mutex> lock(g_setup_mutex);
  if (g_scratch_ptr[dev] == nullptr) {
    void* ptr = nullptr;
    if (cudaGetSymbolAddress(&ptr, g_noalloc_scratch) != cudaSuccess || ptr == nullptr)
      return TTS_ERR_CUDA;
    g_scratch_ptr[dev] = ptr;
  }
  *out = g_scratch_ptr[dev];
  return TTS_OK;
}

}  // namespace

extern "C" tts_status tts_decode_step_noalloc(const float* q, const float* k, const float* v,
                                              int64_t row_stride, const float* gamma_q,
                                              const float* gamma_k, float eps,
                                              const float* rope_cs, int32_t rope_max_pos,
                                              void* k_cache, void* v_cache,
                                              const tts_kv_desc* desc, const int32_t* cur_len,
                                              float scale, float* out, int32_t n_splits,
                                              int32_t* err_flag, void* stream) {
  if (desc == nullptr) return TTS_ERR_NULL;
  const size_t need = tts_decode_attn_workspace_size(desc, n_splits);
  if (need == 0) return TTS_ERR_SHAPE;
  if (need > kNoAllocScratchBytes) return TTS_ERR_WORKSPACE;
  void* scratch = nullptr;
  tts_status st = scratch_for_current_device(&scratch);
  if (st != TTS_OK) return st;
  // The array keeps whatever the previous call (of any shape) left in it, and where the
  // split tickets sit depends on the shape: clear the part this call uses, on its stream.
  st = tts_workspace_init(scratch, need, stream);
  if (st != TTS_OK) return st;
  return tts_decode_step(q, k, v, row_stride, gamma_q, gamma_k, eps, rope_cs, rope_max_pos, k_cache,
                         v_cache, desc, cur_len, scale, out, scratch, kNoAllocScratchBytes, n_splits,
                         err_flag, stream);
}
