// Internal launch interface between the C-ABI layer (api.cu) and the kernels.
#pragma once

#include <cstddef>
#include <cstdint>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "../../include/tts_decode.h"

namespace tts {

struct EmbedParams {
  const void* tab[TTS_MAX_TABLES];  // f32, bf16 or Q8_0 rows (tab_dtype)
  int tab_dtype;                    // tts_dtype
  int n_tables, vocab, hidden;
  const int32_t* ids;
  int64_t ids_stride;
  const float* overlay;
  int64_t overlay_stride;
  float* out;
  int B;
  int32_t* err;
};

struct NormRopeParams {
  float* q;
  int64_t q_stride;
  float* k;
  int64_t k_stride;
  const float* gamma_q;
  const float* gamma_k;
  const int32_t* pos;
  int B, n_q_heads, n_kv_heads, head_dim;
  float eps;
  const float2* cs;
  int max_pos;
  int32_t* err;
};

struct SetRowsParams {
  const float* k;
  const float* v;
  int64_t row_stride;
  void* k_cache;
  void* v_cache;
  int B, n_kv_heads, head_dim, capacity, kv_bf16;
  int paged, page_size, n_pages, bt_stride;
  const int32_t* block_table;
  const int32_t* pos;
  int32_t* err;
};

// Decode attention, standalone (q already normed) or fused with norm+RoPE and the
// new-row write.
struct AttnParams {
  const float* q;       // standalone: normed q; fused: raw projection q
  int64_t q_stride;
  const float* k_new;   // fused only
  const float* v_new;   // fused only
  int64_t kv_new_stride;
  const float* gamma_q;
  const float* gamma_k;
  float eps;
  const float2* cs;
  int max_pos;
  const void* k_cache;
  const void* v_cache;
  void* k_cache_w;      // fused: where the new row goes
  void* v_cache_w;
  int B, n_q_heads, n_kv_heads, capacity;
  int paged, page_size, page_shift, n_pages, bt_stride;
  const int32_t* block_table;
  const int32_t* lens;  // standalone: n_valid; fused: cur_len; prefill: start position
  // Query streams per cache stream (1, or a prefill's T queries) and the constant added
  // to lens[cache stream] + query offset to form the window input (prefill: 1).
  int q_per_stream, lens_add;
  float scale_log2;     // softmax scale * log2(e)
  float* out;
  // optional: the output rounded to bf16 in the projection input layout
  // [Hq D / 8][out_slots][8] (the stream's slot b), written instead of `out`
  __nv_bfloat16* out_packed;
  int out_slots;
  float* ws_o;          // [B][Hq][n_splits][D]
  float* ws_ml;         // [B][Hq][n_splits][2]
  int* ws_cnt;          // [B][Hkv] split tickets
  int* ws_sched;        // [2] persistent mode: work counter, finished-CTA counter
  int n_splits;         // grid.x
  int split_len;        // positions per split, a multiple of the tile
  int n_stages;         // ring stages actually used (set by the launcher)
  int cluster;          // set by the launcher: splits per cluster (>1 = cluster merge)
  int persistent;       // set by the launcher: 1 = fixed grid walking the active items
  int inflight;         // set by the launcher: tiles a producer keeps in flight (0 = ring)
  // set by the launcher: byte offsets in dynamic shared memory of the ring's mbarriers
  // (the ring starts at 0), the per-warp merge scratch, the flag word and item queue,
  // the combine area, the cluster gather area, the persistent work list and the
  // persistent q slots
  uint32_t sm_bar, sm_scratch, sm_flag, sm_comb, sm_gather, sm_list, sm_qbuf;
  uint32_t flags;
  int32_t* err;
};

// Prefill rows: for query row r = b * T + t (position start[b] + t), q RMS-normed and
// rotated in place, k normed and rotated into the cache, v copied into the cache.
struct PrefillRowsParams {
  const float* q;
  float* q_out;         // the normed and rotated q rows [B T][Hq D], dense; nullptr: q skipped
  const float* k;
  const float* v;
  int64_t row_stride;   // floats between consecutive rows r of q, k and v
  const float* gamma_q;
  const float* gamma_k;
  float eps;
  const float2* cs;
  int max_pos;
  void* k_cache;
  void* v_cache;
  int B, T, n_q_heads, n_kv_heads, head_dim, capacity, kv_bf16;
  int paged, page_size, n_pages, bt_stride;
  const int32_t* block_table;
  const int32_t* start;
  int32_t* err;
};

// Sampler: one stream per CTA (see sample.cu).
struct SampleParams {
  const float* logits;
  int64_t stride;       // floats between consecutive streams' logits
  int B, V, top_k;      // top_k 0 or 1: greedy
  float c;              // log2(e) / temperature, rounded once to f32
  uint64_t seed;
  const uint64_t* counter;
  uint32_t draw;        // third counter word: the draw's index within one counter value
  int32_t* out;
  int64_t out_stride;   // int32 elements between consecutive streams' ids
  // optional gather of the drawn token's table row (emb_out == nullptr: none)
  const void* emb_tab;  // f32, bf16 or Q8_0 rows of emb_hidden entries
  int emb_dtype;        // tts_dtype
  int emb_hidden;
  float* emb_out;       // f32 [B][emb_hidden]
};

// bf16-weight GEMV of the decode layer (see layer.cu): y[b][n] = sum_k x[b][k] W[n][k].
constexpr int kGemvMaxB = 8;      // streams per launch
constexpr int kGemvMaxK = 8192;   // row length (a multiple of 256)
struct GemvParams {
  const void* x;        // f32 or bf16 [B][K], rows x_stride elements apart
  int64_t x_stride;
  const float* gamma;   // RMS-norm input mode: gamma [K], and eps
  float eps;
  const void* w;        // bf16 [rows][K]
  int n_out;            // output rows (SiLU-multiply: gate/up pairs)
  int K, B;
  int inter;            // SiLU-multiply: offset of the up rows
  void* y;              // f32 [B][..] (store, residual) or bf16 [B][inter] (SiLU-multiply)
  int64_t y_stride;
  int32_t* err;         // TTS_EFLAG_TIMEOUT when a bounded wait runs out (may be null)
  int seg, stages;      // set by the launcher: row segment length, ring depth,
  uint32_t x_off;       // and the shared-memory offset of the staged activations
};

// Launch helpers (return a cudaError_t from the launch).
cudaError_t launch_frame_embed(const EmbedParams& p, cudaStream_t s);
cudaError_t launch_rope_table(float* cs, int max_pos, int head_dim, double base, cudaStream_t s);
cudaError_t launch_qk_norm_rope(const NormRopeParams& p, cudaStream_t s);
cudaError_t launch_set_rows(const SetRowsParams& p, cudaStream_t s);
cudaError_t launch_zero(void* ptr, size_t bytes, cudaStream_t s);
cudaError_t launch_wait_timeout_probe(int32_t* err, cudaStream_t s);
cudaError_t launch_prefill_rows(const PrefillRowsParams& p, cudaStream_t s);
cudaError_t launch_sample(const SampleParams& p, cudaStream_t s);
cudaError_t launch_counter_advance(uint64_t* counter, uint64_t by, cudaStream_t s);
// x_mode 0: bf16 input, 1: f32 input rounded to bf16, 2: bf16 of the RMS norm of an
// f32 input; epilogue 0: store f32, 1: add into f32 (residual), 2: SiLU-multiply to bf16.
// The pairs built are (2, 0), (1, 1), (2, 2) and (0, 1); B is 1..8.
cudaError_t launch_gemv_bf16(const GemvParams& p, int x_mode, int epilogue, cudaStream_t s);
// The same GEMVs on the tensor cores (gemv_mma.cu) for 1..kGemvMmaMaxB streams, K a
// multiple of 64.  The activations go in packed for the MMA, P[k / 8][slot][k % 8] bf16
// for gemv_mma_slots(B) stream slots: x_mode 0 takes p.x in that layout (what the
// SiLU-multiply epilogue writes, into p.y, y_stride unused); x_mode 1 (f32 rows) and 2
// (RMS norm of f32 rows times gamma) pack p.x into `xpack` (K x slots bf16, 16-byte
// aligned) with a small kernel launched first.
constexpr int kGemvMmaMaxB = 32;
int gemv_mma_slots(int B);
cudaError_t launch_gemv_mma(const GemvParams& p, int x_mode, int epilogue, void* xpack, cudaStream_t s);

// Multi-query prefill attention (prefill_attn.cu): blocks of 64 query rows (64 / G
// queries x the G q heads of a kv head) share every K/V tile of their causal window.
// Query row (b, t, h) reads q at q + (b * T + t) * q_stride + h * D (already normed and
// rotated) and sees cache rows [0, min(max(start[b] + t + 1, 1), capacity)).
constexpr int kPrefillMinT = 8;   // shorter prompts take the per-query decode path
constexpr int kPrefillTile = 64;  // cache rows of a K/V tile (both prefill kernels)
// Rows of each of an item's n_ch chunks: its window [0, nv_max) cut into n_ch parts of
// whole tiles (the last ones may be short or empty).  The window is known only on the
// device (start[] is a device array), so the attention and combine kernels both derive
// the cut from it, the same way.
__host__ __device__ inline int prefill_chunk_len(int nv_max, int n_ch) {
  const int per = (nv_max + n_ch - 1) / n_ch;
  return (per + kPrefillTile - 1) / kPrefillTile * kPrefillTile;
}
struct PrefillAttnParams {
  const float* q;               // the normed and rotated q rows (the rows launch's)
  int64_t q_stride;
  const int32_t* start;         // [B]
  int B, T, n_q_heads, n_kv_heads, capacity;
  int paged, page_size, n_pages, bt_stride;
  const int32_t* block_table;
  float scale_log2;             // scale * log2(e)
  float* out;                   // [B][T][Hq][D]
  float* part;                  // chunk rows [items][n_ch][rows][D] (n_ch > 1)
  float* ml;                    // their (max, sum) [items][n_ch][rows][2]
  int n_qb, n_ch;               // query blocks per (stream, kv head), chunks per item
  int rows;                     // query rows of an item: 64 (CUDA cores) or 128 (tensor cores)
  int merge_in_cluster;         // tensor cores, 1 < n_ch <= 8: an item's chunks form a cluster
                                // and merge there (set by the launcher)
  int32_t* err;
};
bool prefill_attn_supported(int head_dim, int group, int paged, int page_size, int T);
// The tensor-core form (prefill_attn_tc.cu): bf16 caches, head_dim 128, contiguous or
// pages of 64 rows or more; items of 128 query rows.
bool prefill_attn_tc_supported(int kv_bf16, int head_dim, int paged, int page_size);
int prefill_rows_per_item(int kv_bf16, int head_dim, int paged, int page_size);
void prefill_attn_plan(int B, int T, int n_kv_heads, int group, int capacity, int n_splits, int n_sm, int rows,
                       int& n_qb, int& n_ch);
size_t prefill_attn_workspace(int B, int T, int n_kv_heads, int group, int head_dim, int capacity, int n_splits,
                              int n_sm, int rows);
// Clusters of S (2..8) CTAs of the tensor-core kernel the current device keeps resident
// at once (0 if none or S is out of range).
int prefill_tc_active_clusters(int group, int S);
// Whether a tensor-core launch of `items` items in n_ch chunks merges them in clusters
// (2..8 chunks, every item's cluster resident at once).
bool prefill_tc_merges(int items, int group, int n_ch);
// *merged: the chunks were merged inside the launch (no combine launch needed).
cudaError_t launch_prefill_attn_tc(const PrefillAttnParams& p, const void* k_cache, const void* v_cache, int group,
                                   cudaStream_t s, bool* merged);
cudaError_t launch_prefill_attn(const PrefillAttnParams& p, const void* k_cache, const void* v_cache, bool kv_bf16,
                                int head_dim, int group, cudaStream_t s);

// Tile geometry of the attention kernel for a (dtype, head_dim) pair.
struct AttnGeometry {
  int tile_rows;     // positions per pipeline stage
  int max_stages;    // ring depth the kernel is compiled for
  int stage_bytes;   // K tile + V tile
  int threads;       // consumer warps + one producer warp
};
AttnGeometry attn_geometry(int kv_bf16, int head_dim);
cudaError_t launch_decode_attn(const AttnParams& p, int kv_bf16, int head_dim, int group,
                               bool fused, cudaStream_t s);

}  // namespace tts
