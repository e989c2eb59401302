// C ABI of the decode hot path: argument validation on the host, then kernel launches
// on the caller's stream.  Declarations and the full contract are in
// include/tts_decode.h.
#include <cmath>
#include <cstdint>
#include <cuda_runtime.h>

#include "kernels.h"

using namespace tts;

namespace {

bool aligned16(const void* p) { return (reinterpret_cast<uintptr_t>(p) & 15u) == 0; }
bool is_pow2(int x) { return x > 0 && (x & (x - 1)) == 0; }
int log2i(int x) {
  int s = 0;
  while ((1 << s) < x) ++s;
  return s;
}
cudaStream_t as_stream(void* s) { return static_cast<cudaStream_t>(s); }
tts_status from_cuda(cudaError_t e) { return e == cudaSuccess ? TTS_OK : TTS_ERR_CUDA; }

bool head_dim_ok(int d) { return d == 64 || d == 128; }
bool group_ok(int hq, int hkv) {
  if (hq <= 0 || hkv <= 0 || hq % hkv != 0) return false;
  const int g = hq / hkv;
  return g == 1 || g == 2 || g == 4;
}

int sm_count() {
  int dev = 0, n = 0;
  if (cudaGetDevice(&dev) != cudaSuccess) return 152;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) {
    cudaGetLastError();  // clear the sticky-free error this query may leave
    return 152;
  }
  return n;
}

tts_status check_desc(const tts_kv_desc* d) {
  if (d == nullptr) return TTS_ERR_NULL;
  if (d->B < 1 || d->capacity < 1 || !head_dim_ok(d->head_dim) || !group_ok(d->n_q_heads, d->n_kv_heads))
    return TTS_ERR_SHAPE;
  if (d->window_quantum < 1 || d->capacity % d->window_quantum != 0) return TTS_ERR_SHAPE;
  if (d->kv_dtype != TTS_F32 && d->kv_dtype != TTS_BF16) return TTS_ERR_DTYPE;
  if (d->paged != 0 && d->paged != 1) return TTS_ERR_LAYOUT;
  if (d->paged) {
    if (d->block_table == nullptr) return TTS_ERR_NULL;
    if (!is_pow2(d->page_size) || d->page_size > 256 || d->capacity % d->page_size != 0 ||
        d->n_pages < 1 || d->bt_stride < d->capacity / d->page_size)
      return TTS_ERR_LAYOUT;
  }
  return TTS_OK;
}

// Positions per split: a multiple of kSplitQuantum, covering capacity in n_splits
// pieces.  A split's last tile may be partial.
constexpr int kSplitQuantum = 16;
int split_len_for(const tts_kv_desc* d, int n_splits) {
  int per = (d->capacity + n_splits - 1) / n_splits;
  per = ((per + kSplitQuantum - 1) / kSplitQuantum) * kSplitQuantum;
  return per;
}

struct WsLayout {
  size_t o_off, ml_off, cnt_off, total;
};

size_t round256(size_t x) { return (x + 255) & ~static_cast<size_t>(255); }

WsLayout ws_layout(const tts_kv_desc* d, int n_splits) {
  WsLayout w;
  const size_t slots = static_cast<size_t>(d->B) * d->n_q_heads * n_splits;
  w.o_off = 0;
  w.ml_off = round256(slots * d->head_dim * sizeof(float));
  w.cnt_off = w.ml_off + round256(slots * 2 * sizeof(float));
  // split tickets [B][Hkv], then the persistent scheduler's two counters
  w.total = w.cnt_off + round256((static_cast<size_t>(d->B) * d->n_kv_heads + 2) * sizeof(int));
  return w;
}

// Splits actually launched for a requested count (0 = default): at most one per
// kSplitQuantum positions and at most kMaxSplits; each split covers split_len positions.
constexpr int kMaxSplits = 256;
tts_status resolve_splits(const tts_kv_desc* d, int32_t n_splits_req, int& split_len, int& used) {
  int n_splits = n_splits_req == 0 ? tts_decode_attn_default_splits(d) : n_splits_req;
  if (n_splits < 1) return TTS_ERR_SHAPE;
  const int max_splits = (d->capacity + kSplitQuantum - 1) / kSplitQuantum;
  if (n_splits > max_splits) n_splits = max_splits;
  if (n_splits > kMaxSplits) n_splits = kMaxSplits;
  split_len = split_len_for(d, n_splits);
  used = (d->capacity + split_len - 1) / split_len;
  return TTS_OK;
}

// Shared preparation of the attention launch (standalone and fused).
tts_status prepare_attn(const tts_kv_desc* d, const void* k_cache, const void* v_cache,
                        void* workspace, size_t ws_bytes, int32_t n_splits_req, AttnParams& p,
                        int& n_splits_out) {
  tts_status st = check_desc(d);
  if (st != TTS_OK) return st;
  if (k_cache == nullptr || v_cache == nullptr) return TTS_ERR_NULL;
  if (!aligned16(k_cache) || !aligned16(v_cache)) return TTS_ERR_ALIGN;
  int split_len = 0, used = 0;
  st = resolve_splits(d, n_splits_req, split_len, used);
  if (st != TTS_OK) return st;
  if (used > 65535 || d->n_kv_heads > 65535 || d->B > 65535) return TTS_ERR_SHAPE;
  if (used > 1) {
    const WsLayout w = ws_layout(d, used);
    if (workspace == nullptr) return TTS_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return TTS_ERR_ALIGN;
    if (ws_bytes < w.total) return TTS_ERR_WORKSPACE;
    unsigned char* ws = static_cast<unsigned char*>(workspace);
    p.ws_o = reinterpret_cast<float*>(ws + w.o_off);
    p.ws_ml = reinterpret_cast<float*>(ws + w.ml_off);
    p.ws_cnt = reinterpret_cast<int*>(ws + w.cnt_off);
    p.ws_sched = p.ws_cnt + static_cast<size_t>(d->B) * d->n_kv_heads;
  } else {
    p.ws_o = nullptr;
    p.ws_ml = nullptr;
    p.ws_cnt = nullptr;
    p.ws_sched = nullptr;
  }
  p.n_stages = 0;  // chosen by the launcher
  p.q_per_stream = 1;
  p.lens_add = 0;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.B = d->B;
  p.n_q_heads = d->n_q_heads;
  p.n_kv_heads = d->n_kv_heads;
  p.capacity = d->capacity;
  p.paged = d->paged;
  p.page_size = d->paged ? d->page_size : 1;
  p.page_shift = d->paged ? log2i(d->page_size) : 0;
  p.n_pages = d->paged ? d->n_pages : 0;
  p.bt_stride = d->paged ? d->bt_stride : 0;
  p.block_table = d->paged ? d->block_table : nullptr;
  p.flags = d->flags;
  p.n_splits = used;
  p.split_len = split_len;
  n_splits_out = used;
  return TTS_OK;
}

// Prompts of kPrefillMinT rows or more take the multi-query kernel (query blocks share
// every K/V tile); shorter ones run as B x T decode queries.
// Query rows of a multi-query prefill item: 128 on the tensor cores (bf16, head_dim 128,
// contiguous or pages of 64+ rows), else 64.
int prefill_rows(const tts_kv_desc* d) {
  return prefill_rows_per_item(d->kv_dtype == TTS_BF16, d->head_dim, d->paged, d->paged ? d->page_size : 1);
}

bool multi_query_prefill(const tts_kv_desc* d, int T) {
  const int64_t rows = d->paged ? static_cast<int64_t>(d->n_pages) * d->n_kv_heads * d->page_size
                                : static_cast<int64_t>(d->B) * d->n_kv_heads * d->capacity;
  return prefill_attn_supported(d->head_dim, d->n_q_heads / d->n_kv_heads, d->paged, d->paged ? d->page_size : 1, T) &&
         rows < (int64_t{1} << 31);
}

// The prefill workspace: the attention's own part (split or chunk partials), then the
// normed and rotated q rows [B T][Hq D] f32 at a 256-byte boundary (the caller's q rows
// are read only).
struct PrefillWs {
  size_t attn, q_off, total;
  bool q_rows;
};
PrefillWs prefill_ws(const tts_kv_desc* d, int T, int n_splits) {
  PrefillWs w;
  const bool mq = multi_query_prefill(d, T);
  if (mq) {
    w.attn = prefill_attn_workspace(d->B, T, d->n_kv_heads, d->n_q_heads / d->n_kv_heads, d->head_dim, d->capacity,
                                    n_splits, sm_count(), prefill_rows(d));
  } else {
    tts_kv_desc dq = *d;  // the B*T queries take the place of the streams
    dq.B = d->B * T;
    w.attn = tts_decode_attn_workspace_size(&dq, n_splits);
  }
  w.q_rows = true;
  w.q_off = round256(w.attn);
  w.total = w.q_rows ? w.q_off + round256(static_cast<size_t>(d->B) * T * d->n_q_heads * d->head_dim * 4) : w.attn;
  return w;
}

}  // namespace

extern "C" {

int32_t tts_abi_version(void) { return TTS_ABI_VERSION; }
int32_t tts_abi_min_version(void) { return TTS_ABI_MIN_VERSION; }
tts_status tts_abi_check(int32_t caller_version) {
  return (caller_version >= TTS_ABI_MIN_VERSION && caller_version <= TTS_ABI_VERSION) ? TTS_OK
                                                                                      : TTS_ERR_ABI;
}

const char* tts_status_str(int32_t s) {
  switch (s) {
    case TTS_OK: return "TTS_OK";
    case TTS_ERR_NULL: return "TTS_ERR_NULL";
    case TTS_ERR_SHAPE: return "TTS_ERR_SHAPE";
    case TTS_ERR_DTYPE: return "TTS_ERR_DTYPE";
    case TTS_ERR_LAYOUT: return "TTS_ERR_LAYOUT";
    case TTS_ERR_ALIGN: return "TTS_ERR_ALIGN";
    case TTS_ERR_WORKSPACE: return "TTS_ERR_WORKSPACE";
    case TTS_ERR_CUDA: return "TTS_ERR_CUDA";
    case TTS_ERR_ABI: return "TTS_ERR_ABI";
    default: return "TTS_ERR_UNKNOWN";
  }
}

tts_status tts_frame_embed(const tts_tables* t, const int32_t* ids, int64_t ids_stride,
                           const float* overlay, int64_t overlay_stride, float* out, int32_t B,
                           int32_t* err_flag, void* stream) {
  if (t == nullptr || ids == nullptr || out == nullptr) return TTS_ERR_NULL;
  if (t->n_tables < 1 || t->n_tables > TTS_MAX_TABLES || t->vocab < 1 || t->hidden < 4 ||
      t->hidden % 4 != 0 || B < 1 || B > 65535 || ids_stride < t->n_tables)
    return TTS_ERR_SHAPE;
  if (t->dtype != TTS_F32 && t->dtype != TTS_BF16 && t->dtype != TTS_Q8_0) return TTS_ERR_DTYPE;
  if (t->dtype == TTS_Q8_0 && t->hidden % 32 != 0) return TTS_ERR_SHAPE;
  EmbedParams p = {};
  p.tab_dtype = t->dtype;
  for (int i = 0; i < t->n_tables; ++i) {
    if (t->tab[i] == nullptr) return TTS_ERR_NULL;
    if (!aligned16(t->tab[i])) return TTS_ERR_ALIGN;
    p.tab[i] = t->tab[i];
  }
  if (!aligned16(out)) return TTS_ERR_ALIGN;
  if (overlay != nullptr && (!aligned16(overlay) || overlay_stride < t->hidden || overlay_stride % 4 != 0))
    return overlay_stride < t->hidden ? TTS_ERR_SHAPE : TTS_ERR_ALIGN;
  p.n_tables = t->n_tables;
  p.vocab = t->vocab;
  p.hidden = t->hidden;
  p.ids = ids;
  p.ids_stride = ids_stride;
  p.overlay = overlay;
  p.overlay_stride = overlay_stride;
  p.out = out;
  p.B = B;
  p.err = err_flag;
  return from_cuda(launch_frame_embed(p, as_stream(stream)));
}

tts_status tts_rope_table(float* cs, int32_t max_pos, int32_t head_dim, double base, void* stream) {
  if (cs == nullptr) return TTS_ERR_NULL;
  if (max_pos < 1 || !head_dim_ok(head_dim) || !(base > 1.0) || !std::isfinite(base)) return TTS_ERR_SHAPE;
  if (!aligned16(cs)) return TTS_ERR_ALIGN;
  return from_cuda(launch_rope_table(cs, max_pos, head_dim, base, as_stream(stream)));
}

tts_status tts_qk_norm_rope(float* q, int64_t q_row_stride, float* k, int64_t k_row_stride,
                            const float* gamma_q, const float* gamma_k, const int32_t* pos,
                            int32_t B, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                            float eps, const float* rope_cs, int32_t rope_max_pos,
                            int32_t* err_flag, void* stream) {
  if (q == nullptr || k == nullptr || gamma_q == nullptr || gamma_k == nullptr || pos == nullptr ||
      rope_cs == nullptr)
    return TTS_ERR_NULL;
  if (B < 1 || B > 65535 || !head_dim_ok(head_dim) || n_q_heads < 1 || n_kv_heads < 1 ||
      rope_max_pos < 1 || !(eps >= 0.f) || q_row_stride < static_cast<int64_t>(n_q_heads) * head_dim ||
      k_row_stride < static_cast<int64_t>(n_kv_heads) * head_dim)
    return TTS_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(gamma_q) || !aligned16(gamma_k) ||
      !aligned16(rope_cs) || q_row_stride % 4 != 0 || k_row_stride % 4 != 0)
    return TTS_ERR_ALIGN;
  NormRopeParams p = {q, q_row_stride, k, k_row_stride, gamma_q, gamma_k, pos, B, n_q_heads,
                      n_kv_heads, head_dim, eps, reinterpret_cast<const float2*>(rope_cs),
                      rope_max_pos, err_flag};
  return from_cuda(launch_qk_norm_rope(p, as_stream(stream)));
}

tts_status tts_kv_set_rows(const float* k, const float* v, int64_t kv_row_stride, void* k_cache,
                           void* v_cache, const tts_kv_desc* d, const int32_t* dst_pos,
                           int32_t* err_flag, void* stream) {
  tts_status st = check_desc(d);
  if (st != TTS_OK) return st;
  if (k == nullptr || v == nullptr || k_cache == nullptr || v_cache == nullptr || dst_pos == nullptr)
    return TTS_ERR_NULL;
  if (kv_row_stride < static_cast<int64_t>(d->n_kv_heads) * d->head_dim) return TTS_ERR_SHAPE;
  if (!aligned16(k) || !aligned16(v) || !aligned16(k_cache) || !aligned16(v_cache) || kv_row_stride % 4 != 0)
    return TTS_ERR_ALIGN;
  SetRowsParams p = {};
  p.k = k;
  p.v = v;
  p.row_stride = kv_row_stride;
  p.k_cache = k_cache;
  p.v_cache = v_cache;
  p.B = d->B;
  p.n_kv_heads = d->n_kv_heads;
  p.head_dim = d->head_dim;
  p.capacity = d->capacity;
  p.kv_bf16 = d->kv_dtype == TTS_BF16;
  p.paged = d->paged;
  p.page_size = d->paged ? d->page_size : 1;
  p.n_pages = d->n_pages;
  p.bt_stride = d->bt_stride;
  p.block_table = d->block_table;
  p.pos = dst_pos;
  p.err = err_flag;
  return from_cuda(launch_set_rows(p, as_stream(stream)));
}

int32_t tts_decode_attn_default_splits(const tts_kv_desc* d) {
  if (check_desc(d) != TTS_OK) return 1;
  const AttnGeometry geo = attn_geometry(d->kv_dtype == TTS_BF16, d->head_dim);
  const int max_splits = (d->capacity + geo.tile_rows - 1) / geo.tile_rows;
  const int pairs = d->B * d->n_kv_heads;
  const int sms = sm_count();
  int s;
  if (pairs <= 16) {
    // Few (stream, kv head) pairs: about two CTAs per SM over the grid.
    s = (2 * sms + pairs - 1) / pairs;
  } else {
    // Many pairs: windows cut into pieces of at most 512 positions (ragged batches
    // balance; the partials merge through the workspace).
    s = (d->capacity + 511) / 512;
  }
  if (s < 1) s = 1;
  if (s > max_splits) s = max_splits;
  if (s < 1) s = 1;
  return s;
}

size_t tts_decode_attn_workspace_size(const tts_kv_desc* d, int32_t n_splits) {
  if (check_desc(d) != TTS_OK) return 0;
  int split_len = 0, used = 0;
  if (resolve_splits(d, n_splits, split_len, used) != TTS_OK) return 0;
  return ws_layout(d, used).total;
}

tts_status tts_workspace_init(void* workspace, size_t ws_bytes, void* stream) {
  if (workspace == nullptr) return TTS_ERR_NULL;
  if (!aligned16(workspace)) return TTS_ERR_ALIGN;
  return from_cuda(launch_zero(workspace, ws_bytes & ~static_cast<size_t>(15), as_stream(stream)));
}

tts_status tts_decode_attn(const float* q, int64_t q_row_stride, const void* k_cache,
                           const void* v_cache, const tts_kv_desc* d, const int32_t* n_valid,
                           float scale, float* out, void* workspace, size_t ws_bytes,
                           int32_t n_splits, int32_t* err_flag, void* stream) {
  if (q == nullptr || n_valid == nullptr || out == nullptr) return TTS_ERR_NULL;
  AttnParams p = {};
  int used = 0;
  tts_status st = prepare_attn(d, k_cache, v_cache, workspace, ws_bytes, n_splits, p, used);
  if (st != TTS_OK) return st;
  if (q_row_stride < static_cast<int64_t>(d->n_q_heads) * d->head_dim) return TTS_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(out) || q_row_stride % 4 != 0) return TTS_ERR_ALIGN;
  if (!std::isfinite(scale)) return TTS_ERR_SHAPE;
  p.q = q;
  p.q_stride = q_row_stride;
  p.lens = n_valid;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.out = out;
  p.err = err_flag;
  p.flags &= ~TTS_KV_PREFETCH_BEFORE_WAIT;  // only meaningful for the fused step
  return from_cuda(launch_decode_attn(p, d->kv_dtype == TTS_BF16, d->head_dim,
                                      d->n_q_heads / d->n_kv_heads, false, as_stream(stream)));
}

}  // extern "C"

namespace {

// The fused step; with `packed` non-null the output goes there instead of `out`, rounded to
// bf16 in the tensor-core projection's input layout [Hq D / 8][slots][8] (the decode layer's
// o projection then reads it without a packing launch).
tts_status decode_step_impl(const float* q, const float* k, const float* v, int64_t row_stride,
                            const float* gamma_q, const float* gamma_k, float eps,
                            const float* rope_cs, int32_t rope_max_pos, void* k_cache,
                            void* v_cache, const tts_kv_desc* d, const int32_t* cur_len,
                            float scale, float* out, __nv_bfloat16* packed, int slots, void* workspace,
                            size_t ws_bytes, int32_t n_splits, int32_t* err_flag, void* stream) {
  if (q == nullptr || k == nullptr || v == nullptr || gamma_q == nullptr || gamma_k == nullptr ||
      rope_cs == nullptr || cur_len == nullptr || (out == nullptr && packed == nullptr))
    return TTS_ERR_NULL;
  AttnParams p = {};
  int used = 0;
  tts_status st = prepare_attn(d, k_cache, v_cache, workspace, ws_bytes, n_splits, p, used);
  if (st != TTS_OK) return st;
  if (row_stride < static_cast<int64_t>(d->n_q_heads) * d->head_dim || rope_max_pos < 1 || !(eps >= 0.f))
    return TTS_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(packed) ||
      !aligned16(gamma_q) || !aligned16(gamma_k) || !aligned16(rope_cs) || row_stride % 4 != 0)
    return TTS_ERR_ALIGN;
  if (!std::isfinite(scale)) return TTS_ERR_SHAPE;
  p.q = q;
  p.q_stride = row_stride;
  p.k_new = k;
  p.v_new = v;
  p.kv_new_stride = row_stride;
  p.gamma_q = gamma_q;
  p.gamma_k = gamma_k;
  p.eps = eps;
  p.cs = reinterpret_cast<const float2*>(rope_cs);
  p.max_pos = rope_max_pos;
  p.k_cache_w = k_cache;
  p.v_cache_w = v_cache;
  p.lens = cur_len;
  p.scale_log2 = scale * 1.4426950408889634f;
  p.out = out;
  p.out_packed = packed;
  p.out_slots = slots;
  p.err = err_flag;
  return from_cuda(launch_decode_attn(p, d->kv_dtype == TTS_BF16, d->head_dim,
                                      d->n_q_heads / d->n_kv_heads, true, as_stream(stream)));
}

}  // namespace

extern "C" {

tts_status tts_decode_step(const float* q, const float* k, const float* v, int64_t row_stride,
                           const float* gamma_q, const float* gamma_k, float eps,
                           const float* rope_cs, int32_t rope_max_pos, void* k_cache,
                           void* v_cache, const tts_kv_desc* d, const int32_t* cur_len,
                           float scale, float* out, void* workspace, size_t ws_bytes,
                           int32_t n_splits, int32_t* err_flag, void* stream) {
  if (out == nullptr) return TTS_ERR_NULL;
  return decode_step_impl(q, k, v, row_stride, gamma_q, gamma_k, eps, rope_cs, rope_max_pos, k_cache, v_cache, d,
                          cur_len, scale, out, nullptr, 0, workspace, ws_bytes, n_splits, err_flag, stream);
}

size_t tts_prefill_workspace_size(const tts_kv_desc* d, int32_t T, int32_t n_splits) {
  if (check_desc(d) != TTS_OK || T < 1 || static_cast<int64_t>(d->B) * T > 65535) return 0;
  const size_t w = prefill_ws(d, T, n_splits).total;
  return w > 256 ? w : 256;
}

int32_t tts_prefill_launch_count(const tts_kv_desc* d, int32_t T, int32_t n_splits) {
  if (check_desc(d) != TTS_OK || T < 1 || static_cast<int64_t>(d->B) * T > 65535) return 0;
  if (!multi_query_prefill(d, T)) return 2;
  const int rows = prefill_rows(d), group = d->n_q_heads / d->n_kv_heads;
  int n_qb = 0, n_ch = 0;
  prefill_attn_plan(d->B, T, d->n_kv_heads, group, d->capacity, n_splits, sm_count(), rows, n_qb, n_ch);
  if (n_ch == 1) return 2;
  const bool merged = rows == 128 && prefill_tc_merges(d->B * d->n_kv_heads * n_qb, group, n_ch);
  return merged ? 2 : 3;
}

tts_status tts_prefill_step(const float* q, const float* k, const float* v, int64_t row_stride,
                            const float* gamma_q, const float* gamma_k, float eps,
                            const float* rope_cs, int32_t rope_max_pos, void* k_cache,
                            void* v_cache, const tts_kv_desc* d, const int32_t* start_pos,
                            int32_t T, float scale, float* out, void* workspace, size_t ws_bytes,
                            int32_t n_splits, int32_t* err_flag, void* stream) {
  if (q == nullptr || k == nullptr || v == nullptr || gamma_q == nullptr || gamma_k == nullptr ||
      rope_cs == nullptr || start_pos == nullptr || out == nullptr || d == nullptr)
    return TTS_ERR_NULL;
  tts_status st = check_desc(d);
  if (st != TTS_OK) return st;
  if (T < 1 || static_cast<int64_t>(d->B) * T > 65535) return TTS_ERR_SHAPE;
  const bool mq = multi_query_prefill(d, T);
  tts_kv_desc dq = *d;
  dq.B = d->B * T;
  AttnParams p = {};
  int used = 0;
  PrefillAttnParams pp = {};
  const PrefillWs pw = prefill_ws(d, T, n_splits);
  float* q_rows = nullptr;  // the normed q rows, for the paths that read them from memory
  if (pw.q_rows) {
    if (workspace == nullptr) return TTS_ERR_WORKSPACE;
    if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return TTS_ERR_ALIGN;
    if (ws_bytes < pw.total) return TTS_ERR_WORKSPACE;
    q_rows = reinterpret_cast<float*>(static_cast<unsigned char*>(workspace) + pw.q_off);
  }
  if (mq) {
    if (k_cache == nullptr || v_cache == nullptr) return TTS_ERR_NULL;
    if (!aligned16(k_cache) || !aligned16(v_cache)) return TTS_ERR_ALIGN;
    pp.rows = prefill_rows(d);
    prefill_attn_plan(d->B, T, d->n_kv_heads, d->n_q_heads / d->n_kv_heads, d->capacity, n_splits, sm_count(),
                      pp.rows, pp.n_qb, pp.n_ch);
    if (pp.n_ch > 65535) return TTS_ERR_SHAPE;
    if (pp.n_ch > 1) {
      const size_t need = prefill_attn_workspace(d->B, T, d->n_kv_heads, d->n_q_heads / d->n_kv_heads, d->head_dim,
                                                 d->capacity, n_splits, sm_count(), pp.rows);
      if (workspace == nullptr) return TTS_ERR_WORKSPACE;
      if ((reinterpret_cast<uintptr_t>(workspace) & 255u) != 0) return TTS_ERR_ALIGN;
      if (ws_bytes < need) return TTS_ERR_WORKSPACE;
      const size_t rows = static_cast<size_t>(d->B) * d->n_kv_heads * pp.n_qb * pp.n_ch * pp.rows;
      pp.part = static_cast<float*>(workspace);
      pp.ml = pp.part + rows * d->head_dim;
    }
  } else {
    st = prepare_attn(&dq, k_cache, v_cache, workspace, ws_bytes, n_splits, p, used);
    if (st != TTS_OK) return st;
  }
  if (row_stride < static_cast<int64_t>(d->n_q_heads) * d->head_dim || rope_max_pos < 1 || !(eps >= 0.f))
    return TTS_ERR_SHAPE;
  if (!aligned16(q) || !aligned16(k) || !aligned16(v) || !aligned16(out) || !aligned16(gamma_q) ||
      !aligned16(gamma_k) || !aligned16(rope_cs) || row_stride % 4 != 0)
    return TTS_ERR_ALIGN;
  if (!std::isfinite(scale)) return TTS_ERR_SHAPE;
  cudaStream_t s = as_stream(stream);
  PrefillRowsParams rp = {};
  rp.q = q;
  rp.q_out = q_rows;
  rp.k = k;
  rp.v = v;
  rp.row_stride = row_stride;
  rp.gamma_q = gamma_q;
  rp.gamma_k = gamma_k;
  rp.eps = eps;
  rp.cs = reinterpret_cast<const float2*>(rope_cs);
  rp.max_pos = rope_max_pos;
  rp.k_cache = k_cache;
  rp.v_cache = v_cache;
  rp.B = d->B;
  rp.T = T;
  rp.n_q_heads = d->n_q_heads;
  rp.n_kv_heads = d->n_kv_heads;
  rp.head_dim = d->head_dim;
  rp.capacity = d->capacity;
  rp.kv_bf16 = d->kv_dtype == TTS_BF16;
  rp.paged = d->paged;
  rp.page_size = d->paged ? d->page_size : 1;
  rp.n_pages = d->paged ? d->n_pages : 0;
  rp.bt_stride = d->paged ? d->bt_stride : 0;
  rp.block_table = d->paged ? d->block_table : nullptr;
  rp.start = start_pos;
  rp.err = err_flag;
  st = from_cuda(launch_prefill_rows(rp, s));
  if (st != TTS_OK) return st;
  if (mq) {
    pp.q = q_rows;
    pp.q_stride = static_cast<int64_t>(d->n_q_heads) * d->head_dim;
    pp.start = start_pos;
    pp.B = d->B;
    pp.T = T;
    pp.n_q_heads = d->n_q_heads;
    pp.n_kv_heads = d->n_kv_heads;
    pp.capacity = d->capacity;
    pp.paged = d->paged;
    pp.page_size = d->paged ? d->page_size : 1;
    pp.n_pages = d->paged ? d->n_pages : 0;
    pp.bt_stride = d->paged ? d->bt_stride : 0;
    pp.block_table = d->paged ? d->block_table : nullptr;
    pp.scale_log2 = scale * 1.4426950408889634f;
    pp.out = out;
    pp.err = err_flag;
    return from_cuda(launch_prefill_attn(pp, k_cache, v_cache, d->kv_dtype == TTS_BF16, d->head_dim,
                                         d->n_q_heads / d->n_kv_heads, s));
  }
  p.q = q_rows;
  p.q_stride = static_cast<int64_t>(d->n_q_heads) * d->head_dim;
  p.lens = start_pos;
  p.q_per_stream = T;
  p.lens_add = 1;  // query t's window is [0, start + t + 1)
  p.scale_log2 = scale * 1.4426950408889634f;
  p.out = out;
  p.err = err_flag;
  p.flags &= ~TTS_KV_PREFETCH_BEFORE_WAIT;  // the rows launch writes the cache
  return from_cuda(launch_decode_attn(p, d->kv_dtype == TTS_BF16, d->head_dim,
                                      d->n_q_heads / d->n_kv_heads, false, s));
}

tts_status tts_sample(const float* logits, int64_t logits_stride, int32_t B, int32_t vocab,
                      int32_t top_k, float temperature, uint64_t seed, const uint64_t* counter,
                      uint32_t draw, int32_t* out_ids, int64_t out_stride, void* stream) {
  if (logits == nullptr || out_ids == nullptr || (top_k > 1 && counter == nullptr)) return TTS_ERR_NULL;
  if (B < 1 || B > 65535 || vocab < 1 || vocab > TTS_MAX_SAMPLE_VOCAB || logits_stride < vocab ||
      out_stride < 1 || top_k < 0 || top_k > TTS_MAX_TOP_K || top_k > vocab)
    return TTS_ERR_SHAPE;
  if (top_k > 1 && !(temperature > 0.f && std::isfinite(temperature))) return TTS_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(logits) & 3u) != 0 || (reinterpret_cast<uintptr_t>(out_ids) & 3u) != 0 ||
      (counter != nullptr && (reinterpret_cast<uintptr_t>(counter) & 7u) != 0))
    return TTS_ERR_ALIGN;
  SampleParams p = {};
  p.logits = logits;
  p.stride = logits_stride;
  p.B = B;
  p.V = vocab;
  p.top_k = top_k;
  p.c = top_k > 1 ? static_cast<float>(1.4426950408889634 / static_cast<double>(temperature)) : 0.f;
  p.seed = seed;
  p.counter = counter;
  p.draw = draw;
  p.out = out_ids;
  p.out_stride = out_stride;
  return from_cuda(launch_sample(p, as_stream(stream)));
}

tts_status tts_sample_embed(const float* logits, int64_t logits_stride, int32_t B, int32_t vocab,
                            int32_t top_k, float temperature, uint64_t seed, const uint64_t* counter,
                            uint32_t draw, int32_t* out_ids, int64_t out_stride, const tts_tables* table,
                            float* out_rows, void* stream) {
  if (logits == nullptr || out_ids == nullptr || (top_k > 1 && counter == nullptr) || table == nullptr ||
      out_rows == nullptr || table->tab[0] == nullptr)
    return TTS_ERR_NULL;
  if (B < 1 || B > 65535 || vocab < 1 || vocab > TTS_MAX_SAMPLE_VOCAB || logits_stride < vocab ||
      out_stride < 1 || top_k < 0 || top_k > TTS_MAX_TOP_K || top_k > vocab)
    return TTS_ERR_SHAPE;
  if (top_k > 1 && !(temperature > 0.f && std::isfinite(temperature))) return TTS_ERR_SHAPE;
  if (table->n_tables != 1 || table->vocab < vocab || table->hidden < 4 || table->hidden % 4 != 0)
    return TTS_ERR_SHAPE;
  if (table->dtype != TTS_F32 && table->dtype != TTS_BF16 && table->dtype != TTS_Q8_0) return TTS_ERR_DTYPE;
  if (table->dtype == TTS_Q8_0 && table->hidden % 32 != 0) return TTS_ERR_SHAPE;
  if ((reinterpret_cast<uintptr_t>(logits) & 3u) != 0 || (reinterpret_cast<uintptr_t>(out_ids) & 3u) != 0 ||
      (counter != nullptr && (reinterpret_cast<uintptr_t>(counter) & 7u) != 0) || !aligned16(table->tab[0]) ||
      !aligned16(out_rows))
    return TTS_ERR_ALIGN;
  SampleParams p = {};
  p.logits = logits;
  p.stride = logits_stride;
  p.B = B;
  p.V = vocab;
  p.top_k = top_k;
  p.c = top_k > 1 ? static_cast<float>(1.4426950408889634 / static_cast<double>(temperature)) : 0.f;
  p.seed = seed;
  p.counter = counter;
  p.draw = draw;
  p.out = out_ids;
  p.out_stride = out_stride;
  p.emb_tab = table->tab[0];
  p.emb_dtype = table->dtype;
  p.emb_hidden = table->hidden;
  p.emb_out = out_rows;
  return from_cuda(launch_sample(p, as_stream(stream)));
}

tts_status tts_counter_advance(uint64_t* counter, uint64_t by, void* stream) {
  if (counter == nullptr) return TTS_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(counter) & 7u) != 0) return TTS_ERR_ALIGN;
  return from_cuda(launch_counter_advance(counter, by, as_stream(stream)));
}

tts_status tts_check_wait_timeout(int32_t* err_flag, void* stream) {
  if (err_flag == nullptr) return TTS_ERR_NULL;
  if ((reinterpret_cast<uintptr_t>(err_flag) & 3u) != 0) return TTS_ERR_ALIGN;
  return from_cuda(launch_wait_timeout_probe(err_flag, as_stream(stream)));
}

}  // extern "C"

namespace {

// From this many streams on the layer's projections run on the tensor cores (default:
// always; their 64 KB tensor-map stages stream the weights faster than the CUDA-core
// GEMVs of layer.cu even at one stream, where 15 of the MMA's 16 columns are padding).
// A build with a larger value keeps the CUDA-core GEMVs below it.
#ifndef TTS_MMA_MIN_STREAMS
#define TTS_MMA_MIN_STREAMS 1
#endif
constexpr int kMmaMinStreams = TTS_MMA_MIN_STREAMS;

// Scratch of a decode layer, 256-byte regions: a (the SiLU-multiply output, bf16: [B][inter]
// rows below kMmaMinStreams streams, else packed for the tensor-core down projection,
// [inter / 8][slots][8]), the qkv rows (f32), the attention output (f32 [B][Hq D]), the
// attention workspace, then (from kMmaMinStreams streams on) the packed activations of
// the other three projections (bf16, max(hidden, Hq D) x slots).
struct LayerScratch {
  size_t a_off, qkv_off, attn_off, ws_off, xp_off, total;
};
LayerScratch layer_scratch(const tts_kv_desc* d, int hidden, int inter, int n_splits) {
  LayerScratch L;
  const bool mma = d->B >= kMmaMinStreams;
  const size_t B = static_cast<size_t>(d->B);
  const size_t rows = mma ? static_cast<size_t>(gemv_mma_slots(d->B)) : B;
  const int qd = d->n_q_heads * d->head_dim;
  const int width = (d->n_q_heads + 2 * d->n_kv_heads) * d->head_dim;
  L.a_off = 0;
  L.qkv_off = round256(rows * inter * 2);
  L.attn_off = L.qkv_off + round256(B * width * 4);
  L.ws_off = L.attn_off + round256(B * qd * 4);
  L.xp_off = L.ws_off + round256(tts_decode_attn_workspace_size(d, n_splits));
  const size_t kx = static_cast<size_t>(hidden > qd ? hidden : qd);
  L.total = L.xp_off + (mma ? round256(rows * kx * 2) : 0);
  return L;
}

bool layer_dim_ok(int n) { return n >= 256 && n <= kGemvMaxK && n % 256 == 0; }

}  // namespace

extern "C" {

size_t tts_decode_layer_scratch_size(const tts_kv_desc* d, int32_t hidden, int32_t inter,
                                     int32_t n_splits) {
  if (check_desc(d) != TTS_OK || !layer_dim_ok(hidden) || !layer_dim_ok(inter)) return 0;
  return layer_scratch(d, hidden, inter, n_splits).total;
}

int32_t tts_decode_layer_launch_count(const tts_kv_desc* d) {
  if (check_desc(d) != TTS_OK || d->B > kGemvMmaMaxB) return 0;
  // tensor cores: two norm packs, four projections, the decode step; CUDA cores: the
  // projections norm their own inputs
  return d->B >= kMmaMinStreams ? 7 : 5;
}

tts_status tts_decode_layer(float* h, const tts_layer_weights* w, float eps, const float* rope_cs,
                            int32_t rope_max_pos, void* k_cache, void* v_cache, const tts_kv_desc* d,
                            const int32_t* cur_len, float scale, void* scratch, size_t scratch_bytes,
                            int32_t n_splits, int32_t* err_flag, void* stream) {
  if (h == nullptr || w == nullptr || d == nullptr || scratch == nullptr || w->w_qkv == nullptr ||
      w->w_o == nullptr || w->w_gu == nullptr || w->w_down == nullptr || w->gamma_attn == nullptr ||
      w->gamma_mlp == nullptr)
    return TTS_ERR_NULL;
  tts_status st = check_desc(d);
  if (st != TTS_OK) return st;
  const int H = w->hidden, I = w->inter, B = d->B;
  const int qd = d->n_q_heads * d->head_dim;
  const int kd = d->n_kv_heads * d->head_dim;
  const int width = qd + 2 * kd;
  if (B > kGemvMmaMaxB || !layer_dim_ok(H) || !layer_dim_ok(I) || !layer_dim_ok(qd) || !(eps >= 0.f))
    return TTS_ERR_SHAPE;
  if (!aligned16(h) || !aligned16(w->w_qkv) || !aligned16(w->w_o) || !aligned16(w->w_gu) ||
      !aligned16(w->w_down) || !aligned16(w->gamma_attn) || !aligned16(w->gamma_mlp) ||
      (reinterpret_cast<uintptr_t>(scratch) & 255u) != 0)
    return TTS_ERR_ALIGN;
  const LayerScratch L = layer_scratch(d, H, I, n_splits);
  if (scratch_bytes < L.total) return TTS_ERR_WORKSPACE;
  unsigned char* sc = static_cast<unsigned char*>(scratch);
  void* a = sc + L.a_off;
  float* qkv = reinterpret_cast<float*>(sc + L.qkv_off);
  float* attn = reinterpret_cast<float*>(sc + L.attn_off);
  cudaStream_t s = as_stream(stream);
  // from kMmaMinStreams streams on the tensor-core GEMV; below it (a build option) the
  // ring GEMV for one stream and the register GEMV for more
  auto gemv = [&](const GemvParams& g, int x_mode, int epilogue) -> cudaError_t {
    if (B >= kMmaMinStreams) return launch_gemv_mma(g, x_mode, epilogue, sc + L.xp_off, s);
    return launch_gemv_bf16(g, x_mode, epilogue, s);
  };
  // qkv = bf16(rmsnorm(h)) W_qkv^T
  GemvParams g = {};
  g.x = h; g.x_stride = H; g.gamma = w->gamma_attn; g.eps = eps;
  g.w = w->w_qkv; g.n_out = width; g.K = H; g.B = B; g.y = qkv; g.y_stride = width; g.err = err_flag;
  cudaError_t e = gemv(g, 2, 0);
  if (e != cudaSuccess) return from_cuda(e);
  // One stream: the qkv GEMV's CTAs hold one slot of every SM while the attention's
  // first CTAs start, so about 1.4 attention CTAs per SM (fewer, longer splits than the
  // standalone default of about two) finish the layer sooner.
  int32_t splits = n_splits;
  if (splits == 0 && B == 1) {
    const int pairs = d->n_kv_heads;
    splits = (7 * sm_count() + 5 * pairs - 1) / (5 * pairs);
    const int standalone = tts_decode_attn_default_splits(d);
    if (splits > standalone) splits = standalone;
  }
  // on the tensor-core path the attention writes its output already packed for the o
  // projection (bf16, the projection's input layout), so that projection needs no pack
  const bool packed = B >= kMmaMinStreams;
  __nv_bfloat16* xp = reinterpret_cast<__nv_bfloat16*>(sc + L.xp_off);
  st = decode_step_impl(qkv, qkv + qd, qkv + qd + kd, width, w->gamma_q, w->gamma_k, eps, rope_cs,
                        rope_max_pos, k_cache, v_cache, d, cur_len, scale, packed ? nullptr : attn,
                        packed ? xp : nullptr, packed ? gemv_mma_slots(B) : 0, sc + L.ws_off,
                        L.total - L.ws_off, splits, err_flag, stream);
  if (st != TTS_OK) return st;
  // h += bf16(attn) W_o^T
  g = {};
  g.x = packed ? static_cast<const void*>(xp) : attn; g.x_stride = qd; g.w = w->w_o; g.n_out = H; g.K = qd;
  g.B = B; g.y = h; g.y_stride = H; g.err = err_flag;
  if ((e = gemv(g, packed ? 0 : 1, 1)) != cudaSuccess) return from_cuda(e);
  // a = bf16(silu(x W_gate^T) * x W_up^T), x = bf16(rmsnorm(h))
  g = {};
  g.x = h; g.x_stride = H; g.gamma = w->gamma_mlp; g.eps = eps;
  g.w = w->w_gu; g.n_out = I; g.K = H; g.B = B; g.inter = I; g.y = a; g.y_stride = I; g.err = err_flag;
  if ((e = gemv(g, 2, 2)) != cudaSuccess) return from_cuda(e);
  // h += a W_down^T
  g = {};
  g.x = a; g.x_stride = I; g.w = w->w_down; g.n_out = H; g.K = I; g.B = B; g.y = h; g.y_stride = H;
  g.err = err_flag;
  return from_cuda(gemv(g, 0, 1));
}

}  // extern "C"
