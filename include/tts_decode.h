/*
 * tts_decode.h -- C ABI of the GB300 (sm_103a) per-frame decode hot path of a
 * multi-codebook autoregressive TTS transformer (talker + 16-slot code predictor).
 *
 * The operations and where they are defined (page titles as printed on the pages):
 *   [P-pipeline] "qwentts.cpp ... src/pipeline-tts.h" commit page
 *       - fixed-topology section: KV writes through set_rows with the destination rows
 *         carried as data, so every decode graph keeps fixed tensor addresses; per
 *         frame the host uploads 16 code ids and one overlay row and reads back only
 *         results;
 *       - on-device AR input assembly section: the talker gathers and sums the 16 frame
 *         code embeddings plus the trailing text/pad overlay; the code predictor
 *         gathers c0 and each sampled sub-code from its own group table;
 *       - persistent-arenas section: talker attention window padded to 256, predictor
 *         window fixed to the frame cache size, causal mask carrying -inf over the
 *         padded tail;
 *       - KV-cache section: a per-layer K/V buffer sized at init (talker 4096
 *         positions, predictor 16 positions reset every frame); decode appends one
 *         position and reads the [0, cur_len+1) window; the predictor runs a T=2
 *         prefill then 14 single-token decodes.
 *   [P-engine] "minicpm-o-4.5-single-gpu-engine ... docs/optimizations.md",
 *       core-optimisation table: fused q/k norm + RoPE kernels, integer
 *       round-to-nearest-even rounding, paged KV per model; "Lean Talker frame"
 *       option row: q/k/v read as strided views of one projection output.
 *
 * Conventions shared by every call
 *   - Every buffer pointer is a DEVICE pointer owned by the caller (allocated, e.g.,
 *     through PyTorch).  The library never allocates device memory and keeps no state
 *     between calls; descriptor structs are read on the host during the call only.
 *   - `stream` is a cudaStream_t passed as void* (NULL = the legacy default stream).
 *     Every call is asynchronous and stream-ordered; the launch configuration depends
 *     only on shapes and capacity, never on device data such as cur_len, so a
 *     sequence of calls can be captured in a CUDA graph and replayed with fixed
 *     addresses.
 *   - Kernels are launched with programmatic stream serialisation: a call touches its
 *     inputs only after the work enqueued before it on the stream has finished (its
 *     first kernel waits for the previous kernel; a later kernel of the same call may
 *     read the call's inputs as soon as that wait is behind it); one documented opt-in
 *     exception, TTS_KV_PREFETCH_BEFORE_WAIT below.
 *   - The returned tts_status reports errors found on the host, before any launch
 *     (null pointers, bad shapes, misalignment, short workspace, launch failure).
 *     Nothing is launched when it is not TTS_OK.
 *   - Errors only visible on the device (a code id outside the table, a position
 *     outside the cache, a bad page id, an n_valid outside [1, capacity], a bounded
 *     wait that ran out) never trap: the offending index is clamped or the write is
 *     skipped as stated per call, and a bit (TTS_EFLAG_*) is OR-ed into the caller's
 *     int32 `err_flag` (device memory; may be NULL to ignore).  Read it after the
 *     stream synchronises; clear it yourself.
 *   - Alignment: every device pointer must be 16-byte aligned; row strides are given
 *     in elements and must keep each row 16-byte aligned (a multiple of 4 floats).
 *   - head_dim is 64 or 128; n_q_heads / n_kv_heads (the GQA group) is 1, 2 or 4.
 */
#ifndef TTS_DECODE_H
#define TTS_DECODE_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

/* ABI version range (the ABI-bump section of the "qwentts.cpp ... commits/branch/
 * master/tests" page: a version range checked by a probe whose two bounds both
 * reject).  A caller built against version V may use this library iff
 * tts_abi_min_version() <= V <= tts_abi_version(); tts_abi_check(V) makes that test
 * inside the library and returns TTS_OK, or TTS_ERR_ABI for a V below the minimum or
 * above the current version.  (ABI 2 added tts_tables.dtype; ABI 3 added the `draw`
 * argument of tts_sample, tts_abi_check and Q8_0 codebook tables.) */
#define TTS_ABI_VERSION 3
#define TTS_ABI_MIN_VERSION 3
int32_t tts_abi_version(void);
int32_t tts_abi_min_version(void);

typedef enum {
  TTS_OK = 0,
  TTS_ERR_NULL = 1,       /* a required pointer is NULL */
  TTS_ERR_SHAPE = 2,      /* a size or head count outside the supported set */
  TTS_ERR_DTYPE = 3,      /* unknown dtype code */
  TTS_ERR_LAYOUT = 4,     /* inconsistent cache layout (page size, pool, strides) */
  TTS_ERR_ALIGN = 5,      /* a pointer or stride breaks the 16-byte rule */
  TTS_ERR_WORKSPACE = 6,  /* workspace NULL or smaller than required */
  TTS_ERR_CUDA = 7,       /* the CUDA runtime refused the launch */
  TTS_ERR_ABI = 8         /* a caller ABI version outside the supported range */
} tts_status;

/* Human-readable name of a status code (static string). */
const char* tts_status_str(int32_t status);

/* TTS_OK iff tts_abi_min_version() <= caller_version <= tts_abi_version(), else
 * TTS_ERR_ABI.  Pass the TTS_ABI_VERSION of the header the caller was built with. */
tts_status tts_abi_check(int32_t caller_version);

/* Device-side error bits OR-ed into *err_flag. */
#define TTS_EFLAG_ID_RANGE 1    /* code id outside [0, vocab): clamped into range   */
#define TTS_EFLAG_POS_RANGE 2   /* position outside the cache/RoPE table: see call  */
#define TTS_EFLAG_PAGE 4        /* block-table entry outside [0, n_pages): see call */
#define TTS_EFLAG_NVALID 8      /* n_valid outside [1, capacity]: clamped into it   */
#define TTS_EFLAG_TIMEOUT 16    /* a bounded in-kernel wait ran out; output invalid;
                                   re-zero the call's workspace before its next use */

/* Element types.  KV caches: f32 or bf16.  Codebook tables: f32, bf16 or Q8_0. */
typedef enum { TTS_F32 = 0, TTS_BF16 = 1, TTS_Q8_0 = 2 } tts_dtype;

#define TTS_MAX_TABLES 16

/* Codebook tables for the frame-input composition.  tab[g] points to a dense row-major
 * table of `vocab` rows of `hidden` entries of element type `dtype` ([P-pipeline] TTFA /
 * prompt-build section: the tables are gathered whatever their type, "any quant via
 * get_rows"; its TTFA measurements use Q8_0 tables); only the first n_tables entries
 * are read.
 *   TTS_F32:  4 bytes an entry.
 *   TTS_BF16: 2 bytes an entry; an entry enters the sum widened to f32 exactly.
 *   TTS_Q8_0: blocks of 32 consecutive entries of a row, 34 bytes a block (a binary16
 *             scale d, then 32 signed 8-bit quants q); a row is hidden/32 blocks,
 *             hidden a multiple of 32.  An entry is the f32 product d * q, which is
 *             exact (a GGUF Q8_0 tensor has this layout).
 * (ABI 2 added `dtype`; ABI 3 added TTS_Q8_0.) */
typedef struct {
  const void* tab[TTS_MAX_TABLES];
  int32_t n_tables; /* 1..16 */
  int32_t vocab;    /* rows per table */
  int32_t hidden;   /* row length in elements, a multiple of 4 (of 32 for Q8_0) */
  int32_t dtype;    /* tts_dtype of every table: TTS_F32, TTS_BF16 or TTS_Q8_0 */
} tts_tables;

/* Flags of tts_kv_desc.flags */
/* TTS_KV_PREFETCH_BEFORE_WAIT: tts_decode_step may start streaming this layer's cache
 * rows before the previous kernel on the stream has finished.  Set it only when the
 * work enqueued immediately before the call writes neither this cache, nor its block
 * table, nor cur_len (true for a layer loop whose layers own distinct caches). */
#define TTS_KV_PREFETCH_BEFORE_WAIT 1u

/* One layer's K/V cache for B streams, "head-major" so that one kv head's positions
 * are contiguous:
 *   contiguous (paged = 0): K[b][g][j][d], j < capacity, dense; V likewise.
 *   paged      (paged = 1): a pool K[page][g][slot][d], page < n_pages,
 *                           slot < page_size; position j of stream b lives in page
 *                           block_table[b * bt_stride + j / page_size], slot
 *                           j % page_size.  capacity = page_size * pages per stream.
 * Element type f32 or bf16 (kv_dtype).  The window seen by a decode query is
 * [0, n_valid); conceptually it is padded to W = ceil(n_valid / window_quantum) *
 * window_quantum with -inf scores over [n_valid, W), i.e. those rows get weight
 * exactly 0 and are never read, so results do not depend on window_quantum or on what
 * the tail holds. */
typedef struct {
  int32_t B;              /* streams */
  int32_t n_q_heads;      /* Hq */
  int32_t n_kv_heads;     /* Hkv; Hq / Hkv in {1, 2, 4} */
  int32_t head_dim;       /* D in {64, 128} */
  int32_t capacity;       /* positions per stream, >= 1 */
  int32_t window_quantum; /* 256 talker, 16 predictor; divides capacity */
  int32_t kv_dtype;       /* tts_dtype */
  int32_t paged;          /* 0 contiguous, 1 paged */
  int32_t page_size;      /* paged: power of two in [1, 256] */
  int32_t n_pages;        /* paged: pages in the pool */
  int32_t bt_stride;      /* paged: block-table row stride (entries), >= capacity/page_size */
  uint32_t flags;         /* TTS_KV_* */
  const int32_t* block_table; /* paged: device int32 [B][bt_stride]; else NULL */
} tts_kv_desc;

/* ---------------------------------------------------------------------------
 * Step 1: frame-input composition.  [P-pipeline], on-device AR input assembly.
 *   out[b] = ((tab[0][ids[b][0]] + tab[1][ids[b][1]]) + ... ) + overlay[b]
 * in f32, codebooks in ascending order, the overlay added last; the result is
 * bit-identical to that sequence of single f32 additions.  bf16 table entries are
 * widened to f32 exactly, Q8_0 entries are the exact f32 product d * q, before they
 * are added.  For a code-predictor
 * sub-step pass one group table (n_tables = 1) and overlay = NULL.
 *   ids:     device int32 [B][ids_stride], first n_tables entries per row read.
 *   overlay: device f32 rows of `hidden`, row stride overlay_stride; or NULL.
 *   out:     device f32 [B][hidden], dense.
 * An id outside [0, vocab) is clamped into range and sets TTS_EFLAG_ID_RANGE.
 * ------------------------------------------------------------------------- */
tts_status tts_frame_embed(const tts_tables* tables, const int32_t* ids, int64_t ids_stride,
                           const float* overlay, int64_t overlay_stride, float* out, int32_t B,
                           int32_t* err_flag, void* stream);

/* ---------------------------------------------------------------------------
 * RoPE table.  Fills cs[p][i] = (cos theta, sin theta) as float pairs with
 * theta = p * base^(-2i/head_dim), for p < max_pos, i < head_dim/2; the angle and its
 * cos/sin are evaluated in double on the device and rounded to f32 once.  Built once
 * per model (like a model's inverse-frequency buffer) and read by the norm+RoPE calls.
 *   cs: device f32 [max_pos][head_dim/2][2].
 * ------------------------------------------------------------------------- */
tts_status tts_rope_table(float* cs, int32_t max_pos, int32_t head_dim, double base, void* stream);

/* ---------------------------------------------------------------------------
 * Step 2: per-head q/k RMSNorm then rotate-half RoPE, in place.  [P-engine], core
 * table, fused q/k norm + RoPE.  For every head row x of q (Hq heads) and k (Hkv
 * heads) of stream b:
 *   t_d = x_d * (mean_d(x_d^2) + eps)^(-1/2) * gamma_d
 *   y_i = t_i c_i - t_{i+D/2} s_i,  y_{i+D/2} = t_i s_i + t_{i+D/2} c_i
 * with (c_i, s_i) = rope_cs[pos[b]][i].  gamma_q / gamma_k: device f32 [D], shared by
 * the heads.  q rows: stream b at q + b*q_row_stride, heads contiguous (same for k).
 * q and k may be strided views into one fused projection row.  A pos outside
 * [0, rope_max_pos) is clamped and sets TTS_EFLAG_POS_RANGE.
 * ------------------------------------------------------------------------- */
tts_status tts_qk_norm_rope(float* q, int64_t q_row_stride, float* k, int64_t k_row_stride,
                            const float* gamma_q, const float* gamma_k, const int32_t* pos,
                            int32_t B, int32_t n_q_heads, int32_t n_kv_heads, int32_t head_dim,
                            float eps, const float* rope_cs, int32_t rope_max_pos,
                            int32_t* err_flag, void* stream);

/* ---------------------------------------------------------------------------
 * Step 3: KV write by set_rows.  [P-pipeline], fixed-topology section; KV-cache section.
 * For stream b and kv head g the row k[b][g][:] (f32) is written to the K cache at
 * position dst_pos[b] (device data), converted to the cache dtype (identity for f32;
 * bf16 round-to-nearest-even), and likewise v into the V cache.  k/v rows: stream b at
 * k + b*kv_row_stride, heads contiguous.  A position outside [0, capacity) or a page id
 * outside [0, n_pages) skips that stream's write and sets TTS_EFLAG_POS_RANGE /
 * TTS_EFLAG_PAGE.  Nothing else in the caches is touched.
 * ------------------------------------------------------------------------- */
tts_status tts_kv_set_rows(const float* k, const float* v, int64_t kv_row_stride, void* k_cache,
                           void* v_cache, const tts_kv_desc* desc, const int32_t* dst_pos,
                           int32_t* err_flag, void* stream);

/* ---------------------------------------------------------------------------
 * Step 4: single-query GQA decode attention with split-KV partitions.
 * [P-pipeline], persistent-arenas and KV-cache sections.  For stream b and q head h
 * (kv head g = h / (Hq/Hkv)):
 *   s_j = scale * q_h . K[b][g][j],  j < n_valid[b];   rows j >= n_valid[b]: -inf
 *   out[b][h] = sum_j softmax(s)_j V[b][g][j]
 * f32 accumulation.  Each kv head's window is cut into n_splits position ranges that
 * are processed in parallel and merged with a log-sum-exp combine inside the same
 * launch (the last range to finish merges; no kernel waits on another).
 *   q:   device f32, stream b at q + b*q_row_stride, heads contiguous.
 *   out: device f32 [B][Hq][D], dense.
 *   n_valid: device int32 [B] (= cur_len + 1 after the new row is written); an entry
 *        outside [1, capacity] is clamped and sets TTS_EFLAG_NVALID.  In a paged cache
 *        a page id outside [0, n_pages) inside the window reads page 0 instead and sets
 *        TTS_EFLAG_PAGE.
 *   workspace: device scratch of at least tts_decode_attn_workspace_size() bytes,
 *        256-byte aligned, zeroed once before its first use (tts_workspace_init or a
 *        memset); every call that completes without TTS_EFLAG_TIMEOUT leaves it ready
 *        for the next.  After a call that set TTS_EFLAG_TIMEOUT its split tickets and
 *        work counters may hold stale counts: zero it again (tts_workspace_init) before
 *        the next call that uses it.  Calls that overlap in time on the GPU must not
 *        share a workspace.
 *   n_splits: ranges per kv head, >= 1; 0 picks tts_decode_attn_default_splits().
 * ------------------------------------------------------------------------- */
size_t tts_decode_attn_workspace_size(const tts_kv_desc* desc, int32_t n_splits);
int32_t tts_decode_attn_default_splits(const tts_kv_desc* desc);
tts_status tts_workspace_init(void* workspace, size_t ws_bytes, void* stream);

tts_status tts_decode_attn(const float* q, int64_t q_row_stride, const void* k_cache,
                           const void* v_cache, const tts_kv_desc* desc, const int32_t* n_valid,
                           float scale, float* out, void* workspace, size_t ws_bytes,
                           int32_t n_splits, int32_t* err_flag, void* stream);

/* ---------------------------------------------------------------------------
 * Steps 2+3+4 fused: one layer of one decode step for B streams, in the order of the
 * [P-pipeline] KV-cache section.  For stream b with position p = cur_len[b]:
 *   q' = norm_rope(q[b], gamma_q, p), k' = norm_rope(k[b], gamma_k, p)   (as step 2)
 *   K[b][.][p] = cvt(k'), V[b][.][p] = cvt(v[b])                         (as step 3)
 *   out[b] = attention of q' over [0, p + 1)                             (as step 4)
 * q, k, v are read only (they may be strided views of one projection row; each row of
 * stream b starts at ptr + b*row_stride).  The attention uses the converted new row,
 * exactly as if it had been read back from the cache.  Workspace and n_splits as in
 * tts_decode_attn.  The frame-input composition (step 1) is a separate call made once
 * per frame, because the QKV projection sits between it and this step.
 * ------------------------------------------------------------------------- */
tts_status tts_decode_step(const float* q, const float* k, const float* v, int64_t row_stride,
                           const float* gamma_q, const float* gamma_k, float eps,
                           const float* rope_cs, int32_t rope_max_pos, void* k_cache,
                           void* v_cache, const tts_kv_desc* desc, const int32_t* cur_len,
                           float scale, float* out, void* workspace, size_t ws_bytes,
                           int32_t n_splits, int32_t* err_flag, void* stream);

/* ---------------------------------------------------------------------------
 * tts_decode_step without a workspace argument.  The paper has no counterpart: this
 * is a convenience of this library for callers that cannot allocate device memory when
 * they run a step -- e.g. a real-time audio callback that must not enter an allocator,
 * or a host framework that only lends out the tensors it owns.  The caller still passes
 * every input and output; the split-KV scratch comes from a fixed 4 MiB device array
 * inside the library (held on every GPU that loads the library until the process
 * exits), so a configuration needing more (tts_decode_attn_workspace_size() > 4 MiB)
 * is rejected with TTS_ERR_WORKSPACE.  The first call on a device looks the array's
 * device address up (a synchronous runtime call), so make that first call before any
 * stream capture.  Each call first clears the part of the array it uses (one small
 * kernel on `stream`) and then runs the step.  All calls share the one array: calls
 * that can overlap on the GPU (different streams, or different threads) race on it and
 * must be serialised by the caller.  Arguments and results are otherwise those of
 * tts_decode_step.
 * ------------------------------------------------------------------------- */
tts_status tts_decode_step_noalloc(const float* q, const float* k, const float* v,
                                   int64_t row_stride, const float* gamma_q,
                                   const float* gamma_k, float eps, const float* rope_cs,
                                   int32_t rope_max_pos, void* k_cache, void* v_cache,
                                   const tts_kv_desc* desc, const int32_t* cur_len, float scale,
                                   float* out, int32_t n_splits, int32_t* err_flag, void* stream);

/* ---------------------------------------------------------------------------
 * Prefill: T new positions per stream in one call ([P-pipeline], KV-cache section:
 * the prefill writes the prompt's rows from the reset position, causally).  Row t of
 * stream b sits at position p = start_pos[b] + t, t < T:
 *   q'[b][t] = norm_rope(q[b][t], gamma_q, p)
 *   K[b][.][p] = cvt(norm_rope(k[b][t], gamma_k, p)),  V[b][.][p] = cvt(v[b][t])
 *   out[b][t] = attention of q'[b][t] over [0, p + 1)
 * so every query sees the rows before the prompt and the prompt's rows up to its own.
 * With start_pos = 0 it is the prefill after a cache reset.
 *   q, k, v: device f32 rows, row r = b*T + t at ptr + r*row_stride (heads contiguous;
 *        they may be strided views of one projection row), read only.
 *   out: device f32 [B][T][Hq][D], dense.
 *   start_pos: device int32 [B].  A position outside [0, capacity) or [0, rope_max_pos)
 *        is not written and sets TTS_EFLAG_POS_RANGE; a window past capacity is clamped
 *        and sets TTS_EFLAG_NVALID.  Paged: a page id outside [0, n_pages) skips that
 *        row's write and sets TTS_EFLAG_PAGE.
 *   workspace: at least tts_prefill_workspace_size(desc, T, n_splits) bytes, otherwise
 *        as for tts_decode_attn (its B x T queries take the place of its B streams); it
 *        also holds the normed q rows on the paths that read them from memory.
 * Launches on `stream`: the rows, then the attention.  T < 8: the attention runs the
 * B*T queries one by one (as tts_decode_attn).  T >= 8 (and, paged, pages of 8 rows or
 * more): blocks of queries of a stream share every K/V tile of their window (bf16
 * caches with head_dim 128 and contiguous or 64-row-or-larger pages: blocks of
 * 128 / (Hq / Hkv) queries on the tensor cores; otherwise 64 / (Hq / Hkv) queries on
 * the CUDA cores), the windows cut into chunks; with more than one chunk a third launch
 * merges them in chunk order, unless the tensor-core launch merged them itself (2..8
 * chunks that the device keeps resident as one cluster per block).  That path's
 * workspace needs no zeroing.  B*T must not exceed 65535.
 * ------------------------------------------------------------------------- */
size_t tts_prefill_workspace_size(const tts_kv_desc* desc, int32_t T, int32_t n_splits);

/* Kernel launches tts_prefill_step makes for these arguments on the current device (2
 * or 3); 0 for arguments it would reject as shapes.  For counting a graph's nodes. */
int32_t tts_prefill_launch_count(const tts_kv_desc* desc, int32_t T, int32_t n_splits);

tts_status tts_prefill_step(const float* q, const float* k, const float* v, int64_t row_stride,
                            const float* gamma_q, const float* gamma_k, float eps,
                            const float* rope_cs, int32_t rope_max_pos, void* k_cache,
                            void* v_cache, const tts_kv_desc* desc, const int32_t* start_pos,
                            int32_t T, float scale, float* out, void* workspace, size_t ws_bytes,
                            int32_t n_splits, int32_t* err_flag, void* stream);

/* ---------------------------------------------------------------------------
 * In-graph sampler with a counter RNG ([P-pipeline]: the predictor frame unroll and
 * the in-graph sampler; [engine] options table, "Lean Talker frame": one-kernel
 * counter RNG).  For stream b, from its logits row l (vocab entries; NaN counts as
 * -inf):
 *   top_k 0 or 1: the index of the largest logit (the lowest such index on a tie);
 *   top_k = k in [2, TTS_MAX_TOP_K]: candidates are the k largest logits, larger first
 *   and lower index first on a tie, l_0 >= ... >= l_{k-1}; with c = log2(e)/temperature
 *   rounded once to f32, w_i = 2^(f32(f32(l_i - l_0) * c)) in f32 (an exponential of
 *   this library's own: degree-9 Taylor polynomial of 2^f on [0, 1) in Horner form,
 *   times 2^floor, 0 below 2^-126); S = w_0 + ... + w_{k-1} in that order; u = top 24
 *   bits of the first output of Philox4x64-10 at counter words (*counter, b, draw, 0)
 *   and key (seed, 0), times 2^-24; the token is candidate i of the first running sum
 *   (same order) above f32(u * S), else the last candidate.  Every operation is a
 *   single f32 rounding in that order, so the result is exactly reproducible.
 *   logits: device f32, stream b at logits + b*logits_stride.
 *   counter: device uint64 (read only here); advance it between replays with
 *        tts_counter_advance so that a replayed graph draws fresh numbers.
 *   draw: a host constant told apart inside one counter value, e.g. the sub-step of a
 *        code-predictor frame, so that the frame's draws are independent while the
 *        counter moves once per frame.
 *   out_ids: device int32, stream b's token at out_ids + b*out_stride (for example
 *        the column of the next frame's code ids).
 * vocab must not exceed TTS_MAX_SAMPLE_VOCAB.
 * ------------------------------------------------------------------------- */
#define TTS_MAX_TOP_K 64
#define TTS_MAX_SAMPLE_VOCAB 8192
tts_status tts_sample(const float* logits, int64_t logits_stride, int32_t B, int32_t vocab,
                      int32_t top_k, float temperature, uint64_t seed, const uint64_t* counter,
                      uint32_t draw, int32_t* out_ids, int64_t out_stride, void* stream);

/* The sampler and the gather of the drawn codes in one launch: exactly tts_sample(...)
 * followed by tts_frame_embed(table, out_ids, out_stride, NULL, 0, out_rows, B, ...)
 * with one table and no overlay, i.e. out_rows[b] (device f32 [B][table->hidden],
 * dense) is the drawn token's row of table->tab[0], entries widened (bf16) or
 * dequantised (Q8_0) exactly.  table->n_tables must be 1 and table->vocab >= vocab.
 * ([P-pipeline]: the code predictor's in-graph sampler feeds the next sub-step's
 * gather; one launch instead of two per sub-step.) */
tts_status tts_sample_embed(const float* logits, int64_t logits_stride, int32_t B, int32_t vocab,
                            int32_t top_k, float temperature, uint64_t seed, const uint64_t* counter,
                            uint32_t draw, int32_t* out_ids, int64_t out_stride, const tts_tables* table,
                            float* out_rows, void* stream);

/* *counter += by, as one kernel on `stream` (graph-capturable). */
tts_status tts_counter_advance(uint64_t* counter, uint64_t by, void* stream);

/* ---------------------------------------------------------------------------
 * Self-test of the error path of the bounded waits.  Every wait inside this library's
 * kernels (on an mbarrier, a cluster peer or a counter) gives up after a fixed number
 * of SM clock cycles (about a second at the GB300's clocks), sets TTS_EFLAG_TIMEOUT in
 * err_flag and winds its kernel down, so the context stays usable (the workspace of
 * the call must then be re-zeroed before its next use).  This call launches one thread
 * that waits, with that same wait, for an mbarrier phase that nothing completes: after
 * the limit it sets TTS_EFLAG_TIMEOUT in *err_flag (device int32) and returns.  It
 * faults nothing and holds the GPU for about a second; for tests of error handling.
 * ------------------------------------------------------------------------- */
tts_status tts_check_wait_timeout(int32_t* err_flag, void* stream);

/* ---------------------------------------------------------------------------
 * One whole talker decode layer with bf16 weights, for B <= 32 streams ([engine] core
 * table: fused residual add + RMSNorm, q/k norm + RoPE, SiLU-multiply, reproducing the
 * reference rounding with integer round-to-nearest-even; [pipeline] KV-cache section
 * for the step).  In place on the residual stream h [B][hidden] (f32):
 *   x = bf16(rmsnorm(h) * gamma_attn)          (statistics in f32, RNE to bf16)
 *   qkv = x W_qkv^T                             (f32; q, k, v as in tts_decode_step)
 *   attn = tts_decode_step(q, k, v, ...)        (norm + RoPE, new row, attention)
 *   h = h + bf16(attn) W_o^T
 *   x = bf16(rmsnorm(h) * gamma_mlp)
 *   a = bf16(silu(x W_gate^T) * x W_up^T)       (silu in f32)
 *   h = h + a W_down^T
 * Products accumulate in f32; every residual add is one f32 addition.  The projections
 * run on the tensor cores (bf16 x bf16, f32 accumulator).  Each norm input is rounded
 * and packed for them by a small kernel; the decode step writes its output already
 * rounded and packed, and the SiLU-multiply writes `a` packed.  That makes seven
 * launches on `stream` (two packs, four projections, the decode step;
 * tts_decode_layer_launch_count).  The sums of a projection's column ranges are added in
 * a fixed order, so results do not depend on timing.  The weights and the gammas are
 * treated as constants: each launch starts reading them before the preceding kernel on
 * `stream` has finished, so they must not be written by the kernel launched just before
 * this call on the same stream (write them with a copy, or synchronise first).  Weights
 * are bf16, row-major, rows of `hidden` (or `inter`) elements:
 *   w_qkv [(Hq + 2 Hkv) D][hidden], w_o [hidden][Hq D], w_gu [2 inter][hidden] (the
 *   gate rows, then the up rows), w_down [hidden][inter].
 * hidden, inter and Hq*D must be multiples of 256 and at most 8192.
 *   scratch: device memory of tts_decode_layer_scratch_size() bytes, 256-byte aligned,
 *        zeroed once before its first use (it holds the attention workspace).
 * ------------------------------------------------------------------------- */
typedef struct {
  const void* w_qkv;
  const void* w_o;
  const void* w_gu;
  const void* w_down;
  const float* gamma_attn; /* [hidden] */
  const float* gamma_mlp;  /* [hidden] */
  const float* gamma_q;    /* [head_dim] */
  const float* gamma_k;    /* [head_dim] */
  int32_t hidden;
  int32_t inter;
} tts_layer_weights;

size_t tts_decode_layer_scratch_size(const tts_kv_desc* desc, int32_t hidden, int32_t inter,
                                     int32_t n_splits);

/* Kernel launches one tts_decode_layer call makes for this descriptor (7; 5 in a build
 * whose CUDA-core projections serve this stream count); 0 for a descriptor it rejects. */
int32_t tts_decode_layer_launch_count(const tts_kv_desc* desc);

tts_status tts_decode_layer(float* h, const tts_layer_weights* weights, float eps,
                            const float* rope_cs, int32_t rope_max_pos, void* k_cache,
                            void* v_cache, const tts_kv_desc* desc, const int32_t* cur_len,
                            float scale, void* scratch, size_t scratch_bytes, int32_t n_splits,
                            int32_t* err_flag, void* stream);

#ifdef __cplusplus
}
#endif

#endif /* TTS_DECODE_H */
