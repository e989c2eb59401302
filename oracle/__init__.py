"""CPU oracle for the per-frame decode hot path (test infrastructure only).

A plain, slow, single-threaded restatement of what each step of the hot path
computes, compiled from ``oracle.cpp`` with the host compiler and called through
ctypes on numpy arrays.  Only ``tests/``, ``__graft_entry__.smoke()`` and the
CPU-baseline leg of ``bench.py`` may import this package; the CUDA library never
does, and this package imports nothing from the CUDA library.

Steps and the passages they follow (page titles as printed on the pages):

* ``frame_embed`` -- "qwentts.cpp ... src/pipeline-tts.h", on-device AR input
  assembly: 16 code-embedding rows gathered and summed with the trailing text/pad
  overlay; the code predictor gathers one sub-code from its own group table.
* ``rms_norm_rope`` -- "minicpm-o-4.5 ... docs/optimizations.md", core table, fused
  "q/k norm + RoPE" (norm, then rotation).
* ``kv_set_rows`` -- "qwentts.cpp ... src/pipeline-tts.h", fixed topology section:
  KV writes through set_rows with destination rows carried as data; bf16 rounding by
  integer round-to-nearest-even as in the optimizations table.
* ``decode_attn`` -- "qwentts.cpp ... src/pipeline-tts.h", persistent arenas and KV
  cache sections: decode reads the [0, cur_len+1) window, padded tail masked by -inf.
* ``decode_step`` / ``predictor_frame`` -- compositions of the above in the order the
  KV cache section gives (norm+RoPE, write the new row, attend; the predictor resets
  its 16-slot cache, prefills T=2 and then decodes 14 single tokens).
* ``prefill_step`` -- the same section's prefill: T new positions per stream written
  into the cache, each of their queries attending causally over [0, its position],
  i.e. T decode queries whose windows end at their own rows.
* ``rmsnorm_bf16`` / ``gemv_bf16`` / ``decode_layer`` -- one whole talker decode layer
  with bf16 weights (the optimisations table's fused Thinker kernels: residual add +
  RMSNorm, q/k norm + RoPE, SiLU-multiply, "each reproducing the reference rounding with
  integer round-to-nearest-even"): activations rounded to bf16 by RNE where a bf16 model
  would hold them (GEMV inputs), products summed exactly (float64), outputs in f32.
* ``sample`` -- the in-graph sampler with a counter RNG ("qwentts.cpp" pages: the
  predictor frame unroll and the in-graph sampler; the optimisations table's
  "one-kernel counter RNG"): greedy, or temperature/top-k sampling driven by the
  published Philox4x64-10 counter generator, every decision taken in f32 in a fixed
  order (``exp2_f32`` is this oracle's own exponential, see its docstring).
"""
from __future__ import annotations

import ctypes
import math
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")
_lock = threading.Lock()
_lib = None

CFLAGS = ["-O2", "-std=c++17", "-ffp-contract=off", "-fno-fast-math", "-fPIC", "-shared"]


def build(force: bool = False) -> str:
    """Compile ``oracle.cpp`` into ``_build/liboracle.so`` (host compiler, no GPU)."""
    os.makedirs(_BUILD, exist_ok=True)
    if force or not os.path.exists(_LIB_PATH) or os.path.getmtime(_LIB_PATH) < os.path.getmtime(_SRC):
        tmp = _LIB_PATH + f".tmp{os.getpid()}"
        subprocess.check_call(["g++", *CFLAGS, _SRC, "-o", tmp])
        os.replace(tmp, _LIB_PATH)
    return _LIB_PATH


def _load():
    global _lib
    with _lock:
        if _lib is None:
            lib = ctypes.CDLL(build())
            P, I, L, D = ctypes.c_void_p, ctypes.c_int, ctypes.c_int64, ctypes.c_double
            lib.oracle_bf16_rne.argtypes = [ctypes.c_float]
            lib.oracle_bf16_rne.restype = ctypes.c_uint16
            lib.oracle_frame_embed.argtypes = [P, I, I, I, P, L, P, L, P, I]
            lib.oracle_frame_embed.restype = I
            lib.oracle_rms_norm_rope.argtypes = [P, L, P, L, I, I, I, P, ctypes.c_float, P, D]
            lib.oracle_rms_norm_rope.restype = None
            lib.oracle_rope_angle.argtypes = [I, I, I, D, P]
            lib.oracle_rope_angle.restype = None
            lib.oracle_kv_set_rows.argtypes = [P, P, L, P, P, I, I, I, I, I, I, I, I, P, I, P]
            lib.oracle_kv_set_rows.restype = I
            lib.oracle_decode_attn.argtypes = [P, L, P, P, I, I, I, I, I, I, I, I, I, P, I, P, D, P, P]
            lib.oracle_decode_attn.restype = I
            _lib = lib
    return _lib


def _ptr(a):
    return None if a is None else a.ctypes.data


def _c(a, dtype):
    """Contiguous array of the given dtype (no copy when already so)."""
    return np.ascontiguousarray(a, dtype=dtype)


# ---------------------------------------------------------------------------
# bf16 helpers
# ---------------------------------------------------------------------------
def bf16_rne(x: float) -> int:
    """bf16 bit pattern of one f32 value, integer round-to-nearest-even ("minicpm-o-4.5
    ... docs/optimizations.md", core table: the fused kernels reproduce the reference
    rounding with integer round-to-nearest-even)."""
    return int(_load().oracle_bf16_rne(ctypes.c_float(float(np.float32(x)))))


def bf16_rne_array(x) -> np.ndarray:
    """Elementwise bf16 RNE of an f32 array, as uint16 (one oracle call per element;
    the rounding of ``bf16_rne``)."""
    x = _c(x, np.float32)
    lib = _load()
    out = np.empty(x.shape, np.uint16)
    flat_in, flat_out = x.reshape(-1), out.reshape(-1)
    for i in range(flat_in.size):
        flat_out[i] = lib.oracle_bf16_rne(ctypes.c_float(float(flat_in[i])))
    return out


def q8_0_dequant(t) -> np.ndarray:
    """Entries of a Q8_0 table as f32.  t: uint8 [vocab][n_blocks * 34]; each 34-byte block
    holds 32 consecutive entries of a row: a little-endian IEEE binary16 scale d, then 32
    two's-complement int8 quants q; an entry is d * q.  d widens to f32 exactly and the
    product of an 11-bit and an 8-bit significand is exact in f32 ("qwentts.cpp ...
    src/pipeline-tts.h", TTFA / prompt-build section: the tables are gathered whatever
    their quantisation; its TTFA measurements use Q8_0 tables)."""
    t = np.ascontiguousarray(np.asarray(t, dtype=np.uint8))
    vocab, nbytes = t.shape
    if nbytes % 34:
        raise ValueError("a Q8_0 row is a whole number of 34-byte blocks")
    blocks = t.reshape(vocab, nbytes // 34, 34)
    d = np.ascontiguousarray(blocks[:, :, :2]).view("<f2").astype(np.float32)    # [vocab][nb][1]
    q = np.ascontiguousarray(blocks[:, :, 2:]).view(np.int8).astype(np.float32)  # [vocab][nb][32]
    return (d * q).reshape(vocab, -1)


def bf16_bits_to_f32(h) -> np.ndarray:
    """Exact widening of bf16 bit patterns (uint16) to f32: the bf16 bits become the high
    half of the f32 (how a bf16 table entry or cache row enters f32 arithmetic; "qwentts.cpp
    ... src/pipeline-tts.h", on-device AR input assembly: tables of any type read through
    get_rows)."""
    h = np.asarray(h, dtype=np.uint16)
    return (h.astype(np.uint32) << 16).view(np.float32)


# ---------------------------------------------------------------------------
# a1: frame-input composition
# ---------------------------------------------------------------------------
def frame_embed(tables, ids, overlay=None):
    """out[b] = ((E_0[c_b0] + E_1[c_b1]) + ... ) + overlay[b], f32, fixed order.

    tables: list of [vocab][hidden] arrays, f32, or uint16 holding bf16 bit patterns, or
    uint8 Q8_0 rows [vocab][hidden / 32 * 34] (the "TTFA / prompt build" section's gather of
    any table type: a bf16 entry is widened to f32 exactly, a Q8_0 entry is its exact f32
    product d * q, then added like an f32 one); ids: [B][n_tables] int32; overlay:
    [B][hidden] f32 or None.  Returns (out [B][hidden] f32, clamped flag).
    """
    def as_f32(t):
        dt = np.asarray(t).dtype
        if dt == np.uint16:
            return bf16_bits_to_f32(t)
        if dt == np.uint8:
            return q8_0_dequant(t)
        return _c(t, np.float32)
    tabs = [as_f32(t) for t in tables]
    ids = _c(ids, np.int32)
    B, n = ids.shape
    vocab, hidden = tabs[0].shape
    arr = (ctypes.c_void_p * n)(*[t.ctypes.data for t in tabs])
    ov = None if overlay is None else _c(overlay, np.float32)
    out = np.empty((B, hidden), np.float32)
    flag = _load().oracle_frame_embed(arr, n, vocab, hidden, _ptr(ids), n, _ptr(ov),
                                      hidden, _ptr(out), B)
    return out, int(flag)


# ---------------------------------------------------------------------------
# a2: per-head RMSNorm + RoPE
# ---------------------------------------------------------------------------
def rms_norm_rope(x, gamma, eps, pos, base):
    """x: [B][H][D] f32 -> normed and rotated copy (f32): per-head RMSNorm, then
    rotate-half RoPE at pos[b] ("minicpm-o-4.5 ... docs/optimizations.md", core table,
    fused "q/k norm + RoPE"; the formulas are the readings stated in ``oracle.cpp``),
    in double, rounded to f32 once."""
    x = _c(x, np.float32)
    B, H, D = x.shape
    gamma = _c(gamma, np.float32)
    pos = _c(pos, np.int32)
    y = np.empty_like(x)
    _load().oracle_rms_norm_rope(_ptr(x), H * D, _ptr(y), H * D, B, H, D, _ptr(gamma),
                                 ctypes.c_float(eps), _ptr(pos), float(base))
    return y


def rope_angle(pos: int, i: int, head_dim: int, base: float):
    """(cos, sin) of theta = pos * base^(-2i/head_dim) in double: the RoPE angle of
    frequency i (the rotation of ``rms_norm_rope``)."""
    cs = np.empty(2, np.float64)
    _load().oracle_rope_angle(int(pos), int(i), int(head_dim), float(base), _ptr(cs))
    return float(cs[0]), float(cs[1])


# ---------------------------------------------------------------------------
# Cache descriptor shared by a3/a4 on the oracle side
# ---------------------------------------------------------------------------
class KvLayout:
    """Geometry of one layer's K/V cache, head-major (see ``oracle.cpp``)."""

    def __init__(self, B, n_kv_heads, head_dim, capacity, kv_dtype="f32", paged=False,
                 page_size=16, n_pages=0, block_table=None):
        self.B, self.n_kv_heads, self.head_dim, self.capacity = B, n_kv_heads, head_dim, capacity
        self.kv_dtype = kv_dtype
        self.paged = bool(paged)
        self.page_size = page_size
        self.n_pages = n_pages
        self.block_table = None if block_table is None else _c(block_table, np.int32)

    @property
    def dtype_code(self):
        return 0 if self.kv_dtype == "f32" else 1

    @property
    def bt_stride(self):
        return 0 if self.block_table is None else self.block_table.shape[1]


def kv_set_rows(k, v, k_cache, v_cache, layout: KvLayout, dst_pos):
    """Write k[b], v[b] ([B][Hkv][D] f32) into the caches at dst_pos[b], in place
    ("qwentts.cpp ... src/pipeline-tts.h", fixed topology + set_rows section: KV writes
    carry their destination rows as data; bf16 caches round by RNE).

    Caches are numpy arrays (f32, or uint16 holding bf16 bits).  Returns the
    skipped-write flag.
    """
    k = _c(k, np.float32)
    v = _c(v, np.float32)
    B = k.shape[0]
    row = k.shape[1] * k.shape[2]
    dst_pos = _c(dst_pos, np.int32)
    assert k_cache.flags.c_contiguous and v_cache.flags.c_contiguous
    L = layout
    return int(_load().oracle_kv_set_rows(
        _ptr(k), _ptr(v), row, _ptr(k_cache), _ptr(v_cache), L.dtype_code, B, L.n_kv_heads,
        L.head_dim, L.capacity, int(L.paged), L.page_size, L.n_pages, _ptr(L.block_table),
        L.bt_stride, _ptr(dst_pos)))


def decode_attn(q, k_cache, v_cache, layout: KvLayout, n_valid, scale, want_weights=False):
    """Single-query GQA attention over [0, n_valid[b]) per stream, double precision
    ("qwentts.cpp ... src/pipeline-tts.h", persistent arenas and KV cache sections: the
    decode reads the [0, cur_len+1) window, the padded tail masked by -inf, so positions
    past n_valid carry no weight).

    q: [B][Hq][D] f32.  Returns (out [B][Hq][D] f32, weights or None, clamped flag).
    """
    q = _c(q, np.float32)
    B, Hq, D = q.shape
    n_valid = _c(n_valid, np.int32)
    L = layout
    out = np.empty((B, Hq, D), np.float32)
    w = np.empty((B, Hq, L.capacity), np.float64) if want_weights else None
    flag = _load().oracle_decode_attn(
        _ptr(q), Hq * D, _ptr(k_cache), _ptr(v_cache), L.dtype_code, B, Hq, L.n_kv_heads, D,
        L.capacity, int(L.paged), L.page_size, L.n_pages, _ptr(L.block_table), L.bt_stride,
        _ptr(n_valid), float(scale), _ptr(out), _ptr(w))
    return out, w, int(flag)


# ---------------------------------------------------------------------------
# Compositions
# ---------------------------------------------------------------------------
def decode_step(q, k, v, gamma_q, gamma_k, eps, base, k_cache, v_cache, layout: KvLayout,
                cur_len, scale):
    """One layer of one decode step for B streams, in the order the pages give
    ("qwentts.cpp ... src/pipeline-tts.h", KV cache section): q/k RMSNorm + RoPE at
    position cur_len, write the new K/V row at cur_len, attend over [0, cur_len + 1).
    Mutates the caches; returns the attention output."""
    cur_len = _c(cur_len, np.int32)
    qn = rms_norm_rope(q, gamma_q, eps, cur_len, base)
    kn = rms_norm_rope(k, gamma_k, eps, cur_len, base)
    kv_set_rows(kn, v, k_cache, v_cache, layout, cur_len)
    out, _, _ = decode_attn(qn, k_cache, v_cache, layout, cur_len + 1, scale)
    return out


def prefill_step(q, k, v, gamma_q, gamma_k, eps, base, k_cache, v_cache, layout: KvLayout,
                 start, scale):
    """T new positions per stream ("qwentts.cpp", KV cache section: the prefill writes
    the prompt's rows from the reset position, causally).  Stream b's rows t < T sit at
    position start[b] + t.  Every q and k row is RMS-normed and rotated at its own
    position, every k/v row is written into the cache at it, and query t attends over
    the window [0, start[b] + t + 1): the rows before the prompt and the prompt's rows
    up to its own.  Mutates the caches; returns out [B][T][Hq][D] f32.

    q: [B][T][Hq][D], k, v: [B][T][Hkv][D] (f32); start: [B] int32."""
    q = _c(q, np.float32)
    k = _c(k, np.float32)
    v = _c(v, np.float32)
    start = _c(start, np.int32)
    B, T, Hq, D = q.shape
    pos = start[:, None] + np.arange(T, dtype=np.int32)[None, :]
    for t in range(T):  # all of the prompt's rows are in the cache before any query
        kn = rms_norm_rope(k[:, t], gamma_k, eps, pos[:, t], base)
        kv_set_rows(kn, v[:, t], k_cache, v_cache, layout, pos[:, t])
    out = np.empty((B, T, Hq, D), np.float32)
    for t in range(T):
        qn = rms_norm_rope(q[:, t], gamma_q, eps, pos[:, t], base)
        out[:, t], _, _ = decode_attn(qn, k_cache, v_cache, layout, pos[:, t] + 1, scale)
    return out


def predictor_frame(group_tables, codes, bridge, qkv_per_substep, gammas, eps, base,
                    caches, layout: KvLayout, scale):
    """One code-predictor frame for B streams ("qwentts.cpp", KV cache section).

    The 16-slot cache is reset (cur_len = 0; stale rows are masked, not cleared), the
    T=2 prefill writes rows 0 and 1 causally, then 14 single-token decodes write rows
    2..15.  Sub-step j gathers code j from group table j (the bridge row stands in
    front of the c0 row in the prefill).  The QKV projection between the gathered row
    and q/k/v is outside this path, so q/k/v per sub-step and layer are inputs.

    group_tables: 15 arrays [vocab][hidden]; codes: [B][15] int32; bridge: [B][hidden];
    qkv_per_substep[t][l] = (q, k, v) for sub-step t in 0..15 (t=0,1 the prefill rows);
    gammas[l] = (gamma_q, gamma_k); caches[l] = (k_cache, v_cache).
    Returns (embeds, outs): embeds[j] the gathered row for sub-step j (j = 0..14),
    outs[t][l] the attention output of sub-step t at layer l.
    """
    codes = _c(codes, np.int32)
    B = codes.shape[0]
    embeds = []
    for j in range(15):
        e, _ = frame_embed([group_tables[j]], codes[:, j:j + 1], None)
        embeds.append(e)
    outs = []
    n_layers = len(caches)
    for t in range(16):
        cur = np.full(B, t, np.int32)
        per_layer = []
        for l in range(n_layers):
            q, k, v = qkv_per_substep[t][l]
            gq, gk = gammas[l]
            kc, vc = caches[l]
            per_layer.append(decode_step(q, k, v, gq, gk, eps, base, kc, vc, layout, cur, scale))
        outs.append(per_layer)
    return embeds, outs


# ---------------------------------------------------------------------------
# In-graph sampler with a counter RNG
# ---------------------------------------------------------------------------
_M64 = (1 << 64) - 1


def philox4x64_10(counter, key):
    """Philox4x64 with 10 rounds (Salmon, Moraes, Dror, Shaw, "Parallel random numbers:
    as easy as 1, 2, 3", SC 2011): four 64-bit counter words, two 64-bit key words ->
    four 64-bit outputs.  Each round multiplies words 0 and 2 by the two round
    multipliers (high and low halves of the 128-bit products), mixes the high halves
    with words 1 and 3 and the key, and the key is bumped by the two Weyl constants
    between rounds."""
    c = [int(x) & _M64 for x in counter]
    k = [int(x) & _M64 for x in key]
    for r in range(10):
        if r > 0:
            k[0] = (k[0] + 0x9E3779B97F4A7C15) & _M64
            k[1] = (k[1] + 0xBB67AE8584CAA73B) & _M64
        p0 = 0xD2E7470EE14C6C93 * c[0]
        p1 = 0xCA5A826395121157 * c[2]
        c = [(p1 >> 64) ^ c[1] ^ k[0], p1 & _M64, (p0 >> 64) ^ c[3] ^ k[1], p0 & _M64]
    return c


def uniform_f32(seed, counter, b, draw=0):
    """The sampler's uniform for stream b at `counter`: the top 24 bits of the first
    Philox4x64-10 output for counter words (counter, b, draw, 0) and key (seed, 0), times
    2^-24 (exact in f32, in [0, 1)).  The counter RNG is the "one-kernel counter RNG" of
    "minicpm-o-4.5 ... docs/optimizations.md" (options table, "Lean Talker frame");
    `draw` tells apart the draws made at one counter value (the sub-steps of a
    code-predictor frame, each of which samples its own sub-code)."""
    x = philox4x64_10([counter, b, draw, 0], [seed, 0])[0]
    return np.float32((x >> 40) * (1.0 / (1 << 24)))


# 2^f on [0, 1): Taylor coefficients (ln 2)^j / j!, j = 0..9, rounded to f32.
_EXP2_C = [np.float32(math.log(2.0) ** j / math.factorial(j)) for j in range(10)]


def exp2_f32(x):
    """2^x for an f32 x <= 0, in f32 operations in a fixed order: 0 below -126; else
    n = floor(x), f = x - n (exact), p = Horner over the degree-9 Taylor polynomial of
    2^f (each product and sum rounded to f32, no fused multiply-add), times 2^n
    (exact).  The sampler's weights use it ("qwentts.cpp" pages, in-graph sampler), so
    that both sides of the parity tests take every token decision in the same f32
    arithmetic."""
    x = np.float32(x)
    if not x >= np.float32(-126.0):  # also NaN
        return np.float32(0.0)
    n = math.floor(float(x))
    f = np.float32(x - np.float32(n))
    p = _EXP2_C[9]
    for j in range(8, -1, -1):
        p = np.float32(np.float32(p * f) + _EXP2_C[j])
    return np.float32(p * np.float32(2.0 ** n))


def sample(logits, top_k, temperature, seed, counter, draw=0):
    """Token ids [B] int32 from logits [B][V] f32.

    top_k = 0 or 1: greedy, the index of the largest logit (the lowest such index on a
    tie).  top_k = k > 1: the k largest logits (larger first, lower index first on a
    tie) l_0 >= ... >= l_{k-1}; c = f32(log2(e) / temperature) (rounded once from
    double); w_i = exp2_f32(f32(f32(l_i - l_0) * c)); S = w_0 + ... + w_{k-1} summed in
    that order in f32; r = f32(u * S) with u = uniform_f32(seed, counter, b, draw); the result
    is the candidate i of the first running sum (in f32, same order) above r, or the
    last candidate if none is.  NaN logits count as -inf; when the top candidate is not
    finite the result is that candidate.  This is the in-graph sampler of the "qwentts.cpp"
    pages (the code-predictor frame unroll keeps its sampler on the device) on the counter
    RNG of "minicpm-o-4.5 ... docs/optimizations.md" (options table, "Lean Talker
    frame"); the tie and rounding rules are this library's readings."""
    lg = np.array(logits, dtype=np.float32, copy=True)
    lg[np.isnan(lg)] = -np.inf
    B, V = lg.shape
    out = np.empty(B, np.int32)
    c = np.float32(1.4426950408889634 / float(temperature)) if top_k > 1 else np.float32(0)
    for b in range(B):
        row = lg[b]
        if top_k <= 1:
            out[b] = int(np.argmax(row))  # first maximum
            continue
        order = sorted(range(V), key=lambda i: (-float(row[i]), i))[:top_k]
        m = row[order[0]]
        if not np.isfinite(m):  # no finite logit on top: the first candidate
            out[b] = order[0]
            continue
        w = [exp2_f32(np.float32(np.float32(row[i] - m) * c)) for i in order]
        S = np.float32(0.0)
        for wi in w:
            S = np.float32(S + wi)
        r = np.float32(uniform_f32(seed, counter, b, draw) * S)
        acc = np.float32(0.0)
        pick = len(order) - 1
        for j, wi in enumerate(w):
            acc = np.float32(acc + wi)
            if acc > r:
                pick = j
                break
        out[b] = order[pick]
    return out


# ---------------------------------------------------------------------------
# A whole decode layer with bf16 weights
# ---------------------------------------------------------------------------
def bf16_round(x) -> np.ndarray:
    """f32 values rounded to bf16 by round-to-nearest-even, returned as f32 (the
    integer RNE of "minicpm-o-4.5 ... docs/optimizations.md", core table)."""
    return bf16_bits_to_f32(bf16_rne_array(np.asarray(x, np.float32)))


def rmsnorm_bf16(h, gamma, eps):
    """x = h * (mean(h^2) + eps)^-1/2 * gamma per row, in double, rounded once to bf16
    (returned as f32 holding bf16 values).  h: [B][H] f32, gamma: [H] f32.
    ("minicpm-o-4.5 ... docs/optimizations.md", core table: residual add + RMSNorm
    fused, integer RNE; the RMSNorm form is this library's reading.)"""
    h64 = np.asarray(h, np.float64)
    r = 1.0 / np.sqrt((h64 * h64).mean(axis=1, keepdims=True) + float(eps))
    y = (h64 * r * np.asarray(gamma, np.float64)).astype(np.float32)
    return bf16_round(y)


def gemv_bf16(x, w_bits):
    """y[b][n] = sum_k x[b][k] * W[n][k] with x holding bf16 values (f32 arrays) and W
    bf16 bit patterns [N][K]: every product is exact in float64 (two 8-bit significands),
    the sum carries double precision (a library matrix product, ~1e-16 relative), and the
    result is rounded once to f32.  (The QKV / O / gate-up / down projections of a bf16
    decode layer, "minicpm-o-4.5 ... docs/optimizations.md", core table.)"""
    W = bf16_bits_to_f32(w_bits).astype(np.float64)
    return (np.asarray(x, np.float64) @ W.T).astype(np.float32)


def silu_mul_bf16(gate, up):
    """a = silu(gate) * up = gate / (1 + e^-gate) * up in double, rounded once to bf16
    ("minicpm-o-4.5 ... docs/optimizations.md", core table: SiLU-multiply fused)."""
    g = np.asarray(gate, np.float64)
    a = g / (1.0 + np.exp(-g)) * np.asarray(up, np.float64)
    return bf16_round(a.astype(np.float32))


def decode_layer(h, wts, k_cache, v_cache, layout: KvLayout, cur_len, eps, base, scale):
    """One talker decode layer for B streams, in place on the residual stream h ([B][H]
    f32):  x = rmsnorm(h)_bf16;  qkv = x W_qkv^T;  attn = decode_step(q, k, v);
    h = h + bf16(attn) W_o^T;  x2 = rmsnorm(h)_bf16;  gate, up = x2 W_gu^T (rows
    [0, I) and [I, 2I));  h = h + silu_mul(gate, up)_bf16 W_down^T.  The residual adds
    are single f32 additions.  wts: dict with gamma_attn, gamma_mlp (f32 [H]), gamma_q,
    gamma_k (f32 [D]), w_qkv [(Hq + 2 Hkv) D][H], w_o [H][Hq D], w_gu [2I][H],
    w_down [H][I] (bf16 bit patterns).  Mutates h and the caches; returns h.
    ("minicpm-o-4.5 ... docs/optimizations.md", core table: fused residual add +
    RMSNorm, q/k norm + RoPE and SiLU-multiply with integer RNE; "qwentts.cpp ...
    src/pipeline-tts.h", KV cache section, for the decode step.  The layer's structure
    and rounding points are this library's plainest reading of a bf16 transformer
    layer.)"""
    B, H = h.shape
    D = layout.head_dim
    Hkv = layout.n_kv_heads
    Hq = wts["w_o"].shape[1] // D
    x = rmsnorm_bf16(h, wts["gamma_attn"], eps)
    qkv = gemv_bf16(x, wts["w_qkv"])
    q = qkv[:, :Hq * D].reshape(B, Hq, D)
    k = qkv[:, Hq * D:(Hq + Hkv) * D].reshape(B, Hkv, D)
    v = qkv[:, (Hq + Hkv) * D:].reshape(B, Hkv, D)
    attn = decode_step(q, k, v, wts["gamma_q"], wts["gamma_k"], eps, base, k_cache, v_cache,
                       layout, cur_len, scale)
    o = gemv_bf16(bf16_round(attn.reshape(B, Hq * D)), wts["w_o"])
    h[...] = (h + o).astype(np.float32)
    x2 = rmsnorm_bf16(h, wts["gamma_mlp"], eps)
    gu = gemv_bf16(x2, wts["w_gu"])
    I = gu.shape[1] // 2
    a = silu_mul_bf16(gu[:, :I], gu[:, I:])
    d = gemv_bf16(a, wts["w_down"])
    h[...] = (h + d).astype(np.float32)
    return h
