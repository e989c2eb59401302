"""Brute-force decode attention for tiny inputs (test infrastructure only).

A second, independent statement of step a4 written as the plainest per-element loop,
used to pin ``oracle.decode_attn`` on small cases.  It shares no code with
``oracle.cpp``: its own cache addressing, its own bf16 widening, Python floats
(IEEE double) throughout, and the softmax taken straight from its definition with no
max subtraction,

    s_j = scale * sum_d q_d K_jd              (j < n_valid)
    w_j = exp(s_j) / sum_{k < n_valid} exp(s_k)
    o_d = sum_j w_j V_jd

which is only safe while every exp(s_j) stays far from overflow -- hence tiny inputs
(windows of at most 64 rows, scores of order 1).  Positions at or past n_valid are
the -inf tail of the padded window ("qwentts.cpp ... src/pipeline-tts.h", persistent
arenas section): they are simply not visited.  Query head h reads kv head
h // (Hq / Hkv).

Cache layouts (the library's head-major layout):
  contiguous: cache[b][g][j][d];
  paged:      pool[page][g][j % page_size][d] with page = block_table[b][j // page_size].
bf16 caches come as uint16 bit patterns; a bf16 value is the f32 whose upper 16 bits
are those bits, which ``_bf16_value`` builds with ``struct`` rather than numpy views.

Only ``tests/`` may import this module.
"""
from __future__ import annotations

import math
import struct

MAX_BRUTE_ROWS = 64


def _bf16_value(bits: int) -> float:
    return struct.unpack("<f", struct.pack("<I", (int(bits) & 0xFFFF) << 16))[0]


def _element(cache, kv_dtype, b, g, j, d, paged, page_size, block_table):
    if paged:
        page = int(block_table[b][j // page_size])
        x = cache[page][g][j % page_size][d]
    else:
        x = cache[b][g][j][d]
    return _bf16_value(x) if kv_dtype == "bf16" else float(x)


def attn_brute(q, k_cache, v_cache, n_valid, scale, kv_dtype="f32", paged=False,
               page_size=16, block_table=None):
    """q: nested sequence [B][Hq][D] (f32 values); caches as described in the module
    docstring (4-D arrays: [B][Hkv][S][D] or [pages][Hkv][page_size][D]); n_valid: [B].
    Returns out as nested lists [B][Hq][D] of Python floats (double)."""
    B = len(q)
    Hq = len(q[0])
    D = len(q[0][0])
    Hkv = len(k_cache[0])
    group = Hq // Hkv
    out = []
    for b in range(B):
        n = int(n_valid[b])
        if not 1 <= n <= MAX_BRUTE_ROWS:
            raise ValueError("the brute-force loop is for windows of 1..64 rows")
        heads = []
        for h in range(Hq):
            g = h // group
            e = []
            for j in range(n):
                dot = 0.0
                for d in range(D):
                    kx = _element(k_cache, kv_dtype, b, g, j, d, paged, page_size, block_table)
                    dot += float(q[b][h][d]) * kx
                e.append(math.exp(scale * dot))
            total = 0.0
            for j in range(n):
                total += e[j]
            row = []
            for d in range(D):
                acc = 0.0
                for j in range(n):
                    vx = _element(v_cache, kv_dtype, b, g, j, d, paged, page_size, block_table)
                    acc += (e[j] / total) * vx
                row.append(acc)
            heads.append(row)
        out.append(heads)
    return out
