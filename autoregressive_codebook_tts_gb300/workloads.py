"""Seeded synthetic inputs for the per-frame decode hot path.

This module only draws random numbers and lays them out; it holds none of the
method's arithmetic (no sums, norms, rotations or attention).  Both the CUDA
library's tests/bench and the CPU oracle's tests take their inputs from here, so
the two sides always see identical bytes.

The shapes follow the five workloads the library is measured and checked on:

* ``tiny``      -- 1 stream, 1 layer, hidden 1024, 16 q / 8 kv heads, head_dim 128,
  f32; 16 codebook tables of 2048 x 1024 ~N(0, 0.02) plus an overlay row; cache of
  256 slots with cur_len = 37 filled ~N(0, 1); seed 0.
* ``talker``    -- 1 stream, 28 layers, hidden 2048, 16/8 heads, head_dim 128, f32
  KV cache of 4096 positions per layer; 16 codebooks 2048 x 2048; cur_len in
  {255, 1023, 2047, 4095}; eps 1e-6, RoPE base 1e6.
* ``batched``   -- 32 streams, talker shapes, bf16 KV, cur_len ~ U[64, 2048] per stream.
* ``predictor`` -- 32 streams, 5 layers, hidden 1024, 16/8 heads, head_dim 64, f32
  KV; 16-slot cache reset per frame; 15 group tables 2048 x 1024.
* ``paged``     -- 8 streams, talker shapes, bf16 KV in 16-token pages addressed by a
  per-stream block table (a random permutation of a 4096-page pool per layer),
  cur_len ~ U[3072, 4095].
"""
from __future__ import annotations

from dataclasses import dataclass, field, replace

import numpy as np
import torch


@dataclass(frozen=True)
class Workload:
    name: str
    B: int
    layers: int
    hidden: int
    n_q_heads: int
    n_kv_heads: int
    head_dim: int
    capacity: int
    kv_dtype: str          # "f32" | "bf16"
    n_tables: int = 16
    vocab: int = 2048
    table_std: float = 0.02
    eps: float = 1e-6
    rope_base: float = 1e6
    window_quantum: int = 256
    paged: bool = False
    page_size: int = 16
    n_pages: int = 0
    cur_len_lo: int = 0     # inclusive
    cur_len_hi: int = 0     # inclusive
    cur_len_fixed: tuple = field(default=())

    @property
    def group(self):
        return self.n_q_heads // self.n_kv_heads

    @property
    def elem_bytes(self):
        return 4 if self.kv_dtype == "f32" else 2


WORKLOADS = {
    "tiny": Workload("tiny", B=1, layers=1, hidden=1024, n_q_heads=16, n_kv_heads=8,
                     head_dim=128, capacity=256, kv_dtype="f32", cur_len_fixed=(37,)),
    "talker": Workload("talker", B=1, layers=28, hidden=2048, n_q_heads=16, n_kv_heads=8,
                       head_dim=128, capacity=4096, kv_dtype="f32",
                       cur_len_fixed=(255, 1023, 2047, 4095)),
    "batched": Workload("batched", B=32, layers=28, hidden=2048, n_q_heads=16, n_kv_heads=8,
                        head_dim=128, capacity=4096, kv_dtype="bf16",
                        cur_len_lo=64, cur_len_hi=2048),
    "predictor": Workload("predictor", B=32, layers=5, hidden=1024, n_q_heads=16,
                          n_kv_heads=8, head_dim=64, capacity=16, kv_dtype="f32",
                          n_tables=15, window_quantum=16),
    "paged": Workload("paged", B=8, layers=28, hidden=2048, n_q_heads=16, n_kv_heads=8,
                      head_dim=128, capacity=4096, kv_dtype="bf16", paged=True,
                      page_size=16, n_pages=4096, cur_len_lo=3072, cur_len_hi=4095),
}


def workload(name: str, **overrides) -> Workload:
    return replace(WORKLOADS[name], **overrides)


def _gen(seed: int, device="cpu") -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(int(seed))
    return g


# ---------------------------------------------------------------------------
# Frame-input composition inputs
# ---------------------------------------------------------------------------
def tables(n_tables: int, vocab: int, hidden: int, seed: int, std: float = 0.02,
           device="cpu"):
    """n_tables codebook tables [vocab][hidden] f32 ~N(0, std)."""
    g = _gen(seed, device)
    return [torch.randn(vocab, hidden, generator=g, device=device, dtype=torch.float32) * std
            for _ in range(n_tables)]


def q8_0_tables(n_tables: int, vocab: int, hidden: int, seed: int, device="cpu"):
    """n_tables Q8_0 codebook tables as uint8 [vocab][hidden / 32 * 34]: per 34-byte block
    a binary16 scale (random magnitude in [1e-4, 4e-4], random sign) then 32 int8 quants
    uniform in [-127, 127], so entries span about +-0.05 like the f32 tables.  Only random
    bytes laid out in the block format; no quantisation is done here."""
    g = _gen(seed)
    nb = hidden // 32
    out = []
    for _ in range(n_tables):
        mag = torch.rand(vocab, nb, 1, generator=g) * 3e-4 + 1e-4
        sign = torch.randint(0, 2, (vocab, nb, 1), generator=g) * 2 - 1
        d = (mag * sign).to(torch.float16).view(torch.uint8).reshape(vocab, nb, 2)
        q = torch.randint(-127, 128, (vocab, nb, 32), generator=g, dtype=torch.int8).view(torch.uint8)
        out.append(torch.cat([d, q], dim=2).reshape(vocab, nb * 34).contiguous().to(device))
    return out


def code_ids(B: int, n_tables: int, vocab: int, seed: int) -> torch.Tensor:
    """Code ids uniform in [0, vocab), int32 [B][n_tables]."""
    return torch.randint(0, vocab, (B, n_tables), generator=_gen(seed), dtype=torch.int32)


def overlay(B: int, hidden: int, seed: int, std: float = 0.02) -> torch.Tensor:
    """Text/pad overlay rows ~N(0, std), f32 [B][hidden]."""
    return torch.randn(B, hidden, generator=_gen(seed), dtype=torch.float32) * std


# ---------------------------------------------------------------------------
# Per-layer step inputs
# ---------------------------------------------------------------------------
def qkv(B: int, n_q_heads: int, n_kv_heads: int, head_dim: int, seed: int, device="cpu"):
    """One fused projection output per stream, laid out [q | k | v] in one row of
    (Hq + 2 Hkv) * D floats, ~N(0, 1).  Returns (qkv_rows, q_view, k_view, v_view);
    the views are strided slices of the same rows."""
    g = _gen(seed, device)
    width = (n_q_heads + 2 * n_kv_heads) * head_dim
    rows = torch.randn(B, width, generator=g, device=device, dtype=torch.float32)
    qd, kd = n_q_heads * head_dim, n_kv_heads * head_dim
    return rows, rows[:, :qd], rows[:, qd:qd + kd], rows[:, qd + kd:]


def gamma(head_dim: int, seed: int, lo: float = 0.5, hi: float = 1.5) -> torch.Tensor:
    """Per-dimension norm weight, U(lo, hi), f32 [D]."""
    return torch.rand(head_dim, generator=_gen(seed), dtype=torch.float32) * (hi - lo) + lo


def logits(n: int, B: int, vocab: int, seed: int, scale: float = 2.0) -> torch.Tensor:
    """Synthetic sampler inputs ~N(0, scale^2), f32 [n][B][vocab] (the output heads that
    would produce them are outside this path)."""
    return torch.randn(n, B, vocab, generator=_gen(seed), dtype=torch.float32) * scale


def cur_lens(w: Workload, seed: int) -> torch.Tensor:
    """Positions of the token decoded this step, int32 [B] (rows [0, cur_len) are
    already in the cache)."""
    if w.cur_len_fixed:
        vals = [w.cur_len_fixed[b % len(w.cur_len_fixed)] for b in range(w.B)]
        return torch.tensor(vals, dtype=torch.int32)
    return torch.randint(w.cur_len_lo, w.cur_len_hi + 1, (w.B,), generator=_gen(seed),
                         dtype=torch.int32)


def block_table(B: int, pages_per_stream: int, n_pages: int, seed: int) -> torch.Tensor:
    """Each stream's pages drawn without replacement from a shuffled pool, int32
    [B][pages_per_stream]."""
    perm = torch.randperm(n_pages, generator=_gen(seed))
    need = B * pages_per_stream
    if need > n_pages:
        raise ValueError("pool too small for every stream's pages")
    return perm[:need].reshape(B, pages_per_stream).to(torch.int32).contiguous()


POISON_F32 = float("nan")
POISON_BF16_BITS = 0x7FC0   # a quiet NaN in bf16


def cache(w: Workload, filled, seed: int, block_tab=None, poison=True, device="cpu"):
    """One layer's K and V caches in the library's head-major layout.

    Rows [0, filled[b]) of stream b are ~N(0, 1) (f32, or rounded to bf16 by torch's
    own conversion); every other slot holds a poison value (NaN) when ``poison`` is
    set, else more N(0, 1) data.  Contiguous: [B][Hkv][S][D].  Paged: a pool
    [n_pages][Hkv][page_size][D] addressed through ``block_tab``.
    Returns (K, V); bf16 caches come back as torch.bfloat16 tensors.
    """
    g = _gen(seed, device)
    D, Hkv = w.head_dim, w.n_kv_heads
    if w.paged:
        shape = (w.n_pages, Hkv, w.page_size, D)
    else:
        shape = (w.B, Hkv, w.capacity, D)
    out = []
    for _ in range(2):
        t = torch.randn(*shape, generator=g, device=device, dtype=torch.float32)
        if w.kv_dtype == "bf16":
            t = t.to(torch.bfloat16)
        out.append(t)
    if poison:
        filled = [int(x) for x in filled]
        for t in out:
            if w.paged:
                used = torch.zeros(w.n_pages, w.page_size, dtype=torch.bool)
                bt = block_tab.cpu()
                for b in range(w.B):
                    for j0 in range(0, filled[b], w.page_size):
                        n = min(w.page_size, filled[b] - j0)
                        used[int(bt[b, j0 // w.page_size]), :n] = True
                mask = (~used).to(device)[:, None, :, None].expand(shape)
                t.masked_fill_(mask, POISON_F32)
            else:
                for b in range(w.B):
                    t[b, :, filled[b]:, :] = POISON_F32
    return out[0], out[1]
