"""Shared helpers of the GPU parity tests: seeded layer inputs (from the workloads
module), device copies, the per-row error metric, and oracle calls on host copies."""
import math

import numpy as np
import torch

import oracle
from autoregressive_codebook_tts_gb300 import workloads as W


def row_rel_err(got, ref):
    """Per (stream, head) row: max_d |got - ref| / max(max_d |ref|, 1e-30); returns the
    largest over all rows."""
    g = np.asarray(got, np.float64)
    r = np.asarray(ref, np.float64)
    num = np.abs(g - r).max(axis=-1)
    den = np.maximum(np.abs(r).max(axis=-1), 1e-30)
    return float((num / den).max())


ATTN_TOL = {"f32": 1e-5, "bf16": 2e-3}
NORM_TOL = 2e-6


def cache_np(t):
    """Host numpy view of a cache tensor: f32 as float32, bf16 as uint16 bits."""
    t = t.detach().cpu().contiguous()
    if t.dtype == torch.bfloat16:
        return t.view(torch.int16).numpy().view(np.uint16).copy()
    return t.numpy().copy()


def bits(a):
    a = np.ascontiguousarray(a)
    return a.view(np.uint32) if a.dtype == np.float32 else a.view(np.uint16)


class Layer:
    """One layer's worth of inputs for B streams, on the host and on the device."""

    def __init__(self, w: W.Workload, seed: int, cur_len=None, device="cuda", poison=True,
                 block_tab=None):
        self.w = w
        self.cur = (W.cur_lens(w, seed) if cur_len is None
                    else torch.as_tensor(cur_len, dtype=torch.int32)).contiguous()
        if w.paged:
            pages_per = w.capacity // w.page_size
            self.bt = (W.block_table(w.B, pages_per, w.n_pages, seed + 1)
                       if block_tab is None else block_tab)
        else:
            self.bt = None
        self.K, self.V = W.cache(w, self.cur.tolist(), seed + 2, block_tab=self.bt, poison=poison)
        self.qkv, q, k, v = W.qkv(w.B, w.n_q_heads, w.n_kv_heads, w.head_dim, seed + 3)
        self.gq = W.gamma(w.head_dim, seed + 4)
        self.gk = W.gamma(w.head_dim, seed + 5)
        dev = device
        self.d_qkv = self.qkv.to(dev)
        qd, kd = w.n_q_heads * w.head_dim, w.n_kv_heads * w.head_dim
        self.d_q = self.d_qkv[:, :qd]
        self.d_k = self.d_qkv[:, qd:qd + kd]
        self.d_v = self.d_qkv[:, qd + kd:]
        self.d_K, self.d_V = self.K.to(dev), self.V.to(dev)
        self.d_gq, self.d_gk = self.gq.to(dev), self.gk.to(dev)
        self.d_cur = self.cur.to(dev)
        self.d_bt = None if self.bt is None else self.bt.to(dev)

    # host views in oracle shapes
    def q_np(self):
        w = self.w
        return self.qkv[:, :w.n_q_heads * w.head_dim].numpy().reshape(w.B, w.n_q_heads, w.head_dim)

    def k_np(self):
        w = self.w
        qd, kd = w.n_q_heads * w.head_dim, w.n_kv_heads * w.head_dim
        return self.qkv[:, qd:qd + kd].numpy().reshape(w.B, w.n_kv_heads, w.head_dim)

    def v_np(self):
        w = self.w
        qd, kd = w.n_q_heads * w.head_dim, w.n_kv_heads * w.head_dim
        return self.qkv[:, qd + kd:].numpy().reshape(w.B, w.n_kv_heads, w.head_dim)

    def layout(self):
        w = self.w
        return oracle.KvLayout(w.B, w.n_kv_heads, w.head_dim, w.capacity, w.kv_dtype,
                               paged=w.paged, page_size=w.page_size, n_pages=w.n_pages,
                               block_table=None if self.bt is None else self.bt.numpy())

    def desc(self, tts, flags=0, window_quantum=None):
        w = self.w
        return tts.kv_desc(w.B, w.n_q_heads, w.n_kv_heads, w.head_dim, w.capacity, w.kv_dtype,
                           window_quantum=w.window_quantum if window_quantum is None else window_quantum,
                           paged=w.paged, page_size=w.page_size, n_pages=w.n_pages,
                           block_table=self.d_bt, flags=flags)


def rope_table(tts, max_pos, head_dim, base, device="cuda"):
    cs = torch.empty(max_pos, head_dim // 2, 2, dtype=torch.float32, device=device)
    tts.tts_rope_table(cs, max_pos, head_dim, base)
    return cs


def scale_of(w):
    return 1.0 / math.sqrt(w.head_dim)
