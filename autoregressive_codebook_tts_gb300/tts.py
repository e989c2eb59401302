"""Thin ctypes binding of ``libttsdecode.so`` (declared in ``include/tts_decode.h``).

Argument marshalling only: every function takes device tensors, passes their
pointers, strides and the current CUDA stream to the C entry point of the same name,
and raises ``TtsError`` on a non-OK status.  There is no fallback: if the library has
not been built, importing this module raises.
"""
from __future__ import annotations

import ctypes
import math
import os

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.environ.get("TTS_LIBRARY") or os.path.join(_HERE, "_build", "libttsdecode.so")

if not os.path.exists(LIB_PATH):
    raise ImportError(
        f"{LIB_PATH} is missing: build the CUDA library first "
        "(python -m autoregressive_codebook_tts_gb300.build)")

_lib = ctypes.CDLL(LIB_PATH)

TTS_F32, TTS_BF16, TTS_Q8_0 = 0, 1, 2
Q8_0_BLOCK, Q8_0_BYTES = 32, 34  # entries and bytes of a Q8_0 block
TTS_MAX_TABLES = 16
TTS_KV_PREFETCH_BEFORE_WAIT = 1

EFLAG_ID_RANGE = 1
EFLAG_POS_RANGE = 2
EFLAG_PAGE = 4
EFLAG_NVALID = 8
EFLAG_TIMEOUT = 16

EXPORTED = [
    "tts_abi_version", "tts_abi_min_version", "tts_abi_check", "tts_status_str", "tts_frame_embed",
    "tts_rope_table", "tts_qk_norm_rope", "tts_kv_set_rows", "tts_decode_attn_workspace_size",
    "tts_decode_attn_default_splits", "tts_workspace_init", "tts_decode_attn", "tts_decode_step",
    "tts_decode_step_noalloc",
    "tts_prefill_workspace_size",
    "tts_prefill_launch_count",
    "tts_prefill_step",
    "tts_sample",
    "tts_sample_embed",
    "tts_counter_advance",
    "tts_check_wait_timeout",
    "tts_decode_layer_scratch_size",
    "tts_decode_layer_launch_count",
    "tts_decode_layer",
]


class TtsTables(ctypes.Structure):
    _fields_ = [("tab", ctypes.c_void_p * TTS_MAX_TABLES), ("n_tables", ctypes.c_int32),
                ("vocab", ctypes.c_int32), ("hidden", ctypes.c_int32), ("dtype", ctypes.c_int32)]


class TtsKvDesc(ctypes.Structure):
    _fields_ = [("B", ctypes.c_int32), ("n_q_heads", ctypes.c_int32),
                ("n_kv_heads", ctypes.c_int32), ("head_dim", ctypes.c_int32),
                ("capacity", ctypes.c_int32), ("window_quantum", ctypes.c_int32),
                ("kv_dtype", ctypes.c_int32), ("paged", ctypes.c_int32),
                ("page_size", ctypes.c_int32), ("n_pages", ctypes.c_int32),
                ("bt_stride", ctypes.c_int32), ("flags", ctypes.c_uint32),
                ("block_table", ctypes.c_void_p)]


class TtsLayerWeights(ctypes.Structure):
    _fields_ = [("w_qkv", ctypes.c_void_p), ("w_o", ctypes.c_void_p), ("w_gu", ctypes.c_void_p),
                ("w_down", ctypes.c_void_p), ("gamma_attn", ctypes.c_void_p),
                ("gamma_mlp", ctypes.c_void_p), ("gamma_q", ctypes.c_void_p),
                ("gamma_k", ctypes.c_void_p), ("hidden", ctypes.c_int32), ("inter", ctypes.c_int32)]


_P, _I32, _I64, _F, _D, _SZ = (ctypes.c_void_p, ctypes.c_int32, ctypes.c_int64, ctypes.c_float,
                               ctypes.c_double, ctypes.c_size_t)
_sigs = {
    "tts_abi_version": ([], _I32),
    "tts_abi_min_version": ([], _I32),
    "tts_abi_check": ([_I32], _I32),
    "tts_status_str": ([_I32], ctypes.c_char_p),
    "tts_frame_embed": ([ctypes.POINTER(TtsTables), _P, _I64, _P, _I64, _P, _I32, _P, _P], _I32),
    "tts_rope_table": ([_P, _I32, _I32, _D, _P], _I32),
    "tts_qk_norm_rope": ([_P, _I64, _P, _I64, _P, _P, _P, _I32, _I32, _I32, _I32, _F, _P, _I32,
                          _P, _P], _I32),
    "tts_kv_set_rows": ([_P, _P, _I64, _P, _P, ctypes.POINTER(TtsKvDesc), _P, _P, _P], _I32),
    "tts_decode_attn_workspace_size": ([ctypes.POINTER(TtsKvDesc), _I32], _SZ),
    "tts_decode_attn_default_splits": ([ctypes.POINTER(TtsKvDesc)], _I32),
    "tts_workspace_init": ([_P, _SZ, _P], _I32),
    "tts_decode_attn": ([_P, _I64, _P, _P, ctypes.POINTER(TtsKvDesc), _P, _F, _P, _P, _SZ, _I32,
                         _P, _P], _I32),
    "tts_decode_step": ([_P, _P, _P, _I64, _P, _P, _F, _P, _I32, _P, _P,
                         ctypes.POINTER(TtsKvDesc), _P, _F, _P, _P, _SZ, _I32, _P, _P], _I32),
    "tts_decode_step_noalloc": ([_P, _P, _P, _I64, _P, _P, _F, _P, _I32, _P, _P,
                                 ctypes.POINTER(TtsKvDesc), _P, _F, _P, _I32, _P, _P], _I32),
    "tts_prefill_workspace_size": ([ctypes.POINTER(TtsKvDesc), _I32, _I32], _SZ),
    "tts_prefill_launch_count": ([ctypes.POINTER(TtsKvDesc), _I32, _I32], _I32),
    "tts_sample": ([_P, _I64, _I32, _I32, _I32, _F, ctypes.c_uint64, _P, ctypes.c_uint32, _P, _I64, _P],
                   _I32),
    "tts_sample_embed": ([_P, _I64, _I32, _I32, _I32, _F, ctypes.c_uint64, _P, ctypes.c_uint32, _P, _I64,
                          ctypes.POINTER(TtsTables), _P, _P], _I32),
    "tts_counter_advance": ([_P, ctypes.c_uint64, _P], _I32),
    "tts_check_wait_timeout": ([_P, _P], _I32),
    "tts_decode_layer_scratch_size": ([ctypes.POINTER(TtsKvDesc), _I32, _I32, _I32], _SZ),
    "tts_decode_layer_launch_count": ([ctypes.POINTER(TtsKvDesc)], _I32),
    "tts_decode_layer": ([_P, ctypes.POINTER(TtsLayerWeights), _F, _P, _I32, _P, _P,
                          ctypes.POINTER(TtsKvDesc), _P, _F, _P, _SZ, _I32, _P, _P], _I32),
    "tts_prefill_step": ([_P, _P, _P, _I64, _P, _P, _F, _P, _I32, _P, _P,
                          ctypes.POINTER(TtsKvDesc), _P, _I32, _F, _P, _P, _SZ, _I32, _P, _P], _I32),
}
for _name, (_args, _ret) in _sigs.items():
    _fn = getattr(_lib, _name)
    _fn.argtypes = _args
    _fn.restype = _ret


class TtsError(RuntimeError):
    def __init__(self, status: int, where: str):
        self.status = status
        super().__init__(f"{where}: {_lib.tts_status_str(status).decode()}")


def _check(status: int, where: str):
    if status != 0:
        raise TtsError(status, where)


def _ptr(t):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream=None):
    s = torch.cuda.current_stream() if stream is None else stream
    return ctypes.c_void_p(s.cuda_stream)


def _row_stride(t):
    """Elements between consecutive stream rows of a [B, ...] tensor whose rows are
    contiguous inside (e.g. a column slice of a fused projection buffer)."""
    return t.stride(0)


def abi_version() -> int:
    return _lib.tts_abi_version()


def abi_min_version() -> int:
    return _lib.tts_abi_min_version()


def abi_check(caller_version: int) -> int:
    """The library's own range test of a caller's ABI version: 0 (TTS_OK) or TTS_ERR_ABI."""
    return int(_lib.tts_abi_check(int(caller_version)))


def status_str(status: int) -> str:
    return _lib.tts_status_str(status).decode()


# ---------------------------------------------------------------------------
# Descriptors
# ---------------------------------------------------------------------------
def kv_desc(B, n_q_heads, n_kv_heads, head_dim, capacity, kv_dtype="f32", window_quantum=256,
            paged=False, page_size=16, n_pages=0, block_table=None, flags=0) -> TtsKvDesc:
    d = TtsKvDesc()
    d.B, d.n_q_heads, d.n_kv_heads, d.head_dim, d.capacity = B, n_q_heads, n_kv_heads, head_dim, capacity
    d.window_quantum = window_quantum
    d.kv_dtype = TTS_F32 if kv_dtype == "f32" else TTS_BF16
    d.paged = 1 if paged else 0
    d.page_size = page_size if paged else 0
    d.n_pages = n_pages if paged else 0
    d.bt_stride = block_table.stride(0) if (paged and block_table is not None) else 0
    d.flags = flags
    d.block_table = block_table.data_ptr() if (paged and block_table is not None) else None
    return d


def tables(tabs) -> TtsTables:
    """Table descriptor for f32, bf16 or Q8_0 tables (all of one dtype).  A Q8_0 table is
    a uint8 tensor [vocab][hidden / 32 * 34] of 34-byte blocks (binary16 scale, then 32
    int8 quants)."""
    t = TtsTables()
    dts = {x.dtype for x in tabs}
    if len(dts) != 1 or not dts <= {torch.float32, torch.bfloat16, torch.uint8}:
        raise ValueError("codebook tables must all be float32, all bfloat16 or all uint8 (Q8_0)")
    for i, x in enumerate(tabs):
        t.tab[i] = x.data_ptr()
    t.n_tables = len(tabs)
    if tabs[0].dtype == torch.uint8:
        if tabs[0].shape[1] % Q8_0_BYTES:
            raise ValueError("a Q8_0 row is a whole number of 34-byte blocks")
        t.vocab, t.hidden = tabs[0].shape[0], tabs[0].shape[1] // Q8_0_BYTES * Q8_0_BLOCK
        t.dtype = TTS_Q8_0
    else:
        t.vocab, t.hidden = tabs[0].shape
        t.dtype = TTS_BF16 if tabs[0].dtype == torch.bfloat16 else TTS_F32
    return t


# ---------------------------------------------------------------------------
# Entry points
# ---------------------------------------------------------------------------
def tts_frame_embed(tabs, ids, overlay, out, err_flag=None, stream=None):
    """out[b] = ((E_0[ids[b,0]] + ...) + overlay[b]); tabs: list of [vocab, hidden] f32."""
    t = tables(tabs) if not isinstance(tabs, TtsTables) else tabs
    _check(_lib.tts_frame_embed(ctypes.byref(t), _ptr(ids), ids.stride(0), _ptr(overlay),
                                0 if overlay is None else overlay.stride(0), _ptr(out),
                                out.shape[0], _ptr(err_flag), _stream(stream)), "tts_frame_embed")


def tts_rope_table(cs, max_pos, head_dim, base, stream=None):
    _check(_lib.tts_rope_table(_ptr(cs), max_pos, head_dim, float(base), _stream(stream)),
           "tts_rope_table")


def tts_qk_norm_rope(q, k, gamma_q, gamma_k, pos, n_q_heads, n_kv_heads, head_dim, eps, cs,
                     max_pos, err_flag=None, stream=None):
    _check(_lib.tts_qk_norm_rope(_ptr(q), _row_stride(q), _ptr(k), _row_stride(k), _ptr(gamma_q),
                                 _ptr(gamma_k), _ptr(pos), q.shape[0], n_q_heads, n_kv_heads,
                                 head_dim, float(eps), _ptr(cs), max_pos, _ptr(err_flag),
                                 _stream(stream)), "tts_qk_norm_rope")


def tts_kv_set_rows(k, v, k_cache, v_cache, desc: TtsKvDesc, dst_pos, err_flag=None, stream=None):
    assert k.stride(0) == v.stride(0), "k and v rows must share one stride"
    _check(_lib.tts_kv_set_rows(_ptr(k), _ptr(v), _row_stride(k), _ptr(k_cache), _ptr(v_cache),
                                ctypes.byref(desc), _ptr(dst_pos), _ptr(err_flag),
                                _stream(stream)), "tts_kv_set_rows")


def tts_decode_attn_workspace_size(desc: TtsKvDesc, n_splits=0) -> int:
    return int(_lib.tts_decode_attn_workspace_size(ctypes.byref(desc), n_splits))


def tts_decode_attn_default_splits(desc: TtsKvDesc) -> int:
    return int(_lib.tts_decode_attn_default_splits(ctypes.byref(desc)))


def tts_workspace_init(ws, stream=None):
    _check(_lib.tts_workspace_init(_ptr(ws), ws.numel() * ws.element_size(), _stream(stream)),
           "tts_workspace_init")


def workspace(desc: TtsKvDesc, n_splits=0, device="cuda", stream=None):
    """Allocate (through torch) and clear a workspace for desc/n_splits."""
    n = max(tts_decode_attn_workspace_size(desc, n_splits), 256)
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    tts_workspace_init(ws, stream)
    return ws


def tts_decode_attn(q, k_cache, v_cache, desc: TtsKvDesc, n_valid, scale, out, ws, n_splits=0,
                    err_flag=None, stream=None):
    _check(_lib.tts_decode_attn(_ptr(q), _row_stride(q), _ptr(k_cache), _ptr(v_cache),
                                ctypes.byref(desc), _ptr(n_valid), float(scale), _ptr(out),
                                _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                                n_splits, _ptr(err_flag), _stream(stream)), "tts_decode_attn")


def tts_decode_step(q, k, v, gamma_q, gamma_k, eps, cs, max_pos, k_cache, v_cache,
                    desc: TtsKvDesc, cur_len, scale, out, ws, n_splits=0, err_flag=None,
                    stream=None):
    stride = _row_stride(q)
    assert k.stride(0) == stride and v.stride(0) == stride, "q, k, v rows must share one stride"
    _check(_lib.tts_decode_step(_ptr(q), _ptr(k), _ptr(v), stride, _ptr(gamma_q), _ptr(gamma_k),
                                float(eps), _ptr(cs), max_pos, _ptr(k_cache), _ptr(v_cache),
                                ctypes.byref(desc), _ptr(cur_len), float(scale), _ptr(out),
                                _ptr(ws), 0 if ws is None else ws.numel() * ws.element_size(),
                                n_splits, _ptr(err_flag), _stream(stream)), "tts_decode_step")


def tts_decode_step_noalloc(q, k, v, gamma_q, gamma_k, eps, cs, max_pos, k_cache, v_cache,
                            desc: TtsKvDesc, cur_len, scale, out, n_splits=0, err_flag=None,
                            stream=None):
    """tts_decode_step with the library's built-in scratch instead of a workspace (for
    callers that cannot allocate device memory); see include/tts_decode.h."""
    stride = _row_stride(q)
    assert k.stride(0) == stride and v.stride(0) == stride, "q, k, v rows must share one stride"
    _check(_lib.tts_decode_step_noalloc(_ptr(q), _ptr(k), _ptr(v), stride, _ptr(gamma_q),
                                        _ptr(gamma_k), float(eps), _ptr(cs), max_pos,
                                        _ptr(k_cache), _ptr(v_cache), ctypes.byref(desc),
                                        _ptr(cur_len), float(scale), _ptr(out), n_splits,
                                        _ptr(err_flag), _stream(stream)), "tts_decode_step_noalloc")


def tts_prefill_workspace_size(desc: TtsKvDesc, T: int, n_splits=0) -> int:
    return int(_lib.tts_prefill_workspace_size(ctypes.byref(desc), T, n_splits))


def tts_prefill_launch_count(desc: TtsKvDesc, T: int, n_splits=0) -> int:
    return int(_lib.tts_prefill_launch_count(ctypes.byref(desc), T, n_splits))


def prefill_workspace(desc: TtsKvDesc, T: int, n_splits=0, device="cuda", stream=None):
    """Allocate (through torch) and clear a workspace for a prefill of T positions."""
    n = max(tts_prefill_workspace_size(desc, T, n_splits), 256)
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    tts_workspace_init(ws, stream)
    return ws


def tts_prefill_step(q, k, v, gamma_q, gamma_k, eps, cs, max_pos, k_cache, v_cache,
                     desc: TtsKvDesc, start_pos, T, scale, out, ws, n_splits=0, err_flag=None,
                     stream=None):
    """q, k, v: [B*T, ...] row views (row r = b*T + t), read only."""
    stride = _row_stride(q)
    assert k.stride(0) == stride and v.stride(0) == stride, "q, k, v rows must share one stride"
    _check(_lib.tts_prefill_step(_ptr(q), _ptr(k), _ptr(v), stride, _ptr(gamma_q), _ptr(gamma_k),
                                 float(eps), _ptr(cs), max_pos, _ptr(k_cache), _ptr(v_cache),
                                 ctypes.byref(desc), _ptr(start_pos), int(T), float(scale),
                                 _ptr(out), _ptr(ws),
                                 0 if ws is None else ws.numel() * ws.element_size(),
                                 n_splits, _ptr(err_flag), _stream(stream)), "tts_prefill_step")


def tts_sample(logits, top_k, temperature, seed, counter, out_ids, draw=0, stream=None):
    """logits [B, V] f32 (rows may be strided); out_ids: int32 tensor whose first dim
    indexes streams (a column view of an ids buffer is fine); draw: the third Philox
    counter word (e.g. the sub-step within a frame)."""
    B, V = logits.shape
    _check(_lib.tts_sample(_ptr(logits), logits.stride(0), B, V, int(top_k), float(temperature),
                           ctypes.c_uint64(int(seed) & ((1 << 64) - 1)), _ptr(counter),
                           ctypes.c_uint32(int(draw)), _ptr(out_ids), out_ids.stride(0),
                           _stream(stream)), "tts_sample")


def tts_sample_embed(logits, top_k, temperature, seed, counter, out_ids, table, out_rows, draw=0,
                     stream=None):
    """tts_sample, then the drawn tokens' rows of one table into out_rows [B, hidden] f32,
    in one launch; table: a TtsTables of one table or a list of one tensor."""
    B, V = logits.shape
    t = tables(table) if not isinstance(table, TtsTables) else table
    _check(_lib.tts_sample_embed(_ptr(logits), logits.stride(0), B, V, int(top_k), float(temperature),
                                 ctypes.c_uint64(int(seed) & ((1 << 64) - 1)), _ptr(counter),
                                 ctypes.c_uint32(int(draw)), _ptr(out_ids), out_ids.stride(0),
                                 ctypes.byref(t), _ptr(out_rows), _stream(stream)), "tts_sample_embed")


def tts_counter_advance(counter, by=1, stream=None):
    _check(_lib.tts_counter_advance(_ptr(counter), ctypes.c_uint64(int(by)), _stream(stream)),
           "tts_counter_advance")


def tts_check_wait_timeout(err_flag, stream=None):
    """One bounded wait that nothing ends: sets TTS_EFLAG_TIMEOUT in err_flag after about
    a second."""
    _check(_lib.tts_check_wait_timeout(_ptr(err_flag), _stream(stream)), "tts_check_wait_timeout")


def layer_weights(w_qkv, w_o, w_gu, w_down, gamma_attn, gamma_mlp, gamma_q, gamma_k) -> TtsLayerWeights:
    """Descriptor of one layer's weights: bf16 matrices, f32 norm weights (device tensors;
    the caller keeps them alive)."""
    for m in (w_qkv, w_o, w_gu, w_down):
        if m.dtype != torch.bfloat16 or not m.is_contiguous():
            raise ValueError("layer weight matrices must be contiguous bfloat16")
    t = TtsLayerWeights()
    t.w_qkv, t.w_o, t.w_gu, t.w_down = (m.data_ptr() for m in (w_qkv, w_o, w_gu, w_down))
    t.gamma_attn, t.gamma_mlp, t.gamma_q, t.gamma_k = (
        g.data_ptr() for g in (gamma_attn, gamma_mlp, gamma_q, gamma_k))
    t.hidden = w_qkv.shape[1]
    t.inter = w_down.shape[1]
    return t


def tts_decode_layer_launch_count(desc: TtsKvDesc) -> int:
    return int(_lib.tts_decode_layer_launch_count(ctypes.byref(desc)))


def tts_decode_layer_scratch_size(desc: TtsKvDesc, hidden, inter, n_splits=0) -> int:
    return int(_lib.tts_decode_layer_scratch_size(ctypes.byref(desc), hidden, inter, n_splits))


def layer_scratch(desc: TtsKvDesc, hidden, inter, n_splits=0, device="cuda", stream=None):
    """Allocate (through torch) and clear the scratch of a decode layer."""
    n = max(tts_decode_layer_scratch_size(desc, hidden, inter, n_splits), 256)
    ws = torch.empty(n, dtype=torch.uint8, device=device)
    tts_workspace_init(ws, stream)
    return ws


def tts_decode_layer(h, weights: TtsLayerWeights, eps, cs, max_pos, k_cache, v_cache,
                     desc: TtsKvDesc, cur_len, scale, scratch, n_splits=0, err_flag=None,
                     stream=None):
    _check(_lib.tts_decode_layer(_ptr(h), ctypes.byref(weights), float(eps), _ptr(cs), max_pos,
                                 _ptr(k_cache), _ptr(v_cache), ctypes.byref(desc), _ptr(cur_len),
                                 float(scale), _ptr(scratch), scratch.numel() * scratch.element_size(),
                                 n_splits, _ptr(err_flag), _stream(stream)), "tts_decode_layer")


def default_scale(head_dim: int) -> float:
    return 1.0 / math.sqrt(head_dim)
