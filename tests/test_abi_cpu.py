"""Host-side checks of the C ABI that need no GPU: the library builds and loads, it
exports every function that include/tts_decode.h declares, the ABI version range
behaves like the probe described on the "qwentts.cpp" tests page (ABI bump section:
both bounds of [min, max] reject), and argument validation rejects bad calls before
any launch."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


# The validation tests pass fake device addresses that must be rejected on the host.
# They only run where no GPU is visible, so that a validation bug can never turn into
# a launch on fake pointers.
no_gpu = pytest.mark.skipif(
    __import__("torch").cuda.is_available(), reason="host-only validation checks")


@pytest.fixture(scope="module")
def tts():
    from autoregressive_codebook_tts_gb300 import build
    build.build()
    from autoregressive_codebook_tts_gb300 import tts as mod
    return mod


def declared_functions():
    src = open(os.path.join(ROOT, "include", "tts_decode.h")).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    return sorted(set(re.findall(r"\b(tts_[a-z0-9_]+)\s*\(", src)))


def test_library_exports_every_declared_function(tts):
    names = declared_functions()
    assert len(names) >= 12
    lib = ctypes.CDLL(tts.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n
    assert sorted(tts.EXPORTED) == names


def test_abi_version_probe(tts):
    """The probe of the "qwentts.cpp" tests page (ABI bump section): both bounds of the
    supported range accept, and the library itself rejects a caller version one below
    the minimum and one above the current version (tts_abi_check, called through the C
    boundary)."""
    lo, hi = tts.abi_min_version(), tts.abi_version()
    assert 1 <= lo <= hi
    ok, err_abi = 0, 8
    assert tts.abi_check(lo) == ok and tts.abi_check(hi) == ok
    assert tts.abi_check(lo - 1) == err_abi
    assert tts.abi_check(hi + 1) == err_abi
    assert tts.abi_check(-(2 ** 31)) == err_abi and tts.abi_check(2 ** 31 - 1) == err_abi
    assert tts.status_str(tts.abi_check(hi + 1)) == "TTS_ERR_ABI"


def test_status_strings(tts):
    assert tts.status_str(0) == "TTS_OK"
    assert tts.status_str(6) == "TTS_ERR_WORKSPACE"
    assert tts.status_str(99) == "TTS_ERR_UNKNOWN"


def test_decode_layer_launch_count(tts):
    # two norm packs, four projections and the decode step (its output goes to the o
    # projection already packed); shapes the layer rejects count 0
    assert tts.tts_decode_layer_launch_count(tts.kv_desc(32, 16, 8, 128, 4096, "f32")) == 7
    assert tts.tts_decode_layer_launch_count(tts.kv_desc(1, 16, 8, 128, 4096, "bf16")) == 7
    assert tts.tts_decode_layer_launch_count(tts.kv_desc(33, 16, 8, 128, 4096, "f32")) == 0
    assert tts.tts_decode_layer_launch_count(tts.kv_desc(4, 16, 8, 96, 4096, "f32")) == 0


def test_prefill_workspace_holds_the_normed_q_rows(tts):
    # every prefill path reads its normed q rows from the workspace (the caller's q is read
    # only), after the attention's own part, at a 256-byte boundary
    for dt in ("f32", "bf16"):
        for B, T in ((1, 2), (4, 7), (1, 128), (2, 33)):
            d = tts.kv_desc(B, 16, 8, 128, 4096, dt)
            need = tts.tts_prefill_workspace_size(d, T, 0)
            assert need >= B * T * 16 * 128 * 4
            assert tts.tts_prefill_workspace_size(d, T, 1) >= B * T * 16 * 128 * 4
    assert tts.tts_prefill_workspace_size(tts.kv_desc(1, 16, 8, 128, 4096, "f32"), 0, 0) == 0


def _call_attn(tts, desc, q=16, k=16, v=16, nv=16, out=16, ws=256, ws_bytes=1 << 20, n_splits=0):
    P = ctypes.c_void_p
    return tts._lib.tts_decode_attn(P(q) if q else None, desc.n_q_heads * desc.head_dim,
                                    P(k) if k else None, P(v) if v else None, ctypes.byref(desc),
                                    P(nv) if nv else None, 0.1, P(out) if out else None,
                                    P(ws) if ws else None, ws_bytes, n_splits, None, None)


@no_gpu
def test_validation_rejects_before_launch(tts):
    d = tts.kv_desc(1, 16, 8, 128, 4096)
    assert _call_attn(tts, d, q=0) == 1                    # NULL
    assert _call_attn(tts, d, k=0) == 1
    assert _call_attn(tts, tts.kv_desc(1, 16, 8, 96, 4096)) == 2   # head_dim
    assert _call_attn(tts, tts.kv_desc(1, 16, 3, 128, 4096)) == 2  # group
    assert _call_attn(tts, tts.kv_desc(1, 16, 2, 128, 4096)) == 2  # group 8
    assert _call_attn(tts, tts.kv_desc(1, 16, 8, 128, 4000)) == 2  # quantum
    bad = tts.kv_desc(1, 16, 8, 128, 4096)
    bad.kv_dtype = 7
    assert _call_attn(tts, bad) == 3
    assert _call_attn(tts, d, k=24) == 5                   # misaligned cache
    assert _call_attn(tts, d, ws=0) == 6                   # no workspace with splits
    assert _call_attn(tts, d, ws_bytes=16) == 6            # short workspace
    assert _call_attn(tts, d, ws=272) == 5                 # workspace not 256-aligned
    paged = tts.kv_desc(1, 16, 8, 128, 4096, paged=True, page_size=16, n_pages=4)
    assert _call_attn(tts, paged) == 1                     # paged without block table
    paged.block_table = 4096
    paged.bt_stride = 256
    paged.page_size = 12
    assert _call_attn(tts, paged) == 4                     # page size not a power of two


def test_workspace_size_grows_with_splits(tts):
    d = tts.kv_desc(32, 16, 8, 128, 4096, kv_dtype="bf16")
    s1 = tts.tts_decode_attn_workspace_size(d, 1)
    s8 = tts.tts_decode_attn_workspace_size(d, 8)
    s16 = tts.tts_decode_attn_workspace_size(d, 16)
    assert 0 < s1 < s8 < s16
    # o partials + (m, l) + tickets, each rounded to 256 bytes
    assert s8 >= 32 * 16 * 8 * (128 + 2) * 4 + 32 * 8 * 4
    assert tts.tts_decode_attn_default_splits(d) >= 1


@no_gpu
def test_other_entry_points_validate(tts):
    P = ctypes.c_void_p
    t = tts.TtsTables()
    t.n_tables, t.vocab, t.hidden = 16, 2048, 1024
    assert tts._lib.tts_frame_embed(ctypes.byref(t), P(16), 16, None, 0, P(16), 1, None, None) == 1
    t.n_tables = 17
    assert tts._lib.tts_frame_embed(ctypes.byref(t), P(16), 16, None, 0, P(16), 1, None, None) == 2
    assert tts._lib.tts_rope_table(None, 16, 128, 1e6, None) == 1
    assert tts._lib.tts_rope_table(P(16), 16, 100, 1e6, None) == 2
    assert tts._lib.tts_rope_table(P(8), 16, 128, 1e6, None) == 5
    d = tts.kv_desc(1, 16, 8, 128, 4096)
    assert tts._lib.tts_kv_set_rows(P(16), P(16), 1024, P(16), P(16), ctypes.byref(d), None, None, None) == 1
    assert tts._lib.tts_kv_set_rows(P(16), P(16), 1000, P(16), P(16), ctypes.byref(d), P(16), None, None) == 2
    assert tts._lib.tts_qk_norm_rope(P(16), 2048, P(16), 1024, P(16), P(16), None, 1, 16, 8, 128,
                                     1e-6, P(16), 4096, None, None) == 1
    assert tts._lib.tts_qk_norm_rope(P(16), 1000, P(16), 1024, P(16), P(16), P(16), 1, 16, 8, 128,
                                     1e-6, P(16), 4096, None, None) == 2


@no_gpu
def test_prefill_sampler_and_table_dtype_validate(tts):
    P = ctypes.c_void_p
    t = tts.TtsTables()
    t.n_tables, t.vocab, t.hidden, t.dtype = 1, 2048, 1024, 5
    assert tts._lib.tts_frame_embed(ctypes.byref(t), P(16), 16, None, 0, P(16), 1, None, None) == 3
    t.tab[0] = 16
    t.dtype, t.hidden = tts.TTS_Q8_0, 1000                     # Q8_0 rows are whole 32-entry blocks
    assert tts._lib.tts_frame_embed(ctypes.byref(t), P(16), 16, None, 0, P(16), 1, None, None) == 2

    d = tts.kv_desc(2, 16, 8, 128, 4096)

    def prefill(q=16, T=4, stride=4096, ws=256, ws_bytes=1 << 20, start=16):
        return tts._lib.tts_prefill_step(P(q) if q else None, P(16), P(16), stride, P(16), P(16),
                                         1e-6, P(16), 4096, P(16), P(16), ctypes.byref(d),
                                         P(start) if start else None, T, 0.1, P(16),
                                         P(ws) if ws else None, ws_bytes, 8, None, None)
    assert prefill(q=0) == 1
    assert prefill(start=0) == 1
    assert prefill(T=0) == 2
    assert prefill(T=40000) == 2                 # B*T above 65535 queries
    assert prefill(stride=1000) == 2             # row shorter than the q heads
    assert prefill(q=24) == 5                    # misaligned q
    assert prefill(ws_bytes=16) == 6             # workspace too small for 8 splits
    assert tts.tts_prefill_workspace_size(d, 4, 8) > tts.tts_decode_attn_workspace_size(d, 8)
    assert tts.tts_prefill_workspace_size(d, 0, 8) == 0

    def sample(lg=16, V=2048, k=50, T=1.0, ctr=64, out=16, stride=2048):
        return tts._lib.tts_sample(P(lg) if lg else None, stride, 4, V, k, T, 1,
                                   P(ctr) if ctr else None, 0, P(out) if out else None, 1, None)
    assert sample(lg=0) == 1
    assert sample(out=0) == 1
    assert sample(ctr=0) == 1                    # sampling needs the counter
    assert sample(V=9000, stride=9000) == 2      # above TTS_MAX_SAMPLE_VOCAB
    assert sample(k=65) == 2                     # above TTS_MAX_TOP_K
    assert sample(V=32, k=40, stride=32) == 2    # k above the vocabulary
    assert sample(T=0.0) == 2
    assert sample(stride=100) == 2               # rows overlap
    assert sample(lg=18) == 5                    # misaligned logits
    assert sample(ctr=68) == 5                   # misaligned counter
    assert tts._lib.tts_counter_advance(None, 1, None) == 1
    assert tts._lib.tts_counter_advance(P(12), 1, None) == 5


@no_gpu
def test_decode_layer_validates(tts):
    P = ctypes.c_void_p
    d = tts.kv_desc(1, 16, 8, 128, 4096)
    size = tts.tts_decode_layer_scratch_size(d, 2048, 6144, 0)
    assert size > tts.tts_decode_attn_workspace_size(d, 0)
    assert tts.tts_decode_layer_scratch_size(d, 2000, 6144, 0) == 0    # hidden not a multiple of 256
    assert tts.tts_decode_layer_scratch_size(d, 2048, 9216, 0) == 0    # intermediate above 8192

    def weights(hidden=2048, inter=6144, w_qkv=16, gamma_attn=16):
        w = tts.TtsLayerWeights()
        w.w_qkv, w.w_o, w.w_gu, w.w_down = w_qkv, 16, 16, 16
        w.gamma_attn, w.gamma_mlp, w.gamma_q, w.gamma_k = gamma_attn, 16, 16, 16
        w.hidden, w.inter = hidden, inter
        return w

    def layer(h=16, w=None, desc=d, eps=1e-6, sc=256, sc_bytes=None):
        w = weights() if w is None else w
        return tts._lib.tts_decode_layer(P(h) if h else None, ctypes.byref(w), eps, P(16), 4096, P(16),
                                         P(16), ctypes.byref(desc), P(16), 0.1, P(sc) if sc else None,
                                         size if sc_bytes is None else sc_bytes, 0, None, None)
    assert layer(h=0) == 1
    assert layer(w=weights(w_qkv=0)) == 1
    assert layer(w=weights(gamma_attn=0)) == 1
    assert layer(sc=0) == 1
    assert layer(desc=tts.kv_desc(33, 16, 8, 128, 4096)) == 2   # more than 32 streams
    assert layer(w=weights(hidden=2000)) == 2
    assert layer(w=weights(inter=9216)) == 2
    assert layer(eps=-1.0) == 2
    assert layer(h=20) == 5                                        # misaligned residual stream
    assert layer(w=weights(w_qkv=24)) == 5                         # misaligned weights
    assert layer(sc=272) == 5                                      # scratch not 256-byte aligned
    assert layer(sc_bytes=1024) == 6                               # scratch too small


def test_binding_constants_match_the_header(tts):
    """The binding re-declares the header's flag bits, dtype codes and limits; they must
    be the header's values, and the library's status names must match the enum."""
    src = open(os.path.join(ROOT, "include", "tts_decode.h")).read()
    defines = {m.group(1): int(m.group(2)) for m in re.finditer(r"#define (TTS_[A-Z0-9_]+) (\d+)u?\b", src)}
    assert tts.TTS_MAX_TABLES == defines["TTS_MAX_TABLES"]
    assert tts.TTS_KV_PREFETCH_BEFORE_WAIT == defines["TTS_KV_PREFETCH_BEFORE_WAIT"]
    for name in ("ID_RANGE", "POS_RANGE", "PAGE", "NVALID", "TIMEOUT"):
        assert getattr(tts, "EFLAG_" + name) == defines["TTS_EFLAG_" + name]
    assert tts._lib.tts_abi_version() == defines["TTS_ABI_VERSION"]
    assert tts._lib.tts_abi_min_version() == defines["TTS_ABI_MIN_VERSION"]
    dt = dict(re.findall(r"(TTS_F32|TTS_BF16|TTS_Q8_0) = (\d+)", src))
    assert (tts.TTS_F32, tts.TTS_BF16, tts.TTS_Q8_0) == (int(dt["TTS_F32"]), int(dt["TTS_BF16"]),
                                                          int(dt["TTS_Q8_0"]))
    for name, code in re.findall(r"\b(TTS_(?:OK|ERR_[A-Z]+)) = (\d+)", src):
        assert tts._lib.tts_status_str(int(code)).decode() == name
