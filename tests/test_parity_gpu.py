"""GPU parity of every step of the decode hot path against the CPU oracle, called
through the C ABI (ctypes binding) on seeded synthetic inputs.

Bars: bit-exact for the gather-sum, the set_rows write (f32 copy and bf16
round-to-nearest-even) and every byte the kernels must leave alone; per-row max
relative error <= 1e-5 (f32 KV) / 2e-3 (bf16 KV) for attention outputs; <= 2e-6 for
the norm+RoPE rows (f32 arithmetic: ~log2(D) rounding steps in the sum of squares plus
a handful in the scaling and the rotation, each 2^-24, against the oracle's
once-rounded double result).
"""
import math

import numpy as np
import pytest
import torch

import oracle
from autoregressive_codebook_tts_gb300 import workloads as W
from gpu_helpers import (ATTN_TOL, NORM_TOL, Layer, bits, cache_np, rope_table, row_rel_err,
                         scale_of)

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tts(cuda_dev):
    from autoregressive_codebook_tts_gb300 import build
    build.build()
    from autoregressive_codebook_tts_gb300 import tts as mod
    return mod


def err_flag():
    return torch.zeros(1, dtype=torch.int32, device="cuda")


# ---------------------------------------------------------------------------
# Step 1: frame-input composition (bit-exact)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("n_tables,hidden,B,overlay", [
    (16, 1024, 1, True),     # tiny workload
    (16, 2048, 32, True),    # batched talker frame
    (1, 1024, 32, False),    # predictor sub-step: one group table, no overlay
    (5, 36, 3, True),        # ragged hidden (not a multiple of the block)
])
def test_frame_embed_bit_exact(tts, n_tables, hidden, B, overlay):
    tabs = W.tables(n_tables, 2048, hidden, seed=0)
    ids = W.code_ids(B, n_tables, 2048, seed=1)
    ov = W.overlay(B, hidden, seed=2) if overlay else None
    ref, flag = oracle.frame_embed([t.numpy() for t in tabs], ids.numpy(),
                                   None if ov is None else ov.numpy())
    d_tabs = [t.cuda() for t in tabs]
    out = torch.full((B, hidden), float("nan"), device="cuda")
    ef = err_flag()
    tts.tts_frame_embed(d_tabs, ids.cuda(), None if ov is None else ov.cuda(), out, ef)
    torch.cuda.synchronize()
    assert flag == 0 and ef.item() == 0
    assert np.array_equal(bits(out.cpu().numpy()), bits(ref))


@pytest.mark.parametrize("n_tables,hidden,B,overlay", [
    (16, 2048, 32, True),    # batched talker frame from bf16 tables
    (1, 1024, 32, False),    # predictor sub-step
])
def test_frame_embed_bf16_tables_bit_exact(tts, n_tables, hidden, B, overlay):
    """bf16 codebook tables: every entry widened exactly, then the same f32 sum."""
    tabs = [t.to(torch.bfloat16) for t in W.tables(n_tables, 2048, hidden, seed=3)]
    ids = W.code_ids(B, n_tables, 2048, seed=4)
    ov = W.overlay(B, hidden, seed=5) if overlay else None
    ref, flag = oracle.frame_embed([t.view(torch.int16).numpy().view(np.uint16) for t in tabs],
                                   ids.numpy(), None if ov is None else ov.numpy())
    out = torch.full((B, hidden), float("nan"), device="cuda")
    ef = err_flag()
    tts.tts_frame_embed([t.cuda() for t in tabs], ids.cuda(), None if ov is None else ov.cuda(), out, ef)
    torch.cuda.synchronize()
    assert flag == 0 and ef.item() == 0
    assert np.array_equal(bits(out.cpu().numpy()), bits(ref))


@pytest.mark.parametrize("n_tables,hidden,B,overlay", [
    (16, 2048, 32, True),    # batched talker frame from Q8_0 tables
    (1, 1024, 32, False),    # predictor sub-step
    (3, 32, 5, True),        # one block per row
])
def test_frame_embed_q8_0_tables_bit_exact(tts, n_tables, hidden, B, overlay):
    """Q8_0 codebook tables (34-byte blocks: binary16 scale, 32 int8 quants): every entry
    is the exact f32 product scale * quant, then the same f32 sum as for f32 tables."""
    tabs = W.q8_0_tables(n_tables, 2048, hidden, seed=6)
    ids = W.code_ids(B, n_tables, 2048, seed=7)
    ov = W.overlay(B, hidden, seed=8) if overlay else None
    ref, flag = oracle.frame_embed([t.numpy() for t in tabs], ids.numpy(),
                                   None if ov is None else ov.numpy())
    out = torch.full((B, hidden), float("nan"), device="cuda")
    ef = err_flag()
    tts.tts_frame_embed([t.cuda() for t in tabs], ids.cuda(), None if ov is None else ov.cuda(), out, ef)
    torch.cuda.synchronize()
    assert flag == 0 and ef.item() == 0
    assert np.array_equal(bits(out.cpu().numpy()), bits(ref))


def test_frame_embed_clamps_and_flags_bad_ids(tts):
    tabs = W.tables(3, 64, 16, seed=3)
    ids = torch.tensor([[0, 70, 5], [-3, 1, 63]], dtype=torch.int32)
    ref, flag = oracle.frame_embed([t.numpy() for t in tabs], ids.numpy(), None)
    out = torch.empty(2, 16, device="cuda")
    ef = err_flag()
    tts.tts_frame_embed([t.cuda() for t in tabs], ids.cuda(), None, out, ef)
    torch.cuda.synchronize()
    assert flag == 1 and ef.item() & tts.EFLAG_ID_RANGE
    assert np.array_equal(bits(out.cpu().numpy()), bits(ref))


# ---------------------------------------------------------------------------
# RoPE table and step 2: q/k RMSNorm + RoPE
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("head_dim", [64, 128])
def test_rope_table_matches_oracle_angles(tts, head_dim):
    cs = rope_table(tts, 4096, head_dim, 1e6).cpu().numpy()
    for pos in [0, 1, 37, 255, 1023, 2047, 4095]:
        for i in range(0, head_dim // 2, 7):
            c, s = oracle.rope_angle(pos, i, head_dim, 1e6)
            np.testing.assert_array_max_ulp(cs[pos, i], np.array([c, s], np.float32), maxulp=1)


@pytest.mark.parametrize("name", ["tiny", "batched", "predictor"])
def test_qk_norm_rope_matches_oracle(tts, name):
    w = W.workload(name)
    cur = [b % 16 for b in range(w.B)] if name == "predictor" else None
    L = Layer(w, seed=10, cur_len=cur, poison=False)
    cs = rope_table(tts, w.capacity, w.head_dim, w.rope_base)
    ef = err_flag()
    pos = L.d_cur
    tts.tts_qk_norm_rope(L.d_q, L.d_k, L.d_gq, L.d_gk, pos, w.n_q_heads, w.n_kv_heads,
                         w.head_dim, w.eps, cs, w.capacity, ef)
    torch.cuda.synchronize()
    assert ef.item() == 0
    eps = np.float32(w.eps)
    ref_q = oracle.rms_norm_rope(L.q_np(), L.gq.numpy(), eps, L.cur.numpy(), w.rope_base)
    ref_k = oracle.rms_norm_rope(L.k_np(), L.gk.numpy(), eps, L.cur.numpy(), w.rope_base)
    got = L.d_qkv.cpu()
    qd, kd = w.n_q_heads * w.head_dim, w.n_kv_heads * w.head_dim
    got_q = got[:, :qd].numpy().reshape(ref_q.shape)
    got_k = got[:, qd:qd + kd].numpy().reshape(ref_k.shape)
    assert row_rel_err(got_q, ref_q) <= NORM_TOL
    assert row_rel_err(got_k, ref_k) <= NORM_TOL
    # v is not touched
    assert torch.equal(got[:, qd + kd:], L.qkv[:, qd + kd:])


def test_rope_at_position_zero_is_the_norm_alone(tts):
    w = W.workload("tiny")
    L = Layer(w, seed=11, cur_len=[0], poison=False)
    cs = rope_table(tts, w.capacity, w.head_dim, w.rope_base)
    assert torch.equal(cs[0, :, 0].cpu(), torch.ones(w.head_dim // 2))
    assert torch.equal(cs[0, :, 1].cpu(), torch.zeros(w.head_dim // 2))
    tts.tts_qk_norm_rope(L.d_q, L.d_k, L.d_gq, L.d_gk, L.d_cur, w.n_q_heads, w.n_kv_heads,
                         w.head_dim, w.eps, cs, w.capacity)
    ref = torch.nn.functional.rms_norm(torch.from_numpy(L.q_np()).double(), (w.head_dim,),
                                       weight=L.gq.double(), eps=float(np.float32(w.eps)))
    got = L.d_q.cpu().reshape(ref.shape).double()
    assert row_rel_err(got.numpy(), ref.numpy()) <= NORM_TOL


# ---------------------------------------------------------------------------
# Step 3: set_rows (bit-exact, nothing else touched)
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("paged", [False, True])
@pytest.mark.parametrize("kv_dtype", ["f32", "bf16"])
def test_set_rows_bit_exact(tts, paged, kv_dtype):
    w = W.workload("paged" if paged else "batched", kv_dtype=kv_dtype, B=4, n_pages=1100)
    L = Layer(w, seed=20, cur_len=[0, 17, 1000, 4095])
    desc = L.desc(tts)
    ef = err_flag()
    tts.tts_kv_set_rows(L.d_k, L.d_v, L.d_K, L.d_V, desc, L.d_cur, ef)
    torch.cuda.synchronize()
    assert ef.item() == 0
    hk, hv = cache_np(L.K), cache_np(L.V)
    flag = oracle.kv_set_rows(L.k_np(), L.v_np(), hk, hv, L.layout(), L.cur.numpy())
    assert flag == 0
    assert np.array_equal(bits(cache_np(L.d_K)), bits(hk))
    assert np.array_equal(bits(cache_np(L.d_V)), bits(hv))


def test_set_rows_skips_and_flags_out_of_range(tts):
    w = W.workload("batched", kv_dtype="f32", B=3, capacity=256)
    L = Layer(w, seed=21, cur_len=[256, -1, 5])
    before_k = cache_np(L.K)
    ef = err_flag()
    tts.tts_kv_set_rows(L.d_k, L.d_v, L.d_K, L.d_V, L.desc(tts), L.d_cur, ef)
    torch.cuda.synchronize()
    assert ef.item() & tts.EFLAG_POS_RANGE
    hk, hv = before_k.copy(), cache_np(L.V)
    oracle.kv_set_rows(L.k_np(), L.v_np(), hk, hv, L.layout(), L.cur.numpy())
    assert np.array_equal(bits(cache_np(L.d_K)), bits(hk))


# ---------------------------------------------------------------------------
# Step 4: decode attention (standalone)
# ---------------------------------------------------------------------------
ATTN_CASES = [
    # kv_dtype, head_dim, Hq, Hkv, capacity, n_valid per stream, n_splits, paged
    ("f32", 128, 16, 8, 512, [1, 31, 32, 33, 300, 512], 0, False),
    ("f32", 128, 16, 8, 512, [1, 31, 32, 33, 300, 512], 1, False),
    ("f32", 128, 16, 8, 512, [1, 31, 32, 33, 300, 512], 5, False),
    ("bf16", 128, 16, 8, 1024, [1, 63, 64, 65, 700, 1024], 0, False),
    ("bf16", 128, 16, 8, 1024, [2, 129, 1000], 3, True),
    ("f32", 128, 16, 8, 1024, [5, 64, 1023], 7, True),
    ("f32", 64, 16, 8, 16, [1, 2, 9, 16], 0, False),
    ("bf16", 64, 16, 8, 256, [1, 100, 256], 2, False),
    ("f32", 128, 8, 8, 256, [37, 256], 0, False),      # group 1
    ("bf16", 128, 16, 4, 512, [200, 511], 0, False),   # group 4
    ("f32", 64, 16, 4, 256, [255], 3, True),           # group 4, paged, D 64
]


@pytest.mark.parametrize("case", ATTN_CASES, ids=lambda c: f"{c[0]}-D{c[1]}-G{c[2]//c[3]}-S{c[4]}-sp{c[6]}-{'paged' if c[7] else 'contig'}")
def test_decode_attn_matches_oracle(tts, case):
    kv_dtype, D, Hq, Hkv, cap, nv, n_splits, paged = case
    B = len(nv)
    w = W.Workload("case", B=B, layers=1, hidden=Hq * D, n_q_heads=Hq, n_kv_heads=Hkv,
                   head_dim=D, capacity=cap, kv_dtype=kv_dtype, paged=paged, page_size=16,
                   n_pages=B * cap // 16 + 5, window_quantum=16)
    L = Layer(w, seed=30 + B, cur_len=[n - 1 for n in nv])
    # the cache already holds rows [0, cur_len); attend over [0, n_valid) = [0, cur_len + 1):
    # the row at cur_len is written by set_rows first (as the decode step does).
    desc = L.desc(tts)
    ef = err_flag()
    tts.tts_kv_set_rows(L.d_k, L.d_v, L.d_K, L.d_V, desc, L.d_cur, ef)
    n_valid = (L.d_cur + 1).to(torch.int32)
    ws = tts.workspace(desc, n_splits)
    out = torch.full((B, Hq, D), float("nan"), device="cuda")
    tts.tts_decode_attn(L.d_q, L.d_K, L.d_V, desc, n_valid, scale_of(w), out, ws, n_splits, ef)
    torch.cuda.synchronize()
    assert ef.item() == 0
    hk, hv = cache_np(L.d_K), cache_np(L.d_V)
    ref, _, flag = oracle.decode_attn(L.q_np(), hk, hv, L.layout(), np.array(nv, np.int32), scale_of(w))
    assert flag == 0
    assert row_rel_err(out.cpu().numpy(), ref) <= ATTN_TOL[kv_dtype]


def test_decode_attn_poison_padding_and_quantum_invariance(tts):
    """NaN/1e30 past n_valid and the window quantum change nothing: bit-identical."""
    w = W.workload("tiny")
    outs = []
    for poison_val, quantum in [(float("nan"), 256), (1e30, 256), (-1e30, 16), (float("nan"), 128)]:
        L = Layer(w, seed=40, poison=False)
        L.d_K[:, :, 38:] = poison_val
        L.d_V[:, :, 38:] = poison_val
        desc = L.desc(tts, window_quantum=quantum)
        ws = tts.workspace(desc, 0)
        out = torch.empty(1, 16, 128, device="cuda")
        nv = torch.tensor([38], dtype=torch.int32, device="cuda")
        ef = err_flag()
        tts.tts_decode_attn(L.d_q, L.d_K, L.d_V, desc, nv, scale_of(w), out, ws, 0, ef)
        outs.append(out.cpu())
        assert ef.item() == 0
    torch.cuda.synchronize()
    assert all(torch.isfinite(o).all() for o in outs)
    assert all(torch.equal(outs[0], o) for o in outs[1:])


def test_decode_attn_split_counts_agree(tts):
    w = W.workload("talker", layers=1)
    L = Layer(w, seed=41, cur_len=[3000], poison=False)
    desc = L.desc(tts)
    nv = (L.d_cur + 1).to(torch.int32)
    res = []
    # one split; a few; a cluster; a persistent grid with 2-tile and 1-tile splits
    for ns in [1, 2, 16, 64, 128]:
        ws = tts.workspace(desc, ns)
        out = torch.empty(1, 16, 128, device="cuda")
        ef = err_flag()
        tts.tts_decode_attn(L.d_q, L.d_K, L.d_V, desc, nv, scale_of(w), out, ws, ns, ef)
        res.append(out.cpu().numpy())
        assert ef.item() == 0, ns
    torch.cuda.synchronize()
    ref, _, _ = oracle.decode_attn(L.q_np(), cache_np(L.K), cache_np(L.V), L.layout(),
                                   np.array([3001], np.int32), scale_of(w))
    for r in res:
        assert row_rel_err(r, ref) <= ATTN_TOL["f32"]


def test_decode_attn_one_split_over_more_ctas_than_fit(tts):
    """One split per kv head and more (stream, kv head) pairs than the GPU holds at
    once: no workspace, so the grid runs as plain waves (no work counter)."""
    w = W.workload("batched", B=40, layers=1)
    L = Layer(w, seed=45, poison=False)
    desc = L.desc(tts)
    nv = (L.d_cur + 1).to(torch.int32)
    out = torch.empty(w.B, 16, 128, device="cuda")
    ef = err_flag()
    tts.tts_decode_attn(L.d_q, L.d_K, L.d_V, desc, nv, scale_of(w), out, None, 1, ef)
    torch.cuda.synchronize()
    assert ef.item() == 0
    ref, _, _ = oracle.decode_attn(L.q_np(), cache_np(L.K), cache_np(L.V), L.layout(),
                                   nv.cpu().numpy(), scale_of(w))
    assert row_rel_err(out.cpu().numpy(), ref) <= ATTN_TOL["bf16"]


def test_decode_attn_paged_equals_contiguous(tts):
    """The same logical rows through a shuffled block table give bit-identical output
    (same tiles, same arithmetic)."""
    wc = W.workload("batched", B=4, layers=1)
    wp = W.workload("paged", B=4, layers=1, n_pages=1100)
    Lc = Layer(wc, seed=42, cur_len=[100, 2047, 3000, 4095], poison=False)
    Lp = Layer(wp, seed=42, cur_len=[100, 2047, 3000, 4095], poison=False)
    # copy the contiguous rows into the paged pool through the block table
    bt = Lp.bt
    for b in range(4):
        for pg in range(256):
            Lp.d_K[int(bt[b, pg])] = Lc.d_K[b, :, pg * 16:(pg + 1) * 16]
            Lp.d_V[int(bt[b, pg])] = Lc.d_V[b, :, pg * 16:(pg + 1) * 16]
    nv = (Lc.d_cur + 1).to(torch.int32)
    outs = []
    for L in (Lc, Lp):
        desc = L.desc(tts)
        ws = tts.workspace(desc, 8)
        out = torch.empty(4, 16, 128, device="cuda")
        ef = err_flag()
        tts.tts_decode_attn(Lc.d_q, L.d_K, L.d_V, desc, nv, scale_of(wc), out, ws, 8, ef)
        outs.append(out.cpu())
        assert ef.item() == 0
    torch.cuda.synchronize()
    assert torch.equal(outs[0], outs[1])


def test_decode_attn_batched_equals_per_stream(tts):
    """Stream b of a batched call equals a call on stream b alone.  The two launches may
    take different split-merge paths (a one-stream grid fits one wave and merges in a
    thread-block cluster; the batched grid merges through the workspace), which differ
    only in the f32 rounding order of the merge, so the bound is 1e-6 per row."""
    w = W.workload("batched", B=5, layers=1)
    L = Layer(w, seed=43, poison=False)
    desc = L.desc(tts)
    nv = (L.d_cur + 1).to(torch.int32)
    ws = tts.workspace(desc, 8)
    out = torch.empty(5, 16, 128, device="cuda")
    ef = err_flag()
    tts.tts_decode_attn(L.d_q, L.d_K, L.d_V, desc, nv, scale_of(w), out, ws, 8, ef)
    w1 = W.workload("batched", B=1, layers=1)
    for b in range(5):
        d1 = tts.kv_desc(1, 16, 8, 128, 4096, "bf16")
        ws1 = tts.workspace(d1, 8)
        o1 = torch.empty(1, 16, 128, device="cuda")
        tts.tts_decode_attn(L.d_q[b:b + 1], L.d_K[b:b + 1], L.d_V[b:b + 1], d1, nv[b:b + 1],
                            scale_of(w1), o1, ws1, 8, ef)
        torch.cuda.synchronize()
        assert ef.item() == 0
        assert row_rel_err(o1[0].cpu().numpy(), out[b].cpu().numpy()) <= 1e-6


def test_decode_attn_flags_bad_n_valid_and_pages(tts):
    w = W.workload("paged", B=2, layers=1, n_pages=600)
    L = Layer(w, seed=44, cur_len=[100, 200])
    bad_bt = L.d_bt.clone()
    bad_bt[1, 3] = 10_000
    desc = tts.kv_desc(2, 16, 8, 128, 4096, "bf16", paged=True, page_size=16, n_pages=600,
                       block_table=bad_bt)
    ws = tts.workspace(desc, 0)
    out = torch.empty(2, 16, 128, device="cuda")
    ef = err_flag()
    nv = torch.tensor([0, 201], dtype=torch.int32, device="cuda")
    tts.tts_decode_attn(L.d_q, L.d_K, L.d_V, desc, nv, scale_of(w), out, ws, 0, ef)
    torch.cuda.synchronize()
    assert ef.item() & tts.EFLAG_NVALID and ef.item() & tts.EFLAG_PAGE


@pytest.mark.parametrize("n_splits", [0, 4])
def test_paged_entries_past_the_window_are_never_read(tts, n_splits):
    """Block-table entries past each stream's window (from ceil(n_valid / 16) on) hold
    -1: the paged pool is per layer and only a stream's used pages are assigned.  They
    must never be read nor flagged, so the fused step and the standalone attention give
    the same bytes as with a fully assigned table, with err_flag 0.  Default splits run
    the 8-stream workload as a persistent grid whose split length is chosen on the
    device; 4 splits run one item per CTA."""
    w = W.workload("paged", layers=1)
    L = Layer(w, seed=46)
    cs = rope_table(tts, w.capacity, w.head_dim, w.rope_base)
    trimmed = L.d_bt.clone()
    for b in range(w.B):
        used = (int(L.cur[b]) + 1 + w.page_size - 1) // w.page_size
        trimmed[b, used:] = -1
    assert (trimmed == -1).any()
    results = []
    for bt in (L.d_bt, trimmed):
        K, V = L.d_K.clone(), L.d_V.clone()
        desc = tts.kv_desc(w.B, w.n_q_heads, w.n_kv_heads, w.head_dim, w.capacity, w.kv_dtype,
                           paged=True, page_size=w.page_size, n_pages=w.n_pages, block_table=bt)
        ws = tts.workspace(desc, n_splits)
        ef = err_flag()
        step = torch.full((w.B, w.n_q_heads, w.head_dim), float("nan"), device="cuda")
        tts.tts_decode_step(L.d_q, L.d_k, L.d_v, L.d_gq, L.d_gk, w.eps, cs, w.capacity, K, V,
                            desc, L.d_cur, scale_of(w), step, ws, n_splits, ef)
        attn = torch.full_like(step, float("nan"))
        nv = (L.d_cur + 1).to(torch.int32)
        tts.tts_decode_attn(step, K, V, desc, nv, scale_of(w), attn, ws, n_splits, ef)
        torch.cuda.synchronize()
        assert ef.item() == 0
        results.append((step.cpu(), attn.cpu(), K.cpu(), V.cpu()))
    for a, b in zip(*results):
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))


# ---------------------------------------------------------------------------
# Steps 2+3+4 fused: tts_decode_step
# ---------------------------------------------------------------------------
def run_step_and_check(tts, L, n_splits=0, flags=0, tol=None):
    w = L.w
    cs = rope_table(tts, w.capacity, w.head_dim, w.rope_base)
    desc = L.desc(tts, flags=flags)
    ws = tts.workspace(desc, n_splits)
    out = torch.full((w.B, w.n_q_heads, w.head_dim), float("nan"), device="cuda")
    ef = err_flag()
    tts.tts_decode_step(L.d_q, L.d_k, L.d_v, L.d_gq, L.d_gk, w.eps, cs, w.capacity, L.d_K,
                        L.d_V, desc, L.d_cur, scale_of(w), out, ws, n_splits, ef)
    torch.cuda.synchronize()
    assert ef.item() == 0
    hk, hv = cache_np(L.K), cache_np(L.V)
    ref = oracle.decode_step(L.q_np(), L.k_np(), L.v_np(), L.gq.numpy(), L.gk.numpy(),
                             np.float32(w.eps), w.rope_base, hk, hv, L.layout(), L.cur.numpy(),
                             scale_of(w))
    assert row_rel_err(out.cpu().numpy(), ref) <= (tol or ATTN_TOL[w.kv_dtype])
    # cache: every byte except the new rows identical; the new rows within rounding
    gk, gv = cache_np(L.d_K), cache_np(L.d_V)
    changed = bits(gk) != bits(hk)
    changed_v = bits(gv) != bits(hv)
    lay = L.layout()
    newrow_mask = np.zeros(hk.shape, bool)
    for b in range(w.B):
        p = int(L.cur[b])
        for g in range(w.n_kv_heads):
            if w.paged:
                page = int(L.bt[b, p // w.page_size])
                newrow_mask[page, g, p % w.page_size] = True
            else:
                newrow_mask[b, g, p] = True
    assert not (changed & ~newrow_mask).any() and not (changed_v & ~newrow_mask).any()
    if w.kv_dtype == "f32":
        np.testing.assert_allclose(gk[newrow_mask], hk[newrow_mask], rtol=2e-6, atol=2e-6)
        assert np.array_equal(bits(gv[newrow_mask]), bits(hv[newrow_mask]))
    else:
        dk = np.abs(gk[newrow_mask].astype(np.int32) - hk[newrow_mask].astype(np.int32))
        assert dk.max() <= 1  # at most one bf16 ulp where f32 rounding straddles a tie
        assert np.array_equal(gv[newrow_mask], hv[newrow_mask])
    return out


def test_decode_step_tiny_workload(tts):
    """1 stream, 1 layer, hidden 1024, 16/8 heads, D 128, f32, 256 slots, cur_len 37."""
    L = Layer(W.workload("tiny"), seed=0)
    run_step_and_check(tts, L)


@pytest.mark.parametrize("cur_len", [255, 1023, 2047, 4095])
def test_decode_step_talker_sweep(tts, cur_len):
    """Talker shapes (f32 KV, 4096 positions), one layer at each swept cur_len."""
    L = Layer(W.workload("talker", layers=1), seed=cur_len, cur_len=[cur_len])
    run_step_and_check(tts, L)


@pytest.mark.parametrize("flags", [0, 1])
def test_decode_step_batched_ragged_bf16(tts, flags):
    """32 streams, bf16 KV, cur_len ~ U[64, 2048]."""
    L = Layer(W.workload("batched", layers=1), seed=3)
    run_step_and_check(tts, L, flags=flags)


@pytest.mark.parametrize("n_splits", [4, 8, 16])
def test_decode_step_paged_long(tts, n_splits):
    """8 streams, bf16 KV in 16-token pages of a shuffled 4096-page pool, cur_len ~
    U[3072, 4095], 4-16 splits per head."""
    L = Layer(W.workload("paged", layers=1), seed=5)
    run_step_and_check(tts, L, n_splits=n_splits)


def test_decode_step_edges(tts):
    """cur_len 0 (the window is the new row alone), the last slot, tile boundaries."""
    w = W.workload("batched", B=6, layers=1, kv_dtype="f32")
    L = Layer(w, seed=7, cur_len=[0, 1, 31, 32, 4094, 4095])
    run_step_and_check(tts, L)


def test_predictor_frame(tts):
    """Code predictor: 32 streams, 5 layers, D 64, f32 KV, 16-slot cache reset per frame;
    T=2 prefill (rows 0, 1) then 14 single-token decodes; each sub-step gathers its code
    from its own group table.  Two consecutive frames through the same caches."""
    w = W.workload("predictor")
    B, nl = w.B, w.layers
    group_tables = W.tables(15, w.vocab, w.hidden, seed=50)
    d_tables = [t.cuda() for t in group_tables]
    cs = rope_table(tts, w.capacity, w.head_dim, w.rope_base)
    layers = [Layer(w, seed=60 + l, cur_len=[0] * B, poison=True) for l in range(nl)]
    host_caches = [(cache_np(L.K), cache_np(L.V)) for L in layers]
    descs = [L.desc(tts) for L in layers]
    ws = tts.workspace(descs[0], 0)
    ef = err_flag()
    lay = layers[0].layout()
    for frame in range(2):
        codes = W.code_ids(B, 15, w.vocab, seed=70 + frame)
        d_codes = codes.cuda()
        qkv = [[W.qkv(B, w.n_q_heads, w.n_kv_heads, w.head_dim, seed=1000 * frame + 16 * l + t)
                for l in range(nl)] for t in range(16)]
        gammas = [(L.gq.numpy(), L.gk.numpy()) for L in layers]
        ref_e, ref_o = oracle.predictor_frame(
            [t.numpy() for t in group_tables], codes.numpy(), None,
            [[tuple(x.numpy().reshape(B, -1, w.head_dim) for x in qkv[t][l][1:]) for l in range(nl)]
             for t in range(16)],
            gammas, np.float32(w.eps), w.rope_base, host_caches, lay, scale_of(w))
        emb = torch.empty(B, w.hidden, device="cuda")
        for t in range(16):
            cur = torch.full((B,), t, dtype=torch.int32, device="cuda")
            if 1 <= t <= 15:
                j = t - 1
                tts.tts_frame_embed([d_tables[j]], d_codes[:, j:j + 1], None, emb, ef)
                torch.cuda.synchronize()
                assert np.array_equal(bits(emb.cpu().numpy()), bits(ref_e[j]))
            for l in range(nl):
                rows = qkv[t][l][0].cuda()
                qd, kd = w.n_q_heads * w.head_dim, w.n_kv_heads * w.head_dim
                out = torch.empty(B, w.n_q_heads, w.head_dim, device="cuda")
                L = layers[l]
                tts.tts_decode_step(rows[:, :qd], rows[:, qd:qd + kd], rows[:, qd + kd:], L.d_gq,
                                    L.d_gk, w.eps, cs, w.capacity, L.d_K, L.d_V, descs[l], cur,
                                    scale_of(w), out, ws, 0, ef)
                torch.cuda.synchronize()
                assert row_rel_err(out.cpu().numpy(), ref_o[t][l]) <= ATTN_TOL["f32"], (frame, t, l)
    assert ef.item() == 0


def test_decode_step_graph_replay_equals_eager(tts):
    """A captured 4-layer step replays to the same bytes as eager calls."""
    w = W.workload("talker", layers=4)
    cs = rope_table(tts, w.capacity, w.head_dim, w.rope_base)
    layers = [Layer(w, seed=80 + l, cur_len=[1500]) for l in range(4)]
    descs = [L.desc(tts, flags=1) for L in layers]
    ws = tts.workspace(descs[0], 0)
    outs = [torch.empty(1, 16, 128, device="cuda") for _ in range(4)]
    K0 = [(L.d_K.clone(), L.d_V.clone()) for L in layers]

    def step():
        for l, L in enumerate(layers):
            tts.tts_decode_step(L.d_q, L.d_k, L.d_v, L.d_gq, L.d_gk, w.eps, cs, w.capacity, L.d_K,
                                L.d_V, descs[l], L.d_cur, scale_of(w), outs[l], ws)

    step()
    torch.cuda.synchronize()
    eager = [o.clone() for o in outs]
    for (k0, v0), L in zip(K0, layers):
        L.d_K.copy_(k0)
        L.d_V.copy_(v0)
    for o in outs:
        o.fill_(float("nan"))
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        step()
    g.replay()
    torch.cuda.synchronize()
    for a, b in zip(eager, outs):
        assert torch.equal(a, b)
