"""Pins of the CPU oracle against things other than itself.

Each test checks the oracle against a closed form, a hand-derived value (golden
fixtures under tests/golden/), a library routine (torch's rms_norm and
scaled_dot_product_attention in float64, torch's bf16 conversion, sympy's
high-precision cos/sin), or an invariant that the definition implies.  The cases are
chosen so that a plausible slip in the oracle (wrong table or row, wrong summation
order, a dropped eps, a sign or index error in the rotation, a transposed or
mis-mapped head, a softmax over the padded tail) fails at least one of them.
"""
import math
from fractions import Fraction

import numpy as np
import pytest
import sympy as sp
import torch

import oracle
from conftest import read_golden

F = torch.nn.functional


def f32_from_bits(u):
    return np.array([u], dtype=np.uint32).view(np.float32)[0]


# ---------------------------------------------------------------------------
# a1: frame-input composition
# ---------------------------------------------------------------------------
def test_embed_exact_closed_form():
    """Entries chosen so every partial sum is exact in f32: the result must equal the
    exact rational sum of the addressed rows, which pins table/row/column indexing."""
    n, vocab, hidden, B = 16, 64, 32, 3
    tabs = []
    for g in range(n):
        c = np.arange(vocab)[:, None]
        i = np.arange(hidden)[None, :]
        tabs.append((2.0 * g + c * 2.0 ** -6 + i * 2.0 ** -12).astype(np.float32))
    rng = np.random.default_rng(1)
    ids = rng.integers(0, vocab, size=(B, n)).astype(np.int32)
    ov = (np.arange(B)[:, None] * 2.0 ** -8 + np.zeros((1, hidden))).astype(np.float32)
    out, flag = oracle.frame_embed(tabs, ids, ov)
    assert flag == 0
    for b in range(B):
        for i in range(hidden):
            exact = sum(Fraction(2 * g) + Fraction(int(ids[b, g]), 64) + Fraction(i, 4096)
                        for g in range(n)) + Fraction(b, 256)
            assert Fraction(float(out[b, i])) == exact


def test_embed_left_to_right_order_and_overlay_last():
    """Hand-derived: 1.0 followed by fifteen 2^-24 terms, added left to right in f32,
    stays exactly 1.0 (each addition is a tie that rounds to even); the overlay -1.0
    then gives exactly 0.  Any other order (pairwise, reversed, overlay first) keeps
    some of the small terms and gives a nonzero result."""
    vocab, hidden = 4, 8
    tabs = [np.full((vocab, hidden), 2.0 ** -24, np.float32) for _ in range(16)]
    tabs[0][:] = 1.0
    ids = np.zeros((1, 16), np.int32)
    out, _ = oracle.frame_embed(tabs, ids, np.full((1, hidden), -1.0, np.float32))
    assert np.all(out == 0.0)
    out_no_ov, _ = oracle.frame_embed(tabs, ids, None)
    assert np.all(out_no_ov == 1.0)


def test_embed_single_table_is_a_row_copy():
    """Predictor sub-steps gather one row from one group table, no overlay."""
    rng = np.random.default_rng(2)
    tab = rng.standard_normal((50, 16)).astype(np.float32)
    ids = np.array([[7], [49], [0]], np.int32)
    out, _ = oracle.frame_embed([tab], ids, None)
    assert np.array_equal(out, tab[[7, 49, 0]])


def test_embed_clamps_out_of_range_ids():
    tab = np.arange(12, dtype=np.float32).reshape(4, 3)
    out, flag = oracle.frame_embed([tab], np.array([[-1], [4], [2]], np.int32), None)
    assert flag == 1
    assert np.array_equal(out, tab[[0, 3, 2]])


# ---------------------------------------------------------------------------
# a2: RMSNorm + RoPE
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("D", [4, 64, 128])
def test_norm_matches_torch_rms_norm_at_position_zero(D):
    """At position 0 every angle is 0, so the output is the RMSNorm alone; compare with
    torch's rms_norm in float64 (weight = gamma, eps inside the root)."""
    rng = np.random.default_rng(D)
    x = rng.standard_normal((3, 5, D)).astype(np.float32)
    gam = rng.uniform(0.5, 1.5, D).astype(np.float32)
    eps = np.float32(1e-6)
    y = oracle.rms_norm_rope(x, gam, eps, np.zeros(3, np.int32), 1e6)
    ref = F.rms_norm(torch.from_numpy(x).double(), (D,), weight=torch.from_numpy(gam).double(),
                     eps=float(eps)).numpy().astype(np.float32)
    np.testing.assert_array_max_ulp(y, ref, maxulp=1)


def test_norm_constant_row_closed_form():
    """x = c everywhere, gamma = 1, pos 0: every output equals c / sqrt(c^2 + eps)."""
    D = 128
    for c in [3.0, -0.25, 1e-3]:
        x = np.full((1, 1, D), c, np.float32)
        eps = np.float32(1e-6)
        y = oracle.rms_norm_rope(x, np.ones(D, np.float32), eps, np.zeros(1, np.int32), 1e6)
        expect = np.float32(np.float32(c) / math.sqrt(float(np.float32(c)) ** 2 + float(eps)))
        np.testing.assert_array_max_ulp(y, np.full_like(y, expect), maxulp=1)


def test_rope_angles_hand_derived():
    for pos, i, D, base, c, s in read_golden("rope_angles.txt"):
        got = oracle.rope_angle(int(pos), int(i), int(D), float(base))
        assert got[0] == pytest.approx(float(c), abs=1e-15)
        assert got[1] == pytest.approx(float(s), abs=1e-15)


@pytest.mark.parametrize("pos", [1, 37, 255, 4095])
def test_rope_angles_against_sympy(pos):
    """theta_i = pos * base^(-2i/D) evaluated by sympy to 40 digits, base 1e6, D 128,
    at the first, a middle and the last frequency."""
    D, base = 128, 10 ** 6
    for i in [0, 1, 17, 63]:
        theta = sp.Integer(pos) * sp.Integer(base) ** sp.Rational(-2 * i, D)
        c = float(sp.N(sp.cos(theta), 40))
        s = float(sp.N(sp.sin(theta), 40))
        got = oracle.rope_angle(pos, i, D, float(base))
        assert got[0] == pytest.approx(c, abs=1e-12)
        assert got[1] == pytest.approx(s, abs=1e-12)


@pytest.mark.parametrize("D", [64, 128])
def test_rope_is_complex_rotation_of_the_normed_halves(D):
    """Rotate-half RoPE equals multiplying t_i + i t_{i+D/2} by exp(i theta_i).  The
    normed t comes from torch's rms_norm (float64), the angles from sympy."""
    rng = np.random.default_rng(10 + D)
    B, H = 2, 3
    x = rng.standard_normal((B, H, D)).astype(np.float32)
    gam = rng.uniform(0.5, 1.5, D).astype(np.float32)
    pos = np.array([5, 4095], np.int32)
    eps = np.float32(1e-6)
    y = oracle.rms_norm_rope(x, gam, eps, pos, 1e6)
    t = F.rms_norm(torch.from_numpy(x).double(), (D,), weight=torch.from_numpy(gam).double(),
                   eps=float(eps)).numpy()
    for b in range(B):
        ang = np.array([complex(sp.N(sp.exp(sp.I * sp.Integer(int(pos[b])) *
                                            sp.Integer(10 ** 6) ** sp.Rational(-2 * i, D)), 30))
                        for i in range(D // 2)])
        z = (t[b, :, :D // 2] + 1j * t[b, :, D // 2:]) * ang[None, :]
        ref = np.concatenate([z.real, z.imag], axis=-1).astype(np.float32)
        np.testing.assert_allclose(y[b], ref, rtol=0, atol=2e-7 * np.abs(ref).max())


def test_rope_preserves_pair_norms():
    rng = np.random.default_rng(3)
    D = 128
    x = rng.standard_normal((1, 4, D)).astype(np.float32)
    g1 = np.ones(D, np.float32)
    y0 = oracle.rms_norm_rope(x, g1, np.float32(1e-6), np.zeros(1, np.int32), 1e6).astype(np.float64)
    y = oracle.rms_norm_rope(x, g1, np.float32(1e-6), np.array([3001], np.int32), 1e6).astype(np.float64)
    n0 = y0[..., :D // 2] ** 2 + y0[..., D // 2:] ** 2
    n1 = y[..., :D // 2] ** 2 + y[..., D // 2:] ** 2
    np.testing.assert_allclose(n1, n0, rtol=1e-6, atol=1e-12)


# ---------------------------------------------------------------------------
# a3: set_rows and bf16 rounding
# ---------------------------------------------------------------------------
def test_bf16_rne_hand_derived_cases():
    for f_bits, h_bits in read_golden("bf16_rne_cases.txt"):
        assert oracle.bf16_rne(f32_from_bits(int(f_bits, 16))) == int(h_bits, 16), f_bits


def test_bf16_rne_matches_torch_conversion():
    """torch's f32 -> bf16 conversion is round-to-nearest-even; compare on random
    values plus constructed ties (low half exactly 0x8000)."""
    rng = np.random.default_rng(4)
    x = rng.standard_normal(20000).astype(np.float32) * np.float32(10.0) ** rng.integers(-30, 30, 20000).astype(np.float32)
    ties = (rng.integers(0, 2 ** 31, 5000).astype(np.uint32) & np.uint32(0xFFFF0000)) | np.uint32(0x8000)
    x = np.concatenate([x, ties.view(np.float32)])
    x = x[np.isfinite(x)]
    got = oracle.bf16_rne_array(x)
    ref = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    assert np.array_equal(got, ref)


@pytest.mark.parametrize("layout_name", ["contiguous", "paged"])
@pytest.mark.parametrize("kv_dtype", ["f32", "bf16"])
def test_set_rows_hand_derived_offsets(layout_name, kv_dtype):
    """Rows land at the hand-derived flat offsets of the documented layouts; every
    other element keeps its canary value."""
    B, Hkv, D, cap = 2, 2, 2, 4
    paged = layout_name == "paged"
    bt = np.array([[3, 1], [0, 4]], np.int32)
    lay = oracle.KvLayout(B, Hkv, D, cap, kv_dtype, paged=paged, page_size=2, n_pages=5,
                          block_table=bt if paged else None)
    n_el = (5 * Hkv * 2 * D) if paged else (B * Hkv * cap * D)
    dt = np.float32 if kv_dtype == "f32" else np.uint16
    canary = np.float32(-7.0) if kv_dtype == "f32" else np.uint16(0xDEAD)
    kc = np.full(n_el, canary, dt)
    vc = np.full(n_el, canary, dt)
    k = np.array([[[1, 2], [3, 4]], [[5, 6], [7, 8]]], np.float32)
    v = k + np.float32(10)
    flag = oracle.kv_set_rows(k, v, kc, vc, lay, np.array([3, 0], np.int32))
    assert flag == 0
    touched = set()
    for lay_name, b, pos, g, off in read_golden("paged_offsets.txt"):
        if lay_name != layout_name:
            continue
        b, g, off = int(b), int(g), int(off)
        for d in range(D):
            want_k, want_v = k[b, g, d], v[b, g, d]
            if kv_dtype == "bf16":
                want_k = oracle.bf16_rne(want_k)
                want_v = oracle.bf16_rne(want_v)
            assert kc[off + d] == want_k and vc[off + d] == want_v
            touched.add(off + d)
    rest = np.array([i for i in range(n_el) if i not in touched])
    assert np.all(kc[rest] == canary) and np.all(vc[rest] == canary)


def test_set_rows_skips_out_of_range_positions():
    lay = oracle.KvLayout(2, 1, 4, 8, "f32")
    kc = np.zeros(2 * 8 * 4, np.float32)
    vc = np.zeros_like(kc)
    k = np.ones((2, 1, 4), np.float32)
    flag = oracle.kv_set_rows(k, k, kc, vc, lay, np.array([8, -1], np.int32))
    assert flag == 1 and np.all(kc == 0)


# ---------------------------------------------------------------------------
# a4: decode attention
# ---------------------------------------------------------------------------
def _rand_case(rng, B, Hq, Hkv, D, cap, kv_dtype="f32"):
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    kc = rng.standard_normal((B, Hkv, cap, D)).astype(np.float32)
    vc = rng.standard_normal((B, Hkv, cap, D)).astype(np.float32)
    if kv_dtype == "bf16":
        kc = torch.from_numpy(kc).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
        vc = torch.from_numpy(vc).to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    return q, kc, vc


def _as_f64(c, kv_dtype):
    return c.astype(np.float64) if kv_dtype == "f32" else oracle.bf16_bits_to_f32(c).astype(np.float64)


@pytest.mark.parametrize("kv_dtype", ["f32", "bf16"])
@pytest.mark.parametrize("Hq,Hkv", [(16, 8), (4, 1), (8, 8)])
def test_attn_matches_torch_sdpa(kv_dtype, Hq, Hkv):
    """torch scaled_dot_product_attention in float64 with enable_gqa (q head h reads kv
    head h // (Hq/Hkv)) and its default 1/sqrt(D) scale, over the valid rows only."""
    rng = np.random.default_rng(5)
    B, D, cap = 3, 16, 40
    q, kc, vc = _rand_case(rng, B, Hq, Hkv, D, cap, kv_dtype)
    n_valid = np.array([1, 17, 40], np.int32)
    lay = oracle.KvLayout(B, Hkv, D, cap, kv_dtype)
    out, _, flag = oracle.decode_attn(q, kc, vc, lay, n_valid, 1.0 / math.sqrt(D))
    assert flag == 0
    K, V = _as_f64(kc, kv_dtype), _as_f64(vc, kv_dtype)
    for b in range(B):
        n = int(n_valid[b])
        ref = F.scaled_dot_product_attention(
            torch.from_numpy(q[b:b + 1].astype(np.float64))[:, :, None, :],
            torch.from_numpy(K[b:b + 1, :, :n]), torch.from_numpy(V[b:b + 1, :, :n]),
            enable_gqa=True)[0, :, 0, :].numpy()
        np.testing.assert_allclose(out[b], ref, rtol=1e-6, atol=1e-7)


def test_attn_weights_sum_to_one_and_tail_is_exactly_zero():
    rng = np.random.default_rng(6)
    B, Hq, Hkv, D, cap = 2, 4, 2, 8, 64
    q, kc, vc = _rand_case(rng, B, Hq, Hkv, D, cap)
    n_valid = np.array([5, 64], np.int32)
    _, w, _ = oracle.decode_attn(q, kc, vc, oracle.KvLayout(B, Hkv, D, cap), n_valid, 0.3,
                                 want_weights=True)
    assert np.all(np.abs(w.sum(-1) - 1.0) < 1e-12)
    assert np.all(w[0, :, 5:] == 0.0)
    assert np.all(w[0, :, :5] > 0.0)


def test_attn_ignores_poisoned_tail_and_window_padding():
    """Whatever sits past n_valid (NaN, +-1e30) and however far the cache extends, the
    result is bit-identical: the padded tail is never read."""
    rng = np.random.default_rng(7)
    B, Hq, Hkv, D = 1, 4, 2, 8
    q, kc, vc = _rand_case(rng, B, Hq, Hkv, D, 256)
    n_valid = np.array([38], np.int32)
    base, _, _ = oracle.decode_attn(q, kc, vc, oracle.KvLayout(B, Hkv, D, 256), n_valid, 0.35)
    for poison in [np.nan, 1e30, -1e30]:
        kp, vp = kc.copy(), vc.copy()
        kp[:, :, 38:] = poison
        vp[:, :, 38:] = poison
        out, _, _ = oracle.decode_attn(q, kp, vp, oracle.KvLayout(B, Hkv, D, 256), n_valid, 0.35)
        assert np.array_equal(out, base)
    for cap in [38, 64, 512]:
        kp = np.full((B, Hkv, cap, D), np.nan, np.float32)
        vp = kp.copy()
        kp[:, :, :38] = kc[:, :, :38]
        vp[:, :, :38] = vc[:, :, :38]
        out, _, _ = oracle.decode_attn(q, kp, vp, oracle.KvLayout(B, Hkv, D, cap), n_valid, 0.35)
        assert np.array_equal(out, base)


def test_attn_closed_forms():
    rng = np.random.default_rng(8)
    B, Hq, Hkv, D, cap = 1, 2, 1, 8, 32
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    V = rng.standard_normal((B, Hkv, cap, D)).astype(np.float32)
    lay = oracle.KvLayout(B, Hkv, D, cap)
    # All keys equal: uniform weights, output = mean of the valid V rows.
    K = np.repeat(rng.standard_normal((B, Hkv, 1, D)).astype(np.float32), cap, axis=2)
    out, _, _ = oracle.decode_attn(q, K, V, lay, np.array([20], np.int32), 0.5)
    mean = V[0, 0, :20].astype(np.float64).mean(0)
    np.testing.assert_allclose(out[0], np.broadcast_to(mean, (Hq, D)), rtol=1e-6, atol=1e-7)
    # One key dominates by 60 in score: the output is its V row to ~exp(-60).
    K2 = np.zeros((B, Hkv, cap, D), np.float32)
    q2 = np.zeros((B, Hq, D), np.float32)
    q2[..., 0] = 1.0
    K2[0, 0, 3, 0] = 60.0
    out, _, _ = oracle.decode_attn(q2, K2, V, lay, np.array([32], np.int32), 1.0)
    np.testing.assert_allclose(out[0], np.broadcast_to(V[0, 0, 3], (Hq, D)), rtol=1e-6, atol=1e-7)
    # A single valid row: the output is that V row exactly.
    out, _, _ = oracle.decode_attn(q, K, V, lay, np.array([1], np.int32), 0.5)
    assert np.array_equal(out[0], np.broadcast_to(V[0, 0, 0], (Hq, D)))


def test_attn_scale_enters_as_multiplier_of_the_scores():
    """Doubling the scale equals doubling q (the score is scale * q.K)."""
    rng = np.random.default_rng(9)
    q, kc, vc = _rand_case(rng, 1, 2, 1, 8, 16)
    lay = oracle.KvLayout(1, 1, 8, 16)
    a, _, _ = oracle.decode_attn(q, kc, vc, lay, np.array([16], np.int32), 0.4)
    b, _, _ = oracle.decode_attn(q * np.float32(2), kc, vc, lay, np.array([16], np.int32), 0.2)
    np.testing.assert_allclose(a, b, rtol=1e-12, atol=0)


@pytest.mark.parametrize("kv_dtype", ["f32", "bf16"])
def test_attn_paged_equals_contiguous(kv_dtype):
    """Scatter each stream's logical rows into shuffled pages through set_rows; the
    paged result must equal the contiguous one bit for bit."""
    rng = np.random.default_rng(11)
    B, Hq, Hkv, D, ps, pages_per = 2, 4, 2, 8, 16, 4
    cap = ps * pages_per
    n_pages = 11
    bt = np.array([[7, 2, 9, 0], [3, 10, 5, 1]], np.int32)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    kl = rng.standard_normal((B, cap, Hkv, D)).astype(np.float32)
    vl = rng.standard_normal((B, cap, Hkv, D)).astype(np.float32)
    dt = np.float32 if kv_dtype == "f32" else np.uint16
    cont = oracle.KvLayout(B, Hkv, D, cap, kv_dtype)
    pag = oracle.KvLayout(B, Hkv, D, cap, kv_dtype, paged=True, page_size=ps, n_pages=n_pages,
                          block_table=bt)
    kc = np.zeros(B * Hkv * cap * D, dt)
    vc = np.zeros_like(kc)
    kp = np.zeros(n_pages * Hkv * ps * D, dt)
    vp = np.zeros_like(kp)
    n_valid = np.array([37, 64], np.int32)
    for j in range(cap):
        pos = np.full(B, j, np.int32)
        oracle.kv_set_rows(kl[:, j], vl[:, j], kc, vc, cont, pos)
        oracle.kv_set_rows(kl[:, j], vl[:, j], kp, vp, pag, pos)
    a, _, _ = oracle.decode_attn(q, kc, vc, cont, n_valid, 0.3)
    b, _, _ = oracle.decode_attn(q, kp, vp, pag, n_valid, 0.3)
    assert np.array_equal(a, b)


def test_attn_clamps_invalid_n_valid():
    rng = np.random.default_rng(12)
    q, kc, vc = _rand_case(rng, 2, 2, 1, 8, 16)
    lay = oracle.KvLayout(2, 1, 8, 16)
    out, _, flag = oracle.decode_attn(q, kc, vc, lay, np.array([0, 99], np.int32), 0.3)
    ref, _, flag2 = oracle.decode_attn(q, kc, vc, lay, np.array([1, 16], np.int32), 0.3)
    assert flag == 1 and flag2 == 0 and np.array_equal(out, ref)


# Brute-force pins: the oracle's attention against a per-element loop written
# independently in oracle/brute.py (its own addressing, softmax without max
# subtraction, Python doubles).  The oracle rounds its double result to f32 once, so
# the two agree to about one f32 rounding.
BRUTE_RTOL = 2e-7


def _assert_brute(out, ref):
    ref = np.asarray(ref, np.float64)
    err = np.abs(out.astype(np.float64) - ref) / np.maximum(np.abs(ref).max(-1, keepdims=True), 1e-30)
    assert err.max() <= BRUTE_RTOL, err.max()


def test_attn_matches_brute_force_on_the_tiny_workload():
    """The tiny workload's own shapes: 1 stream, 16 q / 8 kv heads, head_dim 128, f32
    cache of 256 slots, window [0, 38) (cur_len 37 after its row is written), the
    rest of the cache poisoned with NaN."""
    from autoregressive_codebook_tts_gb300 import workloads as W
    from oracle.brute import attn_brute
    w = W.workload("tiny")
    n_valid = np.array([38], np.int32)
    K, V = W.cache(w, n_valid.tolist(), seed=21)
    kc, vc = K.numpy(), V.numpy()
    q = W.qkv(w.B, w.n_q_heads, w.n_kv_heads, w.head_dim, seed=22)[1].numpy().reshape(
        w.B, w.n_q_heads, w.head_dim).copy()
    scale = 1.0 / math.sqrt(w.head_dim)
    lay = oracle.KvLayout(w.B, w.n_kv_heads, w.head_dim, w.capacity, "f32")
    out, _, flag = oracle.decode_attn(q, kc, vc, lay, n_valid, scale)
    assert flag == 0
    _assert_brute(out, attn_brute(q, kc, vc, n_valid, scale))


@pytest.mark.parametrize("Hq,Hkv", [(4, 4), (4, 2), (8, 2)])
def test_attn_matches_brute_force_gqa_groups(Hq, Hkv):
    """head_dim 4, windows of 1..64 rows, GQA groups 1, 2 and 4."""
    from oracle.brute import attn_brute
    rng = np.random.default_rng(31 + Hq + Hkv)
    B, D, cap = 4, 4, 64
    q, kc, vc = _rand_case(rng, B, Hq, Hkv, D, cap)
    n_valid = np.array([1, 2, 33, 64], np.int32)
    out, _, flag = oracle.decode_attn(q, kc, vc, oracle.KvLayout(B, Hkv, D, cap), n_valid, 0.5)
    assert flag == 0
    _assert_brute(out, attn_brute(q, kc, vc, n_valid, 0.5))


def test_attn_matches_brute_force_paged_bf16_with_unused_entries_minus_one():
    """A paged bf16 pool of shuffled 16-slot pages; block-table entries past each
    stream's window hold -1 (they are never read, so neither side may touch them)."""
    from oracle.brute import attn_brute
    rng = np.random.default_rng(41)
    B, Hq, Hkv, D, ps, n_pages = 2, 4, 2, 4, 16, 9
    cap = 4 * ps
    bt = np.array([[6, 1, 8, -1], [2, 7, 0, 4]], np.int32)
    n_valid = np.array([37, 64], np.int32)
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    pool = [torch.from_numpy(rng.standard_normal((n_pages, Hkv, ps, D)).astype(np.float32))
            .to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16) for _ in range(2)]
    lay = oracle.KvLayout(B, Hkv, D, cap, "bf16", paged=True, page_size=ps, n_pages=n_pages,
                          block_table=bt)
    out, _, flag = oracle.decode_attn(q, pool[0], pool[1], lay, n_valid, 0.5)
    assert flag == 0
    _assert_brute(out, attn_brute(q, pool[0], pool[1], n_valid, 0.5, kv_dtype="bf16", paged=True,
                                  page_size=ps, block_table=bt))


def test_brute_force_pin_catches_a_swapped_gqa_map():
    """The brute-force comparison is sharp enough to see a plausible mistake: feeding
    the oracle the kv heads in the opposite order (a wrong GQA map) fails it."""
    from oracle.brute import attn_brute
    rng = np.random.default_rng(43)
    B, Hq, Hkv, D, cap = 1, 4, 2, 4, 16
    q, kc, vc = _rand_case(rng, B, Hq, Hkv, D, cap)
    n_valid = np.array([16], np.int32)
    out, _, _ = oracle.decode_attn(q, kc[:, ::-1].copy(), vc[:, ::-1].copy(),
                                   oracle.KvLayout(B, Hkv, D, cap), n_valid, 0.5)
    with pytest.raises(AssertionError):
        _assert_brute(out, attn_brute(q, kc, vc, n_valid, 0.5))


# ---------------------------------------------------------------------------
# Compositions
# ---------------------------------------------------------------------------
def test_decode_step_batched_equals_per_stream():
    rng = np.random.default_rng(13)
    B, Hq, Hkv, D, cap = 3, 4, 2, 16, 32
    q = rng.standard_normal((B, Hq, D)).astype(np.float32)
    k = rng.standard_normal((B, Hkv, D)).astype(np.float32)
    v = rng.standard_normal((B, Hkv, D)).astype(np.float32)
    gq = rng.uniform(0.5, 1.5, D).astype(np.float32)
    gk = rng.uniform(0.5, 1.5, D).astype(np.float32)
    kc0 = rng.standard_normal((B, Hkv, cap, D)).astype(np.float32)
    vc0 = rng.standard_normal((B, Hkv, cap, D)).astype(np.float32)
    cur = np.array([0, 13, 31], np.int32)
    kc, vc = kc0.copy(), vc0.copy()
    out = oracle.decode_step(q, k, v, gq, gk, np.float32(1e-6), 1e6, kc, vc,
                             oracle.KvLayout(B, Hkv, D, cap), cur, 0.25)
    for b in range(B):
        kb, vb = kc0[b:b + 1].copy(), vc0[b:b + 1].copy()
        ob = oracle.decode_step(q[b:b + 1], k[b:b + 1], v[b:b + 1], gq, gk, np.float32(1e-6),
                                1e6, kb, vb, oracle.KvLayout(1, Hkv, D, cap), cur[b:b + 1], 0.25)
        assert np.array_equal(ob[0], out[b])
        assert np.array_equal(kb[0], kc[b]) and np.array_equal(vb[0], vc[b])


def test_decode_step_at_position_zero_attends_to_its_own_value_row():
    """cur_len = 0: the window is the single new row, so the output is v itself."""
    rng = np.random.default_rng(14)
    Hq, Hkv, D = 4, 2, 16
    q = rng.standard_normal((1, Hq, D)).astype(np.float32)
    k = rng.standard_normal((1, Hkv, D)).astype(np.float32)
    v = rng.standard_normal((1, Hkv, D)).astype(np.float32)
    kc = np.full((1, Hkv, 16, D), np.nan, np.float32)
    vc = kc.copy()
    out = oracle.decode_step(q, k, v, np.ones(D, np.float32), np.ones(D, np.float32),
                             np.float32(1e-6), 1e6, kc, vc, oracle.KvLayout(1, Hkv, D, 16),
                             np.array([0], np.int32), 0.25)
    assert np.array_equal(out[0], np.repeat(v[0], Hq // Hkv, axis=0))


def test_predictor_frame_reset_masks_the_previous_frame():
    """Two predictor frames through the same cache: the second frame's outputs equal
    those of the same frame on a fresh (NaN-filled) cache, so stale rows from the
    previous frame never leak (the cache reset is cur_len = 0, not a clear)."""
    rng = np.random.default_rng(15)
    B, L, Hq, Hkv, D, cap, hidden, vocab = 2, 2, 4, 2, 8, 16, 8, 32
    lay = oracle.KvLayout(B, Hkv, D, cap)
    tabs = [rng.standard_normal((vocab, hidden)).astype(np.float32) for _ in range(15)]
    gam = [(np.ones(D, np.float32), np.ones(D, np.float32)) for _ in range(L)]

    def frame_inputs():
        codes = rng.integers(0, vocab, (B, 15)).astype(np.int32)
        qkv = [[tuple(rng.standard_normal(s).astype(np.float32)
                      for s in [(B, Hq, D), (B, Hkv, D), (B, Hkv, D)]) for _ in range(L)]
               for _ in range(16)]
        return codes, qkv

    used = [tuple(rng.standard_normal((B, Hkv, cap, D)).astype(np.float32) for _ in range(2))
            for _ in range(L)]
    c1, qkv1 = frame_inputs()
    oracle.predictor_frame(tabs, c1, None, qkv1, gam, np.float32(1e-6), 1e6, used, lay, 0.3)
    c2, qkv2 = frame_inputs()
    e2, o2 = oracle.predictor_frame(tabs, c2, None, qkv2, gam, np.float32(1e-6), 1e6, used, lay, 0.3)
    fresh = [tuple(np.full((B, Hkv, cap, D), np.nan, np.float32) for _ in range(2)) for _ in range(L)]
    e3, o3 = oracle.predictor_frame(tabs, c2, None, qkv2, gam, np.float32(1e-6), 1e6, fresh, lay, 0.3)
    for t in range(16):
        for l in range(L):
            assert np.array_equal(o2[t][l], o3[t][l])
    for j in range(15):
        assert np.array_equal(e2[j], tabs[j][c2[:, j]])


# ---------------------------------------------------------------------------
# Prefill: T new positions per stream, causal
# ---------------------------------------------------------------------------
def _prefill_case(rng, B, T, Hq, Hkv, D, cap):
    q = rng.standard_normal((B, T, Hq, D)).astype(np.float32)
    k = rng.standard_normal((B, T, Hkv, D)).astype(np.float32)
    v = rng.standard_normal((B, T, Hkv, D)).astype(np.float32)
    gq = rng.uniform(0.5, 1.5, D).astype(np.float32)
    gk = rng.uniform(0.5, 1.5, D).astype(np.float32)
    kc = rng.standard_normal((B, Hkv, cap, D)).astype(np.float32)
    vc = rng.standard_normal((B, Hkv, cap, D)).astype(np.float32)
    return q, k, v, gq, gk, kc, vc


@pytest.mark.parametrize("start", [0, 9])
def test_prefill_matches_torch_causal_sdpa(start):
    """torch scaled_dot_product_attention in float64 over [rows before the prompt | the
    prompt's rows] with a mask that lets prompt query t see every earlier row and the
    prompt's rows 0..t; q and k rows rotated at positions start + t, computed here."""
    rng = np.random.default_rng(21)
    B, T, Hq, Hkv, D, cap = 2, 6, 4, 2, 16, 32
    q, k, v, gq, gk, kc, vc = _prefill_case(rng, B, T, Hq, Hkv, D, cap)
    eps = np.float32(1e-6)
    kc0, vc0 = kc.copy(), vc.copy()
    out = oracle.prefill_step(q, k, v, gq, gk, eps, 1e6, kc, vc, oracle.KvLayout(B, Hkv, D, cap),
                              np.array([start] * B, np.int32), 1.0 / math.sqrt(D))
    n = start + T
    mask = np.zeros((T, n), bool)
    for t in range(T):
        mask[t, :start + t + 1] = True
    for b in range(B):
        qn = np.stack([oracle.rms_norm_rope(q[b, t][None], gq, eps, np.array([start + t], np.int32), 1e6)[0]
                       for t in range(T)])            # [T][Hq][D]
        kn = np.stack([oracle.rms_norm_rope(k[b, t][None], gk, eps, np.array([start + t], np.int32), 1e6)[0]
                       for t in range(T)])            # [T][Hkv][D]
        K = np.concatenate([kc0[b, :, :start], kn.transpose(1, 0, 2)], axis=1).astype(np.float64)
        V = np.concatenate([vc0[b, :, :start], v[b].transpose(1, 0, 2)], axis=1).astype(np.float64)
        ref = F.scaled_dot_product_attention(
            torch.from_numpy(qn.transpose(1, 0, 2).astype(np.float64))[None],
            torch.from_numpy(K)[None], torch.from_numpy(V)[None],
            attn_mask=torch.from_numpy(mask), enable_gqa=True)[0].numpy()   # [Hq][T][D]
        np.testing.assert_allclose(out[b], ref.transpose(1, 0, 2), rtol=1e-6, atol=1e-7)
        # the prompt's rows are in the cache at their positions; the rest is untouched
        assert np.array_equal(kc[b, :, start:n], kn.transpose(1, 0, 2))
        assert np.array_equal(vc[b, :, start:n], v[b].transpose(1, 0, 2))
        assert np.array_equal(kc[b, :, :start], kc0[b, :, :start])
        assert np.array_equal(kc[b, :, n:], kc0[b, :, n:])


@pytest.mark.parametrize("kv_dtype", ["f32", "bf16"])
def test_prefill_equals_decode_steps_one_by_one(kv_dtype):
    """A prompt of T rows in one prefill = T decode steps at start, start + 1, ...: every
    query's window ends at its own row, so writing the later rows first changes nothing.
    Also T = 1 is exactly one decode step."""
    rng = np.random.default_rng(22)
    B, T, Hq, Hkv, D, cap = 3, 5, 4, 2, 16, 24
    q, k, v, gq, gk, kc, vc = _prefill_case(rng, B, T, Hq, Hkv, D, cap)
    if kv_dtype == "bf16":
        kc, vc = oracle.bf16_rne_array(kc), oracle.bf16_rne_array(vc)
    start = np.array([0, 7, 19], np.int32)
    lay = oracle.KvLayout(B, Hkv, D, cap, kv_dtype)
    kp, vp = kc.copy(), vc.copy()
    out = oracle.prefill_step(q, k, v, gq, gk, np.float32(1e-6), 1e6, kp, vp, lay, start, 0.3)
    ks, vs = kc.copy(), vc.copy()
    for t in range(T):
        o = oracle.decode_step(q[:, t], k[:, t], v[:, t], gq, gk, np.float32(1e-6), 1e6, ks, vs,
                               lay, start + t, 0.3)
        assert np.array_equal(o, out[:, t]), t
    assert np.array_equal(kp, ks) and np.array_equal(vp, vs)
    k1, v1 = kc.copy(), vc.copy()
    o1 = oracle.prefill_step(q[:, :1], k[:, :1], v[:, :1], gq, gk, np.float32(1e-6), 1e6, k1, v1,
                             lay, start, 0.3)
    assert np.array_equal(o1[:, 0], out[:, 0])


def test_prefill_first_query_of_an_empty_cache_is_its_own_value_row():
    """start = 0 on a NaN-filled cache: query 0 sees only row 0 (o = v_0 exactly), and no
    query reads past its own row (the NaN rows after the prompt never leak)."""
    rng = np.random.default_rng(23)
    B, T, Hq, Hkv, D, cap = 1, 4, 4, 2, 8, 16
    q, k, v, gq, gk, _, _ = _prefill_case(rng, B, T, Hq, Hkv, D, cap)
    kc = np.full((B, Hkv, cap, D), np.nan, np.float32)
    vc = kc.copy()
    out = oracle.prefill_step(q, k, v, gq, gk, np.float32(1e-6), 1e6, kc, vc,
                              oracle.KvLayout(B, Hkv, D, cap), np.zeros(B, np.int32), 0.5)
    assert np.array_equal(out[0, 0], np.repeat(v[0, 0], Hq // Hkv, axis=0))
    assert np.isfinite(out).all()


def _q8_block(d_bits, qs):
    """One 34-byte Q8_0 block from a binary16 bit pattern and up to 32 quants (rest 0)."""
    q = list(qs) + [0] * (32 - len(qs))
    return bytes([d_bits & 0xFF, d_bits >> 8]) + bytes([v & 0xFF for v in q])


def test_q8_0_entries_hand_derived():
    """Every golden row is its own block in a one-row table; the gathered row holds d * q
    at the block's first entry and 0 at the rest (entry = scale times quant)."""
    rows = read_golden("q8_0_blocks.txt")
    blob = b"".join(_q8_block(int(d, 16), [int(q)]) for d, q, _ in rows)
    tab = np.frombuffer(blob, np.uint8).reshape(1, -1)
    out, flag = oracle.frame_embed([tab], np.zeros((1, 1), np.int32), None)
    assert flag == 0
    got = out.reshape(len(rows), 32)
    for k, (_, _, expect) in enumerate(rows):
        assert got[k, 0] == np.float32(float(expect)), (k, got[k, 0], expect)
        assert np.all(got[k, 1:] == 0.0)


def test_q8_0_block_layout_and_row_addressing():
    """Entry i of a row comes from block i // 32, quant i % 32; row r starts r * 34 *
    hidden / 32 bytes in; scales of 2^k times quants equal to the column index give an
    exact closed form for every entry of every row."""
    vocab, hidden = 5, 96
    nb = hidden // 32
    blob = b""
    for r in range(vocab):
        for k in range(nb):
            # d = 2^(r - k) as binary16: exponent field 15 + r - k, zero mantissa
            d_bits = (15 + r - k) << 10
            blob += _q8_block(d_bits, [(j + 32 * k) % 100 - 50 for j in range(32)])
    tab = np.frombuffer(blob, np.uint8).reshape(vocab, -1)
    ids = np.array([[4], [0], [2]], np.int32)
    out, _ = oracle.frame_embed([tab], ids, None)
    for b, r in enumerate([4, 0, 2]):
        for i in range(hidden):
            k, j = divmod(i, 32)
            assert out[b, i] == np.float32((i % 100 - 50) * 2.0 ** (r - k))


def test_q8_0_sum_of_sixteen_tables_closed_form():
    """Sixteen Q8_0 tables with power-of-two scales and small quants: every partial sum
    is exact in f32, so the gather-sum equals the exact rational sum."""
    vocab, hidden, B = 8, 64, 3
    rng = np.random.default_rng(71)
    tabs, vals = [], []
    for g in range(16):
        blob, v = b"", np.zeros((vocab, hidden))
        for r in range(vocab):
            for k in range(hidden // 32):
                e = int(rng.integers(-6, 3))
                qs = [int(x) for x in rng.integers(-20, 21, 32)]
                blob += _q8_block((15 + e) << 10, qs)
                v[r, 32 * k:32 * k + 32] = np.array(qs) * 2.0 ** e
        tabs.append(np.frombuffer(blob, np.uint8).reshape(vocab, -1))
        vals.append(v)
    ids = rng.integers(0, vocab, (B, 16)).astype(np.int32)
    ov = (rng.integers(-8, 9, (B, hidden)) * 2.0 ** -4).astype(np.float32)
    out, _ = oracle.frame_embed(tabs, ids, ov)
    exact = sum(vals[g][ids[:, g]] for g in range(16)) + ov
    assert np.array_equal(out.astype(np.float64), exact)


def test_embed_bf16_tables_closed_form():
    """bf16 tables (bit patterns): entries (g + 1) + c/8 are exact in bf16 and every
    partial sum is exact in f32, so out = sum_g ((g + 1) + c_g / 8) + overlay exactly."""
    n, vocab, hidden, B = 16, 16, 8, 3
    tabs = []
    for g in range(n):
        vals = np.array([[(g + 1) + c / 8.0] * hidden for c in range(vocab)], np.float32)
        u = vals.view(np.uint32)
        assert (u & 0xFFFF).max() == 0  # exactly representable in bf16
        tabs.append((u >> 16).astype(np.uint16))
    rng = np.random.default_rng(30)
    ids = rng.integers(0, vocab, (B, n)).astype(np.int32)
    ov = np.full((B, hidden), 0.5, np.float32)
    out, flag = oracle.frame_embed(tabs, ids, ov)
    assert flag == 0
    for b in range(B):
        want = sum((g + 1) + ids[b, g] / 8.0 for g in range(n)) + 0.5
        assert np.all(out[b] == np.float32(want))


# ---------------------------------------------------------------------------
# In-graph sampler: counter RNG, own exponential, greedy / top-k
# ---------------------------------------------------------------------------
@pytest.mark.parametrize("key", [(0, 0), (1, 2), (0xDEADBEEF12345678, 0x0123456789ABCDEF)])
def test_philox_matches_numpy_philox(key):
    """numpy's Philox bit generator (Philox4x64-10) steps its counter before each
    block: its outputs 4(n-1)..4n-1 are the block at counter n."""
    bg = np.random.Philox(key=np.array(key, dtype=np.uint64),
                          counter=np.zeros(4, dtype=np.uint64))
    raw = bg.random_raw(12)
    for n in range(1, 4):
        assert [int(x) for x in raw[4 * (n - 1):4 * n]] == oracle.philox4x64_10([n, 0, 0, 0], key)


def test_exp2_f32_accuracy_and_exact_powers():
    xs = np.concatenate([-np.linspace(0, 126, 20001), -np.random.default_rng(31).uniform(0, 126, 2000)])
    got = np.array([oracle.exp2_f32(x) for x in xs.astype(np.float32)], np.float64)
    ref = np.exp2(xs.astype(np.float32).astype(np.float64))
    assert np.max(np.abs(got - ref) / ref) < 3e-7
    for n in range(0, 127):
        assert oracle.exp2_f32(np.float32(-n)) == np.float32(2.0 ** -n)
    assert oracle.exp2_f32(np.float32(-126.5)) == 0.0


def test_philox_all_counter_words_match_numpy_philox():
    """Every counter word enters the generator as numpy's Philox has it: started at
    (c - 1, b, d, 0), numpy's first block is the block at counter (c, b, d, 0) -- the
    words the sampler uses for stream b's draw d at counter value c."""
    key = (0x1234, 0)
    for c, b, d in [(1, 0, 0), (7, 3, 0), (7, 3, 1), (7, 3, 14), (2 ** 40, 31, 9)]:
        bg = np.random.Philox(key=np.array(key, dtype=np.uint64),
                              counter=np.array([c - 1, b, d, 0], dtype=np.uint64))
        assert [int(x) for x in bg.random_raw(4)] == oracle.philox4x64_10([c, b, d, 0], key)


def test_uniform_is_the_top_24_bits():
    x = oracle.philox4x64_10([5, 3, 0, 0], [11, 0])[0]
    assert oracle.uniform_f32(11, 5, 3) == np.float32((x >> 40) / 2.0 ** 24)
    y = oracle.philox4x64_10([5, 3, 7, 0], [11, 0])[0]
    assert oracle.uniform_f32(11, 5, 3, draw=7) == np.float32((y >> 40) / 2.0 ** 24)
    assert x != y


def test_greedy_is_the_first_maximum():
    rng = np.random.default_rng(32)
    lg = rng.standard_normal((6, 300)).astype(np.float32)
    lg[1, [7, 200]] = 9.0   # a tie: the lower index wins
    lg[2, 5] = np.nan       # NaN counts as -inf
    ids = oracle.sample(lg, 0, 1.0, 1, 0)
    ref = np.argmax(np.where(np.isnan(lg), -np.inf, lg), axis=1)
    assert np.array_equal(ids, ref) and ids[1] == 7
    assert np.array_equal(oracle.sample(lg, 1, 0.5, 1, 3), ids)


def test_top_k_draws_follow_the_tempered_softmax():
    """Over many counters the draws of one stream match the softmax of the top-k
    logits at the given temperature (chi-square, fixed seeds), and never leave the
    top k."""
    logits = np.array([[2.0, 1.5, 1.4, 0.3, -1.0, 1.45, -5.0, 0.0]], np.float32)
    k, T, n = 4, 0.7, 3000
    top = sorted(range(8), key=lambda i: (-logits[0, i], i))[:k]
    p = np.exp(logits[0, top].astype(np.float64) / T)
    p /= p.sum()
    counts = {i: 0 for i in range(8)}
    for c in range(n):
        counts[int(oracle.sample(logits, k, T, 99, c)[0])] += 1
    assert all(counts[i] == 0 for i in range(8) if i not in top)
    obs = np.array([counts[i] for i in top], np.float64)
    chi2 = float(((obs - n * p) ** 2 / (n * p)).sum())
    assert chi2 < 16.3  # 3 degrees of freedom, p = 0.001


def test_top_k_ties_at_the_threshold_take_the_lowest_indices():
    """Equal logits at the k-th place: the candidates are the lowest-index ones, equal
    logits are drawn equally often, and an all-equal row is uniform over indices 0..k-1
    (chi-square, fixed seeds)."""
    logits = np.array([[1.0, 5.0, 3.0, 3.0, 3.0, 3.0, 0.0],
                       [2.0, 2.0, 2.0, 2.0, 2.0, 2.0, 2.0]], np.float32)
    k, T, n = 3, 2.0, 4000
    counts = np.zeros((2, 7))
    for c in range(n):
        ids = oracle.sample(logits, k, T, 5, c)
        counts[0, ids[0]] += 1
        counts[1, ids[1]] += 1
    assert counts[0, [0, 4, 5, 6]].sum() == 0 and counts[1, 3:].sum() == 0
    w = np.exp(np.array([5.0, 3.0, 3.0]) / T)
    for row, p in ((0, w / w.sum()), (1, np.full(3, 1.0 / 3.0))):
        obs = counts[row, [1, 2, 3]] if row == 0 else counts[row, :3]
        chi2 = float(((obs - n * p) ** 2 / (n * p)).sum())
        assert chi2 < 13.8  # 2 degrees of freedom, p = 0.001


def test_sample_of_a_row_without_a_finite_logit_is_index_zero():
    lg = np.full((2, 16), -np.inf, np.float32)
    lg[1, :] = np.nan
    assert list(oracle.sample(lg, 0, 1.0, 1, 0)) == [0, 0]
    assert list(oracle.sample(lg, 4, 0.8, 1, 0)) == [0, 0]


# ---------------------------------------------------------------------------
# Whole decode layer with bf16 weights (NEXT-2)
# ---------------------------------------------------------------------------
def _bf16_bits(t):
    return t.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)


def _torch_bf16(x64):
    """float64 tensor -> f32 -> bf16 (round to nearest even) -> back to float64."""
    return x64.float().to(torch.bfloat16).double()


def test_rmsnorm_bf16_matches_torch_rms_norm():
    rng = np.random.default_rng(40)
    h = (rng.standard_normal((3, 64)) * 3).astype(np.float32)
    g = rng.uniform(0.5, 1.5, 64).astype(np.float32)
    got = oracle.rmsnorm_bf16(h, g, 1e-6)
    ref = _torch_bf16(F.rms_norm(torch.from_numpy(h).double(), (64,), torch.from_numpy(g).double(), eps=1e-6))
    assert np.array_equal(got, ref.float().numpy())


def test_gemv_bf16_matches_torch_matmul():
    rng = np.random.default_rng(41)
    x = oracle.bf16_round(rng.standard_normal((4, 96)).astype(np.float32))
    W = torch.from_numpy(rng.standard_normal((40, 96)).astype(np.float32))
    got = oracle.gemv_bf16(x, _bf16_bits(W))
    ref = (torch.from_numpy(x).double() @ W.to(torch.bfloat16).double().T).float().numpy()
    np.testing.assert_array_max_ulp(got, ref, maxulp=1)


def test_silu_mul_matches_torch_silu():
    rng = np.random.default_rng(42)
    g = (rng.standard_normal((2, 500)) * 4).astype(np.float32)
    u = rng.standard_normal((2, 500)).astype(np.float32)
    got = oracle.silu_mul_bf16(g, u)
    ref = _torch_bf16(F.silu(torch.from_numpy(g).double()) * torch.from_numpy(u).double()).float().numpy()
    # one bf16 step where float64 silu formulas round to f32 on either side of a tie
    diff = np.abs(got.view(np.uint32).astype(np.int64) - ref.view(np.uint32).astype(np.int64)) >> 16
    assert diff.max() <= 1 and (diff == 0).mean() > 0.99


def _layer_case(rng, B=2, H=64, Hq=4, Hkv=2, D=16, I=96, cap=32):
    t = lambda *s: torch.from_numpy((rng.standard_normal(s) * 0.2).astype(np.float32))
    wts = dict(gamma_attn=rng.uniform(0.5, 1.5, H).astype(np.float32),
               gamma_mlp=rng.uniform(0.5, 1.5, H).astype(np.float32),
               gamma_q=rng.uniform(0.5, 1.5, D).astype(np.float32),
               gamma_k=rng.uniform(0.5, 1.5, D).astype(np.float32),
               w_qkv=_bf16_bits(t((Hq + 2 * Hkv) * D, H)), w_o=_bf16_bits(t(H, Hq * D)),
               w_gu=_bf16_bits(t(2 * I, H)), w_down=_bf16_bits(t(H, I)))
    h = (rng.standard_normal((B, H)) * 2).astype(np.float32)
    kc = rng.standard_normal((B, Hkv, cap, D)).astype(np.float32)
    vc = rng.standard_normal((B, Hkv, cap, D)).astype(np.float32)
    return wts, h, kc, vc, oracle.KvLayout(B, Hkv, D, cap)


def test_decode_layer_mlp_half_matches_torch():
    """With W_o = 0 the attention half adds exactly nothing, so the layer is the MLP
    half alone: torch rms_norm, matmuls in float64, silu, bf16 roundings by torch."""
    rng = np.random.default_rng(43)
    wts, h, kc, vc, lay = _layer_case(rng)
    wts["w_o"][:] = 0
    h0 = h.copy()
    oracle.decode_layer(h, wts, kc, vc, lay, np.array([5, 30], np.int32), np.float32(1e-6), 1e6, 0.25)
    T = torch.from_numpy
    x2 = _torch_bf16(F.rms_norm(T(h0).double(), (64,), T(wts["gamma_mlp"]).double(), eps=1e-6))
    Wgu = T(oracle.bf16_bits_to_f32(wts["w_gu"])).double()
    gu = (x2 @ Wgu.T).float().double()
    a = _torch_bf16(F.silu(gu[:, :96]) * gu[:, 96:])
    d = (a @ T(oracle.bf16_bits_to_f32(wts["w_down"])).double().T).float()
    ref = (T(h0) + d).numpy()
    np.testing.assert_array_max_ulp(h, ref, maxulp=2)


def test_decode_layer_attention_half_matches_torch():
    """With the up rows of W_gu zero the MLP half adds exactly nothing: h gains
    bf16(attention) W_o^T, where the attention is the pinned decode step of the
    normed-and-projected row."""
    rng = np.random.default_rng(44)
    wts, h, kc, vc, lay = _layer_case(rng)
    wts["w_gu"][96:] = 0
    h0 = h.copy()
    kc0, vc0 = kc.copy(), vc.copy()
    cur = np.array([0, 17], np.int32)
    oracle.decode_layer(h, wts, kc, vc, lay, cur, np.float32(1e-6), 1e6, 0.25)
    T = torch.from_numpy
    x = _torch_bf16(F.rms_norm(T(h0).double(), (64,), T(wts["gamma_attn"]).double(), eps=1e-6))
    qkv = (x @ T(oracle.bf16_bits_to_f32(wts["w_qkv"])).double().T).float().numpy()
    q, k, v = qkv[:, :64].reshape(2, 4, 16), qkv[:, 64:96].reshape(2, 2, 16), qkv[:, 96:].reshape(2, 2, 16)
    attn = oracle.decode_step(q, k, v, wts["gamma_q"], wts["gamma_k"], np.float32(1e-6), 1e6,
                              kc0, vc0, lay, cur, 0.25)
    o = (_torch_bf16(T(attn.reshape(2, 64)).double()) @ T(oracle.bf16_bits_to_f32(wts["w_o"])).double().T).float()
    np.testing.assert_array_max_ulp(h, (T(h0) + o).numpy(), maxulp=2)
    assert np.array_equal(kc, kc0) and np.array_equal(vc, vc0)  # the step wrote the same rows


def test_decode_layer_batched_equals_per_stream():
    rng = np.random.default_rng(45)
    wts, h, kc, vc, lay = _layer_case(rng, B=3)
    cur = np.array([0, 9, 31], np.int32)
    hb, kb, vb = h.copy(), kc.copy(), vc.copy()
    oracle.decode_layer(hb, wts, kb, vb, lay, cur, np.float32(1e-6), 1e6, 0.25)
    for b in range(3):
        h1, k1, v1 = h[b:b + 1].copy(), kc[b:b + 1].copy(), vc[b:b + 1].copy()
        oracle.decode_layer(h1, wts, k1, v1, oracle.KvLayout(1, 2, 16, 32), cur[b:b + 1],
                            np.float32(1e-6), 1e6, 0.25)
        assert np.array_equal(h1[0], hb[b]) and np.array_equal(k1[0], kb[b])
