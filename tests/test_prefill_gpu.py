"""Prefill of T positions per stream (tts_prefill_step) against the oracle: the cache
bytes bit-exact, the q rows left as given, every query's output within the attention
tolerance of the causal definition.  Contiguous and paged, f32 and bf16, a prompt after
a reset (start 0) and after earlier rows, and the error flags of positions past the
cache."""
import numpy as np
import pytest
import torch

import oracle
from autoregressive_codebook_tts_gb300 import workloads as W
from gpu_helpers import ATTN_TOL, Layer, bits, cache_np, rope_table, row_rel_err, scale_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tts(cuda_dev):
    from autoregressive_codebook_tts_gb300 import build
    build.build()
    from autoregressive_codebook_tts_gb300 import tts as mod
    return mod


def _run(tts, w, start, T, seed, n_splits=0, poison=True):
    """Prefill T rows per stream at `start`; returns (layer, rows, out, ef, ref_out, kc, vc, qn)."""
    L = Layer(w, seed=seed, cur_len=start, poison=poison)
    B, Hq, Hkv, D = w.B, w.n_q_heads, w.n_kv_heads, w.head_dim
    rows, _, _, _ = W.qkv(B * T, Hq, Hkv, D, seed + 10)
    qd, kd = Hq * D, Hkv * D
    d_rows = rows.cuda()
    q, k, v = d_rows[:, :qd], d_rows[:, qd:qd + kd], d_rows[:, qd + kd:]
    cs = rope_table(tts, w.capacity, D, w.rope_base)
    desc = L.desc(tts)
    ws = tts.prefill_workspace(desc, T, n_splits)
    out = torch.full((B, T, Hq, D), float("nan"), device="cuda")
    ef = torch.zeros(1, dtype=torch.int32, device="cuda")
    start_d = torch.as_tensor(start, dtype=torch.int32).cuda()
    tts.tts_prefill_step(q, k, v, L.d_gq, L.d_gk, w.eps, cs, w.capacity, L.d_K, L.d_V, desc,
                         start_d, T, scale_of(w), out, ws, n_splits, ef)
    torch.cuda.synchronize()
    # oracle on the host copies of the same inputs
    hr = rows.numpy()
    qh = hr[:, :qd].reshape(B, T, Hq, D)
    kh = hr[:, qd:qd + kd].reshape(B, T, Hkv, D)
    vh = hr[:, qd + kd:].reshape(B, T, Hkv, D)
    kc, vc = cache_np(L.K), cache_np(L.V)
    st = np.asarray(start, np.int32)
    ref = oracle.prefill_step(qh, kh, vh, L.gq.numpy(), L.gk.numpy(), np.float32(w.eps), w.rope_base,
                              kc, vc, L.layout(), st, scale_of(w))
    pos = st[:, None] + np.arange(T, dtype=np.int32)[None, :]
    qn = np.stack([oracle.rms_norm_rope(qh[:, t], L.gq.numpy(), np.float32(w.eps), pos[:, t], w.rope_base)
                   for t in range(T)], axis=1)
    return L, q, out, ef, ref, kc, vc, qn


def _check_caches(L, w, start, T, kc, vc):
    """V: every byte equal.  K: every byte outside the prompt's rows equal; the prompt's
    rows (normed and rotated in f32 on the device, in double by the oracle) within
    2e-6 (f32); bf16 within one ulp of the element plus 1e-6 of its row's largest
    magnitude: where the rotation cancels (x cos - y sin much smaller than x and y) the
    f32 and f64 results may round to bf16 values a few of the small element's ulps
    apart, while any wrong element is off by about its row's scale."""
    gk, gv = cache_np(L.d_K), cache_np(L.d_V)
    assert np.array_equal(bits(gv), bits(vc))
    mask = np.zeros(kc.shape, bool)
    for b in range(w.B):
        for t in range(T):
            p = int(start[b]) + t
            if p >= w.capacity:
                continue
            for g in range(w.n_kv_heads):
                if w.paged:
                    mask[int(L.bt[b, p // w.page_size]), g, p % w.page_size] = True
                else:
                    mask[b, g, p] = True
    assert not ((bits(gk) != bits(kc)) & ~mask).any()
    if w.kv_dtype == "f32":
        np.testing.assert_allclose(gk[mask], kc[mask], rtol=2e-6, atol=2e-6)
    else:
        f = lambda a: (a.astype(np.uint32) << 16).view(np.float32).astype(np.float64)
        got, ref = f(gk), f(kc)
        row_max = np.abs(ref).max(axis=-1, keepdims=True)
        ulp = np.abs(f(kc + 1) - ref)   # the spacing above the oracle's bf16 value
        bound = np.broadcast_to(ulp + 1e-6 * row_max, ref.shape)
        assert (np.abs(got - ref)[mask] <= bound[mask]).all()


# Prompts of 8 rows or more take a multi-query kernel (blocks of queries sharing every
# K/V tile: 128 / G on the tensor cores for bf16 caches with head_dim 128 and contiguous
# or 64-row-or-larger pages, 64 / G on the CUDA cores otherwise), shorter ones the
# per-query decode path.  The multi-query
# cases cover f32 and bf16, head_dim 64 and 128, GQA groups 1, 2 and 4, a ragged last
# query block (T = 130 in blocks of 64, T = 17 in blocks of 16), contiguous caches and
# pages of 8, 16, 64 and 128 rows (one tile split over pages, one box per page, two
# boxes per page).
CASES = [
    ("tiny", dict(), [0], 1),
    ("tiny", dict(), [0], 2),
    ("tiny", dict(), [37], 7),
    ("tiny", dict(), [0], 40),
    ("batched", dict(B=2, layers=1), [100, 3000], 33),
    ("paged", dict(B=2, layers=1, n_pages=600), [50, 1000], 20),
    ("talker", dict(layers=1), [4000], 64),
    ("tiny", dict(head_dim=64, capacity=512), [100], 50),
    ("tiny", dict(n_kv_heads=16, capacity=512), [5], 130),
    ("tiny", dict(n_kv_heads=4, capacity=512), [200], 17),
    ("batched", dict(B=2, layers=1, head_dim=64, capacity=1024), [10, 300], 40),
    ("paged", dict(B=2, layers=1, page_size=64, n_pages=200), [100, 1000], 70),
    ("paged", dict(B=2, layers=1, page_size=128, n_pages=100, kv_dtype="f32"), [0, 2000], 24),
    ("paged", dict(B=2, layers=1, page_size=8, n_pages=300, capacity=1024), [500, 900], 32),
    # bf16, head_dim 128 on the tensor cores with GQA groups 1 and 4 (blocks of 128 and
    # 32 queries, the last ragged), contiguous and 64-row pages
    ("batched", dict(B=2, layers=1, n_kv_heads=16, capacity=2048), [100, 1000], 140),
    ("batched", dict(B=2, layers=1, n_kv_heads=4, capacity=2048), [50, 1900], 70),
    ("paged", dict(B=2, layers=1, n_kv_heads=4, page_size=64, n_pages=200), [300, 2000], 45),
]


@pytest.mark.parametrize("name,over,start,T", CASES)
def test_prefill_matches_oracle(tts, name, over, start, T):
    w = W.workload(name, **over)
    L, q, out, ef, ref, kc, vc, qn = _run(tts, w, start, T, seed=60)
    q_in = W.qkv(w.B * T, w.n_q_heads, w.n_kv_heads, w.head_dim, 70)[0][:, :w.n_q_heads * w.head_dim]
    assert ef.item() == 0
    _check_caches(L, w, start, T, kc, vc)
    # q is read only: the rows are the caller's, bit for bit
    assert np.array_equal(bits(q.cpu().numpy()), bits(q_in.numpy()))
    # every query within the attention tolerance of the causal definition
    o = out.cpu().numpy()
    assert np.isfinite(o).all()
    assert row_rel_err(o.reshape(-1, w.n_q_heads, w.head_dim),
                       ref.reshape(-1, w.n_q_heads, w.head_dim)) <= ATTN_TOL[w.kv_dtype]


@pytest.mark.parametrize("n_splits", [1, 3, 16])
def test_prefill_split_counts_agree(tts, n_splits):
    w = W.workload("talker", layers=1)
    _, _, out, ef, ref, _, _, _ = _run(tts, w, [1500], 24, seed=61, n_splits=n_splits)
    assert ef.item() == 0
    assert row_rel_err(out.cpu().numpy().reshape(-1, 16, 128), ref.reshape(-1, 16, 128)) <= ATTN_TOL["f32"]


# bf16 caches take the tensor-core kernel: 2..8 chunks whose clusters (one per item) all
# fit on the device at once merge inside the launch, 1 chunk normalises in place, other
# counts take the combine launch.  T = 100 gives 16 items of 128 query rows (the second
# ragged), T = 40 gives 8.
@pytest.mark.parametrize("T,n_splits", [(100, 1), (100, 2), (100, 5), (100, 8), (100, 9), (100, 16),
                                        (40, 3), (40, 7), (40, 8)])
def test_tensor_core_prefill_split_counts(tts, T, n_splits):
    w = W.workload("talker", layers=1, kv_dtype="bf16")
    _, _, out, ef, ref, _, _, _ = _run(tts, w, [1500], T, seed=62, n_splits=n_splits)
    assert ef.item() == 0
    assert row_rel_err(out.cpu().numpy().reshape(-1, 16, 128), ref.reshape(-1, 16, 128)) <= ATTN_TOL["bf16"]


def test_prefill_launch_count(tts):
    # the rows and the attention, plus the combine when chunks are merged by a third launch
    w = W.workload("talker", layers=1)
    d16, d32 = (tts.kv_desc(w.B, w.n_q_heads, w.n_kv_heads, w.head_dim, w.capacity, dt,
                            window_quantum=w.window_quantum) for dt in ("bf16", "f32"))
    assert tts.tts_prefill_launch_count(d16, 2) == 2          # per-query decode path
    assert tts.tts_prefill_launch_count(d32, 24, 1) == 2      # one chunk
    assert tts.tts_prefill_launch_count(d32, 24, 3) == 3      # CUDA cores: combine launch
    assert tts.tts_prefill_launch_count(d16, 100, 16) == 3    # more than 8 chunks
    assert tts.tts_prefill_launch_count(d16, 100, 2) == 2     # 16 clusters of 2 fit at once
    assert tts.tts_prefill_launch_count(d16, 0) == 0


def test_prefill_of_one_row_equals_the_decode_step(tts):
    """T = 1 at start c is the decode step at cur_len c: the same cache bytes, outputs
    within rounding of each other (different kernels: the decode step folds the new row
    in from registers, the prefill reads it back from the cache)."""
    w = W.workload("batched", B=3, layers=1)
    cur = [5, 700, 2047]
    L, _, out, ef, _, _, _, _ = _run(tts, w, cur, 1, seed=62, poison=False)
    assert ef.item() == 0
    D2 = Layer(w, seed=62, cur_len=cur, poison=False)
    rows, _, _, _ = W.qkv(w.B, 16, 8, 128, 72)
    d_rows = rows.cuda()
    cs = rope_table(tts, w.capacity, 128, w.rope_base)
    desc = D2.desc(tts)
    o2 = torch.empty(w.B, 16, 128, device="cuda")
    tts.tts_decode_step(d_rows[:, :2048], d_rows[:, 2048:3072], d_rows[:, 3072:], D2.d_gq, D2.d_gk,
                        w.eps, cs, w.capacity, D2.d_K, D2.d_V, desc, D2.d_cur, scale_of(w), o2,
                        tts.workspace(desc, 0), 0, ef)
    torch.cuda.synchronize()
    assert ef.item() == 0
    assert torch.equal(D2.d_K.view(torch.int16), L.d_K.view(torch.int16))
    assert torch.equal(D2.d_V.view(torch.int16), L.d_V.view(torch.int16))
    assert row_rel_err(o2.cpu().numpy(), out[:, 0].cpu().numpy()) <= 1e-3  # bf16 KV, two paths


def test_predictor_two_row_prefill_after_reset(tts):
    """The code predictor's T = 2 prefill at position 0 (16-slot f32 cache, D = 64)."""
    w = W.workload("predictor", layers=1)
    L, _, out, ef, ref, kc, vc, _ = _run(tts, w, [0] * w.B, 2, seed=63)
    assert ef.item() == 0
    _check_caches(L, w, [0] * w.B, 2, kc, vc)
    assert row_rel_err(out.cpu().numpy().reshape(-1, 16, 64), ref.reshape(-1, 16, 64)) <= ATTN_TOL["f32"]


def test_prefill_flags_positions_past_the_cache(tts):
    """A prompt running past capacity: the rows inside are written, the rest skipped
    with TTS_EFLAG_POS_RANGE, and the windows past capacity clamped with
    TTS_EFLAG_NVALID; the queries inside the cache are still exact."""
    w = W.workload("tiny")
    T, start = 6, w.capacity - 3
    L, _, out, ef, ref, kc, vc, _ = _run(tts, w, [start], T, seed=64)
    assert ef.item() & tts.EFLAG_POS_RANGE and ef.item() & tts.EFLAG_NVALID
    _check_caches(L, w, [start], T, kc, vc)
    inside = 3
    assert row_rel_err(out[:, :inside].cpu().numpy().reshape(-1, 16, 128),
                       ref[:, :inside].reshape(-1, 16, 128)) <= ATTN_TOL["f32"]


@pytest.mark.parametrize("T", [2, 48])
def test_paged_prefill_never_reads_entries_past_the_window(tts, T):
    """Block-table entries past each stream's last prompt row hold -1: the prefill (per
    query path for T = 2, multi-query kernel for T = 48) must read none of them and set
    no flag, giving the bytes of a fully assigned table."""
    w = W.workload("paged", B=2, layers=1, n_pages=600)
    start = [300, 2000]
    L = Layer(w, seed=65, cur_len=start, poison=False)
    B, Hq, Hkv, D = w.B, w.n_q_heads, w.n_kv_heads, w.head_dim
    rows, _, _, _ = W.qkv(B * T, Hq, Hkv, D, 75)
    qd, kd = Hq * D, Hkv * D
    cs = rope_table(tts, w.capacity, D, w.rope_base)
    trimmed = L.d_bt.clone()
    for b in range(B):
        used = (start[b] + T + w.page_size - 1) // w.page_size
        trimmed[b, used:] = -1
    assert (trimmed == -1).any()
    start_d = torch.as_tensor(start, dtype=torch.int32).cuda()
    results = []
    for bt in (L.d_bt, trimmed):
        K, V = L.d_K.clone(), L.d_V.clone()
        d_rows = rows.cuda()
        desc = tts.kv_desc(B, Hq, Hkv, D, w.capacity, w.kv_dtype, paged=True, page_size=w.page_size,
                           n_pages=w.n_pages, block_table=bt)
        ws = tts.prefill_workspace(desc, T, 0)
        out = torch.full((B, T, Hq, D), float("nan"), device="cuda")
        ef = torch.zeros(1, dtype=torch.int32, device="cuda")
        tts.tts_prefill_step(d_rows[:, :qd], d_rows[:, qd:qd + kd], d_rows[:, qd + kd:], L.d_gq, L.d_gk, w.eps,
                             cs, w.capacity, K, V, desc, start_d, T, scale_of(w), out, ws, 0, ef)
        torch.cuda.synchronize()
        assert ef.item() == 0
        results.append((out.cpu(), K.cpu(), V.cpu()))
    for a, b in zip(*results):
        assert torch.equal(a.view(torch.int16) if a.dtype == torch.bfloat16 else a.view(torch.int32),
                           b.view(torch.int16) if b.dtype == torch.bfloat16 else b.view(torch.int32))


@pytest.mark.parametrize("kv_dtype,T,n_splits", [("bf16", 100, 0), ("bf16", 100, 16), ("f32", 40, 0)])
def test_prefill_graph_replay_equals_eager(tts, kv_dtype, T, n_splits):
    """Two layers' prefill steps captured in a graph replay to the eager bytes: the
    tensor-core kernel with its chunks merged in clusters (default) or by the combine
    launch (16 chunks), and the CUDA-core kernel."""
    w = W.workload("talker", layers=1, kv_dtype=kv_dtype)
    B, Hq, Hkv, D = w.B, w.n_q_heads, w.n_kv_heads, w.head_dim
    cs = rope_table(tts, w.capacity, D, w.rope_base)
    layers = [Layer(w, seed=90 + l, cur_len=[2000]) for l in range(2)]
    rows = [W.qkv(B * T, Hq, Hkv, D, 95 + l)[0].cuda() for l in range(2)]
    qd, kd = Hq * D, Hkv * D
    desc = layers[0].desc(tts)
    ws = tts.prefill_workspace(desc, T, n_splits)
    outs = [torch.empty(B, T, Hq, D, device="cuda") for _ in range(2)]
    start = torch.full((B,), 2000, dtype=torch.int32, device="cuda")
    ef = torch.zeros(1, dtype=torch.int32, device="cuda")
    caches0 = [(L.d_K.clone(), L.d_V.clone()) for L in layers]

    def step():
        for l, L in enumerate(layers):
            r = rows[l]
            tts.tts_prefill_step(r[:, :qd], r[:, qd:qd + kd], r[:, qd + kd:], L.d_gq, L.d_gk, w.eps, cs,
                                 w.capacity, L.d_K, L.d_V, desc, start, T, scale_of(w), outs[l], ws,
                                 n_splits, ef)

    step()
    torch.cuda.synchronize()
    eager = [o.clone() for o in outs]
    eager_k = [L.d_K.clone() for L in layers]
    for (k0, v0), L in zip(caches0, layers):
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
    assert ef.item() == 0
    for a, b in zip(eager, outs):
        assert torch.equal(a, b)
    # the caches bit for bit (their tails hold NaN poison, so compare the bits)
    ibits = torch.int16 if eager_k[0].dtype == torch.bfloat16 else torch.int32
    for a, L in zip(eager_k, layers):
        assert torch.equal(a.view(ibits), L.d_K.view(ibits))
