"""A whole talker decode layer with bf16 weights (tts_decode_layer) against the
oracle's decode_layer: the residual stream after the layer within 1e-3 per stream row
(max |diff| / max |ref|), the cache rows as for the decode step.  The GPU sums the
products in f32 where the oracle sums them exactly, so a bf16 rounding of an
intermediate (the norm output, the attention output, the SiLU product) can land one
bf16 step apart; such a step moves the layer's output by about 2^-8 of one product
term, far inside the bound.  The projections run on the tensor cores, whose f32
accumulation order differs again; the bound covers it the same way."""
import numpy as np
import pytest
import torch

import oracle
from autoregressive_codebook_tts_gb300 import workloads as W
from gpu_helpers import Layer, bits, cache_np, rope_table, scale_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tts(cuda_dev):
    from autoregressive_codebook_tts_gb300 import build
    build.build()
    from autoregressive_codebook_tts_gb300 import tts as mod
    return mod


def _weights(H, I, Hq, Hkv, D, seed):
    g = torch.Generator().manual_seed(seed)
    m = lambda r, c: (torch.randn(r, c, generator=g) * 0.02).to(torch.bfloat16)
    return dict(w_qkv=m((Hq + 2 * Hkv) * D, H), w_o=m(H, Hq * D), w_gu=m(2 * I, H), w_down=m(H, I),
                gamma_attn=torch.rand(H, generator=g) + 0.5, gamma_mlp=torch.rand(H, generator=g) + 0.5,
                gamma_q=torch.rand(D, generator=g) + 0.5, gamma_k=torch.rand(D, generator=g) + 0.5)


def _bits16(t):
    return t.view(torch.int16).numpy().view(np.uint16)


# The talker shapes, and two smaller layers whose row lengths split into several
# segments of 768 / 1280 elements (hidden 768 / 1280, intermediate 3 x hidden) with
# partial ranges at the ends of the clusters' column splits (1 to 8 streams use the
# MMA's N of 16 with padding slots).
SMALL_768 = dict(hidden=768, n_q_heads=4, n_kv_heads=2, capacity=512)
SMALL_1280 = dict(hidden=1280, n_q_heads=8, n_kv_heads=2, capacity=512)


# 16 and 32 streams use the MMA's N of 16 and 32, the small layers odd tile counts and
# column ranges (hidden 768: six 128-row tiles of the output projections, 2304 SiLU items).
STREAMS_16 = [3, 40, 97, 130, 200, 255, 256, 300, 311, 350, 400, 401, 450, 480, 500, 511]
STREAMS_32 = [(b * 37) % 512 for b in range(32)]


@pytest.mark.parametrize("B,cur,shape", [(1, [4095], {}), (1, [100], {}), (2, [10, 4000], {}), (4, [7, 1000, 2047, 3000], {}),
                                         (8, [300] * 8, {}), (3, [5, 200, 511], SMALL_768),
                                         (5, [0, 1, 64, 300, 511], SMALL_1280), (1, [300], SMALL_768),
                                         (1, [511], SMALL_1280), (16, STREAMS_16, dict(capacity=512)),
                                         (32, STREAMS_32, dict(capacity=512)),
                                         (7, [1, 2, 3, 4, 5, 6, 7], SMALL_768)])
def test_decode_layer_matches_oracle(tts, B, cur, shape):
    w = W.workload("talker", B=B, layers=1, **shape)
    H, I, Hq, Hkv, D = w.hidden, 3 * w.hidden, w.n_q_heads, w.n_kv_heads, w.head_dim
    L = Layer(w, seed=80, cur_len=cur, poison=True)
    wt = _weights(H, I, Hq, Hkv, D, 81)
    d = {k: v.cuda() for k, v in wt.items()}
    lw = tts.layer_weights(d["w_qkv"], d["w_o"], d["w_gu"], d["w_down"], d["gamma_attn"],
                           d["gamma_mlp"], d["gamma_q"], d["gamma_k"])
    g = torch.Generator().manual_seed(82)
    h0 = torch.randn(B, H, generator=g)
    h = h0.cuda()
    cs = rope_table(tts, w.capacity, D, w.rope_base)
    desc = L.desc(tts)
    scratch = tts.layer_scratch(desc, H, I, 0)
    ef = torch.zeros(1, dtype=torch.int32, device="cuda")
    tts.tts_decode_layer(h, lw, w.eps, cs, w.capacity, L.d_K, L.d_V, desc, L.d_cur, scale_of(w),
                         scratch, 0, ef)
    torch.cuda.synchronize()
    assert ef.item() == 0
    hk, hv = cache_np(L.K), cache_np(L.V)
    ref = h0.numpy().copy()
    ow = {k: (_bits16(v) if v.dtype == torch.bfloat16 else v.numpy()) for k, v in wt.items()}
    oracle.decode_layer(ref, ow, hk, hv, L.layout(), L.cur.numpy(), np.float32(w.eps), w.rope_base,
                        scale_of(w))
    got = h.cpu().numpy()
    err = (np.abs(got - ref).max(axis=1) / np.abs(ref).max(axis=1)).max()
    assert err <= 1e-3, err
    # the cache: only the new rows changed; V rows exact, K rows within rounding
    gk, gv = cache_np(L.d_K), cache_np(L.d_V)
    mask = np.zeros(hk.shape, bool)
    for b in range(B):
        mask[b, :, cur[b]] = True
    assert not ((bits(gk) != bits(hk)) & ~mask).any() and not ((bits(gv) != bits(hv)) & ~mask).any()
    np.testing.assert_allclose(gk[mask], hk[mask], rtol=1e-4, atol=1e-4)
    np.testing.assert_allclose(gv[mask], hv[mask], rtol=1e-4, atol=1e-4)


def test_decode_layer_rejects_more_than_32_streams(tts):
    w = W.workload("talker", B=33, layers=1)
    desc = tts.kv_desc(33, 16, 8, 128, 4096)
    assert tts.tts_decode_layer_scratch_size(desc, 2048, 6144) > 0
    wt = {k: v.cuda() for k, v in _weights(2048, 6144, 16, 8, 128, 83).items()}
    lw = tts.layer_weights(wt["w_qkv"], wt["w_o"], wt["w_gu"], wt["w_down"], wt["gamma_attn"],
                           wt["gamma_mlp"], wt["gamma_q"], wt["gamma_k"])
    h = torch.zeros(33, 2048, device="cuda")
    K = torch.zeros(33, 8, 16, 128, device="cuda")  # never read: the call is refused first
    cur = torch.zeros(33, dtype=torch.int32, device="cuda")
    cs = rope_table(tts, 4096, 128, w.rope_base)
    with pytest.raises(tts.TtsError) as e:
        tts.tts_decode_layer(h, lw, 1e-6, cs, 4096, K, K, desc, cur, 0.1,
                             tts.layer_scratch(desc, 2048, 6144), 0)
    assert e.value.status == 2


@pytest.mark.parametrize("B", [1, 32])
def test_decode_layer_graph_replay_equals_eager(tts, B):
    """Two layers captured in a graph replay to the eager bytes: the projections' column
    ranges are summed in a fixed order and the attention's splits merged in a fixed order,
    so nothing depends on timing."""
    w = W.workload("talker", B=B, layers=1, capacity=512)
    H, I, Hq, Hkv, D = w.hidden, 3 * w.hidden, w.n_q_heads, w.n_kv_heads, w.head_dim
    cur = [(b * 37 + 5) % 500 for b in range(B)]
    layers = [Layer(w, seed=120 + l, cur_len=cur, poison=True) for l in range(2)]
    lws, keep = [], []
    for l in range(2):
        d = {k: v.cuda() for k, v in _weights(H, I, Hq, Hkv, D, 130 + l).items()}
        keep.append(d)
        lws.append(tts.layer_weights(d["w_qkv"], d["w_o"], d["w_gu"], d["w_down"], d["gamma_attn"],
                                     d["gamma_mlp"], d["gamma_q"], d["gamma_k"]))
    cs = rope_table(tts, w.capacity, D, w.rope_base)
    descs = [L.desc(tts) for L in layers]
    scratch = tts.layer_scratch(descs[0], H, I, 0)
    ef = torch.zeros(1, dtype=torch.int32, device="cuda")
    h0 = torch.randn(B, H, generator=torch.Generator().manual_seed(140)).cuda()
    h = h0.clone()
    caches0 = [(L.d_K.clone(), L.d_V.clone()) for L in layers]

    def frame():
        for l, L in enumerate(layers):
            tts.tts_decode_layer(h, lws[l], w.eps, cs, w.capacity, L.d_K, L.d_V, descs[l], L.d_cur,
                                 scale_of(w), scratch, 0, ef)

    frame()
    torch.cuda.synchronize()
    eager = h.clone()
    h.copy_(h0)
    for (k0, v0), L in zip(caches0, layers):
        L.d_K.copy_(k0)
        L.d_V.copy_(v0)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        frame()
    g.replay()
    torch.cuda.synchronize()
    assert ef.item() == 0
    assert torch.equal(eager.view(torch.int32), h.view(torch.int32))
