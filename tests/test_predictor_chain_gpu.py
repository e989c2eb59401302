"""A whole code-predictor frame on the GPU against a chain of oracle calls.

Each frame runs the in-graph sampler, which writes every sub-code into the frame's
code ids. The next gather reads that sub-code from its group table, and the decode
steps of all 5 layers run after it. Two frames are captured per graph replay and the
graph is replayed twice, so four frames run at Philox counter values 0..3, each
advanced inside the graph. This is the predictor frame unroll with the in-graph
sampler ("qwentts.cpp -- commits/branch/master/tests" page, fused codec tail) and the
several frames per replay of "minicpm-o-4.5 ... docs/optimizations.md" (core table,
CUDA-graph decode row), at the code-predictor workload's shapes: 32 streams, 5 layers,
16 q / 8 kv heads, head_dim 64, f32 16-slot caches reset per frame, top-50 at
temperature 0.9.

Tokens and gathered rows must be bit-exact. Attention outputs must be within 1e-5 per
(stream, head) row of the oracle's double result.
"""
import numpy as np
import pytest
import torch

import oracle
from autoregressive_codebook_tts_gb300 import workloads as W
from gpu_helpers import ATTN_TOL, row_rel_err

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tts(cuda_dev):
    from autoregressive_codebook_tts_gb300 import build
    build.build()
    from autoregressive_codebook_tts_gb300 import tts as mod
    return mod


def test_predictor_frames_chain_two_per_replay(tts):
    from autoregressive_codebook_tts_gb300.predictor import PredictorFrames
    w = W.workload("predictor")
    B, L, Hq, Hkv, D, V, H = w.B, w.layers, w.n_q_heads, w.n_kv_heads, w.head_dim, w.vocab, w.hidden
    K, top_k, temp, seed = 2, 50, 0.9, 777
    tables = W.tables(15, V, H, seed=50)
    pre = [W.qkv(2 * B, Hq, Hkv, D, seed=60 + l)[0] for l in range(L)]
    width = pre[0].shape[1]
    qkv = torch.zeros(16, L, B, width)
    for t in range(2, 16):
        for l in range(L):
            qkv[t, l] = W.qkv(B, Hq, Hkv, D, seed=100 + 16 * l + t)[0]
    logits = W.logits(15, B, V, seed=80)
    gq = torch.stack([W.gamma(D, 4 + l) for l in range(L)])
    gk = torch.stack([W.gamma(D, 40 + l) for l in range(L)])
    c0 = torch.cat([W.code_ids(B, 1, V, seed=90 + s) for s in range(K)], dim=1).t().contiguous()

    pf = PredictorFrames(B, L, Hq, Hkv, D, H, V, [t.cuda() for t in tables],
                         torch.stack(pre).cuda(), qkv.cuda(), logits.cuda(), gq.cuda(), gk.cuda(),
                         top_k, temp, seed, c0, eps=w.eps, rope_base=w.rope_base,
                         capacity=w.capacity, slots=K)
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        pf.enqueue_frames(K, stream=s)  # outside the capture: sets kernel attributes
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        pf.enqueue_frames(K, stream=s)
    pf.counter.zero_()
    torch.cuda.synchronize()

    # oracle side: per-position q/k/v in oracle shapes, persistent caches
    qd, kd = Hq * D, Hkv * D

    def split(rows):
        rows = rows.numpy()
        return (rows[:, :qd].reshape(-1, Hq, D), rows[:, qd:qd + kd].reshape(-1, Hkv, D),
                rows[:, qd + kd:].reshape(-1, Hkv, D))
    per_t = []
    for t in range(16):
        per_l = []
        for l in range(L):
            if t < 2:
                q, k, v = split(pre[l])
                per_l.append((q[t::2].copy(), k[t::2].copy(), v[t::2].copy()))
            else:
                per_l.append(split(qkv[t, l]))
        per_t.append(per_l)
    gammas = [(gq[l].numpy(), gk[l].numpy()) for l in range(L)]
    caches = [(np.zeros((B, Hkv, w.capacity, D), np.float32),
               np.zeros((B, Hkv, w.capacity, D), np.float32)) for _ in range(L)]
    lay = oracle.KvLayout(B, Hkv, D, w.capacity)
    tabs_np = [t.numpy() for t in tables]
    lg_np = logits.numpy()

    counter = 0
    for replay in range(2):
        g.replay()
        torch.cuda.synchronize()
        assert pf.err.item() == 0
        assert pf.counter.item() == counter + K
        codes_gpu = pf.codes.cpu().numpy()
        emb_gpu = pf.emb.cpu().numpy()
        out_gpu = pf.out.cpu().numpy()
        pout_gpu = pf.pout.cpu().numpy()
        for slot in range(K):
            codes = np.zeros((B, 16), np.int32)
            codes[:, 0] = c0[slot].numpy()
            for j in range(1, 16):
                codes[:, j] = oracle.sample(lg_np[j - 1], top_k, temp, seed, counter, draw=j)
            assert np.array_equal(codes_gpu[slot], codes), (replay, slot)
            embeds, outs = oracle.predictor_frame(tabs_np, codes[:, :15], None, per_t, gammas,
                                                  np.float32(w.eps), w.rope_base, caches, lay,
                                                  1.0 / np.sqrt(D))
            for j in range(15):
                assert np.array_equal(emb_gpu[slot, j].view(np.uint32), embeds[j].view(np.uint32)), j
            for l in range(L):
                for t in range(2):
                    assert row_rel_err(pout_gpu[slot, l, :, t], outs[t][l]) <= ATTN_TOL["f32"]
                for t in range(2, 16):
                    assert row_rel_err(out_gpu[slot, t, l], outs[t][l]) <= ATTN_TOL["f32"]
            counter += 1
    # the frames drew distinct sub-codes: the counter and the draw index both matter
    assert len({tuple(r) for r in codes_gpu[:, :, 1:].reshape(K, -1)}) == K
