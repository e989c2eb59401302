"""The in-graph sampler (tts_sample) against the oracle: the token of every stream
equal, greedy and temperature/top-k, on fresh counters; ties, NaN and -inf rows; the
column of an ids buffer as output; the counter advanced inside a replayed graph."""
import numpy as np
import pytest
import torch

import oracle
from autoregressive_codebook_tts_gb300 import workloads as W

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tts(cuda_dev):
    from autoregressive_codebook_tts_gb300 import build
    build.build()
    from autoregressive_codebook_tts_gb300 import tts as mod
    return mod


def _logits(B, V, seed, scale=2.0):
    g = torch.Generator().manual_seed(seed)
    return torch.randn(B, V, generator=g) * scale


@pytest.mark.parametrize("top_k,temperature", [(0, 1.0), (1, 0.5), (2, 1.0), (8, 0.7), (50, 1.0),
                                               (64, 1.6)])
def test_sample_matches_oracle(tts, top_k, temperature):
    B, V, seed = 32, 2048, 1234
    lg = _logits(B, V, 7)
    d_lg = lg.cuda()
    counter = torch.zeros(1, dtype=torch.int64, device="cuda")
    for c in range(3):
        counter.fill_(c)
        out = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        tts.tts_sample(d_lg, top_k, temperature, seed, counter, out)
        torch.cuda.synchronize()
        ref = oracle.sample(lg.numpy(), top_k, temperature, seed, c)
        assert np.array_equal(out.cpu().numpy(), ref), (top_k, temperature, c)


def test_sample_ties_nan_and_empty_rows(tts):
    B, V = 4, 300
    lg = _logits(B, V, 8)
    lg[0, [10, 250]] = 50.0              # tie on the maximum: lower index
    lg[1, :] = float("-inf")             # nothing finite: the first index
    lg[2, 3] = float("nan")              # NaN counts as -inf
    lg[2, 4] = 40.0
    lg[3, 100:110] = 7.0                 # a block of equal candidates
    for top_k, T in [(0, 1.0), (12, 0.9)]:
        out = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        counter = torch.full((1,), 5, dtype=torch.int64, device="cuda")
        tts.tts_sample(lg.cuda(), top_k, T, 42, counter, out)
        torch.cuda.synchronize()
        ref = oracle.sample(lg.numpy(), top_k, T, 42, 5)
        assert np.array_equal(out.cpu().numpy(), ref), top_k
    assert ref[1] == 0


@pytest.mark.parametrize("top_k", [2, 8, 50, 64])
def test_sample_ties_at_the_threshold(tts, top_k):
    # logits on a grid of quarter steps: many keys equal the k-th largest, so the lowest
    # indices among them must be the ones taken (an odd vocab, not a multiple of 256)
    B, V = 16, 777
    lg = torch.round(_logits(B, V, 9) * 2.0) / 4.0
    lg[0, :] = 1.0                       # every key ties
    lg[1, :] = 0.0
    lg[1, 700:] = 2.0                    # 77 equal maxima, more than any top_k
    for c in range(4):
        out = torch.full((B,), -1, dtype=torch.int32, device="cuda")
        counter = torch.full((1,), c, dtype=torch.int64, device="cuda")
        tts.tts_sample(lg.cuda(), top_k, 0.8, 99, counter, out)
        torch.cuda.synchronize()
        ref = oracle.sample(lg.numpy(), top_k, 0.8, 99, c)
        assert np.array_equal(out.cpu().numpy(), ref), (top_k, c)


def test_sample_writes_a_column_of_the_ids_buffer(tts):
    """Strided logits rows (a slice of a wider buffer) in, one column of a [B][16] code
    id buffer out; the other columns untouched."""
    B, V = 8, 2048
    wide = _logits(B, V + 64, 9).cuda()
    lg = wide[:, 32:32 + V]
    ids = torch.full((B, 16), -7, dtype=torch.int32, device="cuda")
    counter = torch.zeros(1, dtype=torch.int64, device="cuda")
    tts.tts_sample(lg, 8, 1.0, 3, counter, ids[:, 5])
    torch.cuda.synchronize()
    ref = oracle.sample(lg.cpu().numpy(), 8, 1.0, 3, 0)
    got = ids.cpu().numpy()
    assert np.array_equal(got[:, 5], ref)
    assert (np.delete(got, 5, axis=1) == -7).all()


def test_counter_advances_inside_a_replayed_graph(tts):
    B, V, seed = 16, 2048, 77
    lg = _logits(B, V, 10)
    d_lg = lg.cuda()
    counter = torch.zeros(1, dtype=torch.int64, device="cuda")
    outs = torch.full((4, B), -1, dtype=torch.int32, device="cuda")
    slot = torch.zeros(B, dtype=torch.int32, device="cuda")
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        tts.tts_sample(d_lg, 16, 0.8, seed, counter, slot, stream=s)   # warm outside capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        tts.tts_sample(d_lg, 16, 0.8, seed, counter, slot, stream=s)
        tts.tts_counter_advance(counter, 1, stream=s)
    for r in range(4):
        g.replay()
        outs[r].copy_(slot)
    torch.cuda.synchronize()
    assert int(counter.item()) == 4
    for r in range(4):
        assert np.array_equal(outs[r].cpu().numpy(), oracle.sample(lg.numpy(), 16, 0.8, seed, r)), r


@pytest.mark.parametrize("dtype,top_k", [("f32", 50), ("bf16", 0), ("q8_0", 8), ("f32", 1)])
def test_sample_embed_equals_sample_then_gather(tts, dtype, top_k):
    """tts_sample_embed is tts_sample followed by the one-table gather of the drawn codes:
    the same ids (also against the oracle) and the same row bytes."""
    B, V, hidden, seed = 32, 2048, 1024, 99
    lg = _logits(B, V, 11)
    d_lg = lg.cuda()
    if dtype == "q8_0":
        tab = W.q8_0_tables(1, V, hidden, seed=12)[0].cuda()
    else:
        tab = W.tables(1, V, hidden, seed=12)[0]
        tab = (tab.to(torch.bfloat16) if dtype == "bf16" else tab).cuda()
    t = tts.tables([tab])
    counter = torch.full((1,), 5, dtype=torch.int64, device="cuda")
    ids_a = torch.full((B, 3), -1, dtype=torch.int32, device="cuda")
    ids_b = torch.full((B, 3), -1, dtype=torch.int32, device="cuda")
    rows_a = torch.full((B, hidden), float("nan"), device="cuda")
    rows_b = torch.full((B, hidden), float("nan"), device="cuda")
    ef = torch.zeros(1, dtype=torch.int32, device="cuda")
    tts.tts_sample(d_lg, top_k, 0.9, seed, counter, ids_a[:, 1], draw=4)
    tts.tts_frame_embed(t, ids_a[:, 1:2], None, rows_a, ef)
    tts.tts_sample_embed(d_lg, top_k, 0.9, seed, counter, ids_b[:, 1], t, rows_b, draw=4)
    torch.cuda.synchronize()
    assert ef.item() == 0
    assert torch.equal(ids_a, ids_b)
    assert np.array_equal(ids_b[:, 1].cpu().numpy(), oracle.sample(lg.numpy(), top_k, 0.9, seed, 5, draw=4))
    assert torch.equal(rows_a.view(torch.int32), rows_b.view(torch.int32))
