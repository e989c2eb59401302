"""tts_decode_step_noalloc: the fused decode step for callers that cannot allocate
device memory when they run it (a real-time audio callback, a host framework that only
lends out its own tensors).  It takes its split-KV scratch from a fixed array inside the
library instead of a caller workspace.  These tests call it through the C ABI and check
two consecutive calls against tts_decode_step with a normal workspace.  The file sorts
last so that a run stopping at the first failure has already run every other test."""
import numpy as np
import pytest
import torch

from autoregressive_codebook_tts_gb300 import workloads as W
from gpu_helpers import ATTN_TOL, Layer, rope_table, row_rel_err, scale_of

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tts(cuda_dev):
    from autoregressive_codebook_tts_gb300 import build
    build.build()
    from autoregressive_codebook_tts_gb300 import tts as mod
    return mod


@pytest.mark.parametrize("name,n_splits", [("talker", 0), ("batched", 8), ("paged", 12)])
def test_noalloc_step_matches_workspace_step_twice(tts, name, n_splits):
    w = W.workload(name, layers=1)
    L = Layer(w, seed=90)
    cs = rope_table(tts, w.capacity, w.head_dim, w.rope_base)
    desc = L.desc(tts)
    K0, V0 = L.d_K.clone(), L.d_V.clone()

    ws = tts.workspace(desc, n_splits)
    ref = torch.empty(w.B, w.n_q_heads, w.head_dim, device="cuda")
    ef = torch.zeros(1, dtype=torch.int32, device="cuda")
    tts.tts_decode_step(L.d_q, L.d_k, L.d_v, L.d_gq, L.d_gk, w.eps, cs, w.capacity, L.d_K, L.d_V,
                        desc, L.d_cur, scale_of(w), ref, ws, n_splits, ef)
    torch.cuda.synchronize()
    ref_K, ref_V = L.d_K.clone(), L.d_V.clone()

    for call in range(2):
        K, V = K0.clone(), V0.clone()
        out = torch.full_like(ref, float("nan"))
        tts.tts_decode_step_noalloc(L.d_q, L.d_k, L.d_v, L.d_gq, L.d_gk, w.eps, cs, w.capacity,
                                    K, V, desc, L.d_cur, scale_of(w), out, n_splits, ef)
        torch.cuda.synchronize()
        assert ef.item() == 0, call
        assert row_rel_err(out.cpu().numpy(), ref.cpu().numpy()) <= ATTN_TOL[w.kv_dtype], call
        # caches compared as bytes (the unused tail holds NaN poison)
        assert torch.equal(K.view(torch.uint8), ref_K.view(torch.uint8)), call
        assert torch.equal(V.view(torch.uint8), ref_V.view(torch.uint8)), call


def test_noalloc_rejects_configurations_beyond_its_scratch(tts):
    w = W.workload("batched", layers=1)
    L = Layer(w, seed=91, poison=False)
    desc = L.desc(tts)
    assert tts.tts_decode_attn_workspace_size(desc, 128) > 4 << 20
    cs = rope_table(tts, w.capacity, w.head_dim, w.rope_base)
    out = torch.empty(w.B, w.n_q_heads, w.head_dim, device="cuda")
    with pytest.raises(tts.TtsError) as e:
        tts.tts_decode_step_noalloc(L.d_q, L.d_k, L.d_v, L.d_gq, L.d_gk, w.eps, cs, w.capacity,
                                    L.d_K, L.d_V, desc, L.d_cur, scale_of(w), out, 128)
    assert e.value.status == 6  # TTS_ERR_WORKSPACE
