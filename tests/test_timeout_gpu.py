"""The error path of the bounded waits, made to run out without faulting anything: one
thread waits (with the wait every kernel of the library uses) for an mbarrier phase that
nothing completes, gives up after its cycle limit and reports TTS_EFLAG_TIMEOUT to the
host.  The context stays usable: a frame-input composition afterwards is bit-exact."""
import time

import numpy as np
import pytest
import torch

import oracle
from autoregressive_codebook_tts_gb300 import workloads as W
from gpu_helpers import bits

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def tts(cuda_dev):
    from autoregressive_codebook_tts_gb300 import build
    build.build()
    from autoregressive_codebook_tts_gb300 import tts as mod
    return mod


def test_expired_wait_sets_the_timeout_flag_and_the_context_stays_usable(tts):
    ef = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = time.perf_counter()
    tts.tts_check_wait_timeout(ef)
    torch.cuda.synchronize()
    waited = time.perf_counter() - t0
    assert ef.item() == tts.EFLAG_TIMEOUT
    assert waited < 30.0   # about a second of SM cycles, never a hang

    # a library call after the expired wait still gives the oracle's bytes
    tabs = W.tables(4, 512, 256, seed=90)
    ids = W.code_ids(8, 4, 512, seed=91)
    ref, flag = oracle.frame_embed([t.numpy() for t in tabs], ids.numpy(), None)
    out = torch.full((8, 256), float("nan"), device="cuda")
    ef2 = torch.zeros(1, dtype=torch.int32, device="cuda")
    tts.tts_frame_embed([t.cuda() for t in tabs], ids.cuda(), None, out, ef2)
    torch.cuda.synchronize()
    assert flag == 0 and ef2.item() == 0
    assert np.array_equal(bits(out.cpu().numpy()), bits(ref))
