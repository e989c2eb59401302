"""Code-predictor frames enqueued through the public calls, K frames per graph replay.

The "qwentts.cpp" pages keep the code predictor's whole frame on the device: the frame
unroll with an in-graph sampler ("commits/branch/master/tests" page, fused codec tail),
and "minicpm-o-4.5 ... docs/optimizations.md" (core table, CUDA-graph decode row)
replays several frames per graph launch.  One frame of B streams, in the order of the
"src/pipeline-tts.h" KV-cache section:

  * reset: the 16-slot caches are reused from position 0 (stale rows are masked by the
    window, never cleared);
  * the gather of c0 from group table 0, then the T = 2 prefill of every layer (rows 0
    and 1: the bridge row and the c0 row, whose q/k/v come from the projection);
  * for t = 2 .. 15: the sampler draws sub-code j = t - 1 from the logits of the step
    before and writes it into column j of the frame's code ids; the gather reads that
    column from group table j; then one decode step of every layer at position t;
  * the sampler draws sub-code 15 from the last logits, and the counter advances.

Everything here is argument marshalling: buffers are allocated once, and ``enqueue``
only issues ``tts_frame_embed``, ``tts_prefill_step``, ``tts_sample_embed`` (the sampler
with the gather of the drawn code), ``tts_sample``, ``tts_decode_step`` and
``tts_counter_advance`` calls.  The QKV projection and the
output heads sit outside this path, so the q/k/v rows of every (position, layer) and
the logits of every sub-step are inputs.  Sampler draw j of a frame uses the Philox
counter words (counter, stream, j, 0); the counter moves by one per frame.
"""
from __future__ import annotations

import math

import torch

from . import tts


class PredictorFrames:
    """Buffers and enqueue function of code-predictor frames.

    tables: 15 device tensors [vocab][hidden] (group table j for sub-code j).
    pre: [L][2B][width] f32, the prefill rows (row b*2 + t, width = (Hq + 2 Hkv) D,
        laid out [q | k | v]), read only.
    qkv: [16][L][B][width] f32, the rows of positions 2..15 (entries 0 and 1 unused).
    logits: [15][B][vocab] f32 (logits[j - 1] decides sub-code j).
    gq, gk: [L][D] f32.
    slots: sets of output buffers; frame k of a replay writes slot k % slots (codes,
        gathered rows, attention outputs), so a test can read every frame of a replay.
    c0: [slots][B] int32, the code each slot's frame starts from (the talker's code).
    """

    def __init__(self, B, layers, n_q_heads, n_kv_heads, head_dim, hidden, vocab, tables, pre,
                 qkv, logits, gq, gk, top_k, temperature, seed, c0, eps=1e-6, rope_base=1e6,
                 capacity=16, slots=1, device="cuda"):
        self.B, self.L, self.Hq, self.Hkv, self.D = B, layers, n_q_heads, n_kv_heads, head_dim
        self.hidden, self.vocab, self.capacity = hidden, vocab, capacity
        self.top_k, self.temperature, self.seed = top_k, temperature, seed
        self.eps = eps
        self.slots = slots
        self.tabs = [tts.tables([t]) for t in tables]
        self._tables = tables
        self.pre, self.qkv, self.logits, self.gq, self.gk = pre, qkv, logits, gq, gk
        D = head_dim
        self.caches = [(torch.zeros(B, n_kv_heads, capacity, D, device=device),
                        torch.zeros(B, n_kv_heads, capacity, D, device=device)) for _ in range(layers)]
        self.cs = torch.empty(capacity, D // 2, 2, device=device)
        tts.tts_rope_table(self.cs, capacity, D, rope_base)
        # The enqueue order keeps TTS_KV_PREFETCH_BEFORE_WAIT's promise: the launch just
        # before a decode step is the gather or another layer's step, neither of which
        # writes this layer's cache; a layer's rows are written by its own step one
        # sub-step earlier (or by the frame's prefill), launches that have completed by
        # then, and the cur_len tensors are constants.  So the steps may start streaming
        # their cache rows before the preceding launch ends.
        self.desc = tts.kv_desc(B, n_q_heads, n_kv_heads, D, capacity, "f32",
                                window_quantum=capacity, flags=tts.TTS_KV_PREFETCH_BEFORE_WAIT)
        self.ws = tts.workspace(self.desc, 0, device=device)
        self.pws = tts.prefill_workspace(self.desc, 2, 0, device=device)
        self.codes = torch.zeros(slots, B, 16, dtype=torch.int32, device=device)
        self.codes[:, :, 0] = c0.to(device)
        self.emb = torch.empty(slots, 15, B, hidden, device=device)
        self.pout = torch.empty(slots, layers, B, 2, n_q_heads, D, device=device)
        self.out = torch.empty(slots, 16, layers, B, n_q_heads, D, device=device)
        self.zeros = torch.zeros(B, dtype=torch.int32, device=device)
        self.curs = [torch.full((B,), t, dtype=torch.int32, device=device) for t in range(16)]
        self.counter = torch.zeros(1, dtype=torch.int64, device=device)
        self.err = torch.zeros(1, dtype=torch.int32, device=device)
        self.scale = 1.0 / math.sqrt(D)
        self.launches_per_frame = 1 + 2 * layers + 14 * (1 + layers) + 2

    def enqueue(self, k=0, stream=None):
        """One frame into slot k % slots, on `stream` (default: the current stream)."""
        s = k % self.slots
        Hq, Hkv, D, L = self.Hq, self.Hkv, self.D, self.L
        qd, kd = Hq * D, Hkv * D
        codes = self.codes[s]
        ef = self.err
        tts.tts_frame_embed(self.tabs[0], codes[:, 0:1], None, self.emb[s, 0], ef, stream=stream)
        for l in range(L):
            rows = self.pre[l]
            kc, vc = self.caches[l]
            tts.tts_prefill_step(rows[:, :qd], rows[:, qd:qd + kd], rows[:, qd + kd:], self.gq[l],
                                 self.gk[l], self.eps, self.cs, self.capacity, kc, vc, self.desc,
                                 self.zeros, 2, self.scale, self.pout[s, l], self.pws, 0, ef,
                                 stream=stream)
        for t in range(2, 16):
            j = t - 1
            # the sampler draws sub-code j and gathers its row of group table j (one launch)
            tts.tts_sample_embed(self.logits[j - 1], self.top_k, self.temperature, self.seed,
                                 self.counter, codes[:, j], self.tabs[j], self.emb[s, j], draw=j,
                                 stream=stream)
            for l in range(L):
                rows = self.qkv[t, l]
                kc, vc = self.caches[l]
                tts.tts_decode_step(rows[:, :qd], rows[:, qd:qd + kd], rows[:, qd + kd:],
                                    self.gq[l], self.gk[l], self.eps, self.cs, self.capacity, kc,
                                    vc, self.desc, self.curs[t], self.scale, self.out[s, t, l],
                                    self.ws, 0, ef, stream=stream)
        tts.tts_sample(self.logits[14], self.top_k, self.temperature, self.seed, self.counter,
                       codes[:, 15], draw=15, stream=stream)
        tts.tts_counter_advance(self.counter, 1, stream=stream)

    def enqueue_frames(self, n, stream=None):
        for k in range(n):
            self.enqueue(k, stream=stream)
