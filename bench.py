"""Benchmark of the per-frame decode hot path on one GB300 (or N replicas).

Workload (default): the talker single-stream configuration -- 1 stream, 28 layers,
hidden 2048, 16 q / 8 kv heads, head_dim 128, f32 KV cache of 4096 positions per layer
(896 MiB), 16 codebooks of 2048 x 2048 f32, cur_len 4095 (window 4096).  One step is
one frame: the frame-input composition plus 28 fused decode steps (q/k norm + RoPE,
set_rows of the new K/V row, split-KV decode attention), captured once in a CUDA graph
from the public C-ABI calls and replayed.  The KV working set (896 MiB) is larger than
L2, so no flush is needed between steps.

Printed: one JSON line (rank 0).  ``value`` = algorithmic bytes per frame (KV window
read + new-row write + activations + embedding rows) x frames / device time, in GB/s.
``--impl reference`` times the CPU oracle on the same workload instead.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import math
import os
import statistics
import subprocess
import sys
import time

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "decode-attn KV GB/s (% of HBM peak); frame steps/sec at B streams, 1 GB300"
FALLBACK_HBM_GBS = 6800.0
NOMINAL_HBM_GBS = 7900.0
ATTN_SRC = os.path.join(ROOT, "autoregressive_codebook_tts_gb300", "csrc", "attn.cu")


def parse():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=2000)
    ap.add_argument("--warmup", type=int, default=20)
    ap.add_argument("--impl", choices=["native", "reference"], default="native")
    ap.add_argument("--workload", default="batched",
                    choices=["talker", "batched", "paged", "prefill", "predictor", "layer"])
    ap.add_argument("--layer-streams", type=int, default=1, help="layer: streams (1..32)")
    ap.add_argument("--frames-per-replay", type=int, default=4,
                    help="predictor: frames unrolled into one graph replay")
    ap.add_argument("--layers", type=int, default=0,
                    help="layers per frame (0 = the workload's own; fewer only for small profiling cases)")
    ap.add_argument("--prefill-t", type=int, default=128, help="prefill: prompt positions per stream")
    ap.add_argument("--prefill-start", type=int, default=0, help="prefill: first prompt position")
    ap.add_argument("--prefill-kv", default="f32", choices=["f32", "bf16"], help="prefill: cache element type")
    ap.add_argument("--cur-len", type=int, default=4095)
    ap.add_argument("--n-splits", type=int, default=0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--cpu-seconds", type=float, default=10.0)
    ap.add_argument("--sweep", action="store_true", help="talker: also time cur_len 255/1023/2047")
    ap.add_argument("--only", action="store_true",
                    help="batched: skip the paged and talker lines measured in the same run")
    return ap.parse_args()


# ---------------------------------------------------------------------------
# Algorithmic bytes
# ---------------------------------------------------------------------------
def step_bytes(w, cur_lens):
    """Per-layer and per-frame algorithmic bytes (see the module docstring)."""
    e = w.elem_bytes
    Hq, Hkv, D = w.n_q_heads, w.n_kv_heads, w.head_dim
    per_layer = 0
    kv_layer = 0
    for c in cur_lens:
        kv = (c + 1) * Hkv * D * e * 2           # window rows read + new row written
        act = (Hq + 2 * Hkv) * D * 4 + Hq * D * 4  # q, k, v in; out
        const = 2 * D * 4 + (D // 2) * 8           # gammas, RoPE row
        per_layer += kv + act + const
        kv_layer += kv
    embed = len(cur_lens) * (w.n_tables * w.hidden * 4 + 2 * w.hidden * 4 + w.n_tables * 4)
    return per_layer, kv_layer, embed


def hbm_peak():
    path = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(path):
        try:
            with open(path) as f:
                d = json.load(f)
            for key in ("hbm_gbs", "hbm_GBps", "hbm"):
                if key in d and isinstance(d[key], (int, float)):
                    return float(d[key]), "measured"
        except Exception:
            pass
    return FALLBACK_HBM_GBS, "fallback"


def profiled_traffic(summary):
    """dram bytes per launch of the dominant kernel from a committed ncu summary, or None
    when the summary is absent or was taken on a different attn.cu."""
    if not os.path.exists(summary):
        return None
    src_hash = hashlib.sha256(open(ATTN_SRC, "rb").read()).hexdigest()[:16]
    vals = {}
    for line in open(summary):
        if ":" in line:
            k, v = line.split(":", 1)
            vals[k.strip()] = v.strip()
    if vals.get("attn_cu_sha256_16") != src_hash:
        return None
    try:
        return float(vals["traffic_bytes_per_launch_full"])
    except (KeyError, ValueError):
        return None


# ---------------------------------------------------------------------------
# Clock sampling during the timed region
# ---------------------------------------------------------------------------
class ClockSampler:
    QUERY = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
             "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
             "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, gpu_index):
        self.gpu = gpu_index
        self.proc = None
        self.path = os.path.join("/tmp", f"tts_clocks_{os.getpid()}.csv")

    def start(self):
        try:
            self.fh = open(self.path, "w")
            self.proc = subprocess.Popen(
                ["nvidia-smi", f"--id={self.gpu}", f"--query-gpu={self.QUERY}", "--format=csv,noheader,nounits",
                 "-lms", "100"], stdout=self.fh, stderr=subprocess.DEVNULL)
        except Exception:
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.fh.close()
        sms, mx, reasons = [], None, set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for line in open(self.path):
            f = [x.strip() for x in line.split(",")]
            if len(f) < 9:
                continue
            try:
                sms.append(float(f[1]))
                mx = float(f[2])
            except ValueError:
                continue
            for n, v in zip(names, f[5:9]):
                if v.lower().startswith("active"):
                    reasons.add(n)
        os.unlink(self.path)
        if not sms:
            return None
        return {"sm_mhz": statistics.median(sms), "sm_max_mhz": mx, "reasons": sorted(reasons),
                "samples": len(sms)}


# ---------------------------------------------------------------------------
# Native arm
# ---------------------------------------------------------------------------
def build_frame(tts, W, w, cur_len, n_splits, dev, seed=0):
    """Device-resident inputs of one frame and the closure that enqueues it."""
    import torch
    B, L = w.B, w.layers
    g = torch.Generator(device=dev)
    g.manual_seed(seed)
    tabs = [torch.randn(w.vocab, w.hidden, generator=g, device=dev) * w.table_std for _ in range(w.n_tables)]
    ids = torch.randint(0, w.vocab, (B, w.n_tables), generator=g, device=dev, dtype=torch.int32)
    overlay = torch.randn(B, w.hidden, generator=g, device=dev) * w.table_std
    width = (w.n_q_heads + 2 * w.n_kv_heads) * w.head_dim
    qkv = torch.randn(L, B, width, generator=g, device=dev)
    gq = torch.rand(L, w.head_dim, generator=g, device=dev) + 0.5
    gk = torch.rand(L, w.head_dim, generator=g, device=dev) + 0.5
    if isinstance(cur_len, int):
        cur = torch.full((B,), cur_len, dtype=torch.int32, device=dev)
    else:
        cur = cur_len.to(dev)
    kv_dt = torch.float32 if w.kv_dtype == "f32" else torch.bfloat16
    if w.paged:
        pages_per = w.capacity // w.page_size
        bt = torch.randperm(w.n_pages, generator=g, device=dev)[:B * pages_per].reshape(B, pages_per).to(torch.int32).contiguous()
        shape = (w.n_pages, w.n_kv_heads, w.page_size, w.head_dim)
    else:
        bt = None
        shape = (B, w.n_kv_heads, w.capacity, w.head_dim)
    caches = []
    for _ in range(L):
        K = torch.empty(shape, dtype=kv_dt, device=dev)
        V = torch.empty(shape, dtype=kv_dt, device=dev)
        K.normal_(generator=g)
        V.normal_(generator=g)
        caches.append((K, V))
    cs = torch.empty(w.capacity, w.head_dim // 2, 2, device=dev)
    tts.tts_rope_table(cs, w.capacity, w.head_dim, w.rope_base)
    desc = tts.kv_desc(B, w.n_q_heads, w.n_kv_heads, w.head_dim, w.capacity, w.kv_dtype,
                       window_quantum=w.window_quantum, paged=w.paged, page_size=w.page_size,
                       n_pages=w.n_pages, block_table=bt, flags=tts.TTS_KV_PREFETCH_BEFORE_WAIT)
    ws = tts.workspace(desc, n_splits, device=dev)
    emb = torch.empty(B, w.hidden, device=dev)
    outs = torch.empty(L, B, w.n_q_heads, w.head_dim, device=dev)
    ef = torch.zeros(1, dtype=torch.int32, device=dev)
    qd, kd = w.n_q_heads * w.head_dim, w.n_kv_heads * w.head_dim
    scale = 1.0 / math.sqrt(w.head_dim)
    tabs_struct = tts.tables(tabs)

    def layers():
        for l in range(L):
            K, V = caches[l]
            rows = qkv[l]
            tts.tts_decode_step(rows[:, :qd], rows[:, qd:qd + kd], rows[:, qd + kd:], gq[l], gk[l],
                                w.eps, cs, w.capacity, K, V, desc, cur, scale, outs[l], ws,
                                n_splits, ef)

    def frame():
        tts.tts_frame_embed(tabs_struct, ids, overlay, emb, ef)
        layers()

    state = dict(tabs=tabs, ids=ids, overlay=overlay, qkv=qkv, cur=cur, caches=caches, emb=emb,
                 outs=outs, ef=ef, cs=cs, ws=ws, bt=bt, gq=gq, gk=gk, desc=desc)
    return frame, layers, state


def capture(fn, torch):
    s = torch.cuda.Stream()
    s.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(s):
        fn()  # warm (sets kernel attributes outside capture)
    torch.cuda.current_stream().wait_stream(s)
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=s):
        fn()
    torch.cuda.synchronize()
    return g


def timed_replays(g, steps, torch, stream=None):
    st = stream or torch.cuda.current_stream()
    e0 = torch.cuda.Event(enable_timing=True)
    e1 = torch.cuda.Event(enable_timing=True)
    torch.cuda.synchronize()
    e0.record(st)
    with torch.cuda.stream(st):
        for _ in range(steps):
            g.replay()
    e1.record(st)
    torch.cuda.synchronize()
    return e0.elapsed_time(e1) / 1e3


def replay_percentiles(g, steps, torch, flush=None):
    """Per-replay device times (CUDA events around each replay, after the timed region),
    as {"p10", "p50", "p90"} in ms; the L2 flush, when given, runs before each replay."""
    st = torch.cuda.current_stream()
    ev = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(steps)]
    torch.cuda.synchronize()
    for a, b in ev:
        if flush is not None:
            flush.fill_(1)
        a.record(st)
        g.replay()
        b.record(st)
    torch.cuda.synchronize()
    ts = sorted(a.elapsed_time(b) for a, b in ev)
    pick = lambda q: ts[min(len(ts) - 1, int(round(q * (len(ts) - 1))))]
    return {"p10": round(pick(0.1), 5), "p50": round(pick(0.5), 5), "p90": round(pick(0.9), 5)}


class CpuClock:
    """Wall time and the process's CPU time over a timed region of the oracle.  `cores` is
    CPU time / wall time rounded (at least 1): the host threads the oracle actually kept
    busy, e.g. numpy's BLAS threads in its matrix products."""

    def __enter__(self):
        self.w0, self.c0 = time.perf_counter(), time.process_time()
        return self

    def __exit__(self, *exc):
        self.wall = time.perf_counter() - self.w0
        self.cpu = time.process_time() - self.c0
        return False

    @property
    def cores(self):
        return max(1, round(self.cpu / self.wall)) if self.wall > 0 else 1


def host_layer0(state, w):
    """Host (numpy) copies of the frame's inputs that the oracle needs: the tables, ids and
    overlay of the frame-input composition and layer 0's q/k/v, gammas and caches."""
    import numpy as np
    import torch
    K, V = state["caches"][0]
    if w.kv_dtype == "bf16":  # the oracle takes bf16 caches as uint16 bit patterns
        hk = K.cpu().view(torch.int16).numpy().view(np.uint16).copy()
        hv = V.cpu().view(torch.int16).numpy().view(np.uint16).copy()
    else:
        hk = K.cpu().numpy().copy()
        hv = V.cpu().numpy().copy()
    rows = state["qkv"][0].cpu().numpy()
    qd, kd = w.n_q_heads * w.head_dim, w.n_kv_heads * w.head_dim
    B = w.B
    return dict(
        hk=hk, hv=hv, tabs=[t.cpu().numpy() for t in state["tabs"]], ids=state["ids"].cpu().numpy(),
        ov=state["overlay"].cpu().numpy(),
        q=rows[:, :qd].reshape(B, w.n_q_heads, w.head_dim).copy(),
        k=rows[:, qd:qd + kd].reshape(B, w.n_kv_heads, w.head_dim).copy(),
        v=rows[:, qd + kd:].reshape(B, w.n_kv_heads, w.head_dim).copy(),
        gq=state["gq"][0].cpu().numpy(), gk=state["gk"][0].cpu().numpy(),
        cur=state["cur"].cpu().numpy().astype(np.int32),
        bt=None if state["bt"] is None else state["bt"].cpu().numpy())


def oracle_whole(h, w):
    """One sample step of the oracle as it stands: the frame-input composition and layer
    0's fused decode step of every stream, one call each."""
    import numpy as np
    import oracle
    lay = oracle.KvLayout(w.B, w.n_kv_heads, w.head_dim, w.capacity, w.kv_dtype, paged=w.paged,
                          page_size=w.page_size, n_pages=w.n_pages, block_table=h["bt"])
    scale = 1.0 / math.sqrt(w.head_dim)

    def step():
        oracle.frame_embed(h["tabs"], h["ids"], h["ov"])
        oracle.decode_step(h["q"], h["k"], h["v"], h["gq"], h["gk"], np.float32(w.eps), w.rope_base,
                           h["hk"], h["hv"], lay, h["cur"], scale)
    return step


def oracle_units(h, w):
    """The same sample step cut into independent (stream, kv head) units for host threads:
    unit (b, g) runs the oracle's fused decode step on stream b's q heads of kv head g
    (its own cache slice, B = 1 and one kv head), and unit (b, 0) also the stream's
    frame-input composition.  Streams and kv heads never touch each other's data, so the
    units are the whole-batch call's work, split.  The oracle's C calls release the
    interpreter lock, so units run in parallel."""
    import numpy as np
    import oracle
    G, D = w.group, w.head_dim
    scale = 1.0 / math.sqrt(D)
    eps = np.float32(w.eps)
    if w.paged:  # one pool per kv head, so that each unit's pool slice is contiguous
        pools = [(np.ascontiguousarray(h["hk"][:, g:g + 1]), np.ascontiguousarray(h["hv"][:, g:g + 1]))
                 for g in range(w.n_kv_heads)]
    units = []
    for b in range(w.B):
        for g in range(w.n_kv_heads):
            q = np.ascontiguousarray(h["q"][b:b + 1, g * G:(g + 1) * G])
            k = np.ascontiguousarray(h["k"][b:b + 1, g:g + 1])
            v = np.ascontiguousarray(h["v"][b:b + 1, g:g + 1])
            cur = h["cur"][b:b + 1].copy()
            if w.paged:
                kc, vc = pools[g]
                lay = oracle.KvLayout(1, 1, D, w.capacity, w.kv_dtype, paged=True, page_size=w.page_size,
                                      n_pages=w.n_pages, block_table=h["bt"][b:b + 1])
            else:
                kc, vc = h["hk"][b:b + 1, g:g + 1], h["hv"][b:b + 1, g:g + 1]
                lay = oracle.KvLayout(1, 1, D, w.capacity, w.kv_dtype)
            emb = (h["ids"][b:b + 1], h["ov"][b:b + 1]) if g == 0 else None

            def unit(q=q, k=k, v=v, kc=kc, vc=vc, lay=lay, cur=cur, emb=emb):
                if emb is not None:
                    oracle.frame_embed(h["tabs"], emb[0], emb[1])
                oracle.decode_step(q, k, v, h["gq"], h["gk"], eps, w.rope_base, kc, vc, lay, cur, scale)
            units.append(unit)
    return units


def host_threads():
    try:
        return len(os.sched_getaffinity(0))
    except AttributeError:
        return os.cpu_count() or 1


def time_oracle(h, w, sample_bytes, seconds=None, reps=None, threads=1):
    """Runs the oracle sample step (whole-batch calls on one thread, or the
    (stream, kv head) units over `threads` host threads) for about `seconds` or exactly
    `reps` times.  Returns (bytes per second, reps, wall seconds, CpuClock)."""
    from concurrent.futures import ThreadPoolExecutor
    if threads <= 1:
        step = oracle_whole(h, w)
        run = step
        pool = None
    else:
        units = oracle_units(h, w)
        pool = ThreadPoolExecutor(max_workers=threads)

        def run():
            for f in [pool.submit(u) for u in units]:
                f.result()
    n = 0
    try:
        with CpuClock() as clk:
            while True:
                run()
                n += 1
                if reps is not None and n >= reps:
                    break
                if reps is None and time.perf_counter() - clk.w0 >= seconds:
                    break
    finally:
        if pool is not None:
            pool.shutdown()
    return sample_bytes * n / clk.wall, n, clk.wall, clk


def cpu_oracle_sample(state, w, seconds):
    """The oracle as it stands on a bounded sample of the workload (the frame-input
    composition and layer 0's fused decode step, i.e. the same bytes per layer as on the
    device), timed twice on this host: on one thread, and over every host thread the
    process may use.  Returns the cpu_baseline object (all-thread arm, with the
    one-thread arm inside it)."""
    h = host_layer0(state, w)
    per_layer, _, embed = step_bytes(w, [int(c) for c in h["cur"]])
    one, n1, t1, c1 = time_oracle(h, w, embed + per_layer, seconds=seconds, threads=1)
    nt = host_threads()
    allc, na, ta, ca = time_oracle(h, w, embed + per_layer, seconds=seconds, threads=nt)
    lens = (f"cur_len {int(h['cur'][0])}" if w.B == 1
            else f"its cur_len mix ({int(h['cur'].min())}..{int(h['cur'].max())})")
    what = f"(frame-input composition + layer-0 fused decode step) of the {w.name} workload at {lens}"
    return {"value": round(allc / 1e9, 4), "unit": "GB/s", "cores": nt, "kind": "oracle",
            "sample": f"{na} x {what}, units (stream, kv head) over {nt} host threads, {ta:.1f} s",
            "cpu_time_over_wall": round(ca.cpu / ca.wall, 2),
            "single_thread": {"value": round(one / 1e9, 4), "unit": "GB/s", "cores": 1,
                              "sample": f"{n1} x {what}, whole-batch oracle calls, {t1:.1f} s"}}


def max_over_ranks(values, world, device=None):
    """This rank's timings (seconds) -> their maxima over all ranks, on every rank.  The
    ranks are independent replicas (own streams, own caches); this reduction of the
    timings is the only collective of a multi-GPU run."""
    if world == 1:
        return [float(v) for v in values]
    import torch
    import torch.distributed as dist
    t = torch.tensor([float(v) for v in values], dtype=torch.float64, device=device)
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return [float(x) for x in t.tolist()]


def whole_job_gbs(world, bytes_per_step, steps, seconds):
    """Whole-job throughput: every rank moved bytes_per_step per step; the slowest rank's
    time counts."""
    return world * bytes_per_step * steps / seconds / 1e9


def l2_bytes(dev):
    """L2 size of the device, queried at run time."""
    import torch
    n = getattr(torch.cuda.get_device_properties(dev), "L2_cache_size", 0)
    if n:
        return int(n)
    import ctypes
    v = ctypes.c_int(0)
    ctypes.CDLL("libcudart.so").cudaDeviceGetAttribute(ctypes.byref(v), 38, dev.index or 0)  # L2CacheSize
    return int(v.value)


def profile_summary(w, cur_len):
    """The committed ncu summary of the fused step on this workload, if one exists."""
    name = {"talker": "decode_step_talker_f32_cur4095.txt", "batched": "decode_step_batched_bf16.txt",
            "paged": "decode_step_paged_bf16.txt"}.get(w.name)
    if name is None or (w.name == "talker" and cur_len != 4095) or w.layers != W_LAYERS.get(w.name):
        return None
    return os.path.join(ROOT, "profiles", name)


W_LAYERS = {"talker": 28, "batched": 28, "paged": 28}


def measure_frames(args, tts, W, w, cur_arg, cur_list, dev, rank, world, full):
    """Times graph replays of whole frames (frame-input composition + L fused decode
    steps) and, alone, the L decode-step launches of the same frame.  `full` adds the
    end-to-end timing through host buffers.  Returns (result dict, frame state)."""
    import torch
    frame, layers, state = build_frame(tts, W, w, cur_arg, args.n_splits, dev, seed=rank)
    per_layer, kv_layer, embed = step_bytes(w, cur_list)
    frame_bytes = embed + w.layers * per_layer
    L2 = l2_bytes(dev)
    flush = None
    if w.layers * kv_layer < 4 * L2:  # working set within reach of L2: flush it per frame
        flush = torch.empty(2 * L2, dtype=torch.uint8, device=dev)

    g_frame = capture(frame, torch)
    g_layers = capture(layers, torch)
    for _ in range(args.warmup):
        g_frame.replay()
    torch.cuda.synchronize()
    if state["ef"].item() != 0:
        raise RuntimeError(f"device error flag {state['ef'].item()}")

    local = dev.index or 0
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    if flush is None:
        t_frame = timed_replays(g_frame, args.steps, torch)
    else:
        t_frame = 0.0
        for _ in range(args.steps):
            flush.fill_(1)
            t_frame += timed_replays(g_frame, 1, torch)
    if world > 1:
        torch.distributed.barrier()
    # the dominant kernel alone: the L fused decode-step launches of the same frame
    t_layers = timed_replays(g_layers, args.steps, torch)
    clk = clocks.stop()
    # the spread of single frames (outside the timed region above)
    spread = replay_percentiles(g_frame, max(args.steps, 10), torch, flush)

    t_e2e, e2e_steps, h2d, d2h = None, 0, 0, 0
    if full:
        # End to end through the public calls with host buffers, pipelined as a serving
        # loop would run it: two frame states (each its own inputs, caches, outputs and
        # graph) alternate; step k+1's inputs are uploaded from pinned memory on a copy
        # stream while frame k runs, and frame k's outputs (every layer's attention rows,
        # the composed inputs, the error flag) are read back on the copy stream once it
        # ends.  Every step's uploads and read-backs lie inside the timed region.
        frame2, _, state2 = build_frame(tts, W, w, cur_arg, args.n_splits, dev, seed=rank)
        g_frame2 = capture(frame2, torch)
        sets = [(state, g_frame), (state2, g_frame2)]
        h_ids = state["ids"].cpu().pin_memory()
        h_ov = state["overlay"].cpu().pin_memory()
        h_qkv = state["qkv"].cpu().pin_memory()
        h_cur = state["cur"].cpu().pin_memory()
        h_out = torch.empty_like(state["outs"], device="cpu").pin_memory()
        h_emb = torch.empty_like(state["emb"], device="cpu").pin_memory()
        h_ef = [torch.zeros(1, dtype=torch.int32).pin_memory() for _ in range(2)]
        s = torch.cuda.current_stream()
        cp = torch.cuda.Stream(device=dev)
        up = [torch.cuda.Event() for _ in range(2)]
        done = [torch.cuda.Event() for _ in range(2)]

        def upload(j):
            st = sets[j][0]
            st["ids"].copy_(h_ids, non_blocking=True)
            st["overlay"].copy_(h_ov, non_blocking=True)
            st["qkv"].copy_(h_qkv, non_blocking=True)
            st["cur"].copy_(h_cur, non_blocking=True)

        def readback(j):
            st = sets[j][0]
            h_out.copy_(st["outs"], non_blocking=True)
            h_emb.copy_(st["emb"], non_blocking=True)
            h_ef[j].copy_(st["ef"], non_blocking=True)

        def run(n):
            # step k uses set k % 2; its upload waits for frame k - 2 (same set) to end
            with torch.cuda.stream(cp):
                cp.wait_stream(s)
                upload(0)
                up[0].record(cp)
            for k in range(n):
                j = k % 2
                s.wait_event(up[j])
                sets[j][1].replay()
                done[j].record(s)
                with torch.cuda.stream(cp):
                    if k + 1 < n:
                        if k >= 1:
                            cp.wait_event(done[1 - j])
                        upload(1 - j)
                        up[1 - j].record(cp)
                    cp.wait_event(done[j])
                    readback(j)
            s.wait_stream(cp)

        run(4)
        torch.cuda.synchronize()
        e2e_steps = max(10, args.steps)
        e0 = torch.cuda.Event(enable_timing=True)
        e1 = torch.cuda.Event(enable_timing=True)
        e0.record(s)
        run(e2e_steps)
        e1.record(s)
        torch.cuda.synchronize()
        t_e2e = e0.elapsed_time(e1) / 1e3
        h2d = sum(t.numel() * t.element_size() for t in (h_ids, h_ov, h_qkv, h_cur))
        d2h = sum(t.numel() * t.element_size() for t in (h_out, h_emb, h_ef[0]))
        if int(h_ef[0].item()) != 0 or int(h_ef[1].item()) != 0:
            raise RuntimeError(f"device error flag {int(h_ef[0].item())} / {int(h_ef[1].item())}")
        del state2, sets, g_frame2
        t_frame, t_layers, t_e2e = max_over_ranks([t_frame, t_layers, t_e2e], world, dev)
    else:
        t_frame, t_layers = max_over_ranks([t_frame, t_layers], world, dev)

    peak, peak_kind = hbm_peak()
    value = whole_job_gbs(world, frame_bytes, args.steps, t_frame)
    dom_time = t_layers / (args.steps * w.layers)
    achieved = per_layer / dom_time / 1e9
    summary = profile_summary(w, args.cur_len)
    traffic = profiled_traffic(summary) if summary else None
    res = {
        "value": round(value, 2),
        "unit": "GB/s",
        "ms_per_step": round(t_frame / args.steps * 1e3, 5),
        "config": {"workload": (f"{w.name}: B={w.B} streams, {w.layers} layers, hidden {w.hidden}, "
                                f"{w.n_q_heads} q / {w.n_kv_heads} kv heads, head_dim {w.head_dim}, "
                                f"{w.kv_dtype} KV, capacity {w.capacity}"
                                + (f", paged {w.page_size}-token pages" if w.paged else "")
                                + (f", cur_len {cur_list[0]}" if w.name == 'talker'
                                   else f", ragged cur_len {min(cur_list)}..{max(cur_list)}")),
                   "B": w.B, "layers": w.layers, "window_rows_per_layer": sum(c + 1 for c in cur_list),
                   "l2": (f"inputs larger than L2 (KV working set per frame {w.layers * kv_layer / 2 ** 20:.0f} MiB, "
                          f"L2 {L2 / 2 ** 20:.0f} MiB)" if flush is None else
                          f"L2 ({L2 / 2 ** 20:.0f} MiB) flushed before every timed frame "
                          f"(KV working set {w.layers * kv_layer / 2 ** 20:.0f} MiB)"),
                   "frame_step": "graph replay of tts_frame_embed + %d x tts_decode_step" % w.layers,
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "pct_of_hbm_peak": round(100 * value / world / peak, 2),
        "pct_of_nominal_hbm": round(100 * value / world / NOMINAL_HBM_GBS, 2),
        "frame_steps_per_s": round(world * w.B * args.steps / t_frame, 1),
        "ms_per_frame_spread": spread,
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": traffic,
                     "kernel": "decode_attn_kernel<fused> (tts_decode_step)",
                     "peak_source": f"{peak_kind} HBM copy bandwidth",
                     "bytes_per_launch": per_layer, "us_per_launch": round(dom_time * 1e6, 3)},
        "gpu_launches": args.steps * (1 + w.layers),
        "clocks": clk,
    }
    if full:
        res["e2e"] = {"value": round(whole_job_gbs(world, frame_bytes, e2e_steps, t_e2e), 2), "unit": "GB/s",
                      "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                      "ms_per_step": round(t_e2e / e2e_steps * 1e3, 5)}
    return res, state


def run_native(args, rank, world):
    import torch
    from autoregressive_codebook_tts_gb300 import build as b
    b.build()
    from autoregressive_codebook_tts_gb300 import tts
    from autoregressive_codebook_tts_gb300 import workloads as W

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)

    def lens(w):
        if w.name == "talker":
            return args.cur_len, [args.cur_len] * w.B
        c = W.cur_lens(w, seed=0)
        return c, [int(x) for x in c]

    w = W.workload(args.workload, **({"layers": args.layers} if args.layers > 0 else {}))
    cur_arg, cur_list = lens(w)
    body, state = measure_frames(args, tts, W, w, cur_arg, cur_list, dev, rank, world, full=True)
    res = {"metric": METRIC, "value": body.pop("value"), "unit": body.pop("unit"), "n_gpus": world,
           "steps": args.steps, "warmup": args.warmup, "ms_per_step": body.pop("ms_per_step"),
           "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
           "dtype": "f32" if w.kv_dtype == "f32" else "bf16-kv/f32",
           "data": "synthetic (seeded, device-generated; random-init, no weights)"}
    res.update(body)
    if rank == 0 and not args.no_cpu_baseline:
        res["cpu_baseline"] = cpu_oracle_sample(state, w, args.cpu_seconds)
    del state
    # the other decode-attention workloads of the metric, measured in the same run, each
    # with the roofline of its own dominant kernel
    if args.workload == "batched" and args.layers == 0 and not args.only:
        others = {}
        for name in ("paged", "talker"):
            wo = W.workload(name)
            ca, cl = lens(wo)
            torch.cuda.empty_cache()
            r, st = measure_frames(args, tts, W, wo, ca, cl, dev, rank, world, full=False)
            del st
            others[name] = r
            res["gpu_launches"] += r.pop("gpu_launches")
        res["other_workloads"] = others
    if args.sweep and args.workload == "talker" and rank == 0:
        sweep = {}
        for c in (255, 1023, 2047):
            r, st = measure_frames(args, tts, W, W.workload("talker"), c, [c], dev, rank, world, full=False)
            del st
            sweep[str(c)] = {"GB_s": r["value"], "ms_per_step": r["ms_per_step"], "l2": r["config"]["l2"],
                             "roofline_frac": r["roofline"]["frac"]}
        res["sweep_cur_len"] = sweep
    return res


def run_prefill(args, rank, world):
    """Prompt prefill on the talker shapes: T positions per stream from --prefill-start,
    one tts_prefill_step per layer for all 28 layers, captured into a CUDA graph."""
    import torch
    from autoregressive_codebook_tts_gb300 import build as b
    b.build()
    from autoregressive_codebook_tts_gb300 import tts
    from autoregressive_codebook_tts_gb300 import workloads as W

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    w = W.workload("talker", kv_dtype=args.prefill_kv)
    T, start = args.prefill_t, args.prefill_start
    B, L, Hq, Hkv, D = w.B, w.layers, w.n_q_heads, w.n_kv_heads, w.head_dim
    if start < 0 or start + T > w.capacity:
        raise SystemExit("prefill window outside the cache")
    g = torch.Generator(device=dev)
    g.manual_seed(rank)
    qd, kd = Hq * D, Hkv * D
    qkv = torch.randn(L, B * T, qd + 2 * kd, generator=g, device=dev)
    gq = torch.rand(L, D, generator=g, device=dev) + 0.5
    gk = torch.rand(L, D, generator=g, device=dev) + 0.5
    caches = []
    kv_t = torch.float32 if w.kv_dtype == "f32" else torch.bfloat16
    for _ in range(L):
        K = torch.empty(B, Hkv, w.capacity, D, device=dev, dtype=kv_t)
        V = torch.empty_like(K)
        K.normal_(generator=g)
        V.normal_(generator=g)
        caches.append((K, V))
    cs = torch.empty(w.capacity, D // 2, 2, device=dev)
    tts.tts_rope_table(cs, w.capacity, D, w.rope_base)
    desc = tts.kv_desc(B, Hq, Hkv, D, w.capacity, w.kv_dtype, window_quantum=w.window_quantum)
    ws = tts.prefill_workspace(desc, T, args.n_splits, device=dev)
    outs = torch.empty(L, B, T, Hq, D, device=dev)
    ef = torch.zeros(1, dtype=torch.int32, device=dev)
    start_t = torch.full((B,), start, dtype=torch.int32, device=dev)
    scale = 1.0 / math.sqrt(D)

    def layers():
        for l in range(L):
            K, V = caches[l]
            rows = qkv[l]
            tts.tts_prefill_step(rows[:, :qd], rows[:, qd:qd + kd], rows[:, qd + kd:], gq[l], gk[l],
                                 w.eps, cs, w.capacity, K, V, desc, start_t, T, scale, outs[l], ws,
                                 args.n_splits, ef)

    gl = capture(layers, torch)
    for _ in range(args.warmup):
        gl.replay()
    torch.cuda.synchronize()
    if ef.item() != 0:
        raise RuntimeError(f"device error flag {ef.item()}")
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t = timed_replays(gl, args.steps, torch)
    clk = clocks.stop()
    (t,) = max_over_ranks([t], world, dev)
    # bytes a layer must move through HBM at least: the prompt's q/k/v rows read, q
    # written back, its k/v rows written to the cache, the earlier cache rows read once,
    # the output written
    e = w.elem_bytes
    hbm = B * (T * (qd + 2 * kd) * 4 + T * qd * 4 + T * 2 * kd * e + start * 2 * kd * e + T * qd * 4)
    # K/V rows the queries read (the prompt's own rows come back from L2)
    attn_rows = B * sum(start + i + 1 for i in range(T))
    attn_bytes = attn_rows * 2 * kd * e
    peak, peak_kind = hbm_peak()
    t_layer = t / (args.steps * L)
    achieved = hbm / t_layer / 1e9
    value = world * B * T * args.steps / t
    return {
        "metric": "prefill: prompt positions per second (B streams, all 28 layers)",
        "value": round(value, 1), "unit": "positions/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f32" if w.kv_dtype == "f32" else "bf16-kv/f32",
        "data": "synthetic (seeded, device-generated; random-init, no weights)",
        "config": {"workload": f"prefill: talker shapes, B={B}, {T} prompt positions from {start}, "
                               f"28 layers, {w.kv_dtype} KV, capacity {w.capacity}",
                   "frame_step": "graph replay of 28 x tts_prefill_step",
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "us_per_layer": round(t_layer * 1e6, 3),
        "attn_kv_gb_s": round(attn_bytes / t_layer / 1e9, 1),
        "roofline": {"bound": "hbm", "achieved": round(achieved, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(achieved / peak, 4), "traffic": None,
                     "kernel": "tts_prefill_step (rows + attention launches)",
                     "peak_source": "measured HBM copy bandwidth" if peak_kind == "measured"
                     else "fallback HBM copy bandwidth", "bytes_per_launch": hbm},
        "gpu_launches": tts.tts_prefill_launch_count(desc, T, args.n_splits) * L * args.steps,
        "clocks": clk,
    }


def run_predictor(args, rank, world):
    """Code-predictor frames, K per graph replay: per frame the T=2 prefill (rows 0, 1)
    of all layers, then 14 single-token decode steps; before every step after the
    prefill the in-graph sampler draws the next code from that step's logits and the
    frame-input composition gathers it from its group table.  The logits (the output
    heads are outside this path) are fixed synthetic rows, one per sub-step."""
    import torch
    from autoregressive_codebook_tts_gb300 import build as b
    b.build()
    from autoregressive_codebook_tts_gb300 import workloads as W
    from autoregressive_codebook_tts_gb300.predictor import PredictorFrames

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    w = W.workload("predictor")
    B, L, Hq, Hkv, D, V = w.B, w.layers, w.n_q_heads, w.n_kv_heads, w.head_dim, w.vocab
    K = max(1, args.frames_per_replay)
    g = torch.Generator(device=dev)
    g.manual_seed(rank)
    qd, kd = Hq * D, Hkv * D
    tables = [torch.randn(V, w.hidden, generator=g, device=dev) * w.table_std for _ in range(15)]
    qkv = torch.randn(16, L, B, qd + 2 * kd, generator=g, device=dev)   # per position, layer
    pre = torch.randn(L, 2 * B, qd + 2 * kd, generator=g, device=dev)    # prefill rows b*2+t
    logits = torch.randn(15, B, V, generator=g, device=dev) * 2.0
    gq = torch.rand(L, D, generator=g, device=dev) + 0.5
    gk = torch.rand(L, D, generator=g, device=dev) + 0.5
    c0 = torch.randint(0, V, (1, B), generator=g, device=dev, dtype=torch.int32)
    top_k, temp, seed = 50, 0.9, 1234 + rank
    pf = PredictorFrames(B, L, Hq, Hkv, D, w.hidden, V, tables, pre, qkv, logits, gq, gk, top_k, temp,
                         seed, c0, eps=w.eps, rope_base=w.rope_base, capacity=w.capacity, slots=1,
                         device=dev)
    ef = pf.err

    def frames():
        pf.enqueue_frames(K)

    gr = capture(frames, torch)
    for _ in range(args.warmup):
        gr.replay()
    torch.cuda.synchronize()
    if ef.item() != 0:
        raise RuntimeError(f"device error flag {ef.item()}")
    replays = max(1, args.steps // K)
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t = timed_replays(gr, replays, torch)
    clk = clocks.stop()
    (t,) = max_over_ranks([t], world, dev)
    n_frames = replays * K
    # algorithmic bytes per frame: every step's window (rows 0..t) for every layer and
    # stream, the new rows, q/k/v and outputs, the gathered table rows, the logits
    kv = sum(t + 1 for t in range(16)) * L * B * 2 * kd * 4
    act = 16 * L * B * ((qd + 2 * kd) * 4 + qd * 4) + 15 * B * (w.hidden * 4 * 2 + V * 4)
    frame_bytes = kv + act
    peak, peak_kind = hbm_peak()
    launches = pf.launches_per_frame
    value = world * B * n_frames / t
    return {
        "metric": "code-predictor frame steps per second (B streams)",
        "value": round(value, 1), "unit": "frame steps/s", "n_gpus": world, "steps": n_frames,
        "warmup": args.warmup, "ms_per_step": round(t / n_frames * 1e3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
        "data": "synthetic (seeded, device-generated; random-init, no weights; fixed logits)",
        "config": {"workload": f"predictor: B={B} streams, {L} layers, hidden {w.hidden}, 16/8 heads, "
                               f"head_dim {D}, f32 KV, 16-slot cache reset per frame, T=2 prefill + 14 decodes, "
                               f"top-{top_k} sampling at T={temp}",
                   "frames_per_replay": K, "launches_per_frame": launches,
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "us_per_frame": round(t / n_frames * 1e6, 2),
        "roofline": {"bound": "hbm", "achieved": round(frame_bytes / (t / n_frames) / 1e9, 1), "peak": peak,
                     "unit": "GB/s", "frac": round(frame_bytes / (t / n_frames) / 1e9 / peak, 4),
                     "traffic": None, "kernel": "whole predictor frame (launch-bound; the roofline "
                     "fraction is not meaningful at 0.4 MB per launch)",
                     "peak_source": "measured HBM copy bandwidth" if peak_kind == "measured"
                     else "fallback HBM copy bandwidth", "bytes_per_frame": frame_bytes},
        "gpu_launches": launches * n_frames,
        "clocks": clk,
    }


def run_reference_predictor(args, world):
    """The oracle's code-predictor frame (same shapes, fixed codes) as the reference
    arm's step: one step = one frame of all streams."""
    import numpy as np
    from autoregressive_codebook_tts_gb300 import workloads as W
    import oracle
    w = W.workload("predictor")
    B, L, Hq, Hkv, D = w.B, w.layers, w.n_q_heads, w.n_kv_heads, w.head_dim
    tabs = [t.numpy() for t in W.tables(15, w.vocab, w.hidden, seed=50)]
    codes = W.code_ids(B, 15, w.vocab, seed=70).numpy()
    qkv = []
    for t in range(16):
        per_l = []
        for l in range(L):
            _, q, k, v = W.qkv(B, Hq, Hkv, D, seed=16 * l + t)
            per_l.append((q.numpy().reshape(B, Hq, D), k.numpy().reshape(B, Hkv, D),
                          v.numpy().reshape(B, Hkv, D)))
        qkv.append(per_l)
    gam = [(W.gamma(D, 4 + l).numpy(), W.gamma(D, 40 + l).numpy()) for l in range(L)]
    caches = [(np.zeros((B, Hkv, w.capacity, D), np.float32), np.zeros((B, Hkv, w.capacity, D), np.float32))
              for _ in range(L)]
    lay = oracle.KvLayout(B, Hkv, D, w.capacity)

    def step():
        oracle.predictor_frame(tabs, codes, None, qkv, gam, np.float32(w.eps), w.rope_base, caches, lay,
                               1.0 / math.sqrt(D))

    for _ in range(args.warmup):
        step()
    with CpuClock() as clk:
        for _ in range(args.steps):
            step()
    dt = clk.wall
    value = B * args.steps / dt
    return {
        "impl": "reference",
        "metric": "code-predictor frame steps per second (B streams)",
        "value": round(value, 3), "unit": "frame steps/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
        "data": "synthetic (seeded)",
        "config": {"workload": f"predictor: B={B} streams, {L} layers (same shapes as the native arm)",
                   "parallelism": "host threads of the oracle (see cpu_baseline.cores)"},
        "cpu_baseline": {"value": round(value, 3), "unit": "frame steps/s", "cores": clk.cores, "kind": "oracle",
                         "sample": "each step: one whole predictor frame of all streams (fixed codes)"},
        "e2e": {"value": round(value, 3), "unit": "frame steps/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_layer(args, rank, world):
    """Whole talker frames: the frame-input composition, then 28 tts_decode_layer calls
    (norms, bf16-weight GEMVs, the fused decode step, residuals) on random-init bf16
    weights, captured into one CUDA graph."""
    import torch
    from autoregressive_codebook_tts_gb300 import build as b
    b.build()
    from autoregressive_codebook_tts_gb300 import tts
    from autoregressive_codebook_tts_gb300 import workloads as W

    local = int(os.environ.get("LOCAL_RANK", "0"))
    dev = torch.device(f"cuda:{local}")
    torch.cuda.set_device(dev)
    B = args.layer_streams
    w = W.workload("talker", B=B, **({"layers": args.layers} if args.layers > 0 else {}))
    L, H, Hq, Hkv, D = w.layers, w.hidden, w.n_q_heads, w.n_kv_heads, w.head_dim
    I = 3 * H
    g = torch.Generator(device=dev)
    g.manual_seed(rank)
    mat = lambda r, c: (torch.randn(r, c, generator=g, device=dev) * 0.02).to(torch.bfloat16)
    layers_w = []
    keep = []
    for _ in range(L):
        t = dict(w_qkv=mat((Hq + 2 * Hkv) * D, H), w_o=mat(H, Hq * D), w_gu=mat(2 * I, H), w_down=mat(H, I),
                 ga=torch.rand(H, generator=g, device=dev) + 0.5, gm=torch.rand(H, generator=g, device=dev) + 0.5,
                 gq=torch.rand(D, generator=g, device=dev) + 0.5, gk=torch.rand(D, generator=g, device=dev) + 0.5)
        keep.append(t)
        layers_w.append(tts.layer_weights(t["w_qkv"], t["w_o"], t["w_gu"], t["w_down"], t["ga"], t["gm"],
                                          t["gq"], t["gk"]))
    caches = []
    for _ in range(L):
        K = torch.empty(B, Hkv, w.capacity, D, device=dev)
        V = torch.empty_like(K)
        K.normal_(generator=g)
        V.normal_(generator=g)
        caches.append((K, V))
    cs = torch.empty(w.capacity, D // 2, 2, device=dev)
    tts.tts_rope_table(cs, w.capacity, D, w.rope_base)
    desc = tts.kv_desc(B, Hq, Hkv, D, w.capacity, "f32", window_quantum=w.window_quantum,
                       flags=tts.TTS_KV_PREFETCH_BEFORE_WAIT)
    scratch = tts.layer_scratch(desc, H, I, args.n_splits, device=dev)
    tabs = [torch.randn(w.vocab, H, generator=g, device=dev) * w.table_std for _ in range(w.n_tables)]
    tabs_struct = tts.tables(tabs)
    ids = torch.randint(0, w.vocab, (B, w.n_tables), generator=g, device=dev, dtype=torch.int32)
    overlay = torch.randn(B, H, generator=g, device=dev) * w.table_std
    hbuf = torch.empty(B, H, device=dev)
    cur = torch.full((B,), args.cur_len, dtype=torch.int32, device=dev)
    ef = torch.zeros(1, dtype=torch.int32, device=dev)
    scale = 1.0 / math.sqrt(D)

    def frame():
        tts.tts_frame_embed(tabs_struct, ids, overlay, hbuf, ef)
        for l in range(L):
            tts.tts_decode_layer(hbuf, layers_w[l], w.eps, cs, w.capacity, caches[l][0], caches[l][1], desc,
                                 cur, scale, scratch, args.n_splits, ef)

    gr = capture(frame, torch)
    for _ in range(args.warmup):
        gr.replay()
    torch.cuda.synchronize()
    if ef.item() != 0:
        raise RuntimeError(f"device error flag {ef.item()}")
    clocks = ClockSampler(local)
    clocks.start()
    time.sleep(0.3)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    t = timed_replays(gr, args.steps, torch)
    clk = clocks.stop()
    (t,) = max_over_ranks([t], world, dev)
    weights = 2 * ((Hq + 2 * Hkv) * D * H + H * Hq * D + 2 * I * H + H * I)
    per_layer, kv_layer, embed = step_bytes(w, [args.cur_len] * B)
    acts = B * (2 * H * 4 * 4 + H * 2 * 2 + I * 2 * 2)   # h reads/writes, x, a (approximate, small)
    frame_bytes = embed + L * (weights + per_layer + acts)
    peak, peak_kind = hbm_peak()
    value = whole_job_gbs(world, frame_bytes, args.steps, t)
    return {
        "metric": "talker frame GB/s (weights + KV, % of HBM peak); frame steps/sec",
        "value": round(value, 2), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(t / args.steps * 1e3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "bf16-weights/f32",
        "data": "synthetic (seeded, device-generated; random-init bf16 weights)",
        "config": {"workload": f"talker layers: B={B} streams, {L} layers, hidden {H}, intermediate {I}, "
                               f"16/8 heads, head_dim {D}, f32 KV, capacity {w.capacity}, cur_len {args.cur_len}",
                   "frame_step": f"graph replay of tts_frame_embed + {L} x tts_decode_layer",
                   "weights_per_layer_bytes": weights,
                   "parallelism": "replicas" if world > 1 else "single GPU"},
        "frame_steps_per_s": round(world * B * args.steps / t, 1),
        "pct_of_hbm_peak": round(100 * value / world / peak, 2),
        "roofline": {"bound": "hbm", "achieved": round(value / world, 1), "peak": peak, "unit": "GB/s",
                     "frac": round(value / world / peak, 4), "traffic": None,
                     "kernel": "whole frame (GEMVs and the decode step)",
                     "peak_source": "measured HBM copy bandwidth" if peak_kind == "measured"
                     else "fallback HBM copy bandwidth", "bytes_per_frame": frame_bytes},
        "gpu_launches": args.steps * (1 + tts.tts_decode_layer_launch_count(desc) * L),
        "clocks": clk,
    }


def run_reference_prefill(args, world):
    """The oracle's prefill of one layer (talker shapes) as the reference arm's step."""
    import numpy as np
    from autoregressive_codebook_tts_gb300 import workloads as W
    import oracle
    w = W.workload("talker")
    T, start = args.prefill_t, args.prefill_start
    B, Hq, Hkv, D = w.B, w.n_q_heads, w.n_kv_heads, w.head_dim
    rows, _, _, _ = W.qkv(B * T, Hq, Hkv, D, seed=3)
    r = rows.numpy()
    qd, kd = Hq * D, Hkv * D
    q = r[:, :qd].reshape(B, T, Hq, D)
    k = r[:, qd:qd + kd].reshape(B, T, Hkv, D)
    v = r[:, qd + kd:].reshape(B, T, Hkv, D)
    gq, gk = W.gamma(D, 4).numpy(), W.gamma(D, 5).numpy()
    K, V = W.cache(w, [start] * B, seed=7, poison=False)
    kc, vc = K.numpy().copy(), V.numpy().copy()
    lay = oracle.KvLayout(B, Hkv, D, w.capacity, w.kv_dtype)
    st = np.full(B, start, np.int32)

    def step():
        oracle.prefill_step(q, k, v, gq, gk, np.float32(w.eps), w.rope_base, kc, vc, lay, st,
                            1.0 / math.sqrt(D))

    for _ in range(args.warmup):
        step()
    with CpuClock() as clk:
        for _ in range(args.steps):
            step()
    dt = clk.wall
    # one step is one layer of the 28: positions per second of the whole prompt
    value = B * T * args.steps / (dt * w.layers)
    sample = f"each step: one layer's prefill of {T} positions from {start} (1 of {w.layers} layers)"
    return {
        "impl": "reference",
        "metric": "prefill: prompt positions per second (B streams, all 28 layers)",
        "value": round(value, 3), "unit": "positions/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
        "data": "synthetic (seeded)",
        "config": {"workload": f"prefill: talker shapes, B={B}, {T} prompt positions from {start}",
                   "parallelism": "host threads of the oracle (see cpu_baseline.cores)"},
        "cpu_baseline": {"value": round(value, 3), "unit": "positions/s", "cores": clk.cores,
                         "kind": "oracle", "sample": sample},
        "e2e": {"value": round(value, 3), "unit": "positions/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_reference_layer(args, world):
    """The oracle's whole talker decode layer (bf16 weights, same shapes and cur_len as
    the native layer arm) as the reference arm's step: one layer of the frame."""
    import numpy as np
    import torch
    from autoregressive_codebook_tts_gb300 import workloads as W
    import oracle
    B = args.layer_streams
    w = W.workload("talker", B=B)
    H, Hq, Hkv, D = w.hidden, w.n_q_heads, w.n_kv_heads, w.head_dim
    I = 3 * H
    g = torch.Generator().manual_seed(0)
    bits = lambda r, c: ((torch.randn(r, c, generator=g) * 0.02).to(torch.bfloat16)
                         .view(torch.int16).numpy().view(np.uint16))
    wts = dict(w_qkv=bits((Hq + 2 * Hkv) * D, H), w_o=bits(H, Hq * D), w_gu=bits(2 * I, H),
               w_down=bits(H, I), gamma_attn=(torch.rand(H, generator=g) + 0.5).numpy(),
               gamma_mlp=(torch.rand(H, generator=g) + 0.5).numpy(),
               gamma_q=(torch.rand(D, generator=g) + 0.5).numpy(),
               gamma_k=(torch.rand(D, generator=g) + 0.5).numpy())
    cur_list = [args.cur_len] * B
    K, V = W.cache(w, cur_list, seed=7, poison=False)
    kc, vc = K.numpy().copy(), V.numpy().copy()
    lay = oracle.KvLayout(B, Hkv, D, w.capacity, w.kv_dtype)
    cur = np.array(cur_list, np.int32)
    h0 = torch.randn(B, H, generator=g).numpy()

    def step():
        oracle.decode_layer(h0.copy(), wts, kc, vc, lay, cur, np.float32(w.eps), w.rope_base,
                            1.0 / math.sqrt(D))

    for _ in range(args.warmup):
        step()
    with CpuClock() as clk:
        for _ in range(args.steps):
            step()
    dt = clk.wall
    weights = 2 * ((Hq + 2 * Hkv) * D * H + H * Hq * D + 2 * I * H + H * I)
    per_layer, _, _ = step_bytes(w, cur_list)
    value = (weights + per_layer) * args.steps / dt / 1e9
    sample = (f"each step: one whole decode layer of the talker frame (1 of {w.layers} layers), "
              f"B={B}, cur_len {args.cur_len}")
    return {
        "impl": "reference",
        "metric": "talker frame GB/s (weights + KV, % of HBM peak); frame steps/sec",
        "value": round(value, 5), "unit": "GB/s", "n_gpus": world, "steps": args.steps,
        "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
        "data": "synthetic (seeded; random-init bf16 weights)",
        "config": {"workload": f"talker layers: B={B} streams, hidden {H}, intermediate {I}, "
                               f"16/8 heads, head_dim {D}, f32 KV, capacity {w.capacity}, "
                               f"cur_len {args.cur_len}", "parallelism": "host threads of the oracle (see cpu_baseline.cores)"},
        "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": clk.cores, "kind": "oracle",
                         "sample": sample},
        "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def run_reference(args, rank, world):
    """The CPU oracle timed as the reference arm, on the same workload and metric."""
    import numpy as np
    import torch
    from autoregressive_codebook_tts_gb300 import workloads as W
    import oracle
    oracle.build()
    if args.workload == "prefill":
        return run_reference_prefill(args, world)
    if args.workload == "predictor":
        return run_reference_predictor(args, world)
    if args.workload == "layer":
        return run_reference_layer(args, world)
    w = W.workload(args.workload)
    cur_list = [args.cur_len] * w.B if args.workload == "talker" else [int(c) for c in W.cur_lens(w, 0)]
    cur = np.array(cur_list, np.int32)
    tabs = [t.numpy() for t in W.tables(w.n_tables, w.vocab, w.hidden, seed=0)]
    ids = W.code_ids(w.B, w.n_tables, w.vocab, seed=1).numpy()
    ov = W.overlay(w.B, w.hidden, seed=2).numpy()
    rows, q, k, v = W.qkv(w.B, w.n_q_heads, w.n_kv_heads, w.head_dim, seed=3)
    q = q.numpy().reshape(w.B, w.n_q_heads, w.head_dim)
    k = k.numpy().reshape(w.B, w.n_kv_heads, w.head_dim)
    v = v.numpy().reshape(w.B, w.n_kv_heads, w.head_dim)
    gq, gk = W.gamma(w.head_dim, 4).numpy(), W.gamma(w.head_dim, 5).numpy()
    bt = None
    if w.paged:
        bt = W.block_table(w.B, w.capacity // w.page_size, w.n_pages, seed=6)
    K, V = W.cache(w, cur_list, seed=7, block_tab=bt, poison=False)
    if w.kv_dtype == "bf16":
        hk = K.view(torch.int16).numpy().view(np.uint16).copy()
        hv = V.view(torch.int16).numpy().view(np.uint16).copy()
    else:
        hk, hv = K.numpy().copy(), V.numpy().copy()
    h = dict(hk=hk, hv=hv, tabs=tabs, ids=ids, ov=ov, q=q.copy(), k=k.copy(), v=v.copy(), gq=gq, gk=gk,
             cur=cur, bt=None if bt is None else bt.numpy())
    per_layer, _, embed = step_bytes(w, cur_list)
    # one step = the frame-input composition + one layer's fused decode step of every
    # stream (a bounded sample of the frame; the metric is bytes per second, so it
    # carries over), cut into (stream, kv head) units over every host thread
    sample_bytes = embed + per_layer
    nt = host_threads()
    time_oracle(h, w, sample_bytes, reps=args.warmup, threads=nt)
    rate, n, dt, clk = time_oracle(h, w, sample_bytes, reps=args.steps, threads=nt)
    value = rate / 1e9
    sample = (f"each step: frame-input composition + one layer's fused decode step of the "
              f"{w.name} workload (1 of {w.layers} layers), units (stream, kv head) over {nt} host threads")
    return {
        "impl": "reference",
        "metric": METRIC, "value": round(value, 5), "unit": "GB/s", "n_gpus": world,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(dt / args.steps * 1e3, 3),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64 (oracle)",
        "data": "synthetic (seeded)",
        "config": {"workload": f"{w.name} (same shapes as the native arm)", "B": w.B,
                   "layers": w.layers, "parallelism": f"{nt} host threads of the oracle"},
        "cpu_baseline": {"value": round(value, 5), "unit": "GB/s", "cores": nt, "kind": "oracle",
                         "sample": sample, "cpu_time_over_wall": round(clk.cpu / clk.wall, 2)},
        "e2e": {"value": round(value, 5), "unit": "GB/s", "h2d_bytes_per_step": 0,
                "d2h_bytes_per_step": 0},
    }


def main():
    args = parse()
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    if args.impl == "reference":
        if rank != 0:
            return
        print(json.dumps(run_reference(args, rank, world)))
        return
    if world > 1:
        import torch.distributed as dist
        dist.init_process_group("nccl")
    if args.workload == "prefill":
        res = run_prefill(args, rank, world)
    elif args.workload == "predictor":
        res = run_predictor(args, rank, world)
    elif args.workload == "layer":
        res = run_layer(args, rank, world)
    else:
        res = run_native(args, rank, world)
    if rank == 0:
        print(json.dumps(res))
    if world > 1:
        import torch.distributed as dist
        dist.destroy_process_group()


if __name__ == "__main__":
    main()
