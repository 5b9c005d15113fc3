#!/usr/bin/env python
"""Benchmark of the KV-cache attention hot path on one GB300 (or N replicas).

A step is one whole run of the multi-user streaming workload: reset, then for each
of its chunks reserve the slots (advance), write the chunk's K/V at the device-held
slots (write) and attend the chunk's queries over the sink+window ring (attend).
Default workload: 8 users sharing one chunk timeline, bf16, H = 40, D = 128, chunk
4680 tokens, sink 4680, window 32760, 8 chunks (125.6 TFLOP per step).  The K/V
stores (5.4 GB) are far larger than L2, so no flush is needed between steps.

Prints one JSON line.  ``value`` is chunk-attention TFLOP/s over the whole step
(write and advance time included); the line also carries the write and decode
bandwidth, the roofline of the dominant kernel, the end-to-end figure through the
binding with host buffers, and the CPU oracle timed on a bounded sample.

``--impl reference`` times the CPU fp64 oracle as the reference arm instead.
"""
from __future__ import annotations

import argparse
import json
import os
import subprocess
import sys
import tempfile
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from diffusion_serving_gb300 import workloads as wl  # noqa: E402

WORKLOADS = {w.name: w for w in wl.ALL if w.layout == "circular"}
DEFAULT = wl.MULTI_USER.name
METRIC = "chunk-attention TFLOP/s + decode/write HBM GB/s on 1 GB300, as % of roofline"


def load_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return dict(hbm=d["hbm_gbs"], bf16=d["bf16_tflops"], bf16_sust=d["bf16_tflops_sustained"], src="measured")
    return dict(hbm=6800.0, bf16=1900.0, bf16_sust=1700.0, src="fallback")


# ---------------------------------------------------------------------------
# distributed plumbing (replicas only: no data-path collective)
# ---------------------------------------------------------------------------
def dist_init(n_gpus):
    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local = int(os.environ.get("LOCAL_RANK", "0"))
    if world > 1:
        import torch.distributed as dist
        backend = "nccl" if torch.cuda.is_available() else "gloo"
        if torch.cuda.is_available():
            torch.cuda.set_device(local)
        dist.init_process_group(backend)
        return rank, world, dist
    if torch.cuda.is_available():
        torch.cuda.set_device(0)
    return 0, 1, None


def barrier(dist):
    if dist is not None:
        dist.barrier()


def max_over_ranks(x, dist):
    if dist is None:
        return x
    t = torch.tensor([x], dtype=torch.float64, device="cuda" if torch.cuda.is_available() else "cpu")
    dist.all_reduce(t, op=dist.ReduceOp.MAX)
    return float(t.item())


# ---------------------------------------------------------------------------
# clocks sampled during the timed region
# ---------------------------------------------------------------------------
class Clocks:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, device_index):
        self.proc = None
        # raw samples (nvidia-smi CSV); KVC_CLOCKS_DIR keeps them somewhere other than the temp dir
        self.path = os.path.join(os.environ.get("KVC_CLOCKS_DIR", tempfile.gettempdir()),
                                 f"kvc_clocks_{os.getpid()}.csv")
        self.dev = device_index

    def __enter__(self):
        try:
            os.makedirs(os.path.dirname(self.path), exist_ok=True)
            self.f = open(self.path, "w")
            self.proc = subprocess.Popen(["nvidia-smi", f"--id={self.dev}", f"--query-gpu={self.FIELDS}",
                                          "--format=csv,noheader,nounits", "-lms", "200"], stdout=self.f,
                                         stderr=subprocess.DEVNULL)
            time.sleep(0.3)
        except Exception:
            self.proc = None
        return self

    def __exit__(self, *a):
        if self.proc is not None:
            self.proc.terminate()
            try:
                self.proc.wait(timeout=5)
            except Exception:
                self.proc.kill()
            self.f.close()

    def summary(self):
        if self.proc is None or not os.path.exists(self.path):
            return None
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        with open(self.path) as f:
            for line in f:
                parts = [p.strip() for p in line.split(",")]
                if len(parts) < 9:
                    continue
                try:
                    sm.append(float(parts[1]))
                    mx.append(float(parts[2]))
                except ValueError:
                    continue
                for n, v in zip(names, parts[5:9]):
                    if v.lower() == "active":
                        reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": float(max(mx)), "reasons": sorted(reasons),
                "samples": len(sm)}


# ---------------------------------------------------------------------------
# our arm
# ---------------------------------------------------------------------------
def ring_flops(w):
    """Algorithmic flops of one step (every chunk, every rewrite, valid slots only)."""
    total = 0.0
    per_attend, per_kv = [], []
    for c in range(w.n_chunks):
        kv = min((c + 1) * w.chunk, w.window)
        f = wl.attention_flops(w.chunk, kv, w.heads, w.head_dim) * w.batch
        for _ in range(w.rewrites):
            per_attend.append(f)
            per_kv.append(kv)
            total += f
    return total, per_attend, per_kv


def make_inputs(w, device, pool):
    """Distinct (q, k, v) per chunk (and rewrite, up to ``pool`` sets), resident on device."""
    sets = []
    for c in range(w.n_chunks):
        for r in range(w.rewrites):
            if len(sets) < pool:
                sets.append(wl.chunk_inputs(w, c, r, device=device))
    return sets


def run_step(cache, w, inputs, out, stream, ev=None, kvc=None):
    """One step; when ``ev`` is given, record events around each write and attend."""
    launches = 0
    cache.reset(stream=stream)
    launches += 1
    i = 0
    for c in range(w.n_chunks):
        cache.advance(stream=stream)
        launches += 1
        for r in range(w.rewrites):
            q, k, v = inputs[i % len(inputs)]
            i += 1
            if ev is not None:
                ev["w"].append((torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)))
                ev["w"][-1][0].record(stream)
            cache.write(k, v, stream=stream)
            if ev is not None:
                ev["w"][-1][1].record(stream)
                ev["a"].append((torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)))
                ev["a"][-1][0].record(stream)
            cache.attend(q, out, stream=stream)
            if ev is not None:
                ev["a"][-1][1].record(stream)
            launches += 2
    return launches


def decode_bench(kvc, peaks, per_graph=64, replays=5):
    """Split-KV decode on the active-prefix workload shape, timed by replaying a CUDA
    graph of ``per_graph`` attends (host launch cost excluded, as in a captured decode
    loop): a mean-length step (kv_len 490) and a full 32768-slot prefix.  The full-prefix
    point rotates over 4 caches (537 MB of K/V, more than L2) so every read is from HBM."""
    w = wl.DECODE
    caches = []
    g = torch.Generator(device="cuda").manual_seed(w.seed)
    for _ in range(4):
        c = kvc.KVCache(w.batch, w.heads, w.kv_heads, w.head_dim, torch.float16, "linear", capacity=w.capacity)
        c.k_store.normal_(generator=g)
        c.v_store.normal_(generator=g)
        caches.append(c)
    q = torch.randn(1, 1, w.heads, w.head_dim, device="cuda", generator=g).half()
    out = torch.empty_like(q)
    row = w.kv_heads * w.head_dim * 2
    res = {}
    side = torch.cuda.Stream()
    for name, n, ncache in (("mean_step_kv490", wl.DECODE_PROMPT + wl.DECODE_STEPS // 2, 1),
                            ("full_prefix_kv32768", w.capacity, 4)):
        side.wait_stream(torch.cuda.current_stream())
        with torch.cuda.stream(side):
            for c in caches[:ncache]:
                c.set_lengths(kv_len=torch.tensor([n], dtype=torch.int32, device="cuda"), stream=side)
                for _ in range(3):
                    c.attend(q, out, stream=side)
        side.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            for r in range(per_graph):
                caches[r % ncache].attend(q, out, stream=side)
        graph.replay()
        torch.cuda.synchronize()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(replays):
            graph.replay()
        b.record()
        b.synchronize()
        t = a.elapsed_time(b) * 1e-3 / (replays * per_graph)
        nbytes = 2 * n * row
        res[name] = {"kv_len": n, "us": round(t * 1e6, 3), "GB/s": round(nbytes / t / 1e9, 1),
                     "frac": round(nbytes / t / 1e9 / peaks["hbm"], 4), "bytes": nbytes,
                     "timing": f"graph of {per_graph} attends x {replays} replays"}
    # whole decode step (reserve one slot, write its K/V, attend), 64 steps per graph,
    # from a 234-token prompt: kv_len runs 235 .. 618 over the timed replays
    c = caches[0]
    c.reset()
    kp = torch.randn(1, wl.DECODE_PROMPT, w.kv_heads, w.head_dim, device="cuda", generator=g).half()
    k1 = torch.randn(1, 1, w.kv_heads, w.head_dim, device="cuda", generator=g).half()
    c.advance(n_tokens=wl.DECODE_PROMPT)
    c.write(kp, kp)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(graph, stream=side):
        for r in range(per_graph):
            c.advance(n_tokens=1, stream=side)
            c.write(k1, k1, stream=side)
            c.attend(q, out, stream=side)
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(replays):
        graph.replay()
    b.record()
    b.synchronize()
    t = a.elapsed_time(b) * 1e-3 / (replays * per_graph)
    res["step_advance_write_attend"] = {"kv_len": f"{wl.DECODE_PROMPT + 1}..{wl.DECODE_PROMPT + replays * per_graph}",
                                        "us": round(t * 1e6, 3), "tokens_per_s": round(1.0 / t, 1),
                                        "timing": f"graph of {per_graph} steps x {replays} replays"}
    # the same step with the reservation and the write in one launch (kvc_append)
    c.reset()
    c.append(kp, kp)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(graph, stream=side):
        for r in range(per_graph):
            c.append(k1, k1, stream=side)
            c.attend(q, out, stream=side)
    graph.replay()
    c.reset()
    c.append(kp, kp)
    torch.cuda.synchronize()
    a.record()
    for _ in range(replays):
        graph.replay()
    b.record()
    b.synchronize()
    t = a.elapsed_time(b) * 1e-3 / (replays * per_graph)
    res["step_append_attend"] = {"kv_len": f"{wl.DECODE_PROMPT + 1}..{wl.DECODE_PROMPT + replays * per_graph}",
                                 "us": round(t * 1e6, 3), "tokens_per_s": round(1.0 / t, 1),
                                 "timing": f"graph of {per_graph} steps x {replays} replays"}
    # the whole step in one launch (kvc_append_attend_decode)
    c.reset()
    c.append(kp, kp)
    torch.cuda.synchronize()
    graph = torch.cuda.CUDAGraph()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.graph(graph, stream=side):
        for r in range(per_graph):
            c.append_attend(k1, k1, q, out, stream=side)
    graph.replay()
    c.reset()
    c.append(kp, kp)
    torch.cuda.synchronize()
    a.record()
    for _ in range(replays):
        graph.replay()
    b.record()
    b.synchronize()
    t = a.elapsed_time(b) * 1e-3 / (replays * per_graph)
    res["step_fused_append_attend"] = {"kv_len": f"{wl.DECODE_PROMPT + 1}..{wl.DECODE_PROMPT + replays * per_graph}",
                                       "us": round(t * 1e6, 3), "tokens_per_s": round(1.0 / t, 1),
                                       "timing": f"graph of {per_graph} steps x {replays} replays"}
    for c in caches:
        assert c.get_error() == 0
    return res


def _events_time(fn, reps):
    """Seconds per call of fn (which enqueues GPU work on the current stream)."""
    a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
    a.record()
    for _ in range(reps):
        fn()
    b.record()
    b.synchronize()
    return a.elapsed_time(b) * 1e-3 / reps


def dit_bench(kvc, peaks, reps=3):
    """The streaming DiT workload (B2 cond/uncond, H 12, D 128, bf16, chunk 4680, sink
    4680, window 32760, 10 chunks of which 3 evict, 4 denoising rewrites each; 52.75
    TFLOP per run): a whole run (reset, then per chunk advance + 4 x (write + attend))
    launched eagerly and with each chunk's lifecycle replayed from one captured CUDA
    graph, plus one full-window attend alone."""
    w = wl.DIT_STREAM
    cache = kvc.KVCache(w.batch, w.heads, w.kv_heads, w.head_dim, torch.bfloat16, "circular", sink=w.sink,
                        window=w.window, chunk=w.chunk)
    sets = [wl.chunk_inputs(w, 0, r, device="cuda") for r in range(w.rewrites)]
    outs = [torch.empty_like(sets[0][0]) for _ in sets]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())

    def chunk_body(stream):
        cache.advance(stream=stream)
        for (q, k, v), o in zip(sets, outs):
            cache.write(k, v, stream=stream)
            cache.attend(q, o, stream=stream)

    with torch.cuda.stream(side):
        for _ in range(2):
            cache.reset(stream=side)
            for _ in range(w.n_chunks):
                chunk_body(side)
        side.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            chunk_body(side)

        def eager_run():
            cache.reset(stream=side)
            for _ in range(w.n_chunks):
                chunk_body(side)

        def graph_run():
            cache.reset(stream=side)
            for _ in range(w.n_chunks):
                graph.replay()

        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        res = {}
        for name, fn in (("eager", eager_run), ("graph", graph_run)):
            fn()
            a.record(side)
            for _ in range(reps):
                fn()
            b.record(side)
            b.synchronize()
            res[name] = a.elapsed_time(b) * 1e-3 / reps
        # one attend over the full 32760-slot window (the ring is full after a run)
        q, _, _ = sets[0]
        for _ in range(2):
            cache.attend(q, outs[0], stream=side)
        a.record(side)
        for _ in range(reps):
            cache.attend(q, outs[0], stream=side)
        b.record(side)
        b.synchronize()
        t_full = a.elapsed_time(b) * 1e-3 / reps
    assert cache.get_error() == 0
    flops = ring_flops(w)[0]
    f_full = wl.attention_flops(w.chunk, w.window, w.heads, w.head_dim) * w.batch
    cache.close()
    return {"workload": w.name, "tflop_per_run": round(flops / 1e12, 3),
            "run_ms_eager": round(res["eager"] * 1e3, 3), "run_ms_graph": round(res["graph"] * 1e3, 3),
            "TFLOP/s": round(flops / res["graph"] / 1e12, 1),
            "frac": round(flops / res["graph"] / 1e12 / peaks["bf16_sust"], 4),
            "peak_kind": f"bf16 dense sustained, {peaks['src']}",
            "full_window_attend": {"ms": round(t_full * 1e3, 4), "TFLOP/s": round(f_full / t_full / 1e12, 1),
                                   "frac": round(f_full / t_full / 1e12 / peaks["bf16"], 4),
                                   "peak_kind": f"bf16 dense burst, {peaks['src']}"},
            "timing": f"whole run x {reps}; graph = one captured chunk (advance + {w.rewrites} x (write + attend)) "
                      f"replayed per chunk"}


def tiny_bench(kvc, reps=20):
    """The tiny circular workload (fp32, B1 H2 D64, chunk 4, sink 4, window 16, 7 chunks x
    2 rewrites, then reset): absolute time of a chunk step (advance + 2 x (write +
    attend)) and of the whole run with its reset, eager and as a replayed graph."""
    w = wl.TINY_RING
    cache = kvc.KVCache(w.batch, w.heads, w.kv_heads, w.head_dim, torch.float32, "circular", sink=w.sink,
                        window=w.window, chunk=w.chunk)
    sets = [wl.chunk_inputs(w, 0, r, device="cuda") for r in range(w.rewrites)]
    outs = [torch.empty_like(sets[0][0]) for _ in sets]
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())

    def chunk_body(stream):
        cache.advance(stream=stream)
        for (q, k, v), o in zip(sets, outs):
            cache.write(k, v, stream=stream)
            cache.attend(q, o, stream=stream)

    with torch.cuda.stream(side):
        cache.reset(stream=side)
        for _ in range(w.n_chunks):
            chunk_body(side)
        side.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            cache.reset(stream=side)
            for _ in range(w.n_chunks):
                chunk_body(side)
        graph.replay()

        def eager_run():
            cache.reset(stream=side)
            for _ in range(w.n_chunks):
                chunk_body(side)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        times = {}
        for name, fn in (("eager", eager_run), ("graph", graph.replay)):
            fn()
            a.record(side)
            for _ in range(reps):
                fn()
            b.record(side)
            b.synchronize()
            times[name] = a.elapsed_time(b) * 1e-3 / reps
    assert cache.get_error() == 0
    launches = 1 + w.n_chunks * (1 + 2 * w.rewrites)
    return {"workload": w.name, "run_us_eager": round(times["eager"] * 1e6, 2),
            "run_us_graph": round(times["graph"] * 1e6, 2),
            "chunk_step_us_graph": round(times["graph"] / w.n_chunks * 1e6, 2), "launches_per_run": launches,
            "timing": f"reset + {w.n_chunks} chunks x {w.rewrites} rewrites, {reps} runs; latency-bound "
                      f"(no roofline fraction)"}


def decode_schedule_bench(kvc, peaks, reps=5):
    """The active-prefix workload as the pages run it (fp16, H 32 / Hkv 8, D 128, a
    32768-slot store): prefill of 234 tokens (append, causal attend of the 234 queries),
    then 512 decode steps (append the token's K/V and attend, one launch per step), kv_len
    235..746.  The 512 steps are one captured graph; tokens/s = 512 / their time."""
    w = wl.DECODE
    T, N = wl.DECODE_PROMPT, wl.DECODE_STEPS
    c = kvc.KVCache(w.batch, w.heads, w.kv_heads, w.head_dim, torch.float16, "linear", capacity=w.capacity)
    g = torch.Generator(device="cuda").manual_seed(w.seed)
    qp = torch.randn(1, T, w.heads, w.head_dim, device="cuda", generator=g).half()
    kp = torch.randn(1, T, w.kv_heads, w.head_dim, device="cuda", generator=g).half()
    q1 = torch.randn(1, 1, w.heads, w.head_dim, device="cuda", generator=g).half()
    k1 = torch.randn(1, 1, w.kv_heads, w.head_dim, device="cuda", generator=g).half()
    op, o1 = torch.empty_like(qp), torch.empty_like(q1)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())

    def prefill():
        c.reset(stream=side)
        c.append(kp, kp, stream=side)
        c.attend(qp, op, flags=kvc.CAUSAL, stream=side)

    with torch.cuda.stream(side):
        prefill()
        for _ in range(3):
            c.append_attend(k1, k1, q1, o1, stream=side)
        side.synchronize()
        graph = torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph, stream=side):
            for _ in range(N):
                c.append_attend(k1, k1, q1, o1, stream=side)
        a, b, m = (torch.cuda.Event(enable_timing=True) for _ in range(3))
        t_pre = t_dec = 0.0
        for _ in range(reps + 1):
            a.record(side)
            prefill()
            m.record(side)
            graph.replay()
            b.record(side)
            b.synchronize()
            if _ > 0:
                t_pre += a.elapsed_time(m) * 1e-3 / reps
                t_dec += m.elapsed_time(b) * 1e-3 / reps
    assert c.get_error() == 0
    kv_bytes = sum(2 * (T + i + 1) * w.kv_heads * w.head_dim * 2 for i in range(N))
    c.close()
    return {"workload": w.name, "prefill_us": round(t_pre * 1e6, 2), "decode_steps": N,
            "decode_ms": round(t_dec * 1e3, 4), "tokens_per_s": round(N / t_dec, 1),
            "us_per_step": round(t_dec / N * 1e6, 3),
            "kv_GB/s": round(kv_bytes / t_dec / 1e9, 1), "kv_frac": round(kv_bytes / t_dec / 1e9 / peaks["hbm"], 4),
            "timing": f"prefill eager + {N} steps (fused append + attend) as one graph, {reps} runs; "
                      f"kv_len {T + 1}..{T + N}, latency-bound"}


def kernel_code_sha256(path):
    """sha256 of a CUDA source with its // comments and blank lines removed: the code a
    capture was taken of (comment edits do not change the kernel)."""
    import hashlib
    import re
    with open(path) as f:
        text = f.read()
    lines = [re.sub(r"//.*$", "", ln).rstrip() for ln in text.splitlines()]
    return hashlib.sha256("\n".join(ln for ln in lines if ln).encode()).hexdigest()


def tc_traffic_per_launch(w, per_attend_kv):
    """DRAM bytes per attend launch, from the committed capture of the chunk kernel:
    the capture's DRAM / algorithmic ratio times this workload's average algorithmic
    bytes (Q and O once, valid K/V once).  None when the kernel code changed since."""
    path = os.path.join(ROOT, "profiles", "k_attn_tc_traffic.json")
    src = os.path.join(ROOT, "diffusion_serving_gb300", "csrc", "k_attn_tc.cu")
    if not (os.path.exists(path) and os.path.exists(src)):
        return None
    with open(path) as f:
        cap = json.load(f)
    if kernel_code_sha256(src) != cap.get("kernel_code_sha256"):
        return None
    qo = 2 * w.batch * w.chunk * w.heads * w.head_dim * 2
    kv = [2 * w.batch * n * w.kv_heads * w.head_dim * 2 for n in per_attend_kv]
    return round(cap["dram_over_algorithmic"] * (qo + float(np.mean(kv))))


def cross_bench(kvc, peaks, reps=10, lq=None):
    """Ragged cross-attention (2 CFG branches, H 40, D 128, 75600 padded queries, text
    K/V of at most 512 tokens per branch): time per attend for the three length skews in
    two arms that compute the same result, packed K/V by cu_seqlens and a padded 512-slot
    store with per-branch kv_len, plus the padded store attended unmasked (all 512 slots).
    Q and O traffic (3.1 GB) bounds the first two; the roofline time is
    max(bytes / HBM, flops / tensor)."""
    w = wl.CROSS
    B, H, D, Lq = w.batch, w.heads, w.head_dim, lq or wl.CROSS_LQ
    L = wl.CROSS_LKV_MAX
    g = torch.Generator(device="cuda").manual_seed(w.seed)
    q = torch.randn(B, Lq, H, D, device="cuda", generator=g).bfloat16()
    out = torch.empty_like(q)
    kv = torch.randn(B, L, H, D, device="cuda", generator=g).bfloat16()

    def timed(c, lens):
        for _ in range(3):
            c.attend(q, out)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            c.attend(q, out)
        b.record()
        b.synchronize()
        assert c.get_error() == 0
        t = a.elapsed_time(b) * 1e-3 / reps
        nbytes = 2 * q.numel() * 2 + sum(2 * n * H * D * 2 for n in lens)
        flops = sum(wl.attention_flops(Lq, n, H, D) for n in lens)
        roof = max(nbytes / (peaks["hbm"] * 1e9), flops / (peaks["bf16"] * 1e12))
        return {"lens": list(lens), "ms": round(t * 1e3, 4), "GB/s": round(nbytes / t / 1e9, 1),
                "TFLOP/s": round(flops / t / 1e12, 1), "roofline_ms": round(roof * 1e3, 4),
                "frac": round(roof / t, 4)}

    padded = kvc.KVCache(B, H, H, D, torch.bfloat16, "linear", capacity=L)
    padded.advance(n_tokens=L)
    padded.write(kv, kv)
    res = {"padded_512_unmasked": timed(padded, (L, L))}
    for name, lens in wl.CROSS_SKEWS.items():
        packed = kvc.KVCache(B, H, H, D, torch.bfloat16, "packed", capacity=2 * L)
        packed.set_lengths(cu_seqlens=torch.tensor(wl.seqlens_to_cu(lens), dtype=torch.int32, device="cuda"))
        packed.write(kv, kv)
        padded.set_lengths(kv_len=torch.tensor(lens, dtype=torch.int32, device="cuda"))
        res[name] = {"packed": timed(packed, lens), "kv_len": timed(padded, lens)}
        if name == "typical":
            res["metadata"] = metadata_bench(kvc, packed, q, out, lens, reps)
        packed.close()
    return res


def metadata_bench(kvc, packed, q, out, lens, reps, layers=40):
    """The cost of preparing the length metadata, as the pages' cross-attention
    microbenchmark splits it (_total with the per-call metadata preparation, _kernel
    without): per attend, (i) the kernel alone over a layout prepared once, (ii) each
    call copying its cu_seqlens up from pinned host memory and setting them before the
    attend, (iii) one copy and set per step shared by 40 layers' attends."""
    shared = kvc.KVLengths(packed.cfg.batch, "packed", packed.cfg.capacity)
    host_cu = torch.tensor(wl.seqlens_to_cu(lens), dtype=torch.int32).pin_memory()
    dev_cu = torch.empty_like(host_cu, device="cuda")
    packed.use_lengths(shared)

    def prep():
        dev_cu.copy_(host_cu, non_blocking=True)
        shared.set(cu_seqlens=dev_cu)

    def total():
        prep()
        packed.attend(q, out)

    def per_step():
        prep()
        for _ in range(layers):
            packed.attend(q, out)

    prep()
    for fn in (total, lambda: packed.attend(q, out)):
        fn()
    t_kernel = _events_time(lambda: packed.attend(q, out), reps)
    t_total = _events_time(total, reps)
    t_step = _events_time(per_step, max(1, reps // 5)) / layers
    assert packed.get_error() == 0
    packed.use_lengths(None)
    return {"kernel_ms": round(t_kernel * 1e3, 4), "total_ms": round(t_total * 1e3, 4),
            "total_over_kernel": round(t_total / t_kernel, 4),
            "shared_layout_ms_per_layer": round(t_step * 1e3, 4), "layers": layers,
            "note": "total = cu_seqlens copied up + kvc_lengths_set + attend, per call; shared = one copy + "
                    "set per step, read by every layer's attend"}


def cpu_oracle_sample(w, budget_s=12.0):
    """Time the fp64 oracle on sampled query rows of a full-window attend."""
    from oracle import kvc_oracle as orc
    kv = w.window
    rng = np.random.default_rng(0)
    k = rng.standard_normal((kv, 1, w.head_dim)).astype(np.float64)
    v = rng.standard_normal((kv, 1, w.head_dim)).astype(np.float64)
    rows = 64
    flops = 0.0
    t0 = time.perf_counter()
    calls = 0
    while time.perf_counter() - t0 < budget_s:
        q = rng.standard_normal((rows, 1, w.head_dim))
        orc.attend(q, k, v)
        flops += wl.attention_flops(rows, kv, 1, w.head_dim)
        calls += 1
    dt = time.perf_counter() - t0
    return flops / dt / 1e12, dt, calls * rows


def host_cores():
    try:
        return len(os.sched_getaffinity(0))
    except Exception:
        return os.cpu_count() or 1


def blas_threads():
    try:
        from threadpoolctl import threadpool_info
        info = threadpool_info()
        return max((i.get("num_threads", 1) for i in info), default=1)
    except Exception:
        return host_cores()


def ours(args):
    rank, world, dist = dist_init(args.gpus)
    from diffusion_serving_gb300 import kvc
    w = WORKLOADS[args.workload]
    peaks = load_peaks()
    dtype = wl.DTYPES[w.dtype]
    stream = torch.cuda.current_stream()
    cache = kvc.KVCache(w.batch, w.heads, w.kv_heads, w.head_dim, dtype, w.layout, sink=w.sink, window=w.window,
                        chunk=w.chunk)
    inputs = make_inputs(w, "cuda", pool=min(args.pool, w.n_chunks * w.rewrites))
    out = torch.empty_like(inputs[0][0])
    step_flops, per_attend, per_kv = ring_flops(w)

    for _ in range(args.warmup):
        run_step(cache, w, inputs, out, stream)
    torch.cuda.synchronize()
    assert cache.get_error() == 0

    ev = {"w": [], "a": []}
    launches = 0
    with Clocks(torch.cuda.current_device()) as clk:
        barrier(dist)
        torch.cuda.synchronize()
        start, stop = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        start.record(stream)
        for _ in range(args.steps):
            launches += run_step(cache, w, inputs, out, stream, ev)
        stop.record(stream)
        torch.cuda.synchronize()
        barrier(dist)
    elapsed = start.elapsed_time(stop) * 1e-3
    elapsed = max_over_ranks(elapsed, dist)
    err = cache.get_error()
    assert err == 0, f"device error bits {err:#x}"

    attend_t = [a.elapsed_time(b) * 1e-3 for a, b in ev["a"]]
    write_t = [a.elapsed_time(b) * 1e-3 for a, b in ev["w"]]
    attend_flops = per_attend * args.steps
    avg_attend_flops = float(np.mean(attend_flops))
    avg_attend_t = float(np.mean(attend_t))
    achieved = avg_attend_flops / avg_attend_t / 1e12
    row_bytes = w.kv_heads * w.head_dim * 2
    write_bytes = 2 * 2 * w.batch * w.chunk * row_bytes      # K and V, read + write
    write_gbs = write_bytes / float(np.mean(write_t)) / 1e9

    value = world * step_flops * args.steps / elapsed / 1e12
    result = {
        "metric": METRIC,
        "value": round(value, 2),
        "unit": "TFLOP/s",
        "n_gpus": world,
        "steps": args.steps,
        "warmup": args.warmup,
        "ms_per_step": round(elapsed / args.steps * 1e3, 3),
        "higher_is_better": True,
        "scaling": "weak",
        "vs_baseline": None,
        "dtype": w.dtype,
        "data": "synthetic",
        "config": {**workload_config(w),
                   "l2": "inputs larger than L2 (K/V stores %.1f GB)" % (2 * cache.k_store.numel() * 2 / 1e9),
                   "parallelism": f"replicas x{world}"},
        "gpu_launches": launches,
        "roofline": {"bound": "tensor", "achieved": round(achieved, 2), "peak": peaks["bf16_sust"],
                     "unit": "TFLOP/s", "frac": round(achieved / peaks["bf16_sust"], 4),
                     "traffic": tc_traffic_per_launch(w, per_kv),
                     "traffic_note": "bytes per average launch, scaled from profiles/k_attn_tc_traffic.json",
                     "kernel": "chunk attention (attend)", "peak_kind": f"bf16 dense sustained, {peaks['src']}",
                     "attend_ms_avg": round(avg_attend_t * 1e3, 3)},
        "write": {"GB/s": round(write_gbs, 1), "frac": round(write_gbs / peaks["hbm"], 4),
                  "bytes_per_launch": write_bytes, "us_avg": round(float(np.mean(write_t)) * 1e6, 2)},
    }
    if args.step_only:
        clocks = clk.summary()
        if clocks is not None:
            result["clocks"] = clocks
        if rank == 0:
            print(json.dumps(result), flush=True)
        if dist is not None:
            dist.destroy_process_group()
        return
    # the per-step copy a chronological store would make (the circular layout skips it)
    scratch = torch.empty(kvc.kvc_roll_scratch_bytes(cache.cfg), dtype=torch.uint8, device="cuda")
    if scratch.numel() > 0:
        kvc.kvc_roll_window(cache.handle, scratch)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        reps = 5
        a.record()
        for _ in range(reps):
            kvc.kvc_roll_window(cache.handle, scratch)
        b.record()
        b.synchronize()
        roll_t = a.elapsed_time(b) * 1e-3 / reps
        roll_bytes = 8 * w.batch * (w.window - w.sink - w.chunk) * row_bytes
        result["roll_comparator"] = {"us": round(roll_t * 1e6, 1), "GB/s": round(roll_bytes / roll_t / 1e9, 1),
                                     "bytes": roll_bytes, "x_write": round(roll_t / float(np.mean(write_t)), 2),
                                     "note": "clone + copy-back of the retained window, per chunk step; "
                                             "the circular layout does not do it"}
        del scratch
    clocks = clk.summary()
    if clocks is not None:
        result["clocks"] = clocks
    result["decode"] = decode_bench(kvc, peaks)
    result["decode"]["schedule_prefill_512_steps"] = decode_schedule_bench(kvc, peaks)
    result["cross_attention"] = cross_bench(kvc, peaks)
    result["dit_stream"] = dit_bench(kvc, peaks)
    result["tiny_ring"] = tiny_bench(kvc)
    result["next_rows"] = next_rows_bench(kvc, peaks, reps=10)
    # the RoPE write on this workload's chunk (1.53 GB moved), against the plain write
    table = wl.rope_table(w.window, w.head_dim).cuda()
    k0, v0 = inputs[0][1], inputs[0][2]
    cache.reset()
    cache.advance()
    t_plain = _events_time(lambda: cache.write(k0, v0), 5)
    t_rope = _events_time(lambda: cache.write_rope(k0, v0, table), 5)
    assert cache.get_error() == 0
    rope_bytes = write_bytes + w.chunk * (w.head_dim // 2) * 2 * 4
    result["next_rows"]["write_rope_multi_user_chunk"] = {
        "us": round(t_rope * 1e6, 2), "GB/s": round(rope_bytes / t_rope / 1e9, 1),
        "frac": round(rope_bytes / t_rope / 1e9 / peaks["hbm"], 4), "bytes": rope_bytes,
        "x_plain_write": round(t_rope / t_plain, 3), "plain_write_us": round(t_plain * 1e6, 2)}
    del table

    # end to end through the binding: host (pinned) inputs copied in, output read back.
    # A serving loop pipelines the copies: inputs of the coming chunks go up on a copy
    # stream while the compute stream writes and attends the current one, and each
    # output goes down on a second copy stream (inputs and outputs triple-buffered on the
    # device, so that uploads run two chunks ahead of the fill phase's short attends;
    # events order every reuse).  A step's last output goes down while the next step
    # computes; the timed region ends once every output is on the host.
    if True:
        host = [tuple(t.cpu().pin_memory() for t in s) for s in inputs]
        nslot = 3
        dev = [tuple(torch.empty_like(t) for t in inputs[0]) for _ in range(nslot)]
        dev_out = [torch.empty_like(out) for _ in range(nslot)]
        out_host = [torch.empty(out.shape, dtype=out.dtype).pin_memory() for _ in range(nslot)]
        h2d = sum(t.numel() * t.element_size() for t in host[0]) * w.n_chunks * w.rewrites
        d2h = out_host[0].numel() * out_host[0].element_size() * w.n_chunks * w.rewrites
        s_in, s_out = torch.cuda.Stream(), torch.cuda.Stream()
        comp = stream
        ev = lambda: torch.cuda.Event()
        used = [ev() for _ in range(nslot)]      # compute finished reading dev[slot]
        landed = [ev() for _ in range(nslot)]    # inputs of dev[slot] are on the device
        done = [ev() for _ in range(nslot)]      # dev_out[slot] written
        fetched = [ev() for _ in range(nslot)]   # dev_out[slot] copied to the host
        for e in used + fetched:
            e.record(comp)

        turn = [0]   # device slots in use order, counted across steps: a step's first chunks
                     # take the slots its predecessor freed first, not the ones its last
                     # (longest) attends still read

        def e2e_step():
            cache.reset(stream=comp)
            i = 0
            for c in range(w.n_chunks):
                cache.advance(stream=comp)
                for r in range(w.rewrites):
                    slot = turn[0] % nslot
                    turn[0] += 1
                    q, k, v = dev[slot]
                    hq, hk, hv = host[i % len(host)]
                    with torch.cuda.stream(s_in):
                        s_in.wait_event(used[slot])
                        q.copy_(hq, non_blocking=True)
                        k.copy_(hk, non_blocking=True)
                        v.copy_(hv, non_blocking=True)
                        landed[slot].record(s_in)
                    comp.wait_event(landed[slot])
                    comp.wait_event(fetched[slot])
                    cache.write(k, v, stream=comp)
                    cache.attend(q, dev_out[slot], stream=comp)
                    used[slot].record(comp)
                    done[slot].record(comp)
                    with torch.cuda.stream(s_out):
                        s_out.wait_event(done[slot])
                        out_host[slot].copy_(dev_out[slot], non_blocking=True)
                        fetched[slot].record(s_out)
                    i += 1

        e2e_step()
        comp.wait_stream(s_out)
        torch.cuda.synchronize()
        barrier(dist)
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record(comp)
        for _ in range(args.steps):
            e2e_step()
        comp.wait_stream(s_out)         # the timed region ends when the last output is on the host
        b.record(comp)
        torch.cuda.synchronize()
        barrier(dist)
        e2e_t = max_over_ranks(a.elapsed_time(b) * 1e-3, dist)
        # the host link alone, for reading the number above: one chunk's inputs up, one
        # output down, pinned buffers, nothing else running
        # (the best of five rounds: a shared host link varies from one moment to the next)
        hq, hk, hv = host[0]
        q, k, v = dev[0]
        up = down = 0.0
        for _ in range(5):
            a.record(comp)
            for _ in range(3):
                q.copy_(hq, non_blocking=True)
                k.copy_(hk, non_blocking=True)
                v.copy_(hv, non_blocking=True)
            b.record(comp)
            b.synchronize()
            up = max(up, 3 * sum(t.numel() * t.element_size() for t in host[0]) / (a.elapsed_time(b) * 1e-3) / 1e9)
            a.record(comp)
            for _ in range(3):
                out_host[0].copy_(dev_out[0], non_blocking=True)
            b.record(comp)
            b.synchronize()
            down = max(down, 3 * out_host[0].numel() * out_host[0].element_size() / (a.elapsed_time(b) * 1e-3) / 1e9)
        device_ms = elapsed / args.steps * 1e3
        copy_ms = (h2d / up + d2h / down) / 1e6
        e2e_ms = e2e_t / args.steps * 1e3
        result["e2e"] = {"value": round(world * step_flops * args.steps / e2e_t / 1e12, 2), "unit": "TFLOP/s",
                         "h2d_bytes_per_step": h2d, "d2h_bytes_per_step": d2h,
                         "ms_per_step": round(e2e_ms, 3),
                         "pipelining": "inputs up and outputs down on two copy streams, overlapping compute; "
                                       "three device slots, steps back to back",
                         "host_link_GB/s": {"h2d": round(up, 1), "d2h": round(down, 1)},
                         "overlap": {"device_ms_per_step": round(device_ms, 3),
                                     "copies_alone_ms_per_step": round(copy_ms, 3),
                                     "serial_ms": round(device_ms + copy_ms, 3),
                                     "ideal_ms": round(max(device_ms, copy_ms), 3),
                                     "hidden_frac": round((device_ms + copy_ms - e2e_ms) / min(device_ms, copy_ms), 4)}}
    if rank == 0:
        tf, dt, nrows = cpu_oracle_sample(w)
        result["cpu_baseline"] = {"value": round(tf, 6), "unit": "TFLOP/s", "cores": blas_threads(), "kind": "oracle",
                                  "sample": f"{nrows} query rows x {w.window} keys x 1 head (D={w.head_dim}) of a "
                                            f"full-window attend, fp64 NumPy, {dt:.1f} s"}
    if rank == 0:
        print(json.dumps(result), flush=True)
    if dist is not None:
        dist.destroy_process_group()


def next_rows_bench(kvc, peaks, reps):
    """The widening rows on the streaming DiT shapes (B2, Hkv 12, D 128, bf16, 4680-token
    chunks): the write with RoPE fused into K against the plain write of the same chunk
    (HBM: K and V read and written once, plus the (cos, sin) rows of the chunk's
    positions), the two-way LSE merge of one chunk's attention outputs (HBM: two partial
    outputs and LSEs read, one written), and attention with LSE output against plain
    attention over an 8192-slot store.  The write and the merge rotate over three input
    sets (each set 87-115 MB, so a set comes back only after more than L2's worth of other
    traffic)."""
    w = wl.DIT_STREAM
    B, H, Hkv, D, C = w.batch, w.heads, w.kv_heads, w.head_dim, w.chunk
    g = torch.Generator(device="cuda").manual_seed(w.seed)

    def time_it(fn):
        for _ in range(3):
            fn()
        a, b = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        a.record()
        for _ in range(reps):
            fn()
        b.record()
        b.synchronize()
        return a.elapsed_time(b) * 1e-3 / reps

    res = {}
    cache = kvc.KVCache(B, H, Hkv, D, torch.bfloat16, "circular", sink=w.sink, window=w.window, chunk=C)
    cache.advance()
    kv_sets = [(torch.randn(B, C, Hkv, D, device="cuda", generator=g).bfloat16(),
                torch.randn(B, C, Hkv, D, device="cuda", generator=g).bfloat16()) for _ in range(3)]
    table = wl.rope_table(w.window, D).cuda()
    turn = [0]

    def rotating(fn, sets):
        def call():
            fn(*sets[turn[0] % len(sets)])
            turn[0] += 1
        return call

    t_plain = time_it(rotating(lambda k, v: cache.write(k, v), kv_sets))
    t_rope = time_it(rotating(lambda k, v: cache.write_rope(k, v, table), kv_sets))
    assert cache.get_error() == 0
    k = kv_sets[0][0]
    nbytes = 2 * 2 * k.numel() * k.element_size() + C * (D // 2) * 2 * 4
    res["write_rope"] = {"us": round(t_rope * 1e6, 2), "GB/s": round(nbytes / t_rope / 1e9, 1),
                         "frac": round(nbytes / t_rope / 1e9 / peaks["hbm"], 4), "bytes": nbytes,
                         "x_plain_write": round(t_rope / t_plain, 3)}
    cache.close()

    rows = B * C * H
    merge_sets = [(torch.randn(rows, D, device="cuda", generator=g).bfloat16(),
                   torch.randn(rows, device="cuda", generator=g),
                   torch.randn(rows, D, device="cuda", generator=g).bfloat16(),
                   torch.randn(rows, device="cuda", generator=g),
                   torch.empty(rows, D, device="cuda", dtype=torch.bfloat16),
                   torch.empty(rows, device="cuda")) for _ in range(3)]
    t_merge = time_it(rotating(lambda oa, la, ob, lb, out, lo:
                               kvc.kvc_merge(torch.bfloat16, rows, D, oa, la, ob, lb, out, lo), merge_sets))
    nbytes = rows * (3 * D * 2 + 3 * 4)
    res["merge"] = {"rows": rows, "us": round(t_merge * 1e6, 2), "GB/s": round(nbytes / t_merge / 1e9, 1),
                    "frac": round(nbytes / t_merge / 1e9 / peaks["hbm"], 4), "bytes": nbytes}

    cap = 8192
    lin = kvc.KVCache(B, H, Hkv, D, torch.bfloat16, "linear", capacity=cap)
    lin.advance(n_tokens=cap)
    kk = torch.randn(B, cap, Hkv, D, device="cuda", generator=g).bfloat16()
    lin.write(kk, kk)
    q = torch.randn(B, C, H, D, device="cuda", generator=g).bfloat16()
    o = torch.empty_like(q)
    lse = torch.empty(B, C, H, dtype=torch.float32, device="cuda")
    t_att = time_it(lambda: lin.attend(q, o))
    t_lse = time_it(lambda: kvc.kvc_attend_lse(lin.handle, q, o, lse, C))
    assert lin.get_error() == 0
    flops = wl.attention_flops(C, cap, H, D) * B
    res["attend_lse"] = {"kv_len": cap, "ms": round(t_lse * 1e3, 4), "TFLOP/s": round(flops / t_lse / 1e12, 1),
                         "x_attend": round(t_lse / t_att, 4)}
    lin.close()
    return res


def workload_config(w):
    """The workload's shape, the same in both arms' JSON lines."""
    return {"workload": w.name, "batch": w.batch, "heads": w.heads, "kv_heads": w.kv_heads,
            "head_dim": w.head_dim, "chunk": w.chunk, "sink": w.sink, "window": w.window,
            "chunks_per_step": w.n_chunks, "rewrites": w.rewrites, "tflop_per_step": ring_flops(w)[0] / 1e12}


# ---------------------------------------------------------------------------
# reference arm: the CPU fp64 oracle, timed on the host cores
# ---------------------------------------------------------------------------
def reference(args):
    rank = int(os.environ.get("RANK", "0"))
    if rank != 0:
        return
    w = WORKLOADS[args.workload]
    for _ in range(args.warmup):
        cpu_oracle_sample(w, budget_s=min(1.0, args.budget_s))
    t_total, flops_total, rows_total = 0.0, 0.0, 0
    for _ in range(args.steps):
        tf, dt, nrows = cpu_oracle_sample(w, budget_s=args.budget_s)
        t_total += dt
        flops_total += tf * 1e12 * dt
        rows_total += nrows
    value = flops_total / t_total / 1e12
    cores = blas_threads()
    print(json.dumps({
        "impl": "reference", "metric": METRIC, "value": round(value, 6), "unit": "TFLOP/s", "n_gpus": 0,
        "steps": args.steps, "warmup": args.warmup, "ms_per_step": round(t_total / args.steps * 1e3, 1),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f64", "data": "synthetic",
        "config": {**workload_config(w), "l2": "host memory (fp64 oracle on the host cores)",
                   "parallelism": "host cores"},
        "cpu_baseline": {"value": round(value, 6), "unit": "TFLOP/s", "cores": cores, "kind": "oracle",
                         "sample": f"{rows_total} query rows x {w.window} keys x 1 head per run, fp64 NumPy"},
        "e2e": {"value": round(value, 6), "unit": "TFLOP/s", "h2d_bytes_per_step": 0, "d2h_bytes_per_step": 0},
    }), flush=True)


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=10)
    ap.add_argument("--warmup", type=int, default=3)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--workload", default=DEFAULT, choices=sorted(WORKLOADS))
    ap.add_argument("--budget-s", type=float, default=5.0,
                    help="seconds of CPU oracle work per step of the reference arm (a bounded sample)")
    ap.add_argument("--pool", type=int, default=8,
                    help="distinct (q, k, v) input sets, reused cyclically over the chunks")
    ap.add_argument("--cross-only", action="store_true",
                    help="time only the ragged cross-attention attends and print them (profiling aid)")
    ap.add_argument("--cross-lq", type=int, default=None,
                    help="padded query count of the cross-attention timing (default: the full workload)")
    ap.add_argument("--step-only", action="store_true",
                    help="time only the workload step (no extra sections): a profiling aid")
    ap.add_argument("--decode-only", action="store_true",
                    help="time only the decode attends and steps, and print them (profiling aid)")
    ap.add_argument("--next-rows", action="store_true",
                    help="time only the RoPE write, the LSE merge and attention with LSE output, and print them")
    args = ap.parse_args()
    if args.next_rows:
        from diffusion_serving_gb300 import kvc
        print(json.dumps({"next_rows": next_rows_bench(kvc, load_peaks(), reps=max(args.steps, 5))}))
        return
    if args.decode_only:
        from diffusion_serving_gb300 import kvc
        print(json.dumps({"decode": decode_bench(kvc, load_peaks())}))
        return
    if args.cross_only:
        from diffusion_serving_gb300 import kvc
        print(json.dumps({"cross_attention": cross_bench(kvc, load_peaks(), reps=args.steps, lq=args.cross_lq)}))
        return
    if args.impl == "reference":
        reference(args)
    else:
        ours(args)


if __name__ == "__main__":
    main()
