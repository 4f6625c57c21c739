#!/usr/bin/env python
"""Benchmark of the KIVI hot path on one GB300.

Main line (the JSON ``value``): the Llama-3-8B-shaped decode step -- batch 8,
32 query / 8 KV heads, head_dim 128, fp16, 2-bit, group 32, residual 32,
context 4096 -- one step = append one token (flushing when the residual
fills) + fused dequantize decode attention.  ``value`` is the decode
attention's effective HBM bandwidth: algorithmic bytes (packed codes +
scale/zero + fp16 residual + q/out) over the attention time.  Inputs are
larger than L2: every timed workload rotates over enough identical cache
replicas that the one a step reads was last touched more than 1.5 L2 sizes
of reads earlier (as in a model, where the other layers' weights and caches
pass through L2 between two calls of one layer).  Timing: the K launches of
a timed region are captured in one CUDA graph and CUDA events bracket one
replay of it (a decode loop runs this way; events around every launch add
about 5 us per launch on this GPU, reported beside it as
``per_launch_events``).  ``ms_per_step`` and ``tokens_per_s`` time the
one-call decode step (append, then the attention as a programmatic
dependent).  The same line carries the prefill quantizer on the 32k-token
bf16 workload (2- and 4-bit), 3-, 4- and 8-bit attention, the 131k-token
long-context attention and the 2048+512-step streaming decode.

``--impl reference`` times the CPU oracle (the plain C implementation the
tests check against) on the same workload, its (batch, KV head) units split
over one process per host core; ``cpu_baseline`` carries the oracle
single-threaded on batch element 0 and, under ``multicore``, on every core.
"""
from __future__ import annotations

import argparse
import hashlib
import json
import os
import queue
import subprocess
import sys
import threading
import time

import numpy as np

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

METRIC = "2-bit decode-attn effective HBM GB/s (% of peak), tokens/s; quantize GB/s"
WORKLOAD = ("llama3_8b_decode: batch 8, 32 q heads / 8 kv heads, head_dim 128, fp16, "
            "2-bit, group 32, residual 32, context 4096; step = append 1 token + decode attention")
G = 32
L2_BYTES = 129 << 20     # GB300 L2
SPIN_CYCLES = 200_000    # ~0.1 ms GPU spin before a timed step: covers the host enqueue


def n_replicas(cache_bytes: int) -> int:
    """Cache replicas to rotate so that a step's inputs are out of L2."""
    return max(2, -(-int(1.5 * L2_BYTES) // int(cache_bytes)))


# ------------------------------------------------------------------ bytes

def nq(l, R):
    return l - l % R, max(l - R, 0)


def attn_bytes(B, Hkv, Hq, D, l, R, bits, q_bytes=2):
    """Algorithmic bytes of one decode attention: packed codes, fp16 scale/zero,
    fp16 residual rows, the query and the output."""
    nqk, nqv = nq(l, R)
    unit = (nqk * D * bits // 8 + (nqk // G) * D * 4 + (l - nqk) * D * 2
            + nqv * D * bits // 8 + nqv * (D // G) * 4 + (l - nqv) * D * 2)
    return B * Hkv * unit + 2 * B * Hq * D * q_bytes


def append_bytes(B, Hkv, D, t, R, bits, in_bytes=2):
    """Algorithmic bytes of appending token t: read k, v; write two ring rows;
    quantize the value row leaving the window; every R steps the key ring."""
    unit = 2 * D * in_bytes + 2 * D * 2
    if t >= R:
        unit += D * 2 + D * bits // 8 + (D // G) * 4
    if (t + 1) % R == 0:
        unit += R * D * 2 + R * D * bits // 8 + (R // G) * D * 4
    return B * Hkv * unit


def prefill_bytes(B, Hkv, D, T, R, bits, in_bytes):
    """Read K and V once; write codes, scale/zero and the residual rows."""
    nqk, nqv = nq(T, R)
    wr = (nqk * D * bits // 8 + (nqk // G) * D * 4 + nqv * D * bits // 8 + nqv * (D // G) * 4
          + (T - nqk) * D * 2 + (T - nqv) * D * 2)
    return B * Hkv * (2 * T * D * in_bytes + wr)


def peak_hbm():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    try:
        with open(p) as f:
            return float(json.load(f)["hbm_gbs"]), "measured"
    except Exception:
        return 6800.0, "fallback"


def kernel_source_hash() -> str:
    """sha256 of the attention kernel's sources (the kernel and the tile
    layout) with comments and whitespace removed: a comment edit keeps a
    recorded capture valid, a code edit does not."""
    import re
    csrc = os.path.join(ROOT, "bit_kv_cache_kivi_gb300", "csrc")
    h = hashlib.sha256()
    for name in ("attention.cu", "kivi_internal.cuh"):
        src = open(os.path.join(csrc, name)).read()
        src = re.sub(r"/\*.*?\*/", " ", src, flags=re.S)  # block comments
        src = re.sub(r"//[^\n]*", " ", src)                # line comments
        h.update(" ".join(src.split()).encode())
    return h.hexdigest()


def kernel_traffic():
    """Per-launch DRAM bytes of the attention kernel from a committed ncu
    capture, valid only while the kernel's code is unchanged."""
    p = os.path.join(ROOT, "profiles", "attention_traffic.json")
    try:
        with open(p) as f:
            rec = json.load(f)
        return rec["bytes_per_launch"] if rec.get("source_sha256") == kernel_source_hash() else None
    except Exception:
        return None


# ------------------------------------------------------------------ clocks

class ClockSampler:
    """nvidia-smi samples (200 ms) while the GPU work runs."""

    Q = ("clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.hw_slowdown,"
         "clocks_event_reasons.hw_thermal_slowdown,clocks_event_reasons.sw_thermal_slowdown,"
         "clocks_event_reasons.sw_power_cap")

    def __init__(self, index=0):
        self.rows, self.proc = [], None
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(index), f"--query-gpu={self.Q}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
            self.t = threading.Thread(target=self._read, daemon=True)
            self.t.start()
        except Exception:
            self.proc = None

    def _read(self):
        for line in self.proc.stdout:
            self.rows.append([x.strip() for x in line.split(",")])

    def stop(self):
        if self.proc is None:
            return {"sm_mhz": None, "sm_max_mhz": None, "reasons": ["nvidia-smi unavailable"]}
        self.proc.terminate()
        try:
            self.proc.wait(timeout=5)
        except Exception:
            self.proc.kill()
        self.t.join(timeout=2)
        sm, mx, reasons = [], [], set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in self.rows:
            try:
                sm.append(float(r[0]))
                mx.append(float(r[1]))
                for n, v in zip(names, r[3:7]):
                    if v.lower() == "active":
                        reasons.add(n)
            except (ValueError, IndexError):
                continue
        return {"sm_mhz": float(np.median(sm)) if sm else None,
                "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


# ------------------------------------------------------------------ GPU arm

def run_gpu(args):
    import torch
    from bit_kv_cache_kivi_gb300 import build, workloads as W
    from bit_kv_cache_kivi_gb300.kivi import KiviCache

    build.build()
    torch.cuda.set_device(0)
    dev = torch.device("cuda", 0)
    stream = torch.cuda.current_stream()
    peak, peak_src = peak_hbm()
    clocks = ClockSampler(0)

    def ev():
        return torch.cuda.Event(enable_timing=True)

    def fence():
        """Both sides of a timed region: the device idle and, under N ranks,
        every rank at the same point."""
        torch.cuda.synchronize()
        import torch.distributed as dist
        if dist.is_available() and dist.is_initialized():
            dist.barrier()

    # ---------------- main: decode step at context 4096 (+ a rewind window)
    K, Wm = args.steps, args.warmup
    window = 256
    wl = W.llama3_8b_decode(steps=window)
    B, Hq, Hkv, D, R, T0 = wl.B, wl.Hq, wl.Hkv, wl.D, wl.R, wl.T
    def new_cache():
        return KiviCache(batch=B, n_kv_heads=Hkv, n_q_heads=Hq, max_tokens=T0 + window, bits=2,
                         residual=R)
    probe = new_cache()
    probe_bytes = sum(t.numel() * t.element_size() for t in probe.state_views().values())
    n_rep = n_replicas(probe_bytes)
    caches = [probe] + [new_cache() for _ in range(n_rep - 1)]
    k0, v0 = W.to_torch(wl.k, "f16", dev), W.to_torch(wl.v, "f16", dev)
    kn, vn = W.to_torch(wl.k_new, "f16", dev), W.to_torch(wl.v_new, "f16", dev)
    q = W.to_torch(wl.q, "f16", dev)
    out = torch.empty_like(q)

    def rewind_if_needed(c, room=1):
        """Reset a replica that cannot take `room` more appends (outside any
        timed region)."""
        if c.length - T0 + room > window:
            c.reset()
            c.prefill(k0, v0)

    for c in caches:
        c.prefill(k0, v0)
    for step in range(Wm):  # eager warm-up: both call paths
        c = caches[step % n_rep]
        rewind_if_needed(c, 2)
        i = c.length - T0
        c.append(kn[i], vn[i])
        c.attention(q, out)
        i += 1
        c.step(kn[i], vn[i], q, out)
    torch.cuda.synchronize()

    # ---------------- timed (value): one replay of a CUDA graph holding K
    # decode attention launches, launch i on replica i mod n_rep.  The
    # launches may overlap (kivi_set_attention_overlap: no launch writes
    # another's q or cache, so each starts as the one before it drains and
    # waits for it only before its first write); the same graph without the
    # overlap is timed beside it.
    per_rep = -(-K // n_rep)
    for c in caches:
        rewind_if_needed(c, 2 * per_rep + 1)

    outs = [torch.empty_like(q) for _ in range(K)]  # overlapping calls write distinct outputs

    def time_attention_graph(overlap):
        for c in caches:
            c.set_overlap(overlap)
        g = torch.cuda.CUDAGraph()
        with torch.cuda.graph(g):
            for i in range(K):
                caches[i % n_rep].attention(q, outs[i])
        g.replay()  # warm-up replay (attention leaves the caches unchanged)
        fence()
        e0, e1 = ev(), ev()
        e0.record(stream)
        g.replay()
        e1.record(stream)
        fence()
        for c in caches:
            c.set_overlap(False)
        del g
        return e0.elapsed_time(e1) * 1e-3 / K

    ctx_a = [caches[i % n_rep].length for i in range(K)]
    t_att_serial = time_attention_graph(False)
    t_att_graph = time_attention_graph(True)
    att_b = np.array([attn_bytes(B, Hkv, Hq, D, t, R, 2) for t in ctx_a], float)
    attn_gbs = att_b.sum() / (t_att_graph * K) / 1e9

    # ---------------- timed (steps): the one-call decode step (append, then
    # the attention as a programmatic dependent of the append), K steps per
    # graph, launch i on replica i mod n_rep; a first graph of K steps is
    # replayed as warm-up, a second one of the next K steps is timed
    def capture_steps():
        g, ctx = torch.cuda.CUDAGraph(), []
        with torch.cuda.graph(g):
            for i in range(K):
                c = caches[i % n_rep]
                j = c.length - T0
                ctx.append(c.length)
                c.step(kn[j], vn[j], q, out)
        return g, ctx

    gB, _ = capture_steps()
    gB.replay()
    torch.cuda.synchronize()
    del gB
    gB, ctx_b = capture_steps()
    fence()
    e0, e1 = ev(), ev()
    e0.record(stream)
    gB.replay()
    e1.record(stream)
    fence()
    step_graph_s = e0.elapsed_time(e1) * 1e-3 / K
    tokens_per_s = B / step_graph_s
    del gB

    # ---------------- timed (flush window): 32 consecutive one-call steps on
    # every replica from context 4096, so that each replica appends the token
    # that completes a residual of 32 keys and quantizes it (the K flush of
    # Algorithm 1 at l = 4128) inside the timed region; one graph of
    # 32 x n_rep steps, replica-interleaved, warmed up by a first pass over
    # the same lengths
    def flush_window():
        for c in caches:
            c.reset()
            c.prefill(k0, v0)
        g, ctx = torch.cuda.CUDAGraph(), []
        with torch.cuda.graph(g):
            for i in range(32):
                for c in caches:
                    ctx.append(c.length)
                    c.step(kn[i], vn[i], q, out)
        return g, ctx

    gF, _ = flush_window()
    gF.replay()
    torch.cuda.synchronize()
    del gF
    gF, ctx_f = flush_window()
    fence()
    e0, e1 = ev(), ev()
    e0.record(stream)
    gF.replay()
    e1.record(stream)
    fence()
    flush_step_s = e0.elapsed_time(e1) * 1e-3 / len(ctx_f)
    del gF
    assert min(ctx_f) % 32 == 0 and max(ctx_f) - min(ctx_f) == 31  # each replica crosses one K flush

    # ---------------- per-launch event timing (secondary): append and
    # attention as separate calls, events around each launch and a GPU spin
    # before each step so that host latency never falls inside the events
    recs = []
    for step in range(K):
        c = caches[step % n_rep]
        rewind_if_needed(c)
        i = c.length - T0
        t = c.length
        torch.cuda._sleep(SPIN_CYCLES)
        e0, e1, e2 = ev(), ev(), ev()
        e0.record(stream)
        c.append(kn[i], vn[i])
        e1.record(stream)
        c.attention(q, out)
        e2.record(stream)
        recs.append((t, e0, e1, e2))
    torch.cuda.synchronize()
    t_app = np.array([a.elapsed_time(b) for _, a, b, _ in recs]) * 1e-3
    t_att = np.array([b.elapsed_time(c) for _, _, b, c in recs]) * 1e-3
    app_b = np.array([append_bytes(B, Hkv, D, t, R, 2) for t, *_ in recs], float)

    # ---------------- end to end: the step's k, v and q in pinned host memory,
    # read by the kernels directly (the library accepts page-locked host
    # buffers; on a GB300 node they are reached over NVLink-C2C), and the
    # output written to pinned host memory; a host sync per step
    kh = torch.empty((B, Hkv, D), dtype=torch.float16).pin_memory()
    vh = torch.empty_like(kh).pin_memory()
    qh = q.cpu().pin_memory()
    oh = torch.empty_like(qh).pin_memory()
    e2e = []
    for step in range(K):
        c = caches[step % n_rep]
        rewind_if_needed(c)
        i = c.length - T0
        t = c.length
        kh.copy_(kn[i].cpu())  # the host producing this step's input
        vh.copy_(vn[i].cpu())
        e0, e1 = ev(), ev()
        e0.record(stream)
        c.step(kh, vh, qh, oh)
        e1.record(stream)
        e1.synchronize()
        e2e.append((t, e0.elapsed_time(e1) * 1e-3))
    e2e_bytes = sum(attn_bytes(B, Hkv, Hq, D, t + 1, R, 2) for t, _ in e2e)
    e2e_gbs = e2e_bytes / sum(s for _, s in e2e) / 1e9

    result = {
        "metric": METRIC, "value": round(attn_gbs, 2), "unit": "GB/s", "n_gpus": 1,
        "steps": K, "warmup": Wm, "ms_per_step": round(step_graph_s * 1e3, 5),
        "flush_window_ms_per_step": round(flush_step_s * 1e3, 5),
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None,
        "dtype": "f16 (fp16 inputs and outputs; fp16 MMA operands, the key factors as hi/lo pairs; "
                 "fp32 accumulation and softmax)",
        "data": "synthetic (seeded N(0,1) K/V with 4 outlier channels x5 per KV head)",
        "config": {"workload": WORKLOAD,
                   "l2": f"inputs larger than L2: {n_rep} cache replicas rotated "
                         f"({n_rep} x {probe_bytes / 2**20:.0f} MiB), no flush",
                   "context": [int(min(ctx_a + ctx_b)), int(max(ctx_a + ctx_b)) + 1],
                   "timing": "CUDA events around one replay of a CUDA graph of K launches "
                             "(value: K attention launches, each overlapping the one before it "
                             "(kivi_set_attention_overlap), the same without the overlap beside it; "
                             "ms_per_step: K decode steps)"},
        "pct_of_peak": round(100 * attn_gbs / peak, 2),
        "tokens_per_s": round(tokens_per_s, 1),
        "flush_window_tokens_per_s": round(B / flush_step_s, 1),
        "step_us": round(step_graph_s * 1e6, 3),
        "attention_us": round(t_att_graph * 1e6, 3),
        "attention_us_no_overlap": round(t_att_serial * 1e6, 3),
        "per_launch_events": {
            "attention_us": round(float(t_att.mean()) * 1e6, 3),
            "append_us": round(float(t_app.mean()) * 1e6, 3),
            "append_gbs": round(app_b.sum() / t_app.sum() / 1e9, 2),
            "note": "events around every launch add about 5 us per launch on this GPU"},
        # timed regions: the attention graph twice (with and without the
        # overlap), the step graph (2 launches a step), the flush window (2
        # launches a step) and the event-timed steps (2 launches each)
        "gpu_launches": 6 * K + 2 * 32 * n_rep,
    }
    achieved = float(att_b.mean() / t_att_graph / 1e9)
    result["roofline"] = {"kernel": "attn_kernel<2> (fused split-combine)", "bound": "hbm",
                          "achieved": round(achieved, 2), "peak": peak, "unit": "GB/s",
                          "frac": round(achieved / peak, 4), "traffic": kernel_traffic(),
                          "peak_source": f"{peak_src} (MEASURED_PEAKS.json hbm_gbs)"
                          if peak_src == "measured" else "fallback 6800 GB/s",
                          "algorithmic_bytes_per_launch": int(att_b.mean())}
    result["_attn"] = (float(att_b.sum()), t_att_graph * K)  # for the whole-job numbers of N ranks
    result["e2e"] = {"value": round(e2e_gbs, 2), "unit": "GB/s",
                     "h2d_bytes_per_step": int(kh.numel() * 2 * 2 + qh.numel() * 2),
                     "d2h_bytes_per_step": int(oh.numel() * 2)}

    if not args.main_only and args.only is None:
        result["workloads"] = extra_workloads(args, torch, W, KiviCache, dev, stream, ev, peak)
        for bits in (2, 4):
            w = result["workloads"].get(f"prefill_quantize_{bits}bit")
            if w:
                result[f"quantize_{bits}bit_gbs"] = w["gbs"]
                result[f"quantize_{bits}bit_pct"] = w["pct_of_peak"]
    result["clocks"] = clocks.stop()
    del caches, probe
    return result


def graph_per_launch(torch, stream, ev, calls, overlap=()):
    """Per-launch time of `calls` (functions that each enqueue one library
    call on the current stream, replayable: they leave the same state each
    time): captured in one CUDA graph, replayed once as warm-up, then one
    replay timed with CUDA events on `stream`.  The caches in `overlap` let
    their attention launches overlap the launch before them while captured."""
    for c in overlap:
        c.set_overlap(True)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for f in calls:
            f()
    g.replay()
    torch.cuda.synchronize()
    e0, e1 = ev(), ev()
    e0.record(stream)
    g.replay()
    e1.record(stream)
    torch.cuda.synchronize()
    t = e0.elapsed_time(e1) * 1e-3 / len(calls)
    del g
    for c in overlap:
        c.set_overlap(False)
    return t


def plan_splits(c):
    """Splits per unit of the launches graph_per_launch times (overlapped),
    and of ordinary launches."""
    c.set_overlap(True)
    ov = c.splits()
    c.set_overlap(False)
    return {"splits": ov, "splits_ordinary": c.splits()}


def extra_workloads(args, torch, W, KiviCache, dev, stream, ev, peak, which=None):
    res = {}
    want = (lambda n: which is None or which == n)
    # ---- prefill quantizer: batch 4, 8 KV heads, 32768 bf16 tokens
    for bits in ((2, 4) if want("quantize") else ()):
        wl = W.prefill_quantize(bits)
        c = KiviCache(batch=wl.B, n_kv_heads=wl.Hkv, n_q_heads=wl.Hq, max_tokens=wl.T,
                      bits=bits, residual=wl.R)
        k, v = W.to_torch(wl.k, "bf16", dev), W.to_torch(wl.v, "bf16", dev)
        times = []
        for rep in range(3 + args.quant_reps):
            c.reset()
            e0, e1 = ev(), ev()
            e0.record(stream)
            c.prefill(k, v)
            e1.record(stream)
            e1.synchronize()
            if rep >= 3:
                times.append(e0.elapsed_time(e1) * 1e-3)
        nbytes = prefill_bytes(wl.B, wl.Hkv, wl.D, wl.T, wl.R, bits, 2)

        def prefill_once(c=c, k=k, v=v):
            c.reset()
            c.prefill(k, v)
        tg = graph_per_launch(torch, stream, ev, [prefill_once] * args.quant_reps)
        gbs = nbytes / tg / 1e9
        res[f"prefill_quantize_{bits}bit"] = {
            "what": "batch 4, 8 KV heads, 32768 bf16 tokens, V spikes; one quantize/pack launch "
                    "(inputs 537 MB, larger than L2); graph replay of back-to-back launches",
            "gbs": round(gbs, 2), "pct_of_peak": round(100 * gbs / peak, 2),
            "us": round(tg * 1e6, 2), "us_per_launch_events": round(float(np.mean(times)) * 1e6, 2),
            "bytes": nbytes}
        del c, k, v
    if want("attn3"):
        res.update(attention_bits(args, torch, W, KiviCache, dev, stream, ev, peak, 3))
    if want("attn4"):
        res.update(attention_bits(args, torch, W, KiviCache, dev, stream, ev, peak, 4))
    if want("attn8"):
        res.update(attention_bits(args, torch, W, KiviCache, dev, stream, ev, peak, 8))
    if want("outliers"):
        res.update(attention_bits(args, torch, W, KiviCache, dev, stream, ev, peak, 2, outliers=2))
    if want("long"):
        res.update(long_context(args, torch, W, KiviCache, dev, stream, ev, peak))
    if want("streaming"):
        res.update(streaming(args, torch, W, KiviCache, dev, stream, ev, peak))
    return res


def attention_bits(args, torch, W, KiviCache, dev, stream, ev, peak, bits, outliers=0):
    """Decode attention of a 2-, 4- or 8-bit cache on the Llama-3-8B shape
    (context 4097), optionally with fp16 outlier key channels."""
    res = {}
    wl = W.llama3_8b_decode(bits=bits)
    k, v = W.to_torch(wl.k, "f16", dev), W.to_torch(wl.v, "f16", dev)

    def new_cache():
        c = KiviCache(batch=wl.B, n_kv_heads=wl.Hkv, n_q_heads=wl.Hq, max_tokens=wl.capacity,
                      bits=bits, residual=wl.R, outliers=outliers)
        c.prefill(k, v)
        c.append(W.to_torch(wl.k_new[0], "f16", dev), W.to_torch(wl.v_new[0], "f16", dev))
        return c
    c0 = new_cache()
    n_rep = n_replicas(sum(t.numel() * t.element_size() for t in c0.state_views().values()))
    caches = [c0] + [new_cache() for _ in range(n_rep - 1)]
    del k, v
    q = W.to_torch(wl.q, "f16", dev)
    out = torch.empty_like(q)
    for i in range(3):
        caches[i % n_rep].attention(q, out)
    recs = []
    for i in range(args.attn_reps):
        torch.cuda._sleep(SPIN_CYCLES)
        e0, e1 = ev(), ev()
        e0.record(stream)
        caches[i % n_rep].attention(q, out)
        e1.record(stream)
        recs.append((e0, e1))
    torch.cuda.synchronize()
    times = [a.elapsed_time(b) * 1e-3 for a, b in recs]
    tg = graph_per_launch(torch, stream, ev,
                          [lambda c=caches[i % n_rep], o=torch.empty_like(q): c.attention(q, o) for i in range(args.attn_reps)],
                          overlap=caches)
    nbytes = attn_bytes(wl.B, wl.Hkv, wl.Hq, wl.D, wl.T + 1, wl.R, bits)
    if outliers:  # the outlier blocks of the quantized key groups
        nbytes += wl.B * wl.Hkv * (nq(wl.T + 1, wl.R)[0] // G) * (16 + 64 * outliers)
    gbs = nbytes / tg / 1e9
    key = f"attention_{bits}bit_llama3_8b" + (f"_outliers{outliers}" if outliers else "")
    res[key] = {
        "what": f"{bits}-bit decode attention" + (f" with {outliers} fp16 outlier key channels per group"
                                                   if outliers else "")
                + f", batch 8, 32/8 heads, context 4097, R 32; {n_rep} cache replicas rotated; graph replay",
        **plan_splits(caches[0]), "gbs": round(gbs, 2), "pct_of_peak": round(100 * gbs / peak, 2),
        "us": round(tg * 1e6, 2), "us_per_launch_events": round(float(np.mean(times)) * 1e6, 2),
        "bytes": nbytes}
    del caches, c0
    return res


def long_context(args, torch, W, KiviCache, dev, stream, ev, peak):
    res = {}
    # ---- long context attention: batch 1, 32/8 heads, 131072 tokens, R = 128
    wl = W.long_context()
    k, v = W.to_torch(wl.k, "f16", dev), W.to_torch(wl.v, "f16", dev)
    c0 = KiviCache(batch=wl.B, n_kv_heads=wl.Hkv, n_q_heads=wl.Hq, max_tokens=wl.T, bits=2,
                   residual=wl.R)
    n_rep = n_replicas(sum(t.numel() * t.element_size() for t in c0.state_views().values()))
    caches = [c0] + [KiviCache(batch=wl.B, n_kv_heads=wl.Hkv, n_q_heads=wl.Hq, max_tokens=wl.T,
                               bits=2, residual=wl.R) for _ in range(n_rep - 1)]
    for c in caches:
        c.prefill(k, v)
    del k, v
    q = W.to_torch(wl.q, "f16", dev)
    out = torch.empty_like(q)
    for i in range(3):
        caches[i % n_rep].attention(q, out)
    recs = []
    for i in range(args.attn_reps):
        torch.cuda._sleep(SPIN_CYCLES)
        e0, e1 = ev(), ev()
        e0.record(stream)
        caches[i % n_rep].attention(q, out)
        e1.record(stream)
        recs.append((e0, e1))
    torch.cuda.synchronize()
    times = [a.elapsed_time(b) * 1e-3 for a, b in recs]
    tg = graph_per_launch(torch, stream, ev,
                          [lambda c=caches[i % n_rep], o=torch.empty_like(q): c.attention(q, o) for i in range(args.attn_reps)],
                          overlap=caches)
    nbytes = attn_bytes(wl.B, wl.Hkv, wl.Hq, wl.D, wl.T, wl.R, 2)
    gbs = nbytes / tg / 1e9
    res["long_context_attention"] = {
        "what": "batch 1, 32/8 heads, context 131072, R 128; split-K decode attention; "
                f"{n_rep} cache replicas rotated; graph replay",
        **plan_splits(caches[0]), "gbs": round(gbs, 2), "pct_of_peak": round(100 * gbs / peak, 2),
        "us": round(tg * 1e6, 2), "us_per_launch_events": round(float(np.mean(times)) * 1e6, 2),
        "bytes": nbytes}
    del caches, c0
    return res


def streaming(args, torch, W, KiviCache, dev, stream, ev, peak):
    res = {}
    # ---- streaming decode: batch 64, 28/4 heads, 2048 prefill + 512 steps,
    # run on every replica (steps interleaved across replicas)
    wl = W.streaming()
    k, v = W.to_torch(wl.k, "f16", dev), W.to_torch(wl.v, "f16", dev)
    c0 = KiviCache(batch=wl.B, n_kv_heads=wl.Hkv, n_q_heads=wl.Hq, max_tokens=wl.capacity,
                   bits=2, residual=wl.R)
    n_rep = n_replicas(sum(t.numel() * t.element_size() for t in c0.state_views().values()))
    caches = [c0] + [KiviCache(batch=wl.B, n_kv_heads=wl.Hkv, n_q_heads=wl.Hq,
                               max_tokens=wl.capacity, bits=2, residual=wl.R)
                     for _ in range(n_rep - 1)]
    for c in caches:
        c.prefill(k, v)
    del k, v
    kn, vn = W.to_torch(wl.k_new, "f16", dev), W.to_torch(wl.v_new, "f16", dev)
    q = W.to_torch(wl.q, "f16", dev)
    out = torch.empty_like(q)
    # every step of every replica once, in order, through the one-call decode
    # step; chunks of steps captured in CUDA graphs, each replayed once, timed
    chunks = []
    for i0 in range(0, wl.steps, 64):
        g, ctx = torch.cuda.CUDAGraph(), []
        with torch.cuda.graph(g):
            for i in range(i0, min(i0 + 64, wl.steps)):
                for c in caches:
                    ctx.append(c.length)
                    c.step(kn[i], vn[i], q, out)
        e0, e1 = ev(), ev()
        e0.record(stream)
        g.replay()
        e1.record(stream)
        torch.cuda.synchronize()
        chunks.append((ctx, e0.elapsed_time(e1) * 1e-3))
        del g
    t_steps = sum(t for _, t in chunks)
    n_steps = sum(len(ctx) for ctx, _ in chunks)
    # the attention alone at the final context (2560 tokens), replicas rotated
    ta = graph_per_launch(torch, stream, ev,
                          [lambda c=caches[i % n_rep], o=torch.empty_like(q): c.attention(q, o) for i in range(4 * n_rep)],
                          overlap=caches)
    ab = attn_bytes(wl.B, wl.Hkv, wl.Hq, wl.D, caches[0].length, wl.R, 2)
    res["streaming_decode"] = {
        "what": "batch 64, 28/4 heads (GQA 7), 2048 prefill then 512 decode steps (append + "
                f"attention, one-call step) on each of {n_rep} cache replicas rotated step by step; "
                "graph replays",
        "tokens_per_s": round(wl.B * n_steps / t_steps, 1),
        "ms_per_step": round(t_steps / n_steps * 1e3, 5),
        "attention_gbs_at_2560": round(ab / ta / 1e9, 2),
        "pct_of_peak_at_2560": round(100 * ab / ta / 1e9 / peak, 2),
        "attention_us_at_2560": round(ta * 1e6, 2)}
    del caches, c0
    return res


def streaming_attention(args, torch, W, KiviCache, dev, stream, ev, peak):
    """The streaming workload's attention alone at its final context: batch
    64, 28/4 heads (GQA 7), the 2048 + 512 tokens prefilled at once (the same
    cache as the 512 steps leave, see test_streaming_2048_plus_512); for
    profiling captures of the launch the streaming line times."""
    wl = W.streaming()
    k = np.ascontiguousarray(np.concatenate([wl.k, wl.k_new.transpose(1, 2, 0, 3)], axis=2))
    v = np.ascontiguousarray(np.concatenate([wl.v, wl.v_new.transpose(1, 2, 0, 3)], axis=2))
    T = k.shape[2]
    kd, vd = W.to_torch(k, "f16", dev), W.to_torch(v, "f16", dev)

    def new_cache():
        c = KiviCache(batch=wl.B, n_kv_heads=wl.Hkv, n_q_heads=wl.Hq, max_tokens=wl.capacity, bits=2,
                      residual=wl.R)
        c.prefill(kd, vd)
        return c
    c0 = new_cache()
    n_rep = n_replicas(sum(t.numel() * t.element_size() for t in c0.state_views().values()))
    caches = [c0] + [new_cache() for _ in range(n_rep - 1)]
    q = W.to_torch(wl.q, "f16", dev)
    out = torch.empty_like(q)
    for i in range(3):
        caches[i % n_rep].attention(q, out)
    torch.cuda.synchronize()
    tg = graph_per_launch(torch, stream, ev,
                          [lambda c=caches[i % n_rep], o=torch.empty_like(q): c.attention(q, o) for i in range(args.attn_reps)],
                          overlap=caches)
    nbytes = attn_bytes(wl.B, wl.Hkv, wl.Hq, wl.D, T, wl.R, 2)
    gbs = nbytes / tg / 1e9
    return {"streaming_attention_2560": {
        "what": f"batch 64, 28/4 heads (GQA 7), context {T} prefilled, R 32; {n_rep} cache replicas "
                "rotated; graph replay",
        "gbs": round(gbs, 2), "pct_of_peak": round(100 * gbs / peak, 2), "us": round(tg * 1e6, 2),
        "bytes": nbytes}}


def append_window(torch, W, KiviCache, dev, stream, ev):
    """The decode append alone on the Llama-3-8B decode shape: 32 appends
    from context 4096 on one cache, eager, each followed by the attention;
    the last append completes a 32-token key residual and quantizes it (the
    K flush of Algorithm 1).  Events around every append, with a GPU spin
    before it so that host latency stays outside them.  Launch order: the
    prefill, then 32 x (append_kernel, attn_kernel), so that the 31st append
    is a plain step and the 32nd the flush step."""
    wl = W.llama3_8b_decode(steps=32)
    B, Hkv, D, R, T0 = wl.B, wl.Hkv, wl.D, wl.R, wl.T
    c = KiviCache(batch=B, n_kv_heads=Hkv, n_q_heads=wl.Hq, max_tokens=T0 + 32, bits=2, residual=R)
    c.prefill(W.to_torch(wl.k, "f16", dev), W.to_torch(wl.v, "f16", dev))
    kn, vn = W.to_torch(wl.k_new, "f16", dev), W.to_torch(wl.v_new, "f16", dev)
    q = W.to_torch(wl.q, "f16", dev)
    out = torch.empty_like(q)
    recs = []
    for i in range(32):
        t = c.length
        torch.cuda._sleep(SPIN_CYCLES)
        e0, e1 = ev(), ev()
        e0.record(stream)
        c.append(kn[i], vn[i])
        e1.record(stream)
        c.attention(q, out)
        recs.append((t, e0, e1))
    torch.cuda.synchronize()
    us = {t: a.elapsed_time(b) * 1e3 for t, a, b in recs}
    flush_t = [t for t in us if (t + 1) % R == 0]
    assert len(flush_t) == 1 and flush_t[0] == T0 + 31
    plain = np.array([us[t] for t in us if t not in flush_t])
    tf = flush_t[0]
    return {"append_window": {
        "workload": "llama3_8b_decode append: batch 8, 8 kv heads, 2-bit, residual 32; "
                    "32 appends from context 4096, the last one flushing the key residual",
        "plain_us_median": round(float(np.median(plain)), 3),
        "plain_bytes": append_bytes(B, Hkv, D, T0 + 1, R, 2),
        "plain_gbs": round(append_bytes(B, Hkv, D, T0 + 1, R, 2) / (np.median(plain) * 1e-6) / 1e9, 2),
        "flush_us": round(us[tf], 3),
        "flush_bytes": append_bytes(B, Hkv, D, tf, R, 2),
        "flush_gbs": round(append_bytes(B, Hkv, D, tf, R, 2) / (us[tf] * 1e-6) / 1e9, 2),
        "window_us": round(float(sum(us.values())), 3),
        "note": "events around a single launch add a few us on this GPU"}}


def run_only(args):
    """One of the secondary workloads alone (used for profiling captures)."""
    import torch
    from bit_kv_cache_kivi_gb300 import build, workloads as W
    from bit_kv_cache_kivi_gb300.kivi import KiviCache
    build.build()
    dev = torch.device("cuda", 0)
    peak, _ = peak_hbm()

    def ev():
        return torch.cuda.Event(enable_timing=True)

    if args.only == "append":
        return append_window(torch, W, KiviCache, dev, torch.cuda.current_stream(), ev)
    if args.only == "stream_attn":
        return streaming_attention(args, torch, W, KiviCache, dev, torch.cuda.current_stream(), ev, peak)
    return extra_workloads(args, torch, W, KiviCache, dev, torch.cuda.current_stream(), ev, peak,
                           which=args.only)


# ------------------------------------------------------------------ oracle arm

def run_oracle(steps, warmup, budget_s=None):
    """The CPU oracle on a bounded sample of the main workload: the decode
    steps (append + attention) of batch element 0 (8 KV heads, 32 query
    heads) at context ~4096, single-threaded."""
    from bit_kv_cache_kivi_gb300 import workloads as W
    from oracle.kivi_oracle import OracleCache
    wl = W.llama3_8b_decode(steps=warmup + steps)
    o = OracleCache(2, G, wl.R, wl.D, 1, wl.Hkv, wl.capacity)
    o.prefill(np.ascontiguousarray(wl.k[:1]), np.ascontiguousarray(wl.v[:1]))
    q = np.ascontiguousarray(wl.q[:1].astype(np.float32))
    done, t_att, t_app, nbytes = 0, 0.0, 0.0, 0
    t_start = time.perf_counter()
    for i in range(warmup + steps):
        t = o.length
        a0 = time.perf_counter()
        o.append(np.ascontiguousarray(wl.k_new[i, :1]), np.ascontiguousarray(wl.v_new[i, :1]))
        a1 = time.perf_counter()
        o.attention(q)
        a2 = time.perf_counter()
        if i >= warmup:
            done += 1
            t_app += a1 - a0
            t_att += a2 - a1
            nbytes += attn_bytes(1, wl.Hkv, wl.Hq, wl.D, t + 1, wl.R, 2)
        if budget_s is not None and done >= 1 and time.perf_counter() - t_start > budget_s:
            break
    return {"value": round(nbytes / t_att / 1e9, 4), "unit": "GB/s", "cores": 1, "kind": "oracle",
            "sample": f"{done} decode steps (append + attention) of batch element 0 "
                      f"(8 KV heads, 32 query heads) at context ~{wl.T + warmup}; single thread",
            "tokens_per_s": round(done / (t_app + t_att), 3), "steps": done}


def _oracle_units_worker(job, units, cfg, barrier, results, warmup, steps, budget_s):
    """One host process of a multi-process oracle run over (b, kv-head) units,
    each an untouched single-unit oracle cache.  Everything before the shared
    start (a barrier) is untimed.  cfg = (bits, R, D, capacity).

    job "decode": units (k, v, k_new, v_new, q); prefill, `warmup` decode
      steps (append + attention on every unit), then `steps` timed ones, or
      fewer once `budget_s` has passed; bytes are the attention's.
    job "prefill": units (k, v); one unit prefilled as a warm-up, then every
      unit's prefill timed; bytes are the quantizer's.
    job "attention": units (k, v, q); prefill, then `steps` timed attention
      calls per unit."""
    try:
        from oracle.kivi_oracle import OracleCache
        bits, R, D, cap = cfg
        caches = [OracleCache(bits, G, R, D, 1, 1, cap) for _ in units]
        if job == "prefill":
            OracleCache(bits, G, R, D, 1, 1, cap).prefill(units[0][0], units[0][1])
            barrier.wait(timeout=600)
            t0 = time.perf_counter()
            nbytes = 0
            for o, (k, v) in zip(caches, units):
                o.prefill(k, v)
                nbytes += prefill_bytes(1, 1, D, k.shape[2], R, bits, k.dtype.itemsize)
            results.put(("ok", nbytes, time.perf_counter() - t0, 1))
            return
        for o, u in zip(caches, units):
            o.prefill(u[0], u[1])
        if job == "attention":
            barrier.wait(timeout=600)
            t0 = time.perf_counter()
            nbytes = 0
            for _ in range(steps):
                for o, (_, _, q) in zip(caches, units):
                    o.attention(q)
                    nbytes += attn_bytes(1, 1, q.shape[1], D, o.length, R, bits)
            results.put(("ok", nbytes, time.perf_counter() - t0, steps))
            return

        def one(i):
            nb = 0
            for o, (_, _, kn, vn, q) in zip(caches, units):
                t = o.length
                o.append(kn[i], vn[i])
                o.attention(q)
                nb += attn_bytes(1, 1, q.shape[1], D, t + 1, R, bits)
            return nb

        for i in range(warmup):
            one(i)
        barrier.wait(timeout=600)
        t0 = time.perf_counter()
        nbytes, done = 0, 0
        for i in range(warmup, warmup + steps):
            nbytes += one(i)
            done += 1
            if budget_s is not None and time.perf_counter() - t0 > budget_s:
                break
        results.put(("ok", nbytes, time.perf_counter() - t0, done))
    except Exception as e:  # reported to the parent, which fails the run
        barrier.abort()  # the other processes stop waiting for this one
        results.put(("error", repr(e), 0.0, 0))


def host_cores() -> int:
    return len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity") else os.cpu_count()


def oracle_pool(job, units, cfg, nproc, warmup=0, steps=1, budget_s=None):
    """Runs `job` over `units` on `nproc` spawned processes (spawn: the GPU is
    already in use in this process), unit i on process i mod nproc, all
    starting the timed part together.  Returns (bytes of all processes, the
    slowest process's seconds, sorted steps per process)."""
    import multiprocessing as mp
    nproc = max(1, min(nproc, len(units)))
    ctx = mp.get_context("spawn")
    barrier, results = ctx.Barrier(nproc), ctx.Queue()
    procs = []
    for w in range(nproc):
        p = ctx.Process(target=_oracle_units_worker,
                        args=(job, units[w::nproc], cfg, barrier, results, warmup, steps, budget_s))
        p.start()
        procs.append(p)
    got = []
    try:
        deadline = time.monotonic() + 900
        while len(got) < nproc:
            try:
                got.append(results.get(timeout=1.0))
            except queue.Empty:
                # a process that ended without reporting (a crash) fails the run
                dead = [p.exitcode for p in procs if p.exitcode not in (None, 0)]
                if dead or time.monotonic() > deadline:
                    raise RuntimeError(f"oracle {job} run: a process ended without a result "
                                       f"(exit codes {dead})" if dead else f"oracle {job} run timed out")
    finally:
        for p in procs:
            p.join(timeout=30)
            if p.is_alive():
                p.terminate()
                p.join()
    errs = [r[1] for r in got if r[0] != "ok"]
    if errs:
        raise RuntimeError(f"oracle {job} run failed: {errs[0]}")
    return sum(r[1] for r in got), max(r[2] for r in got), sorted(r[3] for r in got)


def _unit(a, b, h):
    return np.ascontiguousarray(a[b:b + 1, h:h + 1])


def _decode_units(wl, pairs):
    g = wl.Hq // wl.Hkv
    return [(_unit(wl.k, b, h), _unit(wl.v, b, h),
             np.ascontiguousarray(wl.k_new[:, b:b + 1, h:h + 1]),
             np.ascontiguousarray(wl.v_new[:, b:b + 1, h:h + 1]),
             np.ascontiguousarray(wl.q[b:b + 1, h * g:(h + 1) * g].astype(np.float32)))
            for b, h in pairs]


def run_oracle_multicore(steps=64, warmup=1, budget_s=None, wl=None, max_procs=None):
    """The CPU oracle on every host core: the main workload's 64 (batch, KV
    head) units split over one process per core, each timing decode steps of
    its units concurrently.  value = attention bytes of all processes / the
    slowest process's wall time."""
    from bit_kv_cache_kivi_gb300 import workloads as W
    if wl is None:
        wl = W.llama3_8b_decode(steps=warmup + steps)
    pairs = [(b, h) for b in range(wl.B) for h in range(wl.Hkv)]
    nproc = max(1, min(host_cores(), len(pairs), max_procs or len(pairs)))
    nbytes, wall, steps = oracle_pool("decode", _decode_units(wl, pairs), (wl.bits, wl.R, wl.D, wl.capacity),
                                      nproc, warmup, steps, budget_s)
    return {"value": round(nbytes / wall / 1e9, 4), "unit": "GB/s", "cores": nproc, "kind": "oracle",
            "sample": f"all {len(pairs)} (batch, KV head) units of {wl.name} at context "
                      f"~{wl.T + warmup}, {len(pairs) // nproc}-{-(-len(pairs) // nproc)} units per process, "
                      f"{nproc} processes, {steps[0]}-{steps[-1]} decode steps (append + attention) each",
            "steps": steps[0], "bytes": nbytes, "tokens_per_s": round(wl.B * sum(steps) / len(steps) / wall, 3)}


def _cpu_entry(nbytes, wall, nproc, sample, unit_tokens=None):
    e = {"gbs": round(nbytes / wall / 1e9, 4), "seconds": round(wall, 3), "cores": nproc,
         "kind": "oracle", "sample": sample}
    if unit_tokens is not None:
        e["tokens_per_s"] = round(unit_tokens / wall, 3)
    return e


def oracle_workload_baselines(res: dict, cores=None, quant_units=2) -> None:
    """The oracle beside the GPU numbers of the other workloads, each on a
    bounded sample: the 32k-token bf16 prefill quantizer (2- and 4-bit) on
    `quant_units` (b, kv-head) units single-threaded and on all 32 units over
    every core; the 131k-token attention on one unit single-threaded and on
    all 8 over the cores; the streaming decode (GQA 7, 2048 + 512 steps of
    append + attention) on one unit per core.  Adds "cpu_oracle" to the
    entries of `res` (a workloads dict) that exist."""
    from bit_kv_cache_kivi_gb300 import workloads as W
    cores = cores or host_cores()
    if any(f"prefill_quantize_{b}bit" in res for b in (2, 4)):
        wl = W.prefill_quantize(2)
        pairs = [(b, h) for b in range(wl.B) for h in range(wl.Hkv)]
        units = [(_unit(wl.k, b, h), _unit(wl.v, b, h)) for b, h in pairs]
        del wl.k, wl.v
        for bits in (2, 4):
            key = f"prefill_quantize_{bits}bit"
            if key not in res:
                continue
            cfg = (bits, wl.R, wl.D, wl.capacity)
            n1, w1, _ = oracle_pool("prefill", units[:quant_units], cfg, 1)
            nm = min(cores, len(units))
            nb, wm, _ = oracle_pool("prefill", units, cfg, nm)
            res[key]["cpu_oracle"] = {
                "single": _cpu_entry(n1, w1, 1, f"prefill of {quant_units} of the {len(units)} "
                                                f"(batch, KV head) units, one thread"),
                "multicore": _cpu_entry(nb, wm, nm, f"prefill of all {len(units)} units, "
                                                    f"{nm} processes")}
        del units
    if "long_context_attention" in res:
        wl = W.long_context()
        g = wl.Hq // wl.Hkv
        units = [(_unit(wl.k, 0, h), _unit(wl.v, 0, h),
                  np.ascontiguousarray(wl.q[0:1, h * g:(h + 1) * g].astype(np.float32)))
                 for h in range(wl.Hkv)]
        del wl.k, wl.v
        cfg = (wl.bits, wl.R, wl.D, wl.capacity)
        n1, w1, _ = oracle_pool("attention", units[:1], cfg, 1)
        nm = min(cores, len(units))
        nb, wm, _ = oracle_pool("attention", units, cfg, nm)
        res["long_context_attention"]["cpu_oracle"] = {
            "single": _cpu_entry(n1, w1, 1, f"one attention over KV head 0 ({g} query heads) at "
                                            f"context {wl.T}, one thread"),
            "multicore": _cpu_entry(nb, wm, nm, f"one attention over all {wl.Hkv} KV heads, {nm} processes")}
        del units
    if "streaming_decode" in res:
        wl = W.streaming()
        pairs = [(b, h) for b in range(wl.B) for h in range(wl.Hkv)]
        nm = min(cores, len(pairs))
        units = _decode_units(wl, pairs[:nm])
        cfg = (wl.bits, wl.R, wl.D, wl.capacity)
        nb, wm, st = oracle_pool("decode", units, cfg, nm, 0, wl.steps)
        res["streaming_decode"]["cpu_oracle"] = {
            "multicore": _cpu_entry(nb, wm, nm, f"{nm} of the {len(pairs)} (batch, KV head) units, one per "
                                                f"process, all {st[0]} steps (append + attention) from "
                                                f"context {wl.T}; tokens_per_s counts a token per "
                                                f"{wl.Hkv} unit-steps", nm * st[0] / wl.Hkv)}


def combine_ranks(result: dict) -> dict:
    """Whole-job numbers of a replicas-only run over the initialised process
    group: the step time is the slowest rank's, and `value` the attention
    bytes of every rank over the slowest rank's attention time (weak
    scaling).  Reads result["_attn"] = (bytes, seconds) of this rank."""
    import torch
    import torch.distributed as dist
    dev = "cuda" if dist.get_backend() == "nccl" else "cpu"
    b, sec = result["_attn"]
    tot = torch.tensor([float(b)], dtype=torch.float64, device=dev)
    mx = torch.tensor([float(sec), float(result["ms_per_step"])], dtype=torch.float64, device=dev)
    dist.all_reduce(tot, op=dist.ReduceOp.SUM)
    dist.all_reduce(mx, op=dist.ReduceOp.MAX)
    out = dict(result)
    out["value"] = round(float(tot[0]) / float(mx[0]) / 1e9, 2)
    out["ms_per_step"] = round(float(mx[1]), 5)
    out["n_gpus"] = dist.get_world_size()
    return out


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=100)
    ap.add_argument("--warmup", type=int, default=5)
    ap.add_argument("--impl", default="ours", choices=["ours", "reference"])
    ap.add_argument("--main-only", action="store_true", help="skip the other workloads")
    ap.add_argument("--only", choices=["main", "quantize", "attn3", "attn4", "attn8", "outliers", "long", "streaming",
                                       "append", "stream_attn"],
                    help="run one workload alone (for profiling); prints its numbers")
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--quant-reps", type=int, default=10)
    ap.add_argument("--attn-reps", type=int, default=30)
    args = ap.parse_args()
    args.warmup = max(args.warmup, 3)
    rank = int(os.environ.get("RANK", "0"))
    world = int(os.environ.get("WORLD_SIZE", "1"))

    if args.impl == "reference":
        if rank != 0:
            return
        cb = run_oracle_multicore(args.steps, args.warmup)
        line = {"impl": "reference", "metric": METRIC, "value": cb["value"], "unit": "GB/s",
                "n_gpus": args.gpus, "steps": cb["steps"], "warmup": args.warmup,
                "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "f32",
                "data": "synthetic", "config": {"workload": WORKLOAD},
                "cpu_baseline": cb,
                "e2e": {"value": cb["value"], "unit": "GB/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if world > 1:
        # Replicas only: every rank runs the same single-GPU workload on its own
        # device; no data-path collective exists.
        import torch
        import torch.distributed as dist
        torch.cuda.set_device(int(os.environ.get("LOCAL_RANK", "0")))
        dist.init_process_group("nccl")
        dist.barrier()
    if args.only and args.only != "main":
        result = run_only(args)
        print(json.dumps(result))
        return
    result = run_gpu(args)
    if world > 1:
        import torch.distributed as dist
        result = combine_ranks(result)
        dist.destroy_process_group()
    result.pop("_attn", None)
    if rank == 0:
        if not args.no_cpu_baseline and world == 1:
            result["cpu_baseline"] = run_oracle(args.steps, 2, budget_s=12.0)
            result["cpu_baseline"]["multicore"] = run_oracle_multicore(budget_s=8.0)
            if "workloads" in result:
                oracle_workload_baselines(result["workloads"])
        if "workloads" in result:  # the long per-workload record goes last
            result["workloads"] = result.pop("workloads")
        print(json.dumps(result))


if __name__ == "__main__":
    main()
