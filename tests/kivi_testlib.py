"""Shared helpers of the parity tests: run a workload through the CUDA path
(via the C ABI binding) and through the oracle, and compare."""
from __future__ import annotations

import numpy as np
import torch

from bit_kv_cache_kivi_gb300 import workloads as W

ATTN_TOL = 2e-3  # max_i |o_i - r_i| / max_i |r_i| per (batch, query head)


ALG1, SHARED = 0, 1  # residual policies


def nq_k(l, R, G=32, policy=ALG1):
    if policy == SHARED:
        return max(l - R, 0) // G * G
    return l - l % R


def nq_v(l, R, G=32, policy=ALG1):
    if policy == SHARED:
        return max(l - R, 0) // G * G
    return max(l - R, 0)


def gpu_cache(wl: W.Workload, capacity: int | None = None, bits: int | None = None,
              policy: int = ALG1, outliers: int = 0):
    from bit_kv_cache_kivi_gb300.kivi import KiviCache
    return KiviCache(batch=wl.B, n_kv_heads=wl.Hkv, n_q_heads=wl.Hq,
                     max_tokens=capacity or wl.capacity, bits=bits or wl.bits,
                     group=wl.G, residual=wl.R, head_dim=wl.D, policy=policy, outliers=outliers)


def oracle_cache(wl: W.Workload, capacity: int | None = None, bits: int | None = None,
                 units=None, policy: int = ALG1, outliers: int = 0):
    """Oracle cache of the whole batch, or of the (b, h) units listed (B=1, H=1 each)."""
    from oracle.kivi_oracle import OracleCache
    cap = capacity or wl.capacity
    if units is None:
        return OracleCache(bits or wl.bits, wl.G, wl.R, wl.D, wl.B, wl.Hkv, cap, policy, outliers)
    return [OracleCache(bits or wl.bits, wl.G, wl.R, wl.D, 1, 1, cap, policy, outliers) for _ in units]


def dev(x: np.ndarray, dtype: str) -> torch.Tensor:
    return W.to_torch(x, dtype, "cuda")


def gpu_state(cache) -> dict:
    torch.cuda.synchronize()
    out = {}
    for n, t in cache.logical_state().items():
        a = t.cpu().numpy()
        out[n] = a.view(np.uint16) if a.dtype == np.int16 else a
    return out


def compare_state(gst: dict, ost: dict, l: int, R: int, G: int, units=None,
                  policy: int = ALG1) -> None:
    """Bit-exact comparison of the live part of two cache states.

    units: optional list of (b, h) selecting GPU units that correspond, in
    order, to oracle states given as a list (one B=1, H=1 state each)."""
    qk, qv = nq_k(l, R, G, policy), nq_v(l, R, G, policy)
    W_ = R + G if policy == SHARED else R  # ring slots
    pairs = []
    if units is None:
        B, H = gst["codes_k"].shape[:2]
        pairs = [((b, h), (ost, b, h)) for b in range(B) for h in range(H)]
    else:
        pairs = [(u, (o, 0, 0)) for u, o in zip(units, ost)]
    for (b, h), (o, ob, oh) in pairs:
        def chk(name, sl_g, sl_o):
            g, r = gst[name][b, h][sl_g], o[name][ob, oh][sl_o]
            if not np.array_equal(g, r):
                idx = np.argwhere(g != r)[:5]
                raise AssertionError(f"{name} differs at unit {(b, h)} l={l}: first {idx.tolist()}")
        chk("codes_k", slice(0, qk), slice(0, qk))
        chk("scale_k", slice(0, qk // G), slice(0, qk // G))
        chk("zero_k", slice(0, qk // G), slice(0, qk // G))
        if "outl_idx" in o:  # outlier-aware keys: the kept channels and values
            chk("outl_idx", slice(0, qk // G), slice(0, qk // G))
            chk("outl_val", slice(0, qk), slice(0, qk))
        chk("codes_v", slice(0, qv), slice(0, qv))
        chk("scale_v", slice(0, qv), slice(0, qv))
        chk("zero_v", slice(0, qv), slice(0, qv))
        for name, lo in (("ring_k", qk), ("ring_v", qv)):
            slots = [t % W_ for t in range(lo, l)]
            if slots:
                chk(name, slots, slots)


def attn_err(out: np.ndarray, ref: np.ndarray, out_dtype: str | None = None) -> float:
    """Worst (over batch, head) of max |o - r| / max |r|.  With out_dtype
    "bf16" the output carries its own rounding, up to half a bf16 ulp of each
    element (8 significant bits), which is taken off each element's error
    first (a comparison with the reference rounded to bf16 would not do: a
    result and a reference on either side of a rounding boundary round a
    whole ulp, 2^-7 of the value, apart)."""
    o = out.astype(np.float64).reshape(-1, out.shape[-1])
    r = ref.astype(np.float64).reshape(-1, ref.shape[-1])
    d = np.abs(o - r)
    if out_dtype == "bf16":
        half_ulp = np.ldexp(1.0, np.frexp(np.maximum(np.abs(r), np.abs(o)))[1] - 9)
        d = np.maximum(d - half_ulp, 0.0)
    return float((d.max(axis=1) / np.abs(r).max(axis=1)).max())


def q_float(q: np.ndarray, dtype: str) -> np.ndarray:
    """The query as the fp32 values the kernel reads."""
    if dtype == "bf16":
        return W.to_torch(q, "bf16").float().numpy()
    return q.astype(np.float32)


def out_float(out: torch.Tensor) -> np.ndarray:
    return out.float().cpu().numpy()


def slice_unit(x: np.ndarray, b: int, h: int) -> np.ndarray:
    """[B, H, ...] -> [1, 1, ...] contiguous copy of one unit."""
    return np.ascontiguousarray(x[b:b + 1, h:h + 1])


# ---------------------------------------------------------------- oracle pool

def _oracle_unit(task):
    """One (batch, kv-head) unit through a B=1, H=1 oracle cache (runs in a
    worker process).  task: dict with bits, G, R, D, cap, k, v and optionally
    kn, vn ([steps][1][1][D]: appended after the prefill), q ({step: [1][grp][D]
    f32}: attention after that append; key -1 = after the prefill)."""
    from oracle.kivi_oracle import OracleCache
    o = OracleCache(task["bits"], task["G"], task["R"], task["D"], 1, 1, task["cap"])
    o.prefill(task["k"], task["v"])
    qs = task.get("q", {})
    outs = {}
    if -1 in qs:
        outs[-1] = o.attention(qs[-1])
    kn, vn = task.get("kn"), task.get("vn")
    if kn is not None:
        for i in range(kn.shape[0]):
            o.append(kn[i], vn[i])
            if i in qs:
                outs[i] = o.attention(qs[i])
    return o.export(), outs


def oracle_units(tasks):
    """_oracle_unit over tasks on a pool of spawned processes (spawned, not
    forked: the parent already uses the GPU), in order."""
    import multiprocessing as mp
    import os
    n = max(1, min(len(tasks), len(os.sched_getaffinity(0)) if hasattr(os, "sched_getaffinity")
                   else os.cpu_count() or 1))
    with mp.get_context("spawn").Pool(n) as pool:
        # bounded: a worker that cannot start makes the pool respawn it
        # forever, so the result is awaited with a time limit
        return pool.map_async(_oracle_unit, tasks, chunksize=1).get(timeout=1800)
