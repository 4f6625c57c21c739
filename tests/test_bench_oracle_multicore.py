"""The multi-process oracle timing of bench.py: the (batch, KV head) units
are split over spawned host processes, each unit exactly once, so the bytes
the processes report add up to the whole batch's -- decode-attention bytes at
every timed step, the quantizer's bytes of a prefill, the attention's bytes
of every timed call.  CPU only (no GPU, no kernel)."""
import sys

from conftest import ROOT

sys.path.insert(0, ROOT)
import bench  # noqa: E402
from bit_kv_cache_kivi_gb300 import workloads as W  # noqa: E402


def test_units_partition_and_bytes():
    wl = W.synthetic("mc", B=3, Hq=8, Hkv=2, T=70, R=32, steps=4, seed=5)
    r = bench.run_oracle_multicore(steps=3, warmup=1, wl=wl, max_procs=4)
    assert r["cores"] == 4 and r["steps"] == 3 and r["kind"] == "oracle"
    # timed steps 1..3 follow one warm-up append: contexts T+2, T+3, T+4
    want = sum(bench.attn_bytes(wl.B, wl.Hkv, wl.Hq, wl.D, wl.T + 2 + i, wl.R, 2) for i in range(3))
    assert r["bytes"] == want
    assert r["value"] > 0 and "6 (batch, KV head) units" in r["sample"]


def test_more_processes_than_units_is_capped():
    wl = W.synthetic("mc1", B=1, Hq=4, Hkv=1, T=40, R=32, steps=2, seed=6)
    r = bench.run_oracle_multicore(steps=1, warmup=1, wl=wl, max_procs=8)
    assert r["cores"] == 1 and r["steps"] == 1
    assert r["bytes"] == bench.attn_bytes(1, 1, 4, wl.D, wl.T + 2, wl.R, 2)


def test_prefill_and_attention_jobs_count_every_unit():
    wl = W.synthetic("mc2", B=2, Hq=6, Hkv=3, T=200, R=64, steps=0, seed=7, dtype="bf16")
    pairs = [(b, h) for b in range(wl.B) for h in range(wl.Hkv)]
    cfg = (4, wl.R, wl.D, wl.capacity)
    units = [(bench._unit(wl.k, b, h), bench._unit(wl.v, b, h)) for b, h in pairs]
    nb, wall, _ = bench.oracle_pool("prefill", units, cfg, 4)
    assert nb == bench.prefill_bytes(wl.B, wl.Hkv, wl.D, wl.T, wl.R, 4, 2) and wall > 0
    g = wl.Hq // wl.Hkv
    qs = [wl.q[b:b + 1, h * g:(h + 1) * g].astype("float32") for b, h in pairs]
    units = [u + (q,) for u, q in zip(units, qs)]
    nb, _, steps = bench.oracle_pool("attention", units, cfg, 3, steps=2)
    assert steps == [2, 2, 2]
    assert nb == 2 * bench.attn_bytes(wl.B, wl.Hkv, wl.Hq, wl.D, wl.T, wl.R, 4)


def test_worker_failure_before_the_start_fails_fast():
    """A process whose prefill fails before the shared start aborts the
    barrier, so the run fails at once instead of after the barrier's
    timeout (a planted error: K and V of different lengths)."""
    import time
    import numpy as np
    import pytest
    wl = W.synthetic("mf", B=2, Hq=4, Hkv=1, T=40, R=32, steps=0, seed=8)
    good = (bench._unit(wl.k, 0, 0), bench._unit(wl.v, 0, 0))
    bad = (bench._unit(wl.k, 1, 0), np.ascontiguousarray(bench._unit(wl.v, 1, 0)[:, :, :39]))
    t0 = time.monotonic()
    with pytest.raises(RuntimeError, match="oracle prefill run failed"):
        bench.oracle_pool("prefill", [good, bad], (2, wl.R, wl.D, wl.capacity), 2)
    assert time.monotonic() - t0 < 60
