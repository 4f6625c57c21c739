"""Decode steps and attention recorded in a CUDA graph (the way a decode loop
runs them, and the way the benchmark times them): one replay of K captured
one-call steps -- each an append and the attention launched as its
programmatic dependent -- must leave the cache and the K outputs of K eager
steps bit for bit, and a replayed attention graph must reproduce its eager
output."""
import numpy as np
import pytest
import torch

from bit_kv_cache_kivi_gb300 import workloads as W
import kivi_testlib as T

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from bit_kv_cache_kivi_gb300 import build, kivi
    build.build()
    kivi.lib()
    torch.cuda.init()


@pytest.mark.parametrize("policy", [T.ALG1, T.SHARED])
@pytest.mark.parametrize("bits", [2, 3])
def test_graph_of_decode_steps_matches_eager_steps(bits, policy):
    wl = W.synthetic("gc", B=2, Hq=8, Hkv=2, T=250, R=32, bits=bits, steps=40, seed=31 + bits + policy)
    cap = 384
    eager = T.gpu_cache(wl, capacity=cap, policy=policy)
    graph = T.gpu_cache(wl, capacity=cap, policy=policy)
    k0, v0 = T.dev(wl.k, "f16"), T.dev(wl.v, "f16")
    eager.prefill(k0, v0)
    graph.prefill(k0, v0)
    q = T.dev(wl.q, wl.q_dtype)
    kn, vn = T.dev(wl.k_new, "f16"), T.dev(wl.v_new, "f16")
    graph.attention(q)  # the first call clears the workspace counters, outside the capture
    torch.cuda.synchronize()
    outs = [torch.empty_like(q) for _ in range(wl.steps)]
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for i in range(wl.steps):
            graph.step(kn[i], vn[i], q, outs[i])
    assert graph.length == wl.T + wl.steps  # the host state advances at capture
    g.replay()
    ref = [eager.step(kn[i], vn[i], q).clone() for i in range(wl.steps)]
    torch.cuda.synchronize()
    for i in range(wl.steps):
        assert torch.equal(outs[i], ref[i]), f"step {i}"
    T.compare_state(T.gpu_state(graph), T.gpu_state(eager), wl.T + wl.steps, wl.R, 32, policy=policy)
    o = T.oracle_cache(wl, capacity=cap, policy=policy)
    o.prefill(wl.k, wl.v)
    for i in range(wl.steps):
        o.append(wl.k_new[i], wl.v_new[i])
    T.compare_state(T.gpu_state(graph), o.export(), wl.T + wl.steps, wl.R, 32, policy=policy)


def test_graph_of_attention_launches_replays_exactly():
    wl = W.synthetic("ga", B=3, Hq=12, Hkv=3, T=700, R=64, steps=0, seed=8)
    c = T.gpu_cache(wl, capacity=768)
    c.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"))
    q = T.dev(wl.q, wl.q_dtype)
    ref = c.attention(q).clone()
    out = torch.empty_like(q)
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g):
        for _ in range(3):
            c.attention(q, out)
    out.zero_()
    g.replay()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(out, ref)
    o = T.oracle_cache(wl, capacity=768)
    o.prefill(wl.k, wl.v)
    assert T.attn_err(T.out_float(out), o.attention(T.q_float(wl.q, wl.q_dtype))) <= T.ATTN_TOL
