"""Attention calls that may overlap the launch before them on the stream
(kivi_set_attention_overlap) give the same outputs, bit for bit, as
ordinary launches of the same split plan: eagerly and inside a CUDA graph,
over several caches and with the same cache (and so the same workspace)
called twice in a row.  Their own automatic plan (fewer, longer splits)
matches the oracle."""
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


def _queries(wl, n):
    rng = np.random.default_rng(1234)
    return [W.cast(rng.standard_normal((wl.B, wl.Hq, wl.D), np.float32), wl.q_dtype) for _ in range(n)]


@pytest.mark.parametrize("bits,Hq,Hkv,T_,R", [(2, 8, 2, 700, 32), (4, 28, 4, 300, 64), (2, 32, 8, 2049, 32)])
def test_overlapping_attention_calls(bits, Hq, Hkv, T_, R):
    wl = W.synthetic("ov", B=2, Hq=Hq, Hkv=Hkv, T=T_, R=R, bits=bits, seed=41 + T_)
    caches = []
    for _ in range(3):
        g = T.gpu_cache(wl)
        g.prefill(T.dev(wl.k, wl.dtype), T.dev(wl.v, wl.dtype))
        caches.append(g)
    qs_np = _queries(wl, 3)
    qs = [T.dev(x, wl.q_dtype) for x in qs_np]
    o = T.oracle_cache(wl)
    o.prefill(wl.k, wl.v)
    refs = [o.attention(T.q_float(x, wl.q_dtype)) for x in qs_np]
    seq = [(0, 0), (0, 1), (1, 2), (2, 0), (1, 1), (0, 2), (0, 0)]

    def run_seq(outs):
        for (ci, qi), out in zip(seq, outs):
            caches[ci].attention(qs[qi], out)

    # An explicit split count plans the same splits with and without the
    # overlap, so the outputs must agree bit for bit.  Ordinary launches
    # first: the reference outputs, and the oracle check.
    for c in caches:
        c.set_splits(3)
    serial = {}
    for ci in range(3):
        for qi in range(3):
            serial[ci, qi] = caches[ci].attention(qs[qi]).clone()
    torch.cuda.synchronize()
    for qi in range(3):
        err = T.attn_err(T.out_float(serial[0, qi]), refs[qi])
        assert err <= T.ATTN_TOL, err
    # overlapping launches: cache 0 twice in a row (one workspace), then the others
    for c in caches:
        c.set_overlap(True)
    outs = [torch.empty_like(qs[0]) for _ in seq]
    run_seq(outs)
    torch.cuda.synchronize()
    for (ci, qi), out in zip(seq, outs):
        assert torch.equal(out, serial[ci, qi]), (ci, qi)
    # the same sequence captured in a CUDA graph, replayed twice
    outs_g = [torch.zeros_like(qs[0]) for _ in seq]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run_seq(outs_g)
    for _ in range(2):
        for out in outs_g:
            out.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for (ci, qi), out in zip(seq, outs_g):
            assert torch.equal(out, serial[ci, qi]), (ci, qi)
    del graph
    # the automatic plan of overlapped launches (fewer, longer splits): the
    # oracle's outputs within tolerance, eagerly and replayed from a graph
    for c in caches:
        c.set_splits(0)
    outs_a = [torch.empty_like(qs[0]) for _ in seq]
    run_seq(outs_a)
    torch.cuda.synchronize()
    for (ci, qi), out in zip(seq, outs_a):
        err = T.attn_err(T.out_float(out), refs[qi])
        assert err <= T.ATTN_TOL, (ci, qi, err)
    outs_ag = [torch.zeros_like(qs[0]) for _ in seq]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run_seq(outs_ag)
    graph.replay()
    torch.cuda.synchronize()
    for a_, b_ in zip(outs_a, outs_ag):
        assert torch.equal(a_, b_)
    for c in caches:
        c.set_overlap(False)
