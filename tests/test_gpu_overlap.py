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


@pytest.mark.parametrize("bits", [2, 4])
def test_overlapping_calls_after_decode_steps(bits):
    """Overlapping attention calls mixed with decode steps and plain appends
    on three caches, across key flushes: an overlapping call that follows a
    step or an append of its own cache (directly, or behind overlapping
    calls on other caches) must see that write.  Against the same sequence
    without the overlap (explicit split counts, so that the plans agree), bit
    for bit, eagerly and replayed from a CUDA graph; the last outputs match
    the oracle."""
    wl = W.synthetic("ovs", B=2, Hq=8, Hkv=2, T=300, R=32, bits=bits, steps=40, seed=5 + bits)
    cap = 384
    # (kind, cache): s = decode step, a = plain append, o = attention call
    ops = [("s", 0), ("o", 1), ("o", 0), ("s", 1), ("s", 1), ("o", 2), ("o", 1), ("a", 2), ("o", 0),
           ("o", 2), ("s", 2), ("o", 2), ("s", 0), ("o", 0)] * 12  # 24 appends a cache: past a key flush
    qs_np = _queries(wl, 2)
    qs = [T.dev(x, wl.q_dtype) for x in qs_np]
    toks = {}
    seen = [0, 0, 0]
    for i, (kind, ci) in enumerate(ops):
        if kind in "sa":
            j = seen[ci] % wl.steps
            toks[i] = (T.dev(wl.k_new[j], "f16"), T.dev(wl.v_new[j], "f16"))
            seen[ci] += 1

    def fresh(overlap):
        cs = []
        for _ in range(3):
            g = T.gpu_cache(wl, capacity=cap)
            g.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"))
            g.set_splits(3)
            g.set_overlap(overlap)
            g.attention(qs[0])  # zeroes the workspace outside any graph
            cs.append(g)
        torch.cuda.synchronize()
        return cs

    def run(cs, outs):
        for i, ((kind, ci), out) in enumerate(zip(ops, outs)):
            if kind == "s":
                cs[ci].step(*toks[i], qs[ci % 2], out)
            elif kind == "a":
                cs[ci].append(*toks[i])
            else:
                cs[ci].attention(qs[ci % 2], out)

    ref_c = fresh(False)
    ref = [torch.zeros_like(qs[0]) for _ in ops]
    run(ref_c, ref)
    torch.cuda.synchronize()
    ov_c = fresh(True)
    outs = [torch.zeros_like(qs[0]) for _ in ops]
    run(ov_c, outs)
    torch.cuda.synchronize()
    for i, (a_, b_) in enumerate(zip(outs, ref)):
        assert torch.equal(a_, b_), (i, ops[i])
    for ci in range(3):
        assert ov_c[ci].length == ref_c[ci].length == wl.T + seen[ci]
        T.compare_state(T.gpu_state(ov_c[ci]), T.gpu_state(ref_c[ci]), ov_c[ci].length, wl.R, 32)
    gr_c = fresh(True)
    outs_g = [torch.zeros_like(qs[0]) for _ in ops]
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run(gr_c, outs_g)
    graph.replay()
    torch.cuda.synchronize()
    for i, (a_, b_) in enumerate(zip(outs_g, ref)):
        assert torch.equal(a_, b_), (i, ops[i])
    for ci in range(3):
        o = T.oracle_cache(wl, capacity=cap)
        o.prefill(wl.k, wl.v)
        for j in range(seen[ci]):
            o.append(wl.k_new[j % wl.steps], wl.v_new[j % wl.steps])
        last = max(i for i, (kind, c) in enumerate(ops) if c == ci and kind in "so")
        err = T.attn_err(T.out_float(outs[last]), o.attention(T.q_float(qs_np[ci % 2], wl.q_dtype)))
        assert err <= T.ATTN_TOL, (ci, err)


def test_overlapping_call_generations_under_replay():
    """Many overlapping calls back to back on two caches (a uniform one and
    one of ragged lengths), the same cache often twice or three times in a
    row, with explicit split counts changing between calls (so the grids
    differ and the generation tickets of a launch are padded differently):
    eagerly and replayed three times from one CUDA graph, every output equals
    the same call made as an ordinary launch, and no bounded wait gives up."""
    wl = W.synthetic("ovg", B=3, Hq=16, Hkv=4, T=1500, R=32, bits=2, seed=77)
    cap = 1536
    lens = [1500, 37, 900]
    cs = []
    for ragged in (False, True):
        g = T.gpu_cache(wl, capacity=cap)
        if ragged:
            g.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"), lengths=lens)
        else:
            g.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"))
        g.attention(T.dev(wl.q, "f16"))  # zeroes the workspace outside any graph
        cs.append(g)
    torch.cuda.synchronize()
    qs_np = _queries(wl, 3)
    qs = [T.dev(x, wl.q_dtype) for x in qs_np]
    # explicit split counts (an automatic count differs between overlapped and
    # ordinary launches, and with it the last bits)
    splits = [1, 3, 2, 9, 2, 6, 17, 5]
    seq = [(i % 7 % 2, i % 3, splits[i % len(splits)]) for i in range(40)]
    seq += [(0, 1, 7)] * 3 + [(1, 2, 4)] * 3

    ref = []
    for ci, qi, sp in seq:
        cs[ci].set_overlap(False)
        cs[ci].set_splits(sp)
        ref.append(cs[ci].attention(qs[qi]).clone())
    torch.cuda.synchronize()

    outs = [torch.zeros_like(qs[0]) for _ in seq]

    def run():
        for (ci, qi, sp), out in zip(seq, outs):
            cs[ci].set_splits(sp)
            cs[ci].attention(qs[qi], out)

    for c in cs:
        c.set_overlap(True)
    run()
    torch.cuda.synchronize()
    for i, (a_, b_) in enumerate(zip(outs, ref)):
        assert torch.equal(a_, b_), (i, seq[i])
    graph = torch.cuda.CUDAGraph()
    with torch.cuda.graph(graph):
        run()
    for rep in range(3):
        for o in outs:
            o.zero_()
        graph.replay()
        torch.cuda.synchronize()
        for i, (a_, b_) in enumerate(zip(outs, ref)):
            assert torch.equal(a_, b_), (rep, i, seq[i])
    for c in cs:
        c.set_overlap(False)
        c.set_splits(0)
    for c in cs:  # the status word (bytes - 16): no bounded wait gave up
        assert c.workspace[c.ws_bytes - 16:c.ws_bytes - 12].view(torch.int32).item() == 0
