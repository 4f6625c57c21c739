"""Guard bytes around every buffer the kernels write (the cache's tiles and
rings, the attention workspace, the output), standing in for a memory
checker: each buffer is the middle of a larger allocation whose head and tail
hold a fixed pattern, and after every call the pattern must be intact and the
inputs unchanged.  Every writing path runs: ragged prefill, single appends
across key and value flushes, multi-token appends, attention and the one-call
decode step; the results are checked against the oracle so that the guarded
cache is known to be the one used."""
import numpy as np
import pytest
import torch

from bit_kv_cache_kivi_gb300 import workloads as W
import kivi_testlib as T

pytestmark = pytest.mark.gpu

GUARD = 4096  # bytes on each side; a multiple of 16 keeps every buffer aligned
PAT = 0xA5


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from bit_kv_cache_kivi_gb300 import build, kivi
    build.build()
    kivi.lib()
    torch.cuda.init()


def _guarded(nbytes: int, device):
    full = torch.full((nbytes + 2 * GUARD,), PAT, dtype=torch.uint8, device=device)
    return full, full[GUARD:GUARD + nbytes]


def _intact(full: torch.Tensor, nbytes: int) -> bool:
    return bool((full[:GUARD] == PAT).all()) and bool((full[GUARD + nbytes:] == PAT).all())


def _rebind(cache) -> dict:
    """Re-creates an empty cache's C handle over guarded buffers and gives it a
    guarded workspace; returns {name: (allocation, bytes)}."""
    from bit_kv_cache_kivi_gb300 import kivi as K
    fulls = {}
    for n, s in zip(K.BUFFER_NAMES, K.kivi_cache_sizes(cache.cfg)):
        full, mid = _guarded(max(s, 16), cache.device)
        fulls[n] = (full, max(s, 16))
        cache.buffers[n] = mid
    K.kivi_cache_destroy(cache.handle)
    cache.handle = K.kivi_cache_init(cache.cfg, K.kivi_buffers(*[cache.buffers[n].data_ptr()
                                                                 for n in K.BUFFER_NAMES]))
    wf, wm = _guarded(max(cache.ws_bytes, 16), cache.device)
    cache.workspace, cache._ws_ptr = wm, wm.data_ptr()
    fulls["workspace"] = (wf, max(cache.ws_bytes, 16))
    return fulls


def _guarded_out(shape, device):
    n = int(np.prod(shape)) * 2
    full, mid = _guarded(n, device)
    return full, n, mid.view(torch.float16).view(*shape)


def _check_guards(fulls: dict, what: str) -> None:
    torch.cuda.synchronize()
    for n, (full, nb) in fulls.items():
        assert _intact(full, nb), f"{what}: guard bytes of {n} overwritten"


def _tok(x, t):
    return np.ascontiguousarray(x[:, :, t])


@pytest.mark.parametrize("policy", [T.ALG1, T.SHARED])
@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_no_write_outside_buffers(bits, policy):
    wl = W.synthetic("gb", B=3, Hq=8, Hkv=2, T=400, R=32, bits=bits, steps=0, seed=60 + bits + policy)
    cap = 512
    g = T.gpu_cache(wl, capacity=cap, policy=policy)
    fulls = _rebind(g)
    o = T.oracle_cache(wl, capacity=cap, policy=policy)
    dev = g.device

    k0, v0 = T.dev(np.ascontiguousarray(wl.k[:, :, :200]), "f16"), T.dev(np.ascontiguousarray(wl.v[:, :, :200]), "f16")
    k0c, v0c = k0.clone(), v0.clone()
    g.prefill(k0, v0)
    o.prefill(np.ascontiguousarray(wl.k[:, :, :200]), np.ascontiguousarray(wl.v[:, :, :200]))
    _check_guards(fulls, "prefill")
    assert torch.equal(k0, k0c) and torch.equal(v0, v0c)

    for t in range(200, 240):  # key flush at 224, value rows every step
        g.append(T.dev(_tok(wl.k, t), "f16"), T.dev(_tok(wl.v, t), "f16"))
        o.append(_tok(wl.k, t), _tok(wl.v, t))
    _check_guards(fulls, "append")

    kc, vc = T.dev(np.ascontiguousarray(wl.k[:, :, 240:310]), "f16"), T.dev(np.ascontiguousarray(wl.v[:, :, 240:310]), "f16")
    g.append_tokens(kc, vc)
    for t in range(240, 310):
        o.append(_tok(wl.k, t), _tok(wl.v, t))
    _check_guards(fulls, "append_tokens")
    T.compare_state(T.gpu_state(g), o.export(), 310, wl.R, wl.G, policy=policy)

    q = T.dev(wl.q, wl.q_dtype)
    qc = q.clone()
    ofull, on, out = _guarded_out(tuple(q.shape), dev)
    fulls["out"] = (ofull, on)
    g.attention(q, out)
    _check_guards(fulls, "attention")
    assert torch.equal(q, qc)
    qf = T.q_float(wl.q, wl.q_dtype)
    assert T.attn_err(T.out_float(out), o.attention(qf)) <= T.ATTN_TOL

    kn, vn = T.dev(_tok(wl.k, 310), "f16"), T.dev(_tok(wl.v, 310), "f16")
    g.step(kn, vn, q, out)
    o.append(_tok(wl.k, 310), _tok(wl.v, 310))
    _check_guards(fulls, "decode step")
    assert T.attn_err(T.out_float(out), o.attention(qf)) <= T.ATTN_TOL
    T.compare_state(T.gpu_state(g), o.export(), 311, wl.R, wl.G, policy=policy)


def test_no_write_outside_buffers_ragged_outliers():
    """Ragged lengths (0, 1, R - 1, R, 2R + 5, 300) with two fp16 outlier key
    channels per group: prefill, 40 single appends, attention and a step."""
    from oracle.kivi_oracle import OracleCache
    lens = [0, 1, 31, 32, 69, 300]
    wl = W.synthetic("gr", B=6, Hq=8, Hkv=2, T=400, R=32, steps=0, seed=71)
    cap = 384
    g = T.gpu_cache(wl, capacity=cap, outliers=2)
    fulls = _rebind(g)
    g.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"), lengths=lens)
    orc = []
    for b, l in enumerate(lens):
        o = OracleCache(2, wl.G, wl.R, wl.D, 1, wl.Hkv, cap, T.ALG1, 2)
        if l:
            o.prefill(np.ascontiguousarray(wl.k[b:b + 1, :, :l]), np.ascontiguousarray(wl.v[b:b + 1, :, :l]))
        orc.append(o)
    _check_guards(fulls, "ragged prefill")
    for i in range(40):
        t = 300 + i  # any token rows serve as the new tokens
        g.append(T.dev(_tok(wl.k, t), "f16"), T.dev(_tok(wl.v, t), "f16"))
        for b, o in enumerate(orc):
            o.append(np.ascontiguousarray(wl.k[b:b + 1, :, t]), np.ascontiguousarray(wl.v[b:b + 1, :, t]))
    _check_guards(fulls, "ragged appends")
    q = T.dev(wl.q, wl.q_dtype)
    ofull, on, out = _guarded_out(tuple(q.shape), g.device)
    fulls["out"] = (ofull, on)
    g.step(T.dev(_tok(wl.k, 399), "f16"), T.dev(_tok(wl.v, 399), "f16"), q, out)
    for b, o in enumerate(orc):
        o.append(np.ascontiguousarray(wl.k[b:b + 1, :, 399]), np.ascontiguousarray(wl.v[b:b + 1, :, 399]))
    _check_guards(fulls, "ragged step")
    gst = T.gpu_state(g)
    qf = T.q_float(wl.q, wl.q_dtype)
    res = T.out_float(out)
    for b, o in enumerate(orc):
        l = lens[b] + 41
        T.compare_state({n: a[b:b + 1] for n, a in gst.items()}, o.export(), l, wl.R, wl.G)
        assert T.attn_err(res[b:b + 1], o.attention(qf[b:b + 1])) <= T.ATTN_TOL, b
