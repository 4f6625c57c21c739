"""Per-sequence lengths in a batch, through the C ABI, against one CPU oracle
cache per sequence.

Each sequence of a ragged batch must hold exactly the state that the
review's Algorithm 1 (or the shared-window policy) leaves for that sequence
alone -- after a ragged prefill, single-token appends and multi-token
appends -- and decode attention must cover each sequence's own tokens."""
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


def _rows(x, b, a, e):
    return np.ascontiguousarray(x[b:b + 1, :, a:e])


def _oracles(wl, lens, cap, bits, policy):
    from oracle.kivi_oracle import OracleCache
    out = []
    for b, l in enumerate(lens):
        o = OracleCache(bits, wl.G, wl.R, wl.D, 1, wl.Hkv, cap, policy)
        if l:
            o.prefill(_rows(wl.k, b, 0, l), _rows(wl.v, b, 0, l))
        out.append(o)
    return out


def _check_state(g, oracles, R, policy):
    gst = T.gpu_state(g)
    lens = g.lengths
    for b, o in enumerate(oracles):
        assert o.length == lens[b]
        T.compare_state({n: a[b:b + 1] for n, a in gst.items()}, o.export(), lens[b], R, 32,
                        policy=policy)


def _check_attention(g, oracles, wl):
    out = T.out_float(g.attention(T.dev(wl.q, wl.q_dtype)))
    qf = T.q_float(wl.q, wl.q_dtype)
    for b, o in enumerate(oracles):
        err = T.attn_err(out[b:b + 1], o.attention(qf[b:b + 1]))
        assert err <= T.ATTN_TOL, (b, g.lengths[b], err)


def _append_all(g, oracles, kn, vn, dtype):
    """One token to every sequence (kn, vn: [B][H][D])."""
    g.append(T.dev(np.ascontiguousarray(kn), dtype), T.dev(np.ascontiguousarray(vn), dtype))
    for b, o in enumerate(oracles):
        o.append(np.ascontiguousarray(kn[b:b + 1]), np.ascontiguousarray(vn[b:b + 1]))


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
@pytest.mark.parametrize("policy", [T.ALG1, T.SHARED])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_ragged_prefill_appends_attention(bits, policy, dtype):
    """Lengths 0, 1, R-1, R, R+1, 2R+5, 300 and 1200 in one batch: the empty
    sequence refuses attention until it has a token; then single appends and
    multi-token appends grow every sequence from its own length."""
    R = 32
    lens = [0, 1, R - 1, R, R + 1, 2 * R + 5, 300, 1200]
    B, steps, chunks = len(lens), 3, [5, 40]
    wl = W.synthetic("vl", B=B, Hq=8, Hkv=2, T=max(lens), R=R, bits=bits, dtype=dtype,
                     steps=steps + sum(chunks), seed=bits * 7 + policy)
    cap = (max(lens) + steps + sum(chunks) + R - 1) // R * R
    g = T.gpu_cache(wl, capacity=cap, bits=bits, policy=policy)
    g.prefill(T.dev(wl.k, dtype), T.dev(wl.v, dtype), lengths=lens)
    assert g.lengths == lens and g.length == -2
    o = _oracles(wl, lens, cap, bits, policy)
    _check_state(g, o, R, policy)
    from bit_kv_cache_kivi_gb300.kivi import KiviError
    with pytest.raises(KiviError) as e:
        g.attention(T.dev(wl.q, wl.q_dtype))
    assert e.value.status == 6  # an empty sequence
    for i in range(steps):
        _append_all(g, o, wl.k_new[i], wl.v_new[i], dtype)
        _check_state(g, o, R, policy)
        _check_attention(g, o, wl)
    i0 = steps
    for c in chunks:
        kc = np.ascontiguousarray(np.moveaxis(wl.k_new[i0:i0 + c], 0, 2))  # [B][H][c][D]
        vc = np.ascontiguousarray(np.moveaxis(wl.v_new[i0:i0 + c], 0, 2))
        g.append_tokens(T.dev(kc, dtype), T.dev(vc, dtype))
        for j in range(c):
            for b, ob in enumerate(o):
                ob.append(np.ascontiguousarray(wl.k_new[i0 + j][b:b + 1]),
                          np.ascontiguousarray(wl.v_new[i0 + j][b:b + 1]))
        i0 += c
        assert g.lengths == [l + steps + (i0 - steps) for l in lens]
        _check_state(g, o, R, policy)
        _check_attention(g, o, wl)


@pytest.mark.parametrize("R", [64, 128])
def test_ragged_large_batch(R):
    """80 sequences of random lengths (several tail splits at R = 128, packed
    splits of different counts per sequence in one grid)."""
    rng = np.random.default_rng(R)
    lens = [int(x) for x in rng.integers(1, 2500, 80)]
    wl = W.synthetic("vb", B=80, Hq=8, Hkv=1, T=max(lens), R=R, seed=R)
    cap = (max(lens) + R - 1) // R * R
    g = T.gpu_cache(wl, capacity=cap)
    g.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"), lengths=lens)
    o = _oracles(wl, lens, cap, 2, T.ALG1)
    _check_state(g, o, R, T.ALG1)
    _check_attention(g, o, wl)


def test_ragged_maximum_batch():
    """The per-sequence length limit, 1024 sequences, lengths 0..300 (some
    empty until the first append), three single-token appends, then every
    sequence against its own oracle cache."""
    rng = np.random.default_rng(1024)
    lens = [int(x) for x in rng.integers(0, 301, 1024)]
    lens[:3] = [0, 31, 32]
    wl = W.synthetic("vm", B=1024, Hq=4, Hkv=1, T=max(lens), R=32, steps=3, seed=77)
    cap = 320
    g = T.gpu_cache(wl, capacity=cap)
    g.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"), lengths=lens)
    o = _oracles(wl, lens, cap, 2, T.ALG1)
    for i in range(wl.steps):
        _append_all(g, o, wl.k_new[i], wl.v_new[i], "f16")
    assert g.lengths == [l + wl.steps for l in lens]
    _check_state(g, o, 32, T.ALG1)
    _check_attention(g, o, wl)


def test_ragged_split_override():
    """A fixed split count with ragged lengths: sequences shorter than the
    count use fewer splits; the merge counts each sequence's own."""
    lens = [40, 700, 2000, 33]
    wl = W.synthetic("vo", B=4, Hq=8, Hkv=2, T=max(lens), R=32, seed=5)
    g = T.gpu_cache(wl, capacity=2016)
    g.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"), lengths=lens)
    o = _oracles(wl, lens, 2016, 2, T.ALG1)
    for n in (1, 3, 9, 40):
        g.set_splits(n)
        _check_attention(g, o, wl)


def test_ragged_restore_and_uniform_lengths():
    """Copying the raw buffers plus set_lengths restores a ragged cache;
    equal lengths given per sequence behave as a uniform cache."""
    lens = [100, 7, 64]
    wl = W.synthetic("vr", B=3, Hq=4, Hkv=2, T=max(lens), R=32, steps=20, seed=8)
    a = T.gpu_cache(wl, capacity=128)
    a.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"), lengths=lens)
    for i in range(5):
        a.append(T.dev(wl.k_new[i], "f16"), T.dev(wl.v_new[i], "f16"))
    b = T.gpu_cache(wl, capacity=128)
    for name, t in a.state_views().items():
        b.state_views()[name].copy_(t)
    b.set_lengths(a.lengths)
    q = T.dev(wl.q, "f16")
    assert b.lengths == [105, 12, 69] and torch.equal(a.attention(q), b.attention(q))
    for i in range(5, 20):
        for c in (a, b):
            c.append(T.dev(wl.k_new[i], "f16"), T.dev(wl.v_new[i], "f16"))
    sa, sb = T.gpu_state(a), T.gpu_state(b)
    for name in sa:
        assert np.array_equal(sa[name], sb[name]), name
    assert torch.equal(a.attention(q), b.attention(q))
    # the same lengths for all: a uniform cache, bit for bit
    u1 = T.gpu_cache(wl, capacity=128)
    u1.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"), lengths=[100, 100, 100])
    u2 = T.gpu_cache(wl, capacity=128)
    u2.prefill(T.dev(np.ascontiguousarray(wl.k[:, :, :100]), "f16"),
               T.dev(np.ascontiguousarray(wl.v[:, :, :100]), "f16"))
    assert u1.length == 100 and u1.lengths == [100] * 3
    assert torch.equal(u1.attention(q), u2.attention(q))
