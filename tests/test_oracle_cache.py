"""Pins of the oracle's grouped + residual cache and of its decode attention."""
import math

import numpy as np
import pytest

from conftest import golden
from bit_kv_cache_kivi_gb300 import workloads as W


def _rand_kv(B, H, T, D, seed, dtype=np.float16):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((B, H, T, D), np.float32)
    v = rng.standard_normal((B, H, T, D), np.float32)
    k[..., 3] *= 5
    return k.astype(dtype), v.astype(dtype)


def test_algorithm1_worked_example(oracle):
    """Review §3.2.3: G=4, R=8, d=8, l=10 -> K grouped [0,8), V grouped [0,2)."""
    g = golden("algorithm1_example.json")
    G, R, D, l = g["G"], g["R"], g["d"], g["l_prompt"]
    assert oracle.nq_k(l, R, G) == g["key_grouped_tokens"][1]
    assert l - oracle.nq_k(l, R, G) == g["key_r"]
    assert oracle.nq_v(l, R, G) == g["value_grouped_tokens"][1]
    k, v = _rand_kv(1, 1, l, D, 0)
    c = oracle.OracleCache(2, G, R, D, 1, 1, 32)
    c.prefill(k, v)
    st = c.export()
    assert st["scale_v"].shape[-1] == g["value_groups_per_token"]
    # V rows 0..1 quantized, the rest not; K rows 0..7 quantized (2 groups)
    assert st["scale_v"][0, 0, :2].all() and not st["scale_v"][0, 0, 2:].any()
    assert st["scale_k"][0, 0, :2].all() and not st["scale_k"][0, 0, 2:].any()
    # residual contents: K tokens 8, 9 and V tokens 2..9, by slot t mod R
    kb, vb = k.view(np.uint16)[0, 0], v.view(np.uint16)[0, 0]
    for t in range(8, 10):
        assert np.array_equal(st["ring_k"][0, 0, t % R], kb[t])
    for t in range(2, 10):
        assert np.array_equal(st["ring_v"][0, 0, t % R], vb[t])
    # decoding: the K residual flushes when it reaches R (at l = 16)
    kn, vn = _rand_kv(8, 1, 1, D, 1)
    for i in range(5):
        c.append(kn[i], vn[i])
        assert oracle.nq_k(c.length, R, G) == 8
        assert oracle.nq_v(c.length, R, G) == c.length - R
    c.append(kn[5], vn[5])
    assert c.length == 16 and oracle.nq_k(16, R, G) == 2 * g["key_flush_when_residual_reaches"]
    st = c.export()
    assert st["scale_k"][0, 0, :4].all()


@pytest.mark.parametrize("policy", [0, 1])
def test_prefill_equals_streaming(oracle, policy):
    """VeloxQuant KIVI item 4: one-shot prefill and token-by-token decode give
    bit-identical caches (group-aligned flushes make the result chunk-free)."""
    B, H, T, D, G, R = 2, 2, 100, 64, 16, 32
    k, v = _rand_kv(B, H, T, D, 42)
    ref = oracle.OracleCache(2, G, R, D, B, H, 128, policy)
    ref.prefill(k, v)
    want = ref.export()
    for T0 in (0, 1, 15, 16, 31, 32, 33, 64, 99, 100):
        c = oracle.OracleCache(2, G, R, D, B, H, 128, policy)
        c.prefill(k[:, :, :T0], v[:, :, :T0])
        for t in range(T0, T):
            c.append(np.ascontiguousarray(k[:, :, t]), np.ascontiguousarray(v[:, :, t]))
        got = c.export()
        for name in want:
            assert np.array_equal(got[name], want[name]), (T0, name)


@pytest.mark.parametrize("policy", [0, 1])
def test_prefill_equals_streaming_three_bit(oracle, policy):
    """The same at 3 bits (the two-plane rows, D = 128, G = 32)."""
    B, H, T, D, G, R = 1, 2, 130, 128, 32, 32
    k, v = _rand_kv(B, H, T, D, 43)
    ref = oracle.OracleCache(3, G, R, D, B, H, 192, policy)
    ref.prefill(k, v)
    want = ref.export()
    for T0 in (0, 1, 31, 32, 33, 64, 97, 129):
        c = oracle.OracleCache(3, G, R, D, B, H, 192, policy)
        c.prefill(k[:, :, :T0], v[:, :, :T0])
        for t in range(T0, T):
            c.append(np.ascontiguousarray(k[:, :, t]), np.ascontiguousarray(v[:, :, t]))
        got = c.export()
        for name in want:
            assert np.array_equal(got[name], want[name]), (T0, name)


def test_determinism(oracle):
    k, v = _rand_kv(1, 2, 70, 128, 9)
    outs = []
    for _ in range(2):
        c = oracle.OracleCache(4, 32, 32, 128, 1, 2, 96)
        c.prefill(k, v)
        outs.append(c.export())
    for name in outs[0]:
        assert np.array_equal(outs[0][name], outs[1][name])


def test_shared_policy_counts(oracle):
    """VeloxQuant KIVI items 3-4: newest R tokens fp16, flushes in multiples of G."""
    for l in range(0, 200):
        nq = oracle.nq_k(l, 32, 16, 1)
        assert nq == oracle.nq_v(l, 32, 16, 1)
        assert nq % 16 == 0 and l - nq >= min(l, 32) and l - nq < 32 + 16


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_cache_dequant_within_bound(oracle, bits):
    """Every quantized element is within its group's bound; residual rows exact."""
    B, H, T, D, G, R = 1, 2, 200, 128, 32, 64
    L = (1 << bits) - 1
    k, v = _rand_kv(B, H, T, D, 5 + bits)
    c = oracle.OracleCache(bits, G, R, D, B, H, 256)
    c.prefill(k, v)
    st = c.export()
    nqk, nqv = oracle.nq_k(T, R, G), oracle.nq_v(T, R, G)
    for h in range(H):
        kh, vh = c.dequant(0, h)
        k32 = k[0, h].astype(np.float32)
        v32 = v[0, h].astype(np.float32)
        sk = st["scale_k"][0, h].view(np.float16).astype(np.float32)
        sv = st["scale_v"][0, h].view(np.float16).astype(np.float32)
        for t in range(nqk):
            s = sk[t // G]
            rng_ = np.array([np.ptp(k32[(t // G) * G:(t // G + 1) * G, d]) for d in range(D)])
            bound = s / 2 + L * np.abs(rng_ / L - s) + 1e-5 * np.abs(k32).max()
            assert (np.abs(kh[t] - k32[t]) <= bound).all()
        assert np.array_equal(kh[nqk:], k32[nqk:])
        for t in range(nqv):
            s = np.repeat(sv[t], G)
            rng_ = np.repeat([np.ptp(v32[t, i * G:(i + 1) * G]) for i in range(D // G)], G)
            bound = s / 2 + L * np.abs(rng_ / L - s) + 1e-5 * np.abs(v32).max()
            assert (np.abs(vh[t] - v32[t]) <= bound).all()
        assert np.array_equal(vh[nqv:], v32[nqv:])


def _live_bytes(oracle, l, D, bits, G, R):
    nqk, nqv = oracle.nq_k(l, R, G), oracle.nq_v(l, R, G)
    kb = nqk * D * bits // 8 + (nqk // G) * D * 2 * 2 + (l - nqk) * D * 2
    vb = nqv * D * bits // 8 + nqv * (D // G) * 2 * 2 + (l - nqv) * D * 2
    return kb, vb


def test_compression_closed_form(oracle):
    """Notebook storage check: 2 bits/element + an fp16 (min, scale) pair per
    group gives >= 4x on K (1024 x 128, all tokens grouped); the ratio depends
    on bits, G, R and l but not on head_dim; 1.0x below the window."""
    g = golden("notebook_checks.json")
    kb, _ = _live_bytes(oracle, 1024, 128, 2, 32, 32)
    fp16 = 1024 * 128 * 2
    assert fp16 == g["k_bytes_fp16_T1024_D128"]
    notebook = int(1024 * 128 * 0.25) + 2 * 2 * math.ceil(1024 / 32) * 128
    assert kb == notebook
    assert fp16 / kb >= g["compression_at_least"]
    assert fp16 / kb == pytest.approx(16 / (2 + 32 / 32))
    # b bits per element + 32 bits of (min, scale) per G elements, every width
    for bits in (2, 3, 4, 8):
        kb_b, _ = _live_bytes(oracle, 1024, 128, bits, 32, 32)
        assert fp16 / kb_b == pytest.approx(16 / (bits + 32 / 32))
        c = oracle.OracleCache(bits, 32, 32, 128, 1, 1, 64)
        c.prefill(*_rand_kv(1, 1, 64, 128, bits))
        assert c.export()["codes_k"].shape[-1] == 128 * bits // 8  # the live row is D*b/8 bytes
    for l in (1, 31, 32, 33, 1000, 4097):
        for bits in (2, 3, 4, 8):
            r64 = sum(_live_bytes(oracle, l, 64, bits, 32, 32)) / (2 * l * 64 * 2)
            r128 = sum(_live_bytes(oracle, l, 128, bits, 32, 32)) / (2 * l * 128 * 2)
            assert r64 == pytest.approx(r128)
    assert sum(_live_bytes(oracle, 20, 128, 2, 32, 32)) == 2 * 20 * 128 * 2
    # and the oracle's own buffers hold exactly the live bytes counted above
    k, v = _rand_kv(1, 1, 100, 128, 3)
    c = oracle.OracleCache(2, 32, 32, 128, 1, 1, 128)
    c.prefill(k, v)
    st = c.export()
    nqk, nqv = oracle.nq_k(100, 32, 32), oracle.nq_v(100, 32, 32)
    assert not st["codes_k"][0, 0, nqk:].any() and not st["scale_v"][0, 0, nqv:].any()
    assert st["scale_k"][0, 0, nqk // 32 - 1].all() and st["scale_v"][0, 0, nqv - 1].all()


# ---------------------------------------------------------------- attention

def test_attention_fp32_matches_double_brute_force(oracle):
    """Decode attention = softmax(q K^T / sqrt(D)) V over the dequantized cache."""
    B, Hq, H, T, D, G, R = 2, 4, 2, 90, 32, 16, 32
    k, v = _rand_kv(B, H, T, D, 11)
    c = oracle.OracleCache(2, G, R, D, B, H, 96)
    c.prefill(k, v)
    rng = np.random.default_rng(12)
    q = rng.standard_normal((B, Hq, D), np.float32)
    out = c.attention(q)
    for b in range(B):
        for j in range(Hq):
            kh, vh = c.dequant(b, j // (Hq // H))
            ref = oracle.attention_f64(q[b, j], kh, vh, 1 / math.sqrt(D))
            err = np.abs(out[b, j] - ref).max() / np.abs(ref).max()
            assert err < 1e-5


def test_attention_below_window_is_plain_softmax(oracle):
    """Below the residual window nothing is quantized: attention over the fp16
    inputs, checked with numpy's softmax in double."""
    B, Hq, H, T, D = 1, 2, 1, 20, 128
    k, v = _rand_kv(B, H, T, D, 13)
    c = oracle.OracleCache(2, 32, 32, D, B, H, 64)
    c.prefill(k, v)
    q = np.random.default_rng(14).standard_normal((B, Hq, D), np.float32)
    out = c.attention(q, 0.1)
    K = k[0, 0].astype(np.float64)
    V = v[0, 0].astype(np.float64)
    for j in range(Hq):
        s = K @ q[0, j].astype(np.float64) * 0.1
        p = np.exp(s - s.max())
        ref = (p / p.sum()) @ V
        assert np.abs(out[0, j] - ref).max() <= 1e-5 * np.abs(ref).max()


def test_split_combine_identity():
    """Splitting the context and merging (m, l, o) partials equals one pass
    (the identity the GPU's split-K combine relies on), in double."""
    rng = np.random.default_rng(15)
    s = rng.standard_normal(1000) * 3
    V = rng.standard_normal((1000, 16))
    p = np.exp(s - s.max())
    ref = p @ V / p.sum()
    edges = [0, 7, 300, 301, 999, 1000]
    parts = []
    for a, b in zip(edges[:-1], edges[1:]):
        m = s[a:b].max()
        e = np.exp(s[a:b] - m)
        parts.append((m, e.sum(), e @ V[a:b]))
    M = max(m for m, _, _ in parts)
    den = sum(l * math.exp(m - M) for m, l, _ in parts)
    num = sum(o * math.exp(m - M) for m, _, o in parts)
    assert np.allclose(num / den, ref, rtol=1e-12, atol=1e-12)


def test_single_head_workload_is_the_notebooks(oracle):
    wl = W.single_head()
    assert wl.k.shape == (1, 1, 1024, 128) and wl.k.dtype == np.float32
    # outlier channels are 5x larger in spread
    sd = wl.k[0, 0].std(axis=0)
    assert set(np.argsort(sd)[-4:]) == {3, 17, 40, 88}
    assert wl.v[0, 0].std() == pytest.approx(0.5, rel=0.05)
