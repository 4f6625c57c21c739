"""Parity of the CUDA path (through the C ABI) against the CPU oracle.

Cache contents (packed codes, fp16 scale/zero, residual rings) must match
bit for bit; decode attention within max relative error 2e-3 per
(batch, query head).  Sizes span several tiles and ragged tails; the
workloads' full sizes are covered in test_gpu_parity_fullsize.py.
"""
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


def run_prefill(wl, bits=None, capacity=None):
    g = T.gpu_cache(wl, capacity, bits)
    g.prefill(T.dev(wl.k, wl.dtype), T.dev(wl.v, wl.dtype))
    o = T.oracle_cache(wl, capacity, bits)
    o.prefill(wl.k, wl.v)
    return g, o


def check_attention(g, o, wl, q=None, splits=None):
    q = wl.q if q is None else q
    if splits is not None:
        g.set_splits(splits)
    out = T.out_float(g.attention(T.dev(q, wl.q_dtype)))
    ref = o.attention(T.q_float(q, wl.q_dtype))
    err = T.attn_err(out, ref, wl.q_dtype)
    assert err <= T.ATTN_TOL, err
    return out


# ---------------------------------------------------------------- quantizer

def test_single_head_notebook_workload():
    """fp32 input, T=1024, R=32: codes bit-exact, then attention."""
    wl = W.single_head()
    g, o = run_prefill(wl)
    T.compare_state(T.gpu_state(g), o.export(), wl.T, wl.R, wl.G)
    check_attention(g, o, wl)


@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
@pytest.mark.parametrize("bits", [2, 3, 4, 8])
@pytest.mark.parametrize("T_,R", [(1000, 32), (777, 64), (95, 32), (32, 32), (20, 32),
                                  (33, 32), (64, 64)])
def test_prefill_state_bit_exact(dtype, bits, T_, R):
    wl = W.synthetic("p", B=2, Hq=4, Hkv=2, T=T_, R=R, bits=bits, dtype=dtype, seed=T_ + R,
                     v_spike_frac=0.01)
    g, o = run_prefill(wl)
    T.compare_state(T.gpu_state(g), o.export(), T_, R, 32)


def test_prefill_extreme_values():
    """Constant groups (zero range), tiny ranges (fp16 subnormal scales), huge
    values, negative zeros and exact ties in one cache."""
    rng = np.random.default_rng(0)
    k = rng.standard_normal((1, 2, 256, 128)).astype(np.float32)
    v = rng.standard_normal((1, 2, 256, 128)).astype(np.float32)
    k[0, 0, :32, :] = 1.5                      # every K group of chunk 0 constant
    v[0, 0, 40, :] = -0.0                      # a V token of negative zeros
    v[0, 0, 41, :32] = 0.0
    v[0, 0, 41, 16] = -0.0
    k[0, 1, 32:64, 5] = rng.integers(0, 4, 32) * 2.0 ** -24   # subnormal range
    v[0, 1, 50, :32] = np.arange(32) * 2.0 ** -20
    k[0, 1, 64:96, 7] = rng.standard_normal(32) * 8e3          # large, within fp16
    v[0, 0, 60, 64:96] = np.array([0, 3] * 16)                  # 2-bit scale exactly 1
    v[0, 0, 60, 70] = 1.5                                       # an exact tie
    for bits in (2, 3, 4):
        wl = W.synthetic("x", B=1, Hq=2, Hkv=2, T=256, bits=bits, seed=1)
        wl.k, wl.v = k.astype(np.float16), v.astype(np.float16)
        g, o = run_prefill(wl)
        T.compare_state(T.gpu_state(g), o.export(), 256, 32, 32)


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_prefill_tie_heavy_lattices(bits, dtype):
    """Inputs on coarse dyadic lattices make (x - z)/s land exactly on, or
    within a few ulps of, half-integers for many elements: every such
    rounding decision must match the oracle's IEEE division bit for bit."""
    rng = np.random.default_rng(77 + bits)
    shape = (2, 2, 320, 128)
    step = 2.0 ** rng.integers(-6, 3, size=(2, 2, 1, 128))
    k = rng.integers(-8, 9, size=shape) * step / 2
    v = rng.integers(-8, 9, size=shape) * (2.0 ** rng.integers(-6, 3, size=(2, 2, 320, 1))) / 4
    k[:, :, ::7] *= 3.0      # ranges that give scales like 2.5 or 3.5
    v[:, :, 1::5] += 0.125
    wl = W.synthetic("ties", B=2, Hq=4, Hkv=2, T=320, bits=bits, dtype=dtype, seed=5)
    wl.k, wl.v = W.cast(k, dtype), W.cast(v, dtype)
    g, o = run_prefill(wl)
    T.compare_state(T.gpu_state(g), o.export(), 320, 32, 32)


# ---------------------------------------------------------------- append

@pytest.mark.parametrize("bits", [2, 3, 4, 8])
@pytest.mark.parametrize("R", [32, 64])
def test_append_crosses_flushes(bits, R):
    """Decode appends through several K flushes and V evictions; state checked
    after every step near the boundaries, attention at a few lengths."""
    wl = W.synthetic("a", B=2, Hq=8, Hkv=2, T=R * 3 - 5, R=R, bits=bits, steps=3 * R + 3,
                     seed=7 + bits)
    g, o = run_prefill(wl)
    l = wl.T
    for i in range(wl.steps):
        kn, vn = wl.k_new[i], wl.v_new[i]
        g.append(T.dev(kn, wl.dtype), T.dev(vn, wl.dtype))
        o.append(kn, vn)
        l += 1
        if l % R in (0, 1, R - 1) or i == wl.steps - 1:
            T.compare_state(T.gpu_state(g), o.export(), l, R, 32)
        if l % R in (0, 1) or i == wl.steps - 1:
            check_attention(g, o, wl, q=wl.q_for_step(i))


def test_stream_equals_prefill_on_gpu():
    """One-shot prefill and token-by-token decode give bit-identical caches."""
    wl = W.synthetic("s", B=2, Hq=4, Hkv=2, T=200, R=32, steps=0, seed=3)
    full = T.gpu_cache(wl)
    full.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"))
    want = T.gpu_state(full)
    for T0 in (0, 1, 31, 32, 100, 199):
        g = T.gpu_cache(wl)
        if T0:
            g.prefill(T.dev(np.ascontiguousarray(wl.k[:, :, :T0]), "f16"),
                      T.dev(np.ascontiguousarray(wl.v[:, :, :T0]), "f16"))
        for t in range(T0, 200):
            g.append(T.dev(np.ascontiguousarray(wl.k[:, :, t]), "f16"),
                     T.dev(np.ascontiguousarray(wl.v[:, :, t]), "f16"))
        assert g.length == 200
        T.compare_state(T.gpu_state(g), want, 200, 32, 32)


def test_capacity_and_state_errors():
    from bit_kv_cache_kivi_gb300.kivi import KiviError
    wl = W.synthetic("c", B=1, Hq=2, Hkv=1, T=64, R=32, steps=1, seed=4)
    g = T.gpu_cache(wl, capacity=64)
    with pytest.raises(KiviError) as e:
        g.attention(T.dev(wl.q, "f16"))
    assert e.value.status == 6  # empty cache
    g.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"))
    with pytest.raises(KiviError) as e:
        g.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"))
    assert e.value.status == 6  # prefill into a non-empty cache
    with pytest.raises(KiviError) as e:
        g.append(T.dev(wl.k_new[0], "f16"), T.dev(wl.v_new[0], "f16"))
    assert e.value.status == 3  # full
    assert g.length == 64
    g.reset()
    assert g.length == 0


# ---------------------------------------------------------------- attention

@pytest.mark.parametrize("Hq,Hkv", [(1, 1), (2, 1), (8, 2), (28, 4), (18, 1), (24, 2)])
@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_attention_gqa_shapes(Hq, Hkv, bits):
    wl = W.synthetic("g", B=2, Hq=Hq, Hkv=Hkv, T=1100, R=32, bits=bits, seed=Hq * 10 + Hkv)
    g, o = run_prefill(wl)
    check_attention(g, o, wl)


@pytest.mark.parametrize("T_", [1, 5, 31, 32, 33, 63, 64, 65, 300])
def test_attention_short_contexts(T_):
    """Below, at and just past the window: ring-only, mixed and packed tiles."""
    wl = W.synthetic("sh", B=1, Hq=4, Hkv=2, T=T_, R=32, seed=T_)
    g, o = run_prefill(wl)
    check_attention(g, o, wl)


@pytest.mark.parametrize("R", [32, 128])
@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_attention_tail_on_last_packed_split(R, bits):
    """320 (batch, kv-head) units leave no room in one wave for a tail split,
    so the last packed split also takes the tail (one or three 64-token
    rounds)."""
    wl = W.synthetic("tf", B=80, Hq=8, Hkv=4, T=450, R=R, bits=bits, seed=R + bits)
    g, o = run_prefill(wl)
    assert g.splits() == 1
    check_attention(g, o, wl)


def test_attention_split_count_invariance():
    wl = W.synthetic("sp", B=1, Hq=8, Hkv=2, T=3000, R=128, seed=11)
    g, o = run_prefill(wl)
    outs = [check_attention(g, o, wl, splits=s) for s in (1, 2, 7, 40)]
    for x in outs[1:]:
        assert T.attn_err(x, outs[0]) <= T.ATTN_TOL


def test_attention_maximum_splits():
    """The split cap: one (batch, kv-head) unit at 65320 tokens (2040 packed
    tiles and a 40-token tail) plans 255 packed splits of 8 tiles and one
    tail split, so 256 partials merge in two full levels of 16.  Overrides
    of 241 and 17 plan 228 splits (a last group of 4) and 17 (a last group
    of one)."""
    wl = W.synthetic("mx", B=1, Hq=4, Hkv=1, T=65320, R=32, seed=29)
    g, o = run_prefill(wl, capacity=65536)
    assert g.splits() == 256
    outs = [check_attention(g, o, wl)]
    for s, planned in ((241, 228), (17, 17)):
        outs.append(check_attention(g, o, wl, splits=s))
        assert g.splits() == planned
    for x in outs[1:]:
        assert T.attn_err(x, outs[0]) <= T.ATTN_TOL


@pytest.mark.parametrize("q_dtype", ["f32", "bf16"])
def test_attention_query_dtypes(q_dtype):
    wl = W.synthetic("qd", B=2, Hq=4, Hkv=2, T=500, R=32, q_dtype=q_dtype, seed=21)
    g, o = run_prefill(wl)
    check_attention(g, o, wl)


def test_attention_softmax_scale_and_sharp_scores():
    """An explicit scale, and large logits (a near one-hot softmax)."""
    wl = W.synthetic("sc", B=1, Hq=4, Hkv=1, T=700, R=32, seed=22)
    g, o = run_prefill(wl)
    for scale in (0.02, 1.0):
        out = T.out_float(g.attention(T.dev(wl.q, "f16"), softmax_scale=scale))
        ref = o.attention(T.q_float(wl.q, "f16"), scale)
        assert T.attn_err(out, ref) <= T.ATTN_TOL


def test_attention_is_deterministic():
    wl = W.synthetic("det", B=2, Hq=8, Hkv=2, T=2000, R=32, seed=23)
    g, _ = run_prefill(wl)
    q = T.dev(wl.q, "f16")
    a = g.attention(q).clone()
    b = g.attention(q)
    assert torch.equal(a, b)
