"""Multi-token append (chunked prefill into a non-empty cache) and state
restore, through the C ABI, against the CPU oracle appending token by token.

The cache left by appending n tokens at once must equal, bit for bit, the one
that n single appends (the review's Algorithm 1, decoding phase) leave; a
cache rebuilt from copies of another's buffers plus its length must behave
identically."""
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


def _chunk(x, a, b):
    return np.ascontiguousarray(x[:, :, a:b])


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
@pytest.mark.parametrize("R", [32, 64, 128])
@pytest.mark.parametrize("dtype", ["f16", "bf16", "f32"])
def test_append_tokens_matches_token_by_token(bits, R, dtype):
    """A prefill, then chunks of 1..200 tokens mixed with single appends;
    the state after every chunk and attention at the end."""
    chunks = [1, 5, 31, 32, 33, 100, 0, 7, 200, 64, 0, 1, 95]  # 0: a single append_decode
    total = 300 + sum(max(c, 1) for c in chunks)
    wl = W.synthetic("at", B=2, Hq=8, Hkv=2, T=total, R=R, bits=bits, dtype=dtype, seed=bits * 10 + R)
    cap = (total + 127) // 128 * 128  # a multiple of every R used here
    g = T.gpu_cache(wl, capacity=cap)
    o = T.oracle_cache(wl, capacity=cap)
    l0 = 300
    g.prefill(T.dev(_chunk(wl.k, 0, l0), dtype), T.dev(_chunk(wl.v, 0, l0), dtype))
    o.prefill(_chunk(wl.k, 0, l0), _chunk(wl.v, 0, l0))
    l = l0
    for c in chunks:
        if c == 0:
            g.append(T.dev(np.ascontiguousarray(wl.k[:, :, l]), dtype), T.dev(np.ascontiguousarray(wl.v[:, :, l]), dtype))
            o.append(np.ascontiguousarray(wl.k[:, :, l]), np.ascontiguousarray(wl.v[:, :, l]))
            l += 1
            continue
        g.append_tokens(T.dev(_chunk(wl.k, l, l + c), dtype), T.dev(_chunk(wl.v, l, l + c), dtype))
        for t in range(l, l + c):
            o.append(np.ascontiguousarray(wl.k[:, :, t]), np.ascontiguousarray(wl.v[:, :, t]))
        l += c
        assert g.length == l == o.length
        T.compare_state(T.gpu_state(g), o.export(), l, R, 32)
    out = T.out_float(g.attention(T.dev(wl.q, wl.q_dtype)))
    assert T.attn_err(out, o.attention(T.q_float(wl.q, wl.q_dtype))) <= T.ATTN_TOL


def test_append_tokens_on_empty_cache_equals_prefill():
    wl = W.synthetic("ae", B=2, Hq=4, Hkv=2, T=777, R=32, seed=3)
    a = T.gpu_cache(wl)
    a.append_tokens(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"))
    b = T.gpu_cache(wl)
    b.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"))
    sa, sb = T.gpu_state(a), T.gpu_state(b)
    T.compare_state(sa, {k: v for k, v in sb.items()}, 777, 32, 32)


def test_append_tokens_capacity():
    from bit_kv_cache_kivi_gb300.kivi import KiviError
    wl = W.synthetic("ac", B=1, Hq=2, Hkv=1, T=64, R=32, seed=4)
    g = T.gpu_cache(wl, capacity=64)
    g.prefill(T.dev(_chunk(wl.k, 0, 40), "f16"), T.dev(_chunk(wl.v, 0, 40), "f16"))
    with pytest.raises(KiviError) as e:
        g.append_tokens(T.dev(_chunk(wl.k, 0, 25), "f16"), T.dev(_chunk(wl.v, 0, 25), "f16"))
    assert e.value.status == 3  # capacity
    assert g.length == 40
    g.append_tokens(T.dev(_chunk(wl.k, 40, 64), "f16"), T.dev(_chunk(wl.v, 40, 64), "f16"))
    assert g.length == 64


def test_state_restore_from_copied_buffers():
    """Copy a cache's eight buffers into a second cache, declare the length:
    attention and the following appends are identical."""
    wl = W.synthetic("st", B=2, Hq=8, Hkv=2, T=1000, R=32, steps=40, seed=9)
    a = T.gpu_cache(wl)
    a.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"))
    for i in range(7):
        a.append(T.dev(wl.k_new[i], "f16"), T.dev(wl.v_new[i], "f16"))
    b = T.gpu_cache(wl)
    for name, t in a.state_views().items():
        b.state_views()[name].copy_(t)
    b.set_length(a.length)
    q = T.dev(wl.q, "f16")
    assert torch.equal(a.attention(q), b.attention(q))
    for i in range(7, 40):
        for c in (a, b):
            c.append(T.dev(wl.k_new[i], "f16"), T.dev(wl.v_new[i], "f16"))
    sa, sb = T.gpu_state(a), T.gpu_state(b)
    for name in sa:
        assert np.array_equal(sa[name], sb[name]), name
    assert torch.equal(a.attention(q), b.attention(q))
