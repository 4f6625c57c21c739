"""The shared-window residual policy (veloxquant-mlx "KIVI", How it works
items 3-4: keys and values keep at least the R most recent tokens in fp16,
aged-out tokens are quantized in whole groups of G) on the CUDA path, against
the oracle's same policy: prefill, appends across flushes, multi-token
appends and decode attention."""
import numpy as np
import pytest
import torch

from bit_kv_cache_kivi_gb300 import workloads as W
import kivi_testlib as T

pytestmark = pytest.mark.gpu
S = T.SHARED


@pytest.fixture(scope="module", autouse=True)
def _lib():
    from bit_kv_cache_kivi_gb300 import build, kivi
    build.build()
    kivi.lib()
    torch.cuda.init()


def _check_attn(g, o, wl):
    out = T.out_float(g.attention(T.dev(wl.q, wl.q_dtype)))
    assert T.attn_err(out, o.attention(T.q_float(wl.q, wl.q_dtype))) <= T.ATTN_TOL


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
@pytest.mark.parametrize("R", [32, 64])
@pytest.mark.parametrize("T_", [1, 31, 33, 63, 64, 65, 95, 96, 97, 500, 1031])
def test_shared_prefill_state_and_attention(bits, R, T_):
    cap = (T_ + 2 * R + 63) // 64 * 64
    wl = W.synthetic("sp", B=2, Hq=8, Hkv=2, T=T_, R=R, bits=bits, seed=T_ + R)
    g = T.gpu_cache(wl, capacity=cap, policy=S)
    g.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"))
    o = T.oracle_cache(wl, capacity=cap, policy=S)
    o.prefill(wl.k, wl.v)
    T.compare_state(T.gpu_state(g), o.export(), T_, R, 32, policy=S)
    _check_attn(g, o, wl)


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
@pytest.mark.parametrize("R", [32, 64])
def test_shared_appends_across_flushes(bits, R):
    wl = W.synthetic("sa", B=2, Hq=8, Hkv=2, T=R + 5, R=R, bits=bits, steps=3 * 32 + 7,
                     seed=3 * bits + R)
    cap = (wl.T + wl.steps + 63) // 64 * 64
    g = T.gpu_cache(wl, capacity=cap, policy=S)
    g.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"))
    o = T.oracle_cache(wl, capacity=cap, policy=S)
    o.prefill(wl.k, wl.v)
    l = wl.T
    for i in range(wl.steps):
        g.append(T.dev(wl.k_new[i], "f16"), T.dev(wl.v_new[i], "f16"))
        o.append(wl.k_new[i], wl.v_new[i])
        l += 1
        if (l - R) % 32 in (0, 1, 31) or i == wl.steps - 1:
            T.compare_state(T.gpu_state(g), o.export(), l, R, 32, policy=S)
        if (l - R) % 32 in (0, 1) or i == wl.steps - 1:
            out = T.out_float(g.attention(T.dev(wl.q_for_step(i), "f16")))
            ref = o.attention(T.q_float(wl.q_for_step(i), "f16"))
            assert T.attn_err(out, ref) <= T.ATTN_TOL


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_shared_append_tokens_and_stream_equals_prefill(bits):
    """Chunks appended at once equal the oracle's token-by-token appends, and
    the final cache equals a one-shot prefill of all the tokens."""
    R = 64
    chunks = [7, 1, 40, 100, 33, 64, 1, 200]
    total = 150 + sum(chunks)
    cap = (total + 63) // 64 * 64
    wl = W.synthetic("st", B=2, Hq=4, Hkv=2, T=total, R=R, bits=bits, seed=40 + bits)
    g = T.gpu_cache(wl, capacity=cap, policy=S)
    o = T.oracle_cache(wl, capacity=cap, policy=S)
    k = lambda a, b: np.ascontiguousarray(wl.k[:, :, a:b])
    v = lambda a, b: np.ascontiguousarray(wl.v[:, :, a:b])
    g.prefill(T.dev(k(0, 150), "f16"), T.dev(v(0, 150), "f16"))
    o.prefill(k(0, 150), v(0, 150))
    l = 150
    for c in chunks:
        g.append_tokens(T.dev(k(l, l + c), "f16"), T.dev(v(l, l + c), "f16"))
        for t in range(l, l + c):
            o.append(np.ascontiguousarray(wl.k[:, :, t]), np.ascontiguousarray(wl.v[:, :, t]))
        l += c
        T.compare_state(T.gpu_state(g), o.export(), l, R, 32, policy=S)
    one = T.gpu_cache(wl, capacity=cap, policy=S)
    one.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"))
    T.compare_state(T.gpu_state(g), T.gpu_state(one), total, R, 32, policy=S)
    _check_attn(g, o, wl)
