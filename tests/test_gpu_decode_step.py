"""The one-call decode step (chooblog KIVI review §1.3, decoding phase: the
new token's key and value join the cache, then the query attends over every
token) on the CUDA path.  kivi_decode_step launches the attention as a
programmatic dependent of the append; its cache and output must be bit for
bit those of kivi_append_decode followed by kivi_decode_attention, and the
cache must equal the oracle's after the same appends."""
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


def _run(wl, steps, policy=T.ALG1, outliers=0, dtype="f16", cap=None, check_every=1):
    cap = cap or -(-(wl.T + steps + 2 * wl.R) // 128) * 128  # a multiple of R (32 or 128)
    a = T.gpu_cache(wl, capacity=cap, policy=policy, outliers=outliers)  # step()
    b = T.gpu_cache(wl, capacity=cap, policy=policy, outliers=outliers)  # append() + attention()
    a.prefill(T.dev(wl.k, dtype), T.dev(wl.v, dtype))
    b.prefill(T.dev(wl.k, dtype), T.dev(wl.v, dtype))
    q = T.dev(wl.q, wl.q_dtype)
    for i in range(steps):
        kn, vn = T.dev(wl.k_new[i], dtype), T.dev(wl.v_new[i], dtype)
        oa = a.step(kn, vn, q)
        b.append(kn, vn)
        ob = b.attention(q)
        if i % check_every == 0 or i == steps - 1:
            torch.cuda.synchronize()
            assert torch.equal(oa, ob), f"step {i}: outputs differ"
    assert a.length == b.length == wl.T + steps
    return a, b


@pytest.mark.parametrize("policy", [T.ALG1, T.SHARED])
@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_step_matches_append_then_attention(bits, policy):
    wl = W.synthetic("ds", B=2, Hq=8, Hkv=2, T=200, R=32, bits=bits, steps=70, seed=7 * bits + policy)
    a, b = _run(wl, wl.steps, policy=policy)
    l = wl.T + wl.steps
    cap = a.cfg.max_tokens
    o = T.oracle_cache(wl, capacity=cap, policy=policy)
    o.prefill(wl.k, wl.v)
    for i in range(wl.steps):
        o.append(wl.k_new[i], wl.v_new[i])
    T.compare_state(T.gpu_state(a), o.export(), l, wl.R, 32, policy=policy)
    out = T.out_float(a.attention(T.dev(wl.q, wl.q_dtype)))
    assert T.attn_err(out, o.attention(T.q_float(wl.q, wl.q_dtype))) <= T.ATTN_TOL


@pytest.mark.parametrize("policy", [T.ALG1, T.SHARED])
def test_steps_from_an_empty_cache(policy):
    """Lengths 1, 2, ... from nothing: only tail splits at first, then the
    first flushes and the first packed tiles."""
    wl = W.synthetic("de", B=2, Hq=8, Hkv=2, T=0, R=32, steps=100, seed=41 + policy)
    cap = 128
    a = T.gpu_cache(wl, capacity=cap, policy=policy)
    b = T.gpu_cache(wl, capacity=cap, policy=policy)
    q = T.dev(wl.q, wl.q_dtype)
    o = T.oracle_cache(wl, capacity=cap, policy=policy)
    for i in range(wl.steps):
        kn, vn = T.dev(wl.k_new[i], "f16"), T.dev(wl.v_new[i], "f16")
        oa = a.step(kn, vn, q)
        b.append(kn, vn)
        ob = b.attention(q)
        o.append(wl.k_new[i], wl.v_new[i])
        torch.cuda.synchronize()
        assert torch.equal(oa, ob), f"step {i}"
        if i in (0, 31, 32, 63, 64, 99):
            T.compare_state(T.gpu_state(a), o.export(), i + 1, wl.R, 32, policy=policy)
            assert T.attn_err(T.out_float(oa), o.attention(T.q_float(wl.q, wl.q_dtype))) <= T.ATTN_TOL


@pytest.mark.parametrize("dtype", ["bf16", "f32"])
def test_step_other_input_dtypes(dtype):
    wl = W.synthetic("dt", B=1, Hq=4, Hkv=1, T=95, R=32, steps=40, seed=3, dtype=dtype)
    _run(wl, wl.steps, dtype=dtype)


@pytest.mark.parametrize("bits", [2, 3])
def test_step_outlier_channels(bits):
    """R = 32, GQA 4, outlier keys: most steps let the packed splits run
    beside the append (only the tail waits), with key flushes that write the
    outlier blocks; the cache must equal the oracle's."""
    wl = W.synthetic("dq", B=2, Hq=8, Hkv=2, T=130, R=32, bits=bits, steps=70, seed=17 + bits)
    a, _ = _run(wl, wl.steps, outliers=2)
    o = T.oracle_cache(wl, capacity=a.cfg.max_tokens, outliers=2)
    o.prefill(wl.k, wl.v)
    for i in range(wl.steps):
        o.append(wl.k_new[i], wl.v_new[i])
    T.compare_state(T.gpu_state(a), o.export(), wl.T + wl.steps, wl.R, 32)


def test_step_outlier_channels_and_long_residual():
    wl = W.synthetic("do", B=2, Hq=8, Hkv=2, T=300, R=128, steps=140, seed=11)
    _run(wl, wl.steps, outliers=2, check_every=7)


def test_step_many_units_tail_on_last_split():
    """Enough (batch, kv-head, head chunk) units that one wave has no room
    for a separate tail split (GQA 7: two head chunks per kv-head)."""
    wl = W.synthetic("du", B=48, Hq=28, Hkv=4, T=300, R=32, steps=36, seed=5)
    a, _ = _run(wl, wl.steps, check_every=5)
    assert a.splits() >= 1


def test_step_ragged_batch():
    wl = W.synthetic("dr", B=3, Hq=8, Hkv=2, T=260, R=32, steps=40, seed=9)
    lens = [260, 31, 97]
    cap = 384
    a = T.gpu_cache(wl, capacity=cap)
    b = T.gpu_cache(wl, capacity=cap)
    k, v = T.dev(wl.k, "f16"), T.dev(wl.v, "f16")
    a.prefill(k, v, lengths=lens)
    b.prefill(k, v, lengths=lens)
    q = T.dev(wl.q, wl.q_dtype)
    for i in range(wl.steps):
        kn, vn = T.dev(wl.k_new[i], "f16"), T.dev(wl.v_new[i], "f16")
        oa = a.step(kn, vn, q)
        b.append(kn, vn)
        ob = b.attention(q)
        torch.cuda.synchronize()
        assert torch.equal(oa, ob), f"step {i}"
    assert a.lengths == b.lengths == [x + wl.steps for x in lens]


def test_step_pinned_host_buffers():
    wl = W.synthetic("dh", B=2, Hq=8, Hkv=2, T=120, R=32, steps=40, seed=13)
    cap = 256
    a = T.gpu_cache(wl, capacity=cap)
    b = T.gpu_cache(wl, capacity=cap)
    a.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"))
    b.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"))
    qh = W.to_torch(wl.q, wl.q_dtype).pin_memory()
    oh = torch.empty_like(qh).pin_memory()
    qd = T.dev(wl.q, wl.q_dtype)
    for i in range(wl.steps):
        kh = W.to_torch(wl.k_new[i], "f16").pin_memory()
        vh = W.to_torch(wl.v_new[i], "f16").pin_memory()
        a.step(kh, vh, qh, oh)
        b.append(T.dev(wl.k_new[i], "f16"), T.dev(wl.v_new[i], "f16"))
        ob = b.attention(qd)
        torch.cuda.synchronize()
        assert torch.equal(oh, ob.cpu()), f"step {i}"


def test_step_refusal_leaves_cache_unchanged():
    from bit_kv_cache_kivi_gb300 import kivi as K
    wl = W.synthetic("dx", B=1, Hq=4, Hkv=1, T=64, R=32, steps=1, seed=1)
    a = T.gpu_cache(wl, capacity=64)
    a.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"))
    with pytest.raises(K.KiviError) as e:
        a.step(T.dev(wl.k_new[0], "f16"), T.dev(wl.v_new[0], "f16"), T.dev(wl.q, wl.q_dtype))
    assert e.value.status == K.KIVI_ECAPACITY and a.length == 64
    page_q = np.ascontiguousarray(W.cast(wl.q, "f16"))
    b = T.gpu_cache(wl, capacity=128)
    b.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"))
    st = K.lib().kivi_decode_step(b.handle, T.dev(wl.k_new[0], "f16").data_ptr(),
                                  T.dev(wl.v_new[0], "f16").data_ptr(), K.KIVI_F16,
                                  page_q.ctypes.data, K.KIVI_F16, b.workspace.data_ptr(), 0.0,
                                  b.workspace.data_ptr(), b.ws_bytes, None)
    assert st == K.KIVI_EINVAL and b.length == 64
