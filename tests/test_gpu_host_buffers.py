"""Per-call inputs and outputs in page-locked host memory.

The C library accepts k, v, k_new, v_new, q and out in pinned host memory
(the kernels read and write them directly); the result must be bit for bit
the one the same call gives with device buffers.  Pageable host memory must
be refused with KIVI_EINVAL before any launch, leaving the cache unchanged."""
import ctypes as C

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


def _pinned(x: np.ndarray, dtype: str) -> torch.Tensor:
    return W.to_torch(x, dtype).pin_memory()


@pytest.mark.parametrize("policy", [T.ALG1, T.SHARED])
@pytest.mark.parametrize("dtype", ["f16", "bf16"])
def test_host_buffers_match_device_buffers(policy, dtype):
    wl = W.synthetic("hb", B=2, Hq=8, Hkv=2, T=300, R=32, steps=40, seed=21 + policy, dtype=dtype)
    a = T.gpu_cache(wl, capacity=384, policy=policy)
    b = T.gpu_cache(wl, capacity=384, policy=policy)
    a.prefill(T.dev(wl.k, dtype), T.dev(wl.v, dtype))
    b.prefill(_pinned(wl.k, dtype), _pinned(wl.v, dtype))
    for i in range(33):  # across a key flush
        a.append(T.dev(wl.k_new[i], dtype), T.dev(wl.v_new[i], dtype))
        b.append(_pinned(wl.k_new[i], dtype), _pinned(wl.v_new[i], dtype))
    kc = np.ascontiguousarray(np.moveaxis(wl.k_new[33:40], 0, 2))
    vc = np.ascontiguousarray(np.moveaxis(wl.v_new[33:40], 0, 2))
    a.append_tokens(T.dev(kc, dtype), T.dev(vc, dtype))
    b.append_tokens(_pinned(kc, dtype), _pinned(vc, dtype))
    # the live part of the two states (rows past it are uninitialized memory)
    T.compare_state(T.gpu_state(b), T.gpu_state(a), 340, 32, 32, policy=policy)
    out_d = a.attention(T.dev(wl.q, wl.q_dtype))
    q_h = _pinned(wl.q, wl.q_dtype)
    out_h = torch.empty_like(q_h).pin_memory()
    b.attention(q_h, out_h)
    torch.cuda.synchronize()
    assert out_h.device.type == "cpu"
    assert torch.equal(out_d.cpu(), out_h)


def test_pageable_host_memory_is_refused():
    from bit_kv_cache_kivi_gb300 import kivi as K
    wl = W.synthetic("hp", B=1, Hq=4, Hkv=2, T=64, R=32, steps=1, seed=5)
    g = T.gpu_cache(wl, capacity=128)
    g.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"))
    lib = K.lib()
    page_k = np.ascontiguousarray(W.cast(wl.k_new[0], "f16"))  # ordinary (pageable) numpy memory
    page_v = np.ascontiguousarray(W.cast(wl.v_new[0], "f16"))
    st = lib.kivi_append_decode(g.handle, page_k.ctypes.data, page_v.ctypes.data, K.KIVI_F16, None)
    assert st == K.KIVI_EINVAL and g.length == 64
    page_q = np.ascontiguousarray(W.cast(wl.q, "f16"))
    page_o = np.zeros_like(page_q)
    st = lib.kivi_decode_attention(g.handle, page_q.ctypes.data, K.KIVI_F16, page_o.ctypes.data, 0.0,
                                   g.workspace.data_ptr(), g.ws_bytes, None)
    assert st == K.KIVI_EINVAL and not page_o.any()
    # through the binding: the library's refusal, before any launch
    with pytest.raises(K.KiviError) as e:
        g.append(torch.from_numpy(page_k), torch.from_numpy(page_v))
    assert e.value.status == K.KIVI_EINVAL and g.length == 64
    with pytest.raises(K.KiviError):
        g.attention(torch.from_numpy(page_q))
    # and the cache still works
    q = T.dev(wl.q, "f16")
    o = T.oracle_cache(wl, capacity=128)
    o.prefill(wl.k, wl.v)
    assert T.attn_err(T.out_float(g.attention(q)), o.attention(T.q_float(wl.q, "f16"))) <= T.ATTN_TOL


def test_cache_buffers_in_pageable_memory_are_refused():
    """The cache's own buffers must be device (or managed) memory: a handle
    over ordinary host memory is refused at its first launching call, before
    any launch."""
    from bit_kv_cache_kivi_gb300 import kivi as K
    cfg = K.kivi_config(2, 32, 32, 128, 1, 1, 4, 64)
    sizes = K.kivi_cache_sizes(cfg)
    host = [np.zeros(n + 16, np.uint8) for n in sizes]
    ptrs = [a.ctypes.data + (-a.ctypes.data) % 16 for a in host]  # 16-byte aligned
    h = K.kivi_cache_init(cfg, K.kivi_buffers(*ptrs))
    try:
        k = T.dev(np.zeros((1, 1, 32, 128), np.float16), "f16")
        st = K.lib().kivi_quantize_prefill(h, k.data_ptr(), k.data_ptr(), K.KIVI_F16, 32, None)
        assert st == K.KIVI_EINVAL and K.kivi_cache_length(h) == 0
    finally:
        K.kivi_cache_destroy(h)
