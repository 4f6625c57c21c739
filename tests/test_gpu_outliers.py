"""Outlier-aware keys (the "KIVI - 2-bit KV cache quantisation" notebook,
Exercises item 2) through the C ABI, against the CPU oracle's same reading:
per key group, the channels with the largest max |k| stay fp16.  The whole
state -- the kept channels and values included -- must match bit for bit
after prefill, single appends and multi-token appends, and attention must
stay within tolerance."""
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


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
@pytest.mark.parametrize("n_out", [1, 2, 4])
@pytest.mark.parametrize("policy", [T.ALG1, T.SHARED])
def test_outliers_prefill_appends_attention(bits, n_out, policy):
    R = 64
    wl = W.synthetic("ol", B=2, Hq=8, Hkv=2, T=500, R=R, bits=bits, steps=140,
                     seed=bits * 100 + n_out * 10 + policy)
    cap = (500 + 140 + R - 1) // R * R
    g = T.gpu_cache(wl, capacity=cap, policy=policy, outliers=n_out)
    o = T.oracle_cache(wl, capacity=cap, policy=policy, outliers=n_out)
    g.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"))
    o.prefill(wl.k, wl.v)
    T.compare_state(T.gpu_state(g), o.export(), 500, R, 32, policy=policy)
    qf = T.q_float(wl.q, wl.q_dtype)
    q = T.dev(wl.q, wl.q_dtype)
    assert T.attn_err(T.out_float(g.attention(q)), o.attention(qf)) <= T.ATTN_TOL
    # single appends across flushes (ALG1 flushes R keys at once), then a chunk
    for i in range(100):
        g.append(T.dev(wl.k_new[i], "f16"), T.dev(wl.v_new[i], "f16"))
        o.append(wl.k_new[i], wl.v_new[i])
    T.compare_state(T.gpu_state(g), o.export(), 600, R, 32, policy=policy)
    kc = np.ascontiguousarray(np.moveaxis(wl.k_new[100:140], 0, 2))
    vc = np.ascontiguousarray(np.moveaxis(wl.v_new[100:140], 0, 2))
    g.append_tokens(T.dev(kc, "f16"), T.dev(vc, "f16"))
    for i in range(100, 140):
        o.append(wl.k_new[i], wl.v_new[i])
    T.compare_state(T.gpu_state(g), o.export(), 640, R, 32, policy=policy)
    assert T.attn_err(T.out_float(g.attention(q)), o.attention(qf)) <= T.ATTN_TOL


@pytest.mark.parametrize("n_out", [2, 4])
def test_outliers_long_context_and_ragged(n_out):
    """Many packed splits and tail splits (R = 128), and a ragged batch."""
    lens = [3000, 17, 1500, 128]
    wl = W.synthetic("olr", B=4, Hq=16, Hkv=4, T=max(lens), R=128, seed=n_out)
    cap = 3072
    g = T.gpu_cache(wl, capacity=cap, outliers=n_out)
    g.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"), lengths=lens)
    from oracle.kivi_oracle import OracleCache
    qf = T.q_float(wl.q, wl.q_dtype)
    out = T.out_float(g.attention(T.dev(wl.q, wl.q_dtype)))
    gst = T.gpu_state(g)
    for b, l in enumerate(lens):
        o = OracleCache(2, 32, 128, 128, 1, 4, cap, 0, n_out)
        o.prefill(np.ascontiguousarray(wl.k[b:b + 1, :, :l]), np.ascontiguousarray(wl.v[b:b + 1, :, :l]))
        T.compare_state({n: a[b:b + 1] for n, a in gst.items()}, o.export(), l, 128, 32)
        assert T.attn_err(out[b:b + 1], o.attention(qf[b:b + 1])) <= T.ATTN_TOL


def test_outliers_lower_the_error_on_outlier_keys():
    """The exercise's claim, on the GPU path: with four planted outlier key
    channels of the synthetic workload, keeping them at fp16 brings the 2-bit
    attention output closer to the fp32 attention of the unquantized cache."""
    wl = W.synthetic("olq", B=2, Hq=8, Hkv=2, T=2048, R=32, seed=3)
    from oracle.kivi_oracle import attention_f64
    qf = T.q_float(wl.q, wl.q_dtype)
    errs = {}
    for n in (0, 4):
        g = T.gpu_cache(wl, outliers=n)
        g.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"))
        out = T.out_float(g.attention(T.dev(wl.q, wl.q_dtype)))
        e = []
        for b in range(2):
            for j in range(8):
                h = j // 4
                ref = attention_f64(qf[b, j], W.cast(wl.k, "f16")[b, h].astype(np.float32),
                                    W.cast(wl.v, "f16")[b, h].astype(np.float32), 1.0 / np.sqrt(128))
                e.append(np.linalg.norm(out[b, j] - ref) / np.linalg.norm(ref))
        errs[n] = float(np.mean(e))
    assert errs[4] < errs[0], errs
