"""kivi_decode_attention_static: decode attention for callers that cannot
allocate device memory where they run it (graph capture, a host framework's
memory pool, latency paths that cannot take cudaMalloc's synchronization).
It uses the library's fixed device scratch area instead of a caller
workspace.  The test drives it through the C ABI and checks two consecutive
calls against the workspace entry point.  It lives in its own file so that
pytest collects it last."""
import numpy as np
import pytest
import torch

from bit_kv_cache_kivi_gb300 import workloads as W
import kivi_testlib as T

pytestmark = pytest.mark.gpu


def test_static_scratch_attention_matches_workspace_attention():
    from bit_kv_cache_kivi_gb300 import build, kivi
    build.build()
    wl = W.synthetic("noalloc", B=4, Hq=32, Hkv=8, T=2000, R=32, seed=31)
    g = T.gpu_cache(wl)
    g.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"))
    assert g.ws_bytes <= 8 << 20
    q = T.dev(wl.q, "f16")
    ref = T.out_float(g.attention(q))
    for call in range(2):
        out = torch.full_like(q, float("nan"))
        kivi.kivi_decode_attention_static(g.handle, q, kivi.KIVI_F16, out, 0.0)
        torch.cuda.synchronize()
        got = T.out_float(out)
        assert np.isfinite(got).all(), call
        assert T.attn_err(got, ref) <= T.ATTN_TOL, call
    # a shape whose split scratch exceeds the fixed area is rejected, not run
    big = kivi.KiviCache(batch=512, n_kv_heads=8, n_q_heads=64, max_tokens=64)
    assert big.ws_bytes > 8 << 20
    kv = torch.zeros((512, 8, 40, 128), dtype=torch.float16, device="cuda")
    big.prefill(kv, kv)
    qb = torch.zeros((512, 64, 128), dtype=torch.float16, device="cuda")
    with pytest.raises(kivi.KiviError) as e:
        kivi.kivi_decode_attention_static(big.handle, qb, kivi.KIVI_F16, qb, 0.0)
    assert e.value.status == kivi.KIVI_EWORKSPACE
