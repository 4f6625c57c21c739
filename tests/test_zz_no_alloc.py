"""kivi_decode_attention_static: decode attention for callers that cannot
allocate device memory where they run it (a plugin whose device memory comes
only from its host framework's pool, or a latency-critical path that cannot
take cudaMalloc's implicit device-wide synchronization).  It uses the
library's fixed device scratch area instead of a caller workspace.

The test drives it through the C ABI: two consecutive calls must give the
workspace entry point's output bit for bit (the same kernel on the same
inputs), the output must match the oracle, and the calls must leave the
device's free memory unchanged.  It lives in its own file so that pytest
collects it last."""
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
    ref = g.attention(q).clone()
    o = T.oracle_cache(wl)
    o.prefill(wl.k, wl.v)
    assert T.attn_err(T.out_float(ref), o.attention(T.q_float(wl.q, "f16"))) <= T.ATTN_TOL
    outs = [torch.full_like(q, float("nan")) for _ in range(2)]
    # the first call on the device looks up the area's address; after it,
    # calls take no device memory
    kivi.kivi_decode_attention_static(g.handle, q, kivi.KIVI_F16, outs[0], 0.0)
    torch.cuda.synchronize()
    free0, _ = torch.cuda.mem_get_info()
    for call, out in enumerate(outs):
        kivi.kivi_decode_attention_static(g.handle, q, kivi.KIVI_F16, out, 0.0)
        torch.cuda.synchronize()
        assert torch.equal(out, ref), call
    free1, _ = torch.cuda.mem_get_info()
    assert free1 == free0
    got = T.out_float(outs[1])
    assert T.attn_err(got, o.attention(T.q_float(wl.q, "f16"))) <= T.ATTN_TOL
    # a shape whose split scratch exceeds the fixed area is rejected, not run
    big = kivi.KiviCache(batch=512, n_kv_heads=8, n_q_heads=64, max_tokens=64)
    assert big.ws_bytes > 8 << 20
    kv = torch.zeros((512, 8, 40, 128), dtype=torch.float16, device="cuda")
    big.prefill(kv, kv)
    qb = torch.zeros((512, 64, 128), dtype=torch.float16, device="cuda")
    with pytest.raises(kivi.KiviError) as e:
        kivi.kivi_decode_attention_static(big.handle, qb, kivi.KIVI_F16, qb, 0.0)
    assert e.value.status == kivi.KIVI_EWORKSPACE
