"""A cache whose packed-tile buffer is larger than 4 GiB: the byte offsets of
the far units pass both 2^31 and 2^32, where 32-bit index arithmetic would
wrap.  Prefill, appends across key flushes and attention run over the whole
batch; units on both sides of each boundary are compared with the oracle
(each alone, as a one-unit oracle cache), bit for bit for the cache and
within the attention tolerance for the output."""
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


def sampled_state(cache, units) -> dict:
    """The logical state of the listed (b, h) units only, as [n][1][...]."""
    torch.cuda.synchronize()
    out = {}
    for n, t in cache.logical_state().items():
        a = torch.stack([t[b, h] for b, h in units]).unsqueeze(1).cpu().numpy()
        out[n] = a.view(np.uint16) if a.dtype == np.int16 else a
    return out


@pytest.mark.parametrize("bits", [2, 4])
def test_tile_offsets_past_4_gib(bits):
    cap = 8192
    wl = W.synthetic("big", B=700, Hq=32, Hkv=8, T=80, R=32, bits=bits, steps=50, seed=23 + bits)
    g = T.gpu_cache(wl, capacity=cap)
    tiles = g.buffers["tiles"]
    unit_bytes = tiles.numel() * tiles.element_size() // (wl.B * wl.Hkv)
    assert tiles.numel() * tiles.element_size() > 2 ** 32
    # units either side of the 2^31 and 2^32 byte offsets, and the last one
    picks = {0, 2 ** 31 // unit_bytes, 2 ** 31 // unit_bytes + 1, 2 ** 32 // unit_bytes,
             2 ** 32 // unit_bytes + 1, wl.B * wl.Hkv - 1}
    units = [(u // wl.Hkv, u % wl.Hkv) for u in sorted(picks)]
    assert any(u * unit_bytes >= 2 ** 32 for u in picks)

    g.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"))
    orc = T.oracle_cache(wl, capacity=cap, units=units)
    for (b, h), o in zip(units, orc):
        o.prefill(T.slice_unit(wl.k, b, h), T.slice_unit(wl.v, b, h))
    T.compare_state(sampled_state(g, units), [o.export() for o in orc], wl.T, wl.R, wl.G,
                    units=[(i, 0) for i in range(len(units))])

    for i in range(wl.steps):  # lengths 81 .. 130: key flushes at 96 and 128
        g.append(T.dev(wl.k_new[i], "f16"), T.dev(wl.v_new[i], "f16"))
        for (b, h), o in zip(units, orc):
            o.append(np.ascontiguousarray(wl.k_new[i, b:b + 1, h:h + 1]),
                     np.ascontiguousarray(wl.v_new[i, b:b + 1, h:h + 1]))
    l = wl.T + wl.steps
    assert g.length == l
    T.compare_state(sampled_state(g, units), [o.export() for o in orc], l, wl.R, wl.G,
                    units=[(i, 0) for i in range(len(units))])

    out = T.out_float(g.attention(T.dev(wl.q, wl.q_dtype)))
    grp = wl.Hq // wl.Hkv
    qf = T.q_float(wl.q, wl.q_dtype)
    for (b, h), o in zip(units, orc):
        ref = o.attention(np.ascontiguousarray(qf[b:b + 1, h * grp:(h + 1) * grp]))
        assert T.attn_err(out[b:b + 1, h * grp:(h + 1) * grp], ref) <= T.ATTN_TOL, (b, h)
