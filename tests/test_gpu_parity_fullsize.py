"""Parity at the full sizes of the five workloads, in the launch configuration
the benchmark times: every (batch, kv-head) unit against the oracle (the
larger workloads run the oracle one unit per process)."""
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


def unit_oracles(wl, units, capacity=None, bits=None, T_=None):
    """One B=1, H=1 oracle cache per sampled unit, prefilled with that unit."""
    outs = T.oracle_cache(wl, capacity, bits, units=units)
    for (b, h), o in zip(units, outs):
        k, v = T.slice_unit(wl.k, b, h), T.slice_unit(wl.v, b, h)
        if T_ is not None:
            k, v = np.ascontiguousarray(k[:, :, :T_]), np.ascontiguousarray(v[:, :, :T_])
        o.prefill(k, v)
    return outs


def unit_attention_err(out, wl, units, oracles, q):
    grp = wl.Hq // wl.Hkv
    worst = 0.0
    for (b, h), o in zip(units, oracles):
        qs = np.ascontiguousarray(T.q_float(q, wl.q_dtype)[b:b + 1, h * grp:(h + 1) * grp])
        ref = o.attention(qs)
        worst = max(worst, T.attn_err(out[b:b + 1, h * grp:(h + 1) * grp], ref))
    return worst


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_llama3_8b_decode_step(bits):
    """batch 8, 32/8 heads, context 4096 fp16: prefill, one append, attention;
    the whole batch against the oracle (2 bits, and the same step at 4 bits)."""
    wl = W.llama3_8b_decode(bits=bits)
    g = T.gpu_cache(wl)
    g.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"))
    o = T.oracle_cache(wl)
    o.prefill(wl.k, wl.v)
    T.compare_state(T.gpu_state(g), o.export(), 4096, 32, 32)
    g.append(T.dev(wl.k_new[0], "f16"), T.dev(wl.v_new[0], "f16"))
    o.append(wl.k_new[0], wl.v_new[0])
    T.compare_state(T.gpu_state(g), o.export(), 4097, 32, 32)
    out = T.out_float(g.attention(T.dev(wl.q, "f16")))
    assert T.attn_err(out, o.attention(T.q_float(wl.q, "f16"))) <= T.ATTN_TOL


def _unit_task(wl, b, h, bits=None, cap=None):
    return {"bits": bits or wl.bits, "G": wl.G, "R": wl.R, "D": wl.D, "cap": cap or wl.capacity,
            "k": T.slice_unit(wl.k, b, h), "v": T.slice_unit(wl.v, b, h)}


@pytest.mark.parametrize("bits", [2, 4])
def test_prefill_quantize_bf16_32k(bits):
    """batch 4, 8 KV heads, 32768 tokens of bf16 with V spikes, 2 and 4 bits:
    the state of every unit bit for bit."""
    wl = W.prefill_quantize(bits)
    g = T.gpu_cache(wl)
    g.prefill(T.dev(wl.k, "bf16"), T.dev(wl.v, "bf16"))
    units = [(b, h) for b in range(wl.B) for h in range(wl.Hkv)]
    res = T.oracle_units([_unit_task(wl, b, h) for b, h in units])
    T.compare_state(T.gpu_state(g), [st for st, _ in res], wl.T, wl.R, wl.G, units=units)


@pytest.mark.parametrize("bits", [3, 8])
def test_prefill_quantize_bf16_32k_other_widths(bits):
    """The same workload at 3 and 8 bits: sampled units."""
    wl = W.prefill_quantize(bits)
    g = T.gpu_cache(wl)
    g.prefill(T.dev(wl.k, "bf16"), T.dev(wl.v, "bf16"))
    units = [(0, 0), (3, 7), (1, 5)]
    orc = unit_oracles(wl, units)
    T.compare_state(T.gpu_state(g), [o.export() for o in orc], wl.T, wl.R, wl.G, units=units)


def test_long_context_131k():
    """batch 1, 32/8 heads, 131072 tokens, R=128: every unit's state bit for
    bit and its split-K attention in tolerance."""
    wl = W.long_context()
    g = T.gpu_cache(wl)
    g.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"))
    assert g.splits() > 16
    grp = wl.Hq // wl.Hkv
    units = [(0, h) for h in range(wl.Hkv)]
    qf = T.q_float(wl.q, wl.q_dtype)
    tasks = []
    for b, h in units:
        t = _unit_task(wl, b, h)
        t["q"] = {-1: np.ascontiguousarray(qf[b:b + 1, h * grp:(h + 1) * grp])}
        tasks.append(t)
    res = T.oracle_units(tasks)
    T.compare_state(T.gpu_state(g), [st for st, _ in res], wl.T, wl.R, wl.G, units=units)
    out = T.out_float(g.attention(T.dev(wl.q, "f16")))
    for (b, h), (_, outs) in zip(units, res):
        assert T.attn_err(out[b:b + 1, h * grp:(h + 1) * grp], outs[-1]) <= T.ATTN_TOL, h


def test_streaming_2048_plus_512():
    """batch 64, 28/4 heads: 512 decode steps after a 2048 prefill.  Attention
    of every unit at the flush boundaries against the oracle; the final state
    of every unit bit for bit against the oracle, and against a one-shot
    prefill of the same 2560 tokens."""
    wl = W.streaming()
    g = T.gpu_cache(wl)
    g.prefill(T.dev(wl.k, "f16"), T.dev(wl.v, "f16"))
    grp = wl.Hq // wl.Hkv
    units = [(b, h) for b in range(wl.B) for h in range(wl.Hkv)]
    check_at = [0, 1, 31, 32, 63, 64, 255, 511]
    qs = {i: T.q_float(wl.q_for_step(i), wl.q_dtype) for i in check_at}
    tasks = []
    for b, h in units:
        t = _unit_task(wl, b, h)
        t["kn"] = np.ascontiguousarray(wl.k_new[:, b:b + 1, h:h + 1])
        t["vn"] = np.ascontiguousarray(wl.v_new[:, b:b + 1, h:h + 1])
        t["q"] = {i: np.ascontiguousarray(qs[i][b:b + 1, h * grp:(h + 1) * grp]) for i in check_at}
        tasks.append(t)
    res = T.oracle_units(tasks)
    kn_all = T.dev(wl.k_new, "f16")
    vn_all = T.dev(wl.v_new, "f16")
    for i in range(wl.steps):
        g.append(kn_all[i], vn_all[i])
        if i in qs:
            out = T.out_float(g.attention(T.dev(wl.q_for_step(i), "f16")))
            worst = max(T.attn_err(out[b:b + 1, h * grp:(h + 1) * grp], outs[i])
                        for (b, h), (_, outs) in zip(units, res))
            assert worst <= T.ATTN_TOL, (i, worst)
        else:
            g.attention(T.dev(wl.q, "f16"))
    l = wl.T + wl.steps
    st = T.gpu_state(g)
    T.compare_state(st, [s_ for s_, _ in res], l, wl.R, wl.G, units=units)
    k_all = np.concatenate([wl.k, wl.k_new.transpose(1, 2, 0, 3)], axis=2)
    v_all = np.concatenate([wl.v, wl.v_new.transpose(1, 2, 0, 3)], axis=2)
    one = T.gpu_cache(wl)
    one.prefill(T.dev(np.ascontiguousarray(k_all), "f16"), T.dev(np.ascontiguousarray(v_all), "f16"))
    T.compare_state(st, T.gpu_state(one), l, wl.R, wl.G)
