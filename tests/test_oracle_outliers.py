"""Pins of the oracle's outlier-aware keys (the "KIVI - 2-bit KV cache
quantisation" notebook, Exercises item 2: keep the top-1% of K channels at
fp16 and quantise the rest).

Reading: per key group of G tokens, the n_out channels with the largest
max |k| over the group are kept as fp16 (largest first, ties to the lower
channel); their codes, scales and zeros are 0; the other channels are
quantized exactly as without outliers."""
import numpy as np
import pytest

from bit_kv_cache_kivi_gb300 import workloads as W


def _kv(B, H, T, D, seed, outl=(3, 17, 40, 88), scale=8.0):
    rng = np.random.default_rng(seed)
    k = rng.standard_normal((B, H, T, D), np.float32)
    v = rng.standard_normal((B, H, T, D), np.float32)
    for c in outl:
        k[..., c] *= scale
    return k.astype(np.float16), v.astype(np.float16)


def _brute_outliers(kg: np.ndarray, n: int) -> list:
    """Top-n channels of one group [G, D] by max |x| (ties: lower channel),
    by sorting -- independent of the oracle's selection loop."""
    amax = np.abs(kg.astype(np.float32)).max(axis=0)
    order = sorted(range(kg.shape[1]), key=lambda d: (-amax[d], d))
    return order[:n]


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
@pytest.mark.parametrize("n_out", [1, 2, 4])
def test_outlier_selection_and_storage(oracle, bits, n_out):
    B, H, T, D, G, R = 2, 2, 200, 128, 32, 64
    k, v = _kv(B, H, T, D, bits * 10 + n_out)
    plain = oracle.OracleCache(bits, G, R, D, B, H, 256)
    plain.prefill(k, v)
    c = oracle.OracleCache(bits, G, R, D, B, H, 256, outliers=n_out)
    c.prefill(k, v)
    sp, so = plain.export(), c.export()
    nqk = oracle.nq_k(T, R, G)
    assert so["outl_idx"].shape == (B, H, 256 // G, n_out)
    for b in range(B):
        for h in range(H):
            for g in range(nqk // G):
                kg = k[b, h, g * G:(g + 1) * G]
                want = _brute_outliers(kg, n_out)
                assert list(so["outl_idx"][b, h, g]) == want
                # kept values: the fp16 inputs, bit for bit
                assert np.array_equal(so["outl_val"][b, h, g * G:(g + 1) * G],
                                      kg.view(np.uint16)[:, want])
                # their scale / zero are 0; every other channel as without outliers
                keep = [d for d in range(D) if d not in want]
                assert not so["scale_k"][b, h, g, want].any() and not so["zero_k"][b, h, g, want].any()
                assert np.array_equal(so["scale_k"][b, h, g, keep], sp["scale_k"][b, h, g, keep])
                assert np.array_equal(so["zero_k"][b, h, g, keep], sp["zero_k"][b, h, g, keep])
                codes_o = np.array([oracle.unpack_row(so["codes_k"][b, h, t], D, bits)
                                    for t in range(g * G, (g + 1) * G)])
                codes_p = np.array([oracle.unpack_row(sp["codes_k"][b, h, t], D, bits)
                                    for t in range(g * G, (g + 1) * G)])
                assert not codes_o[:, want].any()
                assert np.array_equal(codes_o[:, keep], codes_p[:, keep])
            # values, rings and the unquantized part are untouched
            for name in ("codes_v", "scale_v", "zero_v", "ring_k", "ring_v"):
                assert np.array_equal(so[name], sp[name]), name
            assert not so["outl_idx"][b, h, nqk // G:].any() and not so["outl_val"][b, h, nqk:].any()


def test_outlier_ties_go_to_the_lower_channel(oracle):
    G, D = 32, 128
    k = np.zeros((1, 1, G, D), np.float16)
    k[0, 0, 5, [90, 7, 60]] = 3.0      # three-way tie
    k[0, 0, 9, 100] = -3.5             # the largest |x| (negative)
    v = np.zeros_like(k)
    c = oracle.OracleCache(2, G, G, D, 1, 1, 64, outliers=3)
    c.prefill(k, v)
    assert list(c.export()["outl_idx"][0, 0, 0]) == [100, 7, 60]


def test_outlier_dequant_is_exact(oracle):
    """Decoded keys of the kept channels equal the fp16 inputs."""
    B, H, T, D, G, R = 1, 2, 96, 128, 32, 32
    k, v = _kv(B, H, T, D, 7)
    c = oracle.OracleCache(2, G, R, D, B, H, 128, outliers=2)
    c.prefill(k, v)
    st = c.export()
    for h in range(H):
        kh, _ = c.dequant(0, h)
        for t in range(oracle.nq_k(T, R, G)):
            for o in range(2):
                ch = st["outl_idx"][0, h, t // G, o]
                assert kh[t, ch] == np.float32(k[0, h, t, ch])


@pytest.mark.parametrize("policy", [0, 1])
def test_outliers_prefill_equals_streaming(oracle, policy):
    """Group-local selection keeps prefill and token-by-token appends
    bit-identical."""
    B, H, T, D, G, R = 1, 2, 130, 128, 32, 32
    k, v = _kv(B, H, T, D, 11)
    ref = oracle.OracleCache(2, G, R, D, B, H, 160, policy, outliers=2)
    ref.prefill(k, v)
    want = ref.export()
    for T0 in (0, 31, 33, 100):
        c = oracle.OracleCache(2, G, R, D, B, H, 160, policy, outliers=2)
        c.prefill(k[:, :, :T0], v[:, :, :T0])
        for t in range(T0, T):
            c.append(np.ascontiguousarray(k[:, :, t]), np.ascontiguousarray(v[:, :, t]))
        got = c.export()
        for name in want:
            assert np.array_equal(got[name], want[name]), (T0, name)


def test_outliers_reduce_attention_error(oracle):
    """The exercise's claim on the notebook's single-head workload (four
    planted outlier key channels): keeping them at fp16 lowers the 2-bit
    attention error against the double-precision reference."""
    wl = W.single_head()
    q = wl.q.astype(np.float32)
    ref = oracle.attention_f64(q[0, 0], wl.k[0, 0].astype(np.float32),
                               wl.v[0, 0].astype(np.float32), 1.0 / np.sqrt(wl.D))
    errs = {}
    for n in (0, 2, 4):
        c = oracle.OracleCache(2, 32, 32, wl.D, 1, 1, wl.capacity, outliers=n)
        c.prefill(W.cast(wl.k, "f16"), W.cast(wl.v, "f16"))
        out = c.attention(q)[0, 0]
        errs[n] = float(np.linalg.norm(out - ref) / np.linalg.norm(ref))
    assert errs[2] < errs[0] and errs[4] < errs[2], errs
