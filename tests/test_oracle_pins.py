"""Pins of the CPU oracle against what the pages and the mathematics fix.

No GPU is involved.  Each test names the passage it checks; together they are
meant to catch a dropped term, a wrong sign or index, or a swapped axis
anywhere in the oracle.
"""
import math

import numpy as np
import pytest
import torch

from conftest import golden
from bit_kv_cache_kivi_gb300 import workloads as W


def f16(a):
    return np.asarray(a, np.float32).astype(np.float16).view(np.uint16)


# ---------------------------------------------------------------- conversions

def test_f16_conversion_matches_numpy(oracle):
    """Rounding to fp16 (RNE, subnormals, overflow) equals numpy's cast."""
    rng = np.random.default_rng(0)
    vals = (rng.standard_normal(20000) * 10.0 ** rng.integers(-9, 6, 20000)).astype(np.float32)
    edge = np.array([0.0, -0.0, 65504, 65519.99, 65520, 1e6, 6.0e-8, 2.98e-8, 2.99e-8,
                     5.96e-8, 1e-45, 6.1035156e-05, 6.1035152e-05, 1.0009765625,
                     1.00048828125, 1.00146484375, -2049.0, 2049.0, 2051.0], np.float32)
    vals = np.concatenate([vals, edge, -edge])
    with np.errstate(over="ignore"):
        expect = vals.astype(np.float16).view(np.uint16)
    got = np.array([oracle.f32_to_f16_bits(v) for v in vals], np.uint16)
    assert np.array_equal(got, expect)
    # and back: every finite fp16 pattern widens exactly
    pats = np.arange(0, 65536, dtype=np.uint32).astype(np.uint16)
    finite = pats[(pats & 0x7C00) != 0x7C00]
    back = np.array([oracle.f16_bits_to_f32(int(h)) for h in finite[::7]], np.float32)
    assert np.array_equal(back, finite[::7].view(np.float16).astype(np.float32))


def test_bf16_widening_matches_torch(oracle):
    x = torch.randn(4096) * 100
    bits = x.to(torch.bfloat16).view(torch.int16).numpy().view(np.uint16)
    got = np.array([oracle.lib().orc_bf16_to_f32(int(b)) for b in bits], np.float32)
    assert np.array_equal(got, x.to(torch.bfloat16).float().numpy())


# ---------------------------------------------------------------- quantizer

def test_worked_example_from_review(oracle):
    """[0.1, 0.2, 0.15, 50.0] per token at 2 bits: s ~ 16.63, small values -> 0."""
    g = golden("worked_example.json")
    codes, s16, z16, s32 = oracle.quantize_group(f16(g["group"]), g["bits"])
    assert round(s32, g["scale_printed_decimals"]) == pytest.approx(g["scale_printed"])
    assert list(codes[:3]) == g["codes_of_small_values"]
    assert codes[3] == (1 << g["bits"]) - 1
    # stored fp16 scale is the fp16 rounding of the fp32 scale
    assert oracle.f16_bits_to_f32(s16) == np.float32(s32).astype(np.float16).astype(np.float32)
    # zero point is the minimum, exact
    assert oracle.f16_bits_to_f32(z16) == np.float16(0.1).astype(np.float32)


def _brute_codes(x32, z, s, L):
    """argmin_k |y - k| over k in [0, L], ties to the even k (brute force)."""
    y = (np.float32(x32) - np.float32(z)) / np.float32(s)
    ks = np.arange(L + 1, dtype=np.float64)
    out = []
    for yy in np.atleast_1d(y).astype(np.float64):
        dist = np.abs(yy - ks)
        best = np.flatnonzero(dist == dist.min())
        out.append(int(best[0]) if len(best) == 1 else int([k for k in best if k % 2 == 0][0]))
    return np.array(out)


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_rounding_is_nearest_even_brute_force(oracle, bits):
    L = (1 << bits) - 1
    rng = np.random.default_rng(bits)
    for trial in range(300):
        n = int(rng.integers(2, 9))
        x = rng.standard_normal(n).astype(np.float32) * float(rng.choice([1e-3, 1, 7, 300]))
        xb = f16(x)
        codes, s16, z16, _ = oracle.quantize_group(xb, bits)
        s = oracle.f16_bits_to_f32(s16)
        z = oracle.f16_bits_to_f32(z16)
        xv = xb.view(np.float16).astype(np.float32)
        assert np.array_equal(codes, _brute_codes(xv, z, s, L)), (x, codes)


def test_exact_ties_round_to_even(oracle):
    # 2-bit, range 3 -> scale exactly 1, zero 0: 0.5 -> 0, 1.5 -> 2, 2.5 -> 2
    codes, s16, z16, _ = oracle.quantize_group(f16([0.0, 0.5, 1.5, 2.5, 3.0]), 2)
    assert oracle.f16_bits_to_f32(s16) == 1.0 and oracle.f16_bits_to_f32(z16) == 0.0
    assert list(codes) == [0, 0, 2, 2, 3]
    # 3-bit, range 7 -> scale 1: 2.5 -> 2, 3.5 -> 4, 6.5 -> 6
    codes, s16, _, _ = oracle.quantize_group(f16([0.0, 2.5, 3.5, 6.5, 7.0]), 3)
    assert oracle.f16_bits_to_f32(s16) == 1.0 and list(codes) == [0, 2, 4, 6, 7]
    # 4-bit, range 15 -> scale 1: 6.5 -> 6, 7.5 -> 8
    codes, _, _, _ = oracle.quantize_group(f16([0.0, 6.5, 7.5, 15.0]), 4)
    assert list(codes) == [0, 6, 8, 15]
    # 8-bit, range 255 -> scale 1: 0.5 -> 0, 1.5 -> 2, 254.5 -> 254, 127.5 -> 128
    codes, s16, _, _ = oracle.quantize_group(f16([0.0, 0.5, 1.5, 127.5, 254.5, 255.0]), 8)
    assert oracle.f16_bits_to_f32(s16) == 1.0 and list(codes) == [0, 0, 2, 128, 254, 255]


@pytest.mark.parametrize("bits", [2, 3, 4, 8])
def test_codes_in_range_and_error_bound(oracle, bits):
    """codes in [0, 2^b-1]; |x - xhat| <= s16/2 + L|s32 - s16| (+ fp32 rounding)."""
    L = (1 << bits) - 1
    rng = np.random.default_rng(10 + bits)
    for trial in range(200):
        x = rng.standard_normal(32).astype(np.float32)
        x[rng.integers(0, 32)] *= float(rng.choice([1, 5, 40]))
        xb = f16(x)
        codes, s16, z16, s32 = oracle.quantize_group(xb, bits)
        assert codes.min() >= 0 and codes.max() <= L
        s = oracle.f16_bits_to_f32(s16)
        xv = xb.view(np.float16).astype(np.float64)
        xhat = np.array([oracle.dequant(int(c), s16, z16) for c in codes], np.float64)
        bound = s / 2 + L * abs(s32 - s) + 4 * np.finfo(np.float32).eps * np.abs(xv).max()
        assert np.abs(xv - xhat).max() <= bound


def test_zero_range_and_underflowing_scale(oracle):
    codes, s16, z16, _ = oracle.quantize_group(f16([1.25] * 32), 2)
    assert s16 == 0x3C00 and not codes.any()
    assert oracle.dequant(0, s16, z16) == 1.25
    # range 2^-24: fp32 scale 2^-24/3 rounds to fp16 zero -> stored scale 1
    tiny = np.array([0, 1] * 16, np.uint16)  # fp16 patterns 0 and 2^-24
    codes, s16, z16, _ = oracle.quantize_group(tiny, 2)
    assert s16 == 0x3C00 and not codes.any() and z16 == 0


def test_pack_layout_lsb_first(oracle):
    """Channel e of a packed row occupies bits [e*bits, e*bits + bits), LSB
    first, keys and values alike, at every width (the plain reading of
    "codes packed to uint8")."""
    assert list(oracle.pack_row(np.array([0, 1, 2, 3] * 4, np.uint8), 2)) == [0xE4] * 4
    assert list(oracle.pack_row(np.array([1, 2] * 4, np.uint8), 4)) == [0x21] * 4
    # 8 bits: one byte per channel, in channel order
    c8 = np.arange(128, dtype=np.uint8) * 2 + 1
    assert np.array_equal(oracle.pack_row(c8, 8), c8)
    # 3 bits: codes 1..7, 0 of channels 0..7 fill three bytes; channel 2
    # (bits 6..8) and channel 5 (bits 15..17) cross a byte boundary
    c3 = np.array([1, 2, 3, 4, 5, 6, 7, 0], np.uint8)
    bits = sum(int(c) << (3 * e) for e, c in enumerate(c3))
    assert list(oracle.pack_row(c3, 3)) == [bits & 0xFF, (bits >> 8) & 0xFF, (bits >> 16) & 0xFF]
    one = np.zeros(128, np.uint8)
    one[2] = 4  # the high bit of channel 2 is bit 8: byte 1, bit 0
    row = oracle.pack_row(one, 3)
    assert row.size == 48 and row[1] == 1 and np.count_nonzero(row) == 1
    # against numpy's little-endian bit packing of the codes' bits
    rng = np.random.default_rng(3)
    for b_ in (2, 3, 4, 8):
        c = rng.integers(0, 1 << b_, 128).astype(np.uint8)
        lsb = ((c[:, None] >> np.arange(b_)) & 1).astype(np.uint8).reshape(-1)
        assert np.array_equal(oracle.pack_row(c, b_), np.packbits(lsb, bitorder="little"))
        assert np.array_equal(oracle.unpack_row(oracle.pack_row(c, b_), 128, b_), c)


def test_key_per_channel_value_per_token_orientation(oracle):
    """Structured K/V whose per-channel (K) and per-token (V) ranges are known.

    K[t, d] = (t mod 32) * 2^(d mod 4): the range of every 32-token channel
    group is 31 * 2^(d mod 4).  V[t, d] = (d mod 32) * 2^(t mod 4): the range
    of every 32-channel token group is 31 * 2^(t mod 4).  A swapped axis or a
    wrong group index changes the stored scales.
    """
    T, D = 96, 128
    t = np.arange(T)[:, None]
    d = np.arange(D)[None, :]
    K = ((t % 32) * 2.0 ** (d % 4)).astype(np.float32)
    V = ((d % 32) * 2.0 ** (t % 4)).astype(np.float32)
    c = oracle.OracleCache(2, 32, 32, D, 1, 1, 128)
    c.prefill(K[None, None].astype(np.float16), V[None, None].astype(np.float16))
    st = c.export()
    # Algorithm 1 at l=96, R=32: K fully quantized, V quantized for t < 64
    sk = st["scale_k"][0, 0, :3].view(np.float16).astype(np.float32)
    want_k = (31.0 * 2.0 ** (np.arange(D) % 4) / 3.0).astype(np.float32).astype(np.float16).astype(np.float32)
    assert np.array_equal(sk, np.broadcast_to(want_k, sk.shape))
    assert not st["zero_k"][0, 0, :3].any()
    sv = st["scale_v"][0, 0, :64].view(np.float16).astype(np.float32)
    want_v = (31.0 * 2.0 ** (np.arange(64) % 4) / 3.0).astype(np.float32).astype(np.float16).astype(np.float32)
    assert np.array_equal(sv, np.broadcast_to(want_v[:, None], sv.shape))
    # codes of K depend only on t mod 32: rint(i / s') with s' = fp16(31/3)
    ck = np.array([oracle.unpack_row(st["codes_k"][0, 0, i], D, 2) for i in range(32)])
    expect = np.array([0] * 6 + [1] * 10 + [2] * 10 + [3] * 6)
    assert np.array_equal(ck, np.broadcast_to(expect[:, None], ck.shape))
    # codes of V depend only on d mod 32, the same pattern along channels
    cv = oracle.unpack_row(st["codes_v"][0, 0, 5], D, 2)
    assert np.array_equal(cv, np.tile(expect, 4))


# ---------------------------------------------------------------- statistics

def test_per_tensor_and_per_head_statistics(oracle):
    """Cache Quantization page: per-tensor 8/4/2-bit and per-head 4-bit keys.

    The page's keys are unseeded, so the per-tensor numbers carry the sample's
    extreme values.  Scale-free consequences are pinned: the 8-bit/4-bit MSE
    ratio and the 2-bit/4-bit ratio; the per-head statistic averages 32 heads
    and is pinned directly.
    """
    g = golden("cache_quantization_tables.json")
    rng = np.random.default_rng(12345)
    keys = rng.standard_normal((1, 32, 512, 128), np.float32)
    x16 = f16(keys).ravel()

    def mse_cos(bits, groups):
        xs = []
        for part in np.split(x16, groups):
            codes, s, z, _ = oracle.quantize_group(part, bits)
            xs.append(codes.astype(np.float32) * np.float32(oracle.f16_bits_to_f32(s))
                      + np.float32(oracle.f16_bits_to_f32(z)))
        xh = np.concatenate(xs).astype(np.float64)
        k = keys.ravel().astype(np.float64)
        return np.mean((xh - k) ** 2), xh @ k / np.linalg.norm(xh) / np.linalg.norm(k)

    pt = {b: mse_cos(b, 1) for b in (8, 4, 2)}
    page = g["per_tensor"]
    r84 = page["8"]["key_mse"] / page["4"]["key_mse"]
    assert pt[8][0] / pt[4][0] == pytest.approx(r84, rel=0.05)
    r24 = page["2"]["key_mse"] / page["4"]["key_mse"]
    assert pt[2][0] / pt[4][0] == pytest.approx(r24, rel=g["tolerance"]["mse_rel"])
    assert pt[8][1] == pytest.approx(page["8"]["key_cos"], abs=g["tolerance"]["cos_abs"])
    assert pt[4][1] == pytest.approx(page["4"]["key_cos"], abs=g["tolerance"]["cos_abs"])
    # The 2-bit per-tensor cosine is not pinned to the page's 0.8037: one
    # scale spans the whole tensor, so the value follows the sample's two
    # extreme elements (0.78 to 0.80 over seeds of this generator), and the
    # page's keys are unseeded.  What holds for any sample is the order.
    assert pt[2][1] < pt[4][1] < pt[8][1]
    ph = mse_cos(4, 32)
    assert ph[0] == pytest.approx(g["per_head_4bit"]["key_mse"], rel=g["tolerance"]["mse_rel"])
    assert ph[1] == pytest.approx(g["per_head_4bit"]["key_cos"], abs=g["tolerance"]["cos_abs"])
    assert ph[0] < pt[4][0]  # per-head beats per-tensor at the same width


def test_two_bit_key_cosine(oracle):
    """VeloxQuant KIVI page: 2-bit raw-key cosine ~0.93 on unit-norm Gaussian keys."""
    g = golden("veloxquant_cosine.json")
    rng = np.random.default_rng(7)
    k = rng.standard_normal((1, 1, 1024, 128), np.float32)
    k /= np.linalg.norm(k, axis=-1, keepdims=True)
    c = oracle.OracleCache(g["bits"], g["group"], 32, 128, 1, 1, 1024)
    c.prefill(k.astype(np.float16), k.astype(np.float16))
    kh, _ = c.dequant(0, 0)
    kk = k[0, 0].astype(np.float64)
    cos = (kh * kk).sum() / np.linalg.norm(kh) / np.linalg.norm(kk)
    assert cos == pytest.approx(g["cosine"], abs=g["tolerance_abs"])


def _grouped_fake_quant(oracle, X, axis, bits, G=32):
    """Quantize every group of the notebook's layout with the oracle primitive."""
    x16 = f16(X)
    T, D = X.shape
    out = np.zeros((T, D), np.float32)
    if axis == 0:  # K: each channel, groups of G tokens
        for d in range(D):
            for t0 in range(0, T, G):
                codes, s, z, _ = oracle.quantize_group(x16[t0:t0 + G, d], bits)
                out[t0:t0 + G, d] = [oracle.dequant(int(c), s, z) for c in codes]
    else:          # V: each token, groups of G channels
        for t in range(T):
            for d0 in range(0, D, G):
                codes, s, z, _ = oracle.quantize_group(x16[t, d0:d0 + G], bits)
                out[t, d0:d0 + G] = [oracle.dequant(int(c), s, z) for c in codes]
    return out


def test_notebook_quality_checks(oracle):
    """The notebook's own checks on its seeded data (2-bit and 4-bit)."""
    g = golden("notebook_checks.json")
    wl = W.single_head()
    K, V, Q = wl.k[0, 0], wl.v[0, 0], wl.notebook_Q
    Kh2 = _grouped_fake_quant(oracle, K, 0, 2)
    Vh2 = _grouped_fake_quant(oracle, V, 1, 2)
    Kh4 = _grouped_fake_quant(oracle, K, 0, 4)
    Vh4 = _grouped_fake_quant(oracle, V, 1, 4)
    frac = g["max_abs_error_fraction_of_max"]
    assert np.abs(K - Kh2).max() < frac * np.abs(K).max()
    assert np.abs(V - Vh2).max() < frac * np.abs(V).max()

    def attn(Kx, Vx):
        s = Q.astype(np.float64) @ Kx.T.astype(np.float64) / math.sqrt(K.shape[1])
        s -= s.max(axis=1, keepdims=True)
        p = np.exp(s)
        p /= p.sum(axis=1, keepdims=True)
        return p @ Vx.astype(np.float64)

    Y = attn(K, V)
    e2 = np.linalg.norm(Y - attn(Kh2, Vh2)) / np.linalg.norm(Y)
    e4 = np.linalg.norm(Y - attn(Kh4, Vh4)) / np.linalg.norm(Y)
    assert e4 < g["rel_err_4bit_below"]
    assert g["rel_err_2bit_above"] < e2 < g["rel_err_2bit_below"]
    assert e4 < e2
    # the notebook's bit-width sweep (16, 8, 4, 3, 2): the error grows as the
    # width falls, and the step from 3 to 2 bits is the largest
    e3 = np.linalg.norm(Y - attn(_grouped_fake_quant(oracle, K, 0, 3),
                                 _grouped_fake_quant(oracle, V, 1, 3))) / np.linalg.norm(Y)
    e8 = np.linalg.norm(Y - attn(_grouped_fake_quant(oracle, K, 0, 8),
                                 _grouped_fake_quant(oracle, V, 1, 8))) / np.linalg.norm(Y)
    assert e8 < e4 < e3 < e2
    assert e2 - e3 > e3 - e4
