"""ctypes front end of the C oracle (``kivi_oracle.c``).

TEST INFRASTRUCTURE ONLY: imported by the tests, ``__graft_entry__.smoke()``
and the CPU-baseline leg of ``bench.py``; the product path never loads it.

Inputs are numpy arrays; fp16 and bf16 tensors travel as their uint16 bit
patterns.  Every function here is argument marshalling: the arithmetic lives
in the C file, which follows the pages step by step.
"""
from __future__ import annotations

import ctypes as C
import os
import subprocess
import threading

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "kivi_oracle.c")
_HDR = os.path.join(_HERE, "kivi_oracle.h")
_LIB = os.path.join(_HERE, "libkivi_oracle.so")

F32, F16, BF16 = 0, 1, 2
POLICY_ALG1, POLICY_SHARED = 0, 1

_lock = threading.Lock()
_lib = None


def build(force: bool = False) -> str:
    """Compile the oracle with gcc (fp32 strict: no contraction, no fast-math)."""
    stale = (not os.path.exists(_LIB)) or any(
        os.path.getmtime(p) > os.path.getmtime(_LIB) for p in (_SRC, _HDR))
    if force or stale:
        tmp = _LIB + f".tmp{os.getpid()}"
        cmd = ["gcc", "-O2", "-std=c11", "-ffp-contract=off", "-fno-fast-math",
               "-fPIC", "-shared", "-o", tmp, _SRC, "-lm"]
        subprocess.run(cmd, check=True)
        os.replace(tmp, _LIB)
    return _LIB


def lib():
    global _lib
    with _lock:
        if _lib is None:
            build()
            L = C.CDLL(_LIB)
            vp, i32, i64, f32 = C.c_void_p, C.c_int, C.c_long, C.c_float
            sig = {
                "orc_f32_to_f16": (C.c_uint16, [f32]),
                "orc_f16_to_f32": (f32, [C.c_uint16]),
                "orc_bf16_to_f32": (f32, [C.c_uint16]),
                "orc_quantize_group": (None, [vp, i64, i64, i32, vp, i64, vp, vp, vp]),
                "orc_dequant": (f32, [i32, C.c_uint16, C.c_uint16]),
                "orc_pack_row": (None, [vp, i32, i32, vp]),
                "orc_unpack_row": (None, [vp, i32, i32, vp]),
                "orc_nq_k": (i64, [i64, i32, i32, i32]),
                "orc_nq_v": (i64, [i64, i32, i32, i32]),
                "orc_cache_new": (vp, [i32, i32, i32, i32, i32, i32, i64, i32]),
                "orc_cache_free": (None, [vp]),
                "orc_cache_length": (i64, [vp]),
                "orc_cache_prefill": (i32, [vp, vp, vp, i32, i64]),
                "orc_cache_append": (i32, [vp, vp, vp, i32]),
                "orc_cache_export": (None, [vp] * 9),
                "orc_cache_set_outliers": (i32, [vp, i32]),
                "orc_cache_outliers": (i32, [vp]),
                "orc_cache_export_outliers": (None, [vp, vp, vp]),
                "orc_cache_dequant": (None, [vp, i32, i32, vp, vp]),
                "orc_decode_attention": (i32, [vp, vp, i32, f32, vp]),
                "orc_attention_f64": (None, [vp, vp, vp, i64, i32, C.c_double, vp]),
            }
            for name, (res, args) in sig.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _p(a: np.ndarray):
    assert a.flags["C_CONTIGUOUS"]
    return a.ctypes.data_as(C.c_void_p)


def _as_input(x: np.ndarray):
    """(array, dtype code) for an input tensor given as f32 / f16 / bf16-bits."""
    if x.dtype == np.float32:
        return np.ascontiguousarray(x), F32
    if x.dtype == np.float16:
        return np.ascontiguousarray(x).view(np.uint16), F16
    if x.dtype == np.uint16:  # bfloat16 bit patterns
        return np.ascontiguousarray(x), BF16
    raise TypeError(f"unsupported input dtype {x.dtype}")


# ---------------------------------------------------------------- primitives

def f32_to_f16_bits(x: float) -> int:
    return int(lib().orc_f32_to_f16(float(x)))


def f16_bits_to_f32(h: int) -> float:
    return float(lib().orc_f16_to_f32(int(h)))


def quantize_group(x16_bits: np.ndarray, bits: int):
    """One group (1-D fp16 bit patterns) -> (codes, scale16, zero16, scale32)."""
    x = np.ascontiguousarray(x16_bits, dtype=np.uint16)
    n = x.size
    codes = np.zeros(n, np.uint8)
    s16, z16, s32 = C.c_uint16(), C.c_uint16(), C.c_float()
    lib().orc_quantize_group(_p(x), n, 1, bits, _p(codes), 1, C.byref(s16),
                             C.byref(z16), C.byref(s32))
    return codes, int(s16.value), int(z16.value), float(s32.value)


def dequant(q: int, s16: int, z16: int) -> float:
    return float(lib().orc_dequant(int(q), int(s16), int(z16)))


def pack_row(codes: np.ndarray, bits: int) -> np.ndarray:
    c = np.ascontiguousarray(codes, dtype=np.uint8)
    out = np.zeros((c.size * bits + 7) // 8, np.uint8)
    lib().orc_pack_row(_p(c), c.size, bits, _p(out))
    return out


def unpack_row(packed: np.ndarray, D: int, bits: int) -> np.ndarray:
    p = np.ascontiguousarray(packed, dtype=np.uint8)
    out = np.zeros(D, np.uint8)
    lib().orc_unpack_row(_p(p), D, bits, _p(out))
    return out


def nq_k(l: int, R: int, G: int, policy: int = POLICY_ALG1) -> int:
    return int(lib().orc_nq_k(l, R, G, policy))


def nq_v(l: int, R: int, G: int, policy: int = POLICY_ALG1) -> int:
    return int(lib().orc_nq_v(l, R, G, policy))


def attention_f64(q: np.ndarray, k: np.ndarray, v: np.ndarray, scale: float) -> np.ndarray:
    q = np.ascontiguousarray(q, np.float32)
    k = np.ascontiguousarray(k, np.float32)
    v = np.ascontiguousarray(v, np.float32)
    l, D = k.shape
    out = np.zeros(D, np.float64)
    lib().orc_attention_f64(_p(q), _p(k), _p(v), l, D, float(scale), _p(out))
    return out


# ---------------------------------------------------------------- the cache

class OracleCache:
    """The oracle's grouped + residual cache for a batch of (b, kv-head) units."""

    def __init__(self, bits: int, group: int, residual: int, head_dim: int,
                 batch: int, n_kv_heads: int, max_tokens: int,
                 policy: int = POLICY_ALG1, outliers: int = 0):
        self.bits, self.G, self.R, self.D = bits, group, residual, head_dim
        self.B, self.H, self.Tcap, self.policy = batch, n_kv_heads, max_tokens, policy
        self._h = lib().orc_cache_new(bits, group, residual, head_dim, batch,
                                      n_kv_heads, max_tokens, policy)
        if not self._h:
            raise ValueError("oracle rejected the cache configuration")
        self.outliers = outliers
        if outliers and lib().orc_cache_set_outliers(self._h, outliers) != 0:
            raise ValueError("oracle rejected the outlier count")

    def __del__(self):
        h = getattr(self, "_h", None)
        if h:
            lib().orc_cache_free(h)
            self._h = None

    @property
    def length(self) -> int:
        return int(lib().orc_cache_length(self._h))

    @property
    def ring_slots(self) -> int:
        return self.R + (self.G if self.policy == POLICY_SHARED else 0)

    def prefill(self, k: np.ndarray, v: np.ndarray) -> None:
        ka, dt = _as_input(k)
        va, dt2 = _as_input(v)
        assert dt == dt2 and ka.shape == va.shape and ka.ndim == 4
        T = ka.shape[2]
        if lib().orc_cache_prefill(self._h, _p(ka), _p(va), dt, T) != 0:
            raise RuntimeError("oracle prefill rejected")

    def append(self, k1: np.ndarray, v1: np.ndarray) -> None:
        ka, dt = _as_input(k1)
        va, _ = _as_input(v1)
        if lib().orc_cache_append(self._h, _p(ka), _p(va), dt) != 0:
            raise RuntimeError("oracle append rejected (capacity)")

    def export(self) -> dict:
        B, H, T, D, G = self.B, self.H, self.Tcap, self.D, self.G
        rb = D * self.bits // 8
        W = self.ring_slots
        st = {
            "codes_k": np.zeros((B, H, T, rb), np.uint8),
            "scale_k": np.zeros((B, H, T // G, D), np.uint16),
            "zero_k": np.zeros((B, H, T // G, D), np.uint16),
            "codes_v": np.zeros((B, H, T, rb), np.uint8),
            "scale_v": np.zeros((B, H, T, D // G), np.uint16),
            "zero_v": np.zeros((B, H, T, D // G), np.uint16),
            "ring_k": np.zeros((B, H, W, D), np.uint16),
            "ring_v": np.zeros((B, H, W, D), np.uint16),
        }
        order = ["codes_k", "scale_k", "zero_k", "codes_v", "scale_v", "zero_v",
                 "ring_k", "ring_v"]
        lib().orc_cache_export(self._h, *[_p(st[n]) for n in order])
        if self.outliers:
            n = self.outliers
            st["outl_idx"] = np.zeros((B, H, T // G, n), np.uint8)
            st["outl_val"] = np.zeros((B, H, T, n), np.uint16)
            lib().orc_cache_export_outliers(self._h, _p(st["outl_idx"]), _p(st["outl_val"]))
        return st

    def dequant(self, b: int, h: int):
        l = self.length
        kh = np.zeros((l, self.D), np.float32)
        vh = np.zeros((l, self.D), np.float32)
        lib().orc_cache_dequant(self._h, b, h, _p(kh), _p(vh))
        return kh, vh

    def attention(self, q: np.ndarray, scale: float = 0.0) -> np.ndarray:
        qa = np.ascontiguousarray(q, np.float32)
        assert qa.ndim == 3 and qa.shape[0] == self.B and qa.shape[2] == self.D
        out = np.zeros_like(qa)
        if lib().orc_decode_attention(self._h, _p(qa), qa.shape[1], float(scale), _p(out)) != 0:
            raise RuntimeError("oracle attention rejected")
        return out
