"""Seeded synthetic inputs shaped like the pages' workloads.

This module only draws random numbers and casts them to the input dtype; it
holds none of the method's arithmetic.  The tests, the oracle runs and the
benchmark all take their inputs from here, so both sides of every parity
check see identical bytes.

Recipes
-------
* ``single_head`` -- the notebook "KIVI - 2-bit KV cache quantisation",
  section "K (per-channel) and V (per-token) quantisation": torch CPU
  generator seeded 0, K and V = randn(1024, 128) * 0.5, K channels
  3, 17, 40, 88 scaled by 5; the query comes from the same notebook's
  attention section (seed 1, randn(1, T, 128)), its first row.  fp32.
* everything else -- ``numpy.random.default_rng(seed)``; draw order: the
  outlier channels (4 per KV head, distinct, shared by batch and tokens),
  K, V, the query, then the decode tokens.  Entries N(0, 1), outlier
  channels x5 in K and in the appended K tokens; optional V token spikes
  (a fraction of (b, h, t) rows chosen without replacement, whole row x8).
  Drawn in fp32, then cast (round to nearest even) to the input dtype.

bf16 tensors are returned as their uint16 bit patterns (numpy has no bf16).
"""
from __future__ import annotations

from dataclasses import dataclass, field

import numpy as np
import torch

OUTLIER_SCALE = 5.0
SPIKE_SCALE = 8.0


def cast(x: np.ndarray, dtype: str) -> np.ndarray:
    """fp32 array -> the input dtype (RNE).  'bf16' yields uint16 bit patterns."""
    x = np.ascontiguousarray(x, np.float32)
    if dtype == "f32":
        return x
    if dtype == "f16":
        return x.astype(np.float16)
    if dtype == "bf16":
        t = torch.from_numpy(x).to(torch.bfloat16).view(torch.int16)
        return t.numpy().view(np.uint16)
    raise ValueError(dtype)


def to_torch(x: np.ndarray, dtype: str, device=None) -> torch.Tensor:
    """numpy input (as produced by ``cast``) -> torch tensor of the input dtype."""
    if dtype == "bf16":
        t = torch.from_numpy(np.ascontiguousarray(x).view(np.int16)).view(torch.bfloat16)
    else:
        t = torch.from_numpy(np.ascontiguousarray(x))
    return t.to(device) if device is not None else t


@dataclass
class Workload:
    name: str
    B: int
    Hq: int
    Hkv: int
    D: int
    T: int            # prefill length
    R: int            # residual length
    G: int            # group size
    bits: int
    dtype: str        # dtype of K/V inputs: 'f32', 'f16' or 'bf16'
    q_dtype: str      # dtype of the query / output
    steps: int        # decode appends after the prefill
    seed: int
    k: np.ndarray = field(repr=False)        # [B, Hkv, T, D]
    v: np.ndarray = field(repr=False)        # [B, Hkv, T, D]
    q: np.ndarray = field(repr=False)        # [B, Hq, D]
    k_new: np.ndarray = field(repr=False)    # [steps, B, Hkv, D]
    v_new: np.ndarray = field(repr=False)    # [steps, B, Hkv, D]
    outlier_channels: np.ndarray = field(repr=False)  # [Hkv, 4]

    @property
    def capacity(self) -> int:
        need = self.T + self.steps
        return ((need + self.R - 1) // self.R) * self.R

    def q_for_step(self, i: int) -> np.ndarray:
        """A fresh N(0,1) query for decode step i (its own sub-stream)."""
        rng = np.random.default_rng([self.seed, 1000 + i])
        return cast(rng.standard_normal((self.B, self.Hq, self.D), np.float32), self.q_dtype)


def single_head(bits: int = 2) -> Workload:
    """The notebook's single-head K/V pair and query (fp32, T=1024, D=128)."""
    T, D = 1024, 128
    torch.manual_seed(0)
    K = torch.randn(T, D) * 0.5
    V = torch.randn(T, D) * 0.5
    for c in (3, 17, 40, 88):
        K[:, c] *= OUTLIER_SCALE
    torch.manual_seed(1)
    Q = torch.randn(1, T, D)
    k = K.numpy().reshape(1, 1, T, D).copy()
    v = V.numpy().reshape(1, 1, T, D).copy()
    q = Q[0, :1].numpy().reshape(1, 1, D).copy()
    empty = np.zeros((0, 1, 1, D), np.float32)
    wl = Workload("single_head", 1, 1, 1, D, T, 32, 32, bits, "f32", "f32", 0, 0,
                  k, v, q, empty, empty.copy(), np.array([[3, 17, 40, 88]]))
    wl.notebook_Q = Q.numpy()[0].copy()  # [T, D], the notebook's full query block
    return wl


def synthetic(name: str, *, B: int, Hq: int, Hkv: int, T: int, D: int = 128,
              R: int = 32, G: int = 32, bits: int = 2, dtype: str = "f16",
              q_dtype: str = "f16", steps: int = 0, seed: int = 0,
              v_spike_frac: float = 0.0) -> Workload:
    rng = np.random.default_rng(seed)
    outl = np.stack([rng.choice(D, 4, replace=False) for _ in range(Hkv)])
    k = rng.standard_normal((B, Hkv, T, D), np.float32)
    v = rng.standard_normal((B, Hkv, T, D), np.float32)
    for h in range(Hkv):
        k[:, h, :, outl[h]] *= OUTLIER_SCALE
    if v_spike_frac > 0.0:
        rows = B * Hkv * T
        n = int(round(rows * v_spike_frac))
        pick = rng.choice(rows, n, replace=False)
        v.reshape(rows, D)[pick] *= SPIKE_SCALE
    q = rng.standard_normal((B, Hq, D), np.float32)
    k_new = rng.standard_normal((steps, B, Hkv, D), np.float32)
    v_new = rng.standard_normal((steps, B, Hkv, D), np.float32)
    for h in range(Hkv):
        k_new[:, :, h, outl[h]] *= OUTLIER_SCALE
    return Workload(name, B, Hq, Hkv, D, T, R, G, bits, dtype, q_dtype, steps, seed,
                    cast(k, dtype), cast(v, dtype), cast(q, q_dtype),
                    cast(k_new, dtype), cast(v_new, dtype), outl)


# The five workloads of the benchmark description, at full size.
def llama3_8b_decode(**kw) -> Workload:
    """batch 8, 32 q heads / 8 KV heads, context 4096, fp16, one append + attention."""
    args = dict(B=8, Hq=32, Hkv=8, T=4096, R=32, dtype="f16", q_dtype="f16",
                steps=1, seed=2)
    args.update(kw)
    return synthetic("llama3_8b_decode", **args)


def prefill_quantize(bits: int = 2, **kw) -> Workload:
    """batch 4, 8 KV heads, context 32768, bf16, 0.1% V token spikes x8."""
    args = dict(B=4, Hq=8, Hkv=8, T=32768, R=32, bits=bits, dtype="bf16",
                q_dtype="f16", steps=0, seed=3, v_spike_frac=0.001)
    args.update(kw)
    return synthetic(f"prefill_quantize_{bits}bit", **args)


def long_context(**kw) -> Workload:
    """batch 1, 32 q heads / 8 KV heads, context 131072, residual 128, fp16."""
    args = dict(B=1, Hq=32, Hkv=8, T=131072, R=128, dtype="f16", q_dtype="f16",
                steps=0, seed=4)
    args.update(kw)
    return synthetic("long_context", **args)


def streaming(**kw) -> Workload:
    """batch 64, 28 q heads / 4 KV heads, prefill 2048 then 512 decode steps."""
    args = dict(B=64, Hq=28, Hkv=4, T=2048, R=32, dtype="f16", q_dtype="f16",
                steps=512, seed=5)
    args.update(kw)
    return synthetic("streaming", **args)
