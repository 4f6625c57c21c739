"""GB300-native KIVI KV cache: 2/4-bit grouped quantization with an fp16
residual window, and fused dequantize + decode attention over the packed
cache.  The compute runs in the CUDA library ``libkivi_gb300.so`` (built from
``csrc/``); ``kivi`` is its thin ctypes binding.

Importing this package loads nothing; ``bit_kv_cache_kivi_gb300.kivi``
loads the shared library on first use and raises if it is missing.
"""

__all__ = ["kivi", "workloads"]
