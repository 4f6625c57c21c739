"""Thin Python binding of the C ABI in ``include/kivi.h`` (ctypes).

The functions named ``kivi_*`` mirror the C entry points one to one and do
argument marshalling only: every step of the hot path runs in the CUDA
library.  ``KiviCache`` bundles a handle with its device buffers, allocated
with PyTorch (PyTorch provides device memory and streams, nothing else).

There is no fallback: if ``libkivi_gb300.so`` is missing this module raises
on first use; build it with ``python -m bit_kv_cache_kivi_gb300.build``.
"""
from __future__ import annotations

import ctypes as C
import os
import threading

import torch

LIB_PATH = os.path.join(os.path.dirname(os.path.abspath(__file__)), "libkivi_gb300.so")

KIVI_OK, KIVI_EINVAL, KIVI_ESHAPE, KIVI_ECAPACITY = 0, 1, 2, 3
KIVI_EDTYPE, KIVI_ECUDA, KIVI_ESTATE, KIVI_EWORKSPACE = 4, 5, 6, 7
KIVI_F32, KIVI_F16, KIVI_BF16 = 0, 1, 2

BUFFER_NAMES = ("tiles", "ring_k", "ring_v")

_TORCH_DTYPE = {torch.float32: KIVI_F32, torch.float16: KIVI_F16, torch.bfloat16: KIVI_BF16}


class KiviError(RuntimeError):
    def __init__(self, status: int, what: str):
        self.status = status
        msg = f"{what}: {kivi_status_string(status)} (status {status})"
        if status == KIVI_ECUDA:
            msg += f", cudaError {lib().kivi_last_cuda_error()}"
        super().__init__(msg)


KIVI_POLICY_ALG1, KIVI_POLICY_SHARED = 0, 1


class kivi_config(C.Structure):
    _fields_ = [("bits", C.c_int), ("group", C.c_int), ("residual", C.c_int),
                ("head_dim", C.c_int), ("batch", C.c_int), ("n_kv_heads", C.c_int),
                ("n_q_heads", C.c_int), ("max_tokens", C.c_int), ("policy", C.c_int),
                ("outlier_channels", C.c_int)]


class kivi_buffers(C.Structure):
    _fields_ = [(n, C.c_void_p) for n in BUFFER_NAMES]


_lock = threading.Lock()
_lib = None


def lib() -> C.CDLL:
    """Load the CUDA library (raises if it has not been built)."""
    global _lib
    with _lock:
        if _lib is None:
            if not os.path.exists(LIB_PATH):
                raise ImportError(f"{LIB_PATH} is missing; build it with "
                                  "`python -m bit_kv_cache_kivi_gb300.build`")
            L = C.CDLL(LIB_PATH)
            vp, i32, sz, f32 = C.c_void_p, C.c_int, C.c_size_t, C.c_float
            sigs = {
                "kivi_cache_sizes": (i32, [C.POINTER(kivi_config), C.POINTER(sz)]),
                "kivi_cache_init": (i32, [C.POINTER(kivi_config), C.POINTER(kivi_buffers),
                                          C.POINTER(vp)]),
                "kivi_quantize_prefill": (i32, [vp, vp, vp, i32, i32, vp]),
                "kivi_quantize_prefill_varlen": (i32, [vp, vp, vp, i32, i32, C.POINTER(i32), vp]),
                "kivi_cache_set_lengths": (i32, [vp, C.POINTER(i32)]),
                "kivi_cache_lengths": (i32, [vp, C.POINTER(i32)]),
                "kivi_append_decode": (i32, [vp, vp, vp, i32, vp]),
                "kivi_append_tokens": (i32, [vp, vp, vp, i32, i32, vp]),
                "kivi_cache_set_length": (i32, [vp, i32]),
                "kivi_attention_workspace_bytes": (sz, [vp]),
                "kivi_decode_attention": (i32, [vp, vp, i32, vp, f32, vp, sz, vp]),
                "kivi_set_attention_splits": (i32, [vp, i32]),
                "kivi_attention_splits": (i32, [vp, i32]),
                "kivi_set_attention_overlap": (i32, [vp, i32]),
                "kivi_cache_length": (i32, [vp]),
                "kivi_cache_reset": (i32, [vp]),
                "kivi_cache_destroy": (None, [vp]),
                "kivi_status_string": (C.c_char_p, [i32]),
                "kivi_last_cuda_error": (i32, []),
                "kivi_decode_attention_static": (i32, [vp, vp, i32, vp, f32, vp]),
                "kivi_decode_step": (i32, [vp, vp, vp, i32, vp, i32, vp, f32, vp, sz, vp]),
                "kivi_check_bounded_wait": (i32, [vp, vp]),
            }
            for name, (res, args) in sigs.items():
                fn = getattr(L, name)
                fn.restype = res
                fn.argtypes = args
            _lib = L
    return _lib


def _check(status: int, what: str) -> None:
    if status != KIVI_OK:
        raise KiviError(status, what)


_raw_stream = getattr(torch._C, "_cuda_getCurrentRawStream", None)


def _stream(stream, device_index: int | None = None) -> int:
    """The cudaStream_t to launch on: the given stream, else the current
    stream of the device (read without building a Stream object)."""
    if stream is None:
        if _raw_stream is not None:
            return _raw_stream(torch.cuda.current_device() if device_index is None else device_index)
        return torch.cuda.current_stream().cuda_stream
    return stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream)


def _ptr(t) -> int:
    return t.data_ptr() if isinstance(t, torch.Tensor) else int(t)


# ------------------------------------------------------------ C entry points

def kivi_status_string(status: int) -> str:
    return lib().kivi_status_string(status).decode()


def kivi_check_bounded_wait(status: torch.Tensor, stream=None) -> None:
    """Runs the attention's bounded wait on a barrier phase nothing completes;
    ORs 1 into status (one int32 on the current device) when it gives up."""
    if not (isinstance(status, torch.Tensor) and status.dtype == torch.int32 and status.numel() >= 1):
        raise KiviError(KIVI_EINVAL, "kivi_check_bounded_wait: status must be an int32 tensor")
    _check(lib().kivi_check_bounded_wait(status.data_ptr(), _stream(stream)), "kivi_check_bounded_wait")


def kivi_cache_sizes(cfg: kivi_config) -> list[int]:
    out = (C.c_size_t * len(BUFFER_NAMES))()
    _check(lib().kivi_cache_sizes(C.byref(cfg), out), "kivi_cache_sizes")
    return list(out)


def kivi_cache_init(cfg: kivi_config, bufs: kivi_buffers) -> C.c_void_p:
    h = C.c_void_p()
    _check(lib().kivi_cache_init(C.byref(cfg), C.byref(bufs), C.byref(h)), "kivi_cache_init")
    return h


def kivi_quantize_prefill(h, k, v, dtype: int, n_tokens: int, stream=None) -> None:
    _check(lib().kivi_quantize_prefill(h, _ptr(k), _ptr(v), dtype, n_tokens, _stream(stream)),
           "kivi_quantize_prefill")


def kivi_quantize_prefill_varlen(h, k, v, dtype: int, max_len: int, lengths, stream=None) -> None:
    arr = (C.c_int * len(lengths))(*[int(x) for x in lengths])
    _check(lib().kivi_quantize_prefill_varlen(h, _ptr(k), _ptr(v), dtype, max_len, arr, _stream(stream)),
           "kivi_quantize_prefill_varlen")


def kivi_cache_set_lengths(h, lengths) -> None:
    arr = (C.c_int * len(lengths))(*[int(x) for x in lengths])
    _check(lib().kivi_cache_set_lengths(h, arr), "kivi_cache_set_lengths")


def kivi_cache_lengths(h, batch: int) -> list[int]:
    arr = (C.c_int * batch)()
    _check(lib().kivi_cache_lengths(h, arr), "kivi_cache_lengths")
    return list(arr)


def kivi_append_decode(h, k_new, v_new, dtype: int, stream=None) -> None:
    _check(lib().kivi_append_decode(h, _ptr(k_new), _ptr(v_new), dtype, _stream(stream)),
           "kivi_append_decode")


def kivi_append_tokens(h, k, v, dtype: int, n_tokens: int, stream=None) -> None:
    _check(lib().kivi_append_tokens(h, _ptr(k), _ptr(v), dtype, n_tokens, _stream(stream)),
           "kivi_append_tokens")


def kivi_cache_set_length(h, length: int) -> None:
    _check(lib().kivi_cache_set_length(h, length), "kivi_cache_set_length")


def kivi_attention_workspace_bytes(h) -> int:
    return int(lib().kivi_attention_workspace_bytes(h))


def kivi_decode_attention(h, q, q_dtype: int, out, softmax_scale: float, workspace,
                          ws_bytes: int, stream=None) -> None:
    _check(lib().kivi_decode_attention(h, _ptr(q), q_dtype, _ptr(out), float(softmax_scale),
                                       _ptr(workspace), ws_bytes, _stream(stream)),
           "kivi_decode_attention")


def kivi_decode_step(h, k_new, v_new, kv_dtype: int, q, q_dtype: int, out, softmax_scale: float,
                     workspace, ws_bytes: int, stream=None) -> None:
    """Append one token, then decode attention over the grown cache, the
    attention launched as a programmatic dependent of the append (the C
    header describes which of its CTAs wait for the append)."""
    _check(lib().kivi_decode_step(h, _ptr(k_new), _ptr(v_new), kv_dtype, _ptr(q), q_dtype, _ptr(out),
                                  float(softmax_scale), _ptr(workspace), ws_bytes, _stream(stream)),
           "kivi_decode_step")


def kivi_decode_attention_static(h, q, q_dtype: int, out, softmax_scale: float,
                                 stream=None) -> None:
    """Decode attention using the library's fixed device scratch area instead
    of a workspace argument (for callers that cannot allocate; see kivi.h)."""
    _check(lib().kivi_decode_attention_static(h, _ptr(q), q_dtype, _ptr(out),
                                              float(softmax_scale), _stream(stream)),
           "kivi_decode_attention_static")


def kivi_set_attention_splits(h, n_splits: int) -> None:
    _check(lib().kivi_set_attention_splits(h, n_splits), "kivi_set_attention_splits")


def kivi_attention_splits(h, l: int) -> int:
    return int(lib().kivi_attention_splits(h, l))


def kivi_set_attention_overlap(h, enable: int) -> None:
    _check(lib().kivi_set_attention_overlap(h, int(enable)), "kivi_set_attention_overlap")


def kivi_cache_length(h) -> int:
    return int(lib().kivi_cache_length(h))


def kivi_cache_reset(h) -> None:
    _check(lib().kivi_cache_reset(h), "kivi_cache_reset")


def kivi_cache_destroy(h) -> None:
    lib().kivi_cache_destroy(h)


# ------------------------------------------------------------ convenience

class KiviCache:
    """A KIVI cache: C handle + the three device buffers + attention workspace."""

    def __init__(self, *, batch: int, n_kv_heads: int, n_q_heads: int, max_tokens: int,
                 bits: int = 2, group: int = 32, residual: int = 32, head_dim: int = 128,
                 policy: int = 0, outliers: int = 0, device="cuda"):
        self.cfg = kivi_config(bits, group, residual, head_dim, batch, n_kv_heads,
                               n_q_heads, max_tokens, policy, outliers)
        d = torch.device(device)
        if d.type == "cuda" and d.index is None:
            d = torch.device("cuda", torch.cuda.current_device())
        self.device = d
        sizes = kivi_cache_sizes(self.cfg)
        self.buffers = {n: torch.empty(max(s, 16), dtype=torch.uint8, device=self.device)
                        for n, s in zip(BUFFER_NAMES, sizes)}
        bufs = kivi_buffers(*[self.buffers[n].data_ptr() for n in BUFFER_NAMES])
        self.handle = kivi_cache_init(self.cfg, bufs)
        self.ws_bytes = kivi_attention_workspace_bytes(self.handle)
        self._tok_shape = torch.Size((batch, n_kv_heads, head_dim))
        self._q_shape = torch.Size((batch, n_q_heads, head_dim))
        self.workspace = torch.empty(max(self.ws_bytes, 16), dtype=torch.uint8, device=self.device)
        self._ws_ptr = self.workspace.data_ptr()
        self._step_fn = lib().kivi_decode_step  # the per-step call, looked up once

    def __del__(self):
        h = getattr(self, "handle", None)
        if h:
            kivi_cache_destroy(h)
            self.handle = None

    # -- shape helpers
    @property
    def length(self) -> int:
        """Every sequence's length; -2 when the sequences' lengths differ."""
        return kivi_cache_length(self.handle)

    @property
    def lengths(self) -> list[int]:
        """Per-sequence lengths."""
        return kivi_cache_lengths(self.handle, self.cfg.batch)

    def _reachable(self, x: torch.Tensor) -> bool:
        """On the cache's device, or host memory.  Host tensors must be
        page-locked (the kernels read and write them in place); the C
        library checks that with one pointer query per buffer and refuses
        pageable memory with KIVI_EINVAL before any launch, so it is not
        queried a second time here."""
        return x.device == self.device or x.device.type == "cpu"

    def _check_kv(self, x: torch.Tensor, T: int | None) -> int:
        c = self.cfg
        if not self._reachable(x) or not x.is_contiguous():
            raise ValueError("K/V must be contiguous tensors on the cache's device or in pinned host memory")
        want = (c.batch, c.n_kv_heads, T, c.head_dim) if T is not None else self._tok_shape
        if x.shape != want:
            raise ValueError(f"expected shape {want}, got {tuple(x.shape)}")
        if x.dtype not in _TORCH_DTYPE:
            raise ValueError(f"unsupported dtype {x.dtype}")
        return _TORCH_DTYPE[x.dtype]

    # -- the hot path
    def prefill(self, k: torch.Tensor, v: torch.Tensor, lengths=None, stream=None) -> None:
        """Prefill an empty cache from k, v [B][H][T][D]; with ``lengths``
        (B ints), sequence b takes only its first lengths[b] rows."""
        T = k.shape[2]
        dt = self._check_kv(k, T)
        if self._check_kv(v, T) != dt:
            raise ValueError("K and V dtypes differ")
        if lengths is None:
            kivi_quantize_prefill(self.handle, k, v, dt, T, stream)
        else:
            if len(lengths) != self.cfg.batch:
                raise ValueError(f"expected {self.cfg.batch} lengths")
            kivi_quantize_prefill_varlen(self.handle, k, v, dt, T, lengths, stream)

    def append(self, k_new: torch.Tensor, v_new: torch.Tensor, stream=None) -> None:
        shape = self._tok_shape
        if k_new.shape != shape:
            k_new = k_new.reshape(shape)
        if v_new.shape != shape:
            v_new = v_new.reshape(shape)
        dt = self._check_kv(k_new, None)
        if self._check_kv(v_new, None) != dt:
            raise ValueError("K and V dtypes differ")
        kivi_append_decode(self.handle, k_new, v_new, dt, _stream(stream, self.device.index))

    def append_tokens(self, k: torch.Tensor, v: torch.Tensor, stream=None) -> None:
        """Append k, v [B][H][n][D] (n >= 1) to a cache of any length."""
        n = k.shape[2]
        dt = self._check_kv(k, n)
        if self._check_kv(v, n) != dt:
            raise ValueError("K and V dtypes differ")
        kivi_append_tokens(self.handle, k, v, dt, n, stream)

    def set_length(self, length: int) -> None:
        """The length of a state whose buffers were just restored."""
        kivi_cache_set_length(self.handle, length)

    def set_lengths(self, lengths) -> None:
        """Per-sequence lengths of a state whose buffers were just restored."""
        if len(lengths) != self.cfg.batch:
            raise ValueError(f"expected {self.cfg.batch} lengths")
        kivi_cache_set_lengths(self.handle, lengths)

    def _check_q_out(self, q: torch.Tensor, out: torch.Tensor | None) -> torch.Tensor:
        if q.shape != self._q_shape or not q.is_contiguous():
            raise ValueError(f"q must be contiguous {tuple(self._q_shape)}")
        if not self._reachable(q):
            raise ValueError("q must be on the cache's device or in pinned host memory")
        if q.dtype not in _TORCH_DTYPE:
            raise ValueError(f"unsupported q dtype {q.dtype}")
        if out is None:
            out = torch.empty_like(q, pin_memory=q.device.type == "cpu")
        elif (out.shape != q.shape or out.dtype != q.dtype or not out.is_contiguous()
              or not self._reachable(out)):
            raise ValueError("out must match q (and be on the device or in pinned host memory)")
        return out

    def attention(self, q: torch.Tensor, out: torch.Tensor | None = None,
                  softmax_scale: float = 0.0, stream=None) -> torch.Tensor:
        out = self._check_q_out(q, out)
        kivi_decode_attention(self.handle, q, _TORCH_DTYPE[q.dtype], out, softmax_scale,
                              self.workspace, self.ws_bytes, _stream(stream, self.device.index))
        return out

    def step(self, k_new: torch.Tensor, v_new: torch.Tensor, q: torch.Tensor,
             out: torch.Tensor | None = None, softmax_scale: float = 0.0, stream=None) -> torch.Tensor:
        """One decode step: append k_new, v_new ([B][H][D]), then decode
        attention of q over the grown cache, in one call; the attention is
        launched as a programmatic dependent of the append, so its launch,
        its query tables and (on most steps) its packed splits overlap the
        append.  Same cache and output as append() followed by attention()."""
        shape = self._tok_shape
        if k_new.shape != shape:
            k_new = k_new.reshape(shape)
        if v_new.shape != shape:
            v_new = v_new.reshape(shape)
        dt = self._check_kv(k_new, None)
        if self._check_kv(v_new, None) != dt:
            raise ValueError("K and V dtypes differ")
        out = self._check_q_out(q, out)
        st = self._step_fn(self.handle, k_new.data_ptr(), v_new.data_ptr(), dt, q.data_ptr(),
                           _TORCH_DTYPE[q.dtype], out.data_ptr(), float(softmax_scale), self._ws_ptr,
                           self.ws_bytes, _stream(stream, self.device.index))
        if st != KIVI_OK:
            raise KiviError(st, "kivi_decode_step")
        return out

    def set_splits(self, n: int) -> None:
        kivi_set_attention_splits(self.handle, n)

    def set_overlap(self, enable: bool) -> None:
        """Let attention() calls overlap the kernel before them on the stream
        (see kivi_set_attention_overlap in kivi.h for when that is safe)."""
        kivi_set_attention_overlap(self.handle, 1 if enable else 0)

    def splits(self, l: int | None = None) -> int:
        return kivi_attention_splits(self.handle, self.length if l is None else l)

    def reset(self) -> None:
        kivi_cache_reset(self.handle)

    def _tile_bytes(self) -> int:
        c = self.cfg
        n = c.outlier_channels
        return 2 * c.group * (c.head_dim * c.bits // 8) + 8 * c.head_dim + (16 + 64 * n if n else 0)

    def _ring_slots(self) -> int:
        c = self.cfg
        return c.residual + c.group if c.policy == KIVI_POLICY_SHARED else c.residual

    def state_views(self) -> dict:
        """The cache's state as its three raw buffers (saving and restoring a
        cache is copying these plus ``length``): the packed tiles as bytes
        [B][H][T/G][tile bytes], the rings as fp16 bit patterns (int16)."""
        c = self.cfg
        B, H, T, D, G = c.batch, c.n_kv_heads, c.max_tokens, c.head_dim, c.group
        tb = self._tile_bytes()
        W = self._ring_slots()
        return {"tiles": self.buffers["tiles"][:B * H * (T // G) * tb].view(B, H, T // G, tb),
                "ring_k": self.buffers["ring_k"][:2 * B * H * W * D].view(torch.int16).view(B, H, W, D),
                "ring_v": self.buffers["ring_v"][:2 * B * H * W * D].view(torch.int16).view(B, H, W, D)}

    def layout_views(self) -> dict:
        """Strided views of the arrays inside the tiles (no copies), with the
        tile axis kept: codes_k / codes_v [B][H][T/G][G][RB] (u8), scale_k /
        zero_k [B][H][T/G][D] in channel-pair order (see ``key_scale_pos``),
        scale_v / zero_v [B][H][T/G][G * D/G] in token-pair order (see
        ``value_scale_pos``), fp16 bit patterns as int16; plus the rings.  At
        8 bits the code rows are stored rotated by 16-byte chunks (see
        ``row_chunk_rotation``)."""
        c = self.cfg
        B, H, T, D, G = c.batch, c.n_kv_heads, c.max_tokens, c.head_dim, c.group
        rb = D * c.bits // 8
        tb = self._tile_bytes()
        nt = T // G
        u8 = self.buffers["tiles"]
        i16 = u8[:(u8.numel() // 2) * 2].view(torch.int16)
        st8 = (H * nt * tb, nt * tb, tb)
        st16 = tuple(x // 2 for x in st8)
        # as_strided offsets count from the start of the storage, and the
        # tile buffer may itself be a view into a larger allocation
        b8, b16 = u8.storage_offset(), i16.storage_offset()
        # byte offsets in a tile: key zeros, key codes, value codes, key
        # scales, value scales, value zeros
        o_kc = 2 * D
        o_sk = o_kc + 2 * G * rb
        out = {"codes_k": u8.as_strided((B, H, nt, G, rb), st8 + (rb, 1), b8 + o_kc),
               "codes_v": u8.as_strided((B, H, nt, G, rb), st8 + (rb, 1), b8 + o_kc + G * rb),
               "scale_k": i16.as_strided((B, H, nt, D), st16 + (1,), b16 + o_sk // 2),
               "zero_k": i16.as_strided((B, H, nt, D), st16 + (1,), b16),
               "scale_v": i16.as_strided((B, H, nt, D), st16 + (1,), b16 + (o_sk + 2 * D) // 2),
               "zero_v": i16.as_strided((B, H, nt, D), st16 + (1,), b16 + (o_sk + 4 * D) // 2)}
        n = c.outlier_channels
        if n:  # the outlier block after the base tile: indices, then values [G][n]
            o_ob = 2 * G * rb + 8 * D
            out["outl_idx"] = u8.as_strided((B, H, nt, n), st8 + (1,), b8 + o_ob)
            out["outl_val"] = i16.as_strided((B, H, nt, G, n), st16 + (n, 1), b16 + (o_ob + 16) // 2)
        sv = self.state_views()
        out["ring_k"], out["ring_v"] = sv["ring_k"], sv["ring_v"]
        return out

    def logical_state(self) -> dict:
        """The arrays in token-major shapes and channel order (device
        copies): codes_k / codes_v [B][H][T][RB] as plain rows (channel e at
        bits [e*bits, e*bits + bits), LSB first), scale_k / zero_k
        [B][H][T/G][D], scale_v / zero_v [B][H][T][D/G], ring_k / ring_v
        [B][H][W][D]."""
        c = self.cfg
        B, H, T, D, G = c.batch, c.n_kv_heads, c.max_tokens, c.head_dim, c.group
        lv = self.layout_views()
        dev = self.buffers["tiles"].device
        kidx = torch.tensor([key_scale_pos(ch, c.bits) for ch in range(D)], device=dev)
        vidx = torch.tensor([value_scale_pos(t, gp) for t in range(G) for gp in range(D // G)], device=dev)
        out = {}
        for n, t in lv.items():
            if n in ("codes_k", "codes_v"):
                if c.bits == 8:  # undo the rows' chunk rotation
                    idx = torch.tensor([[16 * ((ch + row_chunk_rotation(8, n == "codes_k", r)) % 8) + i
                                         for ch in range(8) for i in range(16)] for r in range(G)],
                                       device=dev)
                    t = torch.gather(t, 4, idx.expand(B, H, t.shape[2], G, 128))
                out[n] = plain_rows(t.reshape(B, H, T, t.shape[-1]), c.bits, n == "codes_v")
            elif n in ("scale_k", "zero_k"):
                out[n] = t.index_select(3, kidx)
            elif n in ("scale_v", "zero_v"):
                out[n] = t.index_select(3, vidx).reshape(B, H, T, D // G)
            elif n == "outl_val":
                out[n] = t.reshape(B, H, T, t.shape[-1])
            else:
                out[n] = t.clone()
        return out


def _hi_bit3(s: int, i: int) -> int:
    """Bit of (set s, index i) inside a 16-bit unit of a 3-bit row's high plane."""
    p = 2 * (i % 4) + 2 + (1 if i >= 4 else 0)
    return (p + 8) % 16 if s else p


def tile_row_bit(e: int, j: int, bits: int, value: bool, D: int = 128, G: int = 32) -> int:
    """Bit (from the row start) holding bit j of channel e's code in a code
    row of a tile (after undoing the 8-bit chunk rotation).  Key rows at 2, 4
    and 8 bits are plain (channel e at bits e*bits + j).  Value rows keep the
    same order inside units of 4 channels and interleave the units by group:
    the unit of channels G*gp + 4w .. +3 sits at unit position 4w + gp.  A
    3-bit row is two planes: the low two bits as a 2-bit row of the same
    kind, then the high bits in 16-bit units (keys: unit 2(m mod 4) + h
    holds channels 16m + 8h + i, set m // 4; values: unit w holds channels
    32gp + 4w + c, set gp // 2, index 4(gp mod 2) + c)."""
    lbits = 2 if bits == 3 else bits
    if bits == 3 and j == 2:
        if value:
            gp, w, c = e // 32, (e % 32) // 4, e % 4
            return D * 2 + 16 * w + _hi_bit3(gp // 2, 4 * (gp % 2) + c)
        m, h, i = e // 16, (e % 16) // 8, e % 8
        return D * 2 + 16 * (2 * (m % 4) + h) + _hi_bit3(m // 4, i)
    if not value:
        return e * lbits + j
    u, c = e // 4, e % 4
    pos = 4 * (u % (G // 4)) + u // (G // 4)
    return pos * 4 * lbits + c * lbits + j


_PLAIN_MAPS: dict = {}


def plain_rows(rows: torch.Tensor, bits: int, value: bool) -> torch.Tensor:
    """Code rows of a tile ([..., D*bits/8] u8) as plain rows: channel e at
    bits [e*bits, e*bits + bits), LSB first (a fresh tensor)."""
    RB = rows.shape[-1]
    D = RB * 8 // bits
    if bits != 3 and not value:
        return rows.clone()
    key = (bits, value, D, rows.device)
    if key not in _PLAIN_MAPS:
        src = [tile_row_bit(e, j, bits, value, D) for e in range(D) for j in range(bits)]
        _PLAIN_MAPS[key] = torch.tensor(src, dtype=torch.long, device=rows.device)
    src = _PLAIN_MAPS[key]
    shifts = torch.arange(8, dtype=torch.uint8, device=rows.device)
    flat = rows.reshape(-1, RB)
    out = torch.empty_like(flat)
    step = max(1, (64 << 20) // (RB * 8))  # rows per chunk: about 64 MB of bits
    for i in range(0, flat.shape[0], step):
        blk = flat[i:i + step]
        b = ((blk.unsqueeze(-1) >> shifts) & 1).reshape(blk.shape[0], RB * 8)
        p = b.index_select(1, src).reshape(blk.shape[0], RB, 8)
        out[i:i + step] = (p << shifts).sum(dim=-1, dtype=torch.uint8)
    return out.reshape(rows.shape)


def key_scale_pos(c: int, bits: int) -> int:
    """fp16 slot of channel c in a tile's key scale / zero block: 32-bit word
    i of pair block m holds channels (P m + i, P m + i + P/2), P = 16 at 2 and
    3 bits, 8 at 4 bits (the pairs the score product's B fragments take)."""
    P = {2: 16, 3: 16, 4: 8, 8: 4}[bits]
    return P * (c // P) + 2 * (c % (P // 2)) + (c % P) // (P // 2)


def row_chunk_rotation(bits: int, key: bool, r: int) -> int:
    """16-byte chunks by which code row r of a tile is rotated: at 8 bits key
    rows by r & 1, value rows by 2 (r & 3) (logical chunk c sits at chunk
    (c + rotation) mod 8); none at 2 and 4 bits."""
    if bits != 8:
        return 0
    return (r & 1) if key else 2 * (r & 3)


def value_scale_pos(t: int, gp: int) -> int:
    """fp16 slot of token t (within its tile), value group gp in a tile's
    value scale / zero block: tokens (8a + r, 8a + r + 4), r < 4, share the
    32-bit word 4 (4a + r) + gp."""
    return 32 * (t // 8) + 8 * (t % 4) + 2 * gp + (t // 4) % 2
