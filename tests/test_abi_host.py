"""Host-side checks of the C-ABI library: it builds, loads, exports every
entry point the header declares, and its host logic (sizes, validation,
state checks, split plan) behaves as documented.  No GPU is needed: nothing
here launches a kernel."""
import ctypes as C
import os
import re

import pytest

from conftest import ROOT


@pytest.fixture(scope="module")
def K():
    from bit_kv_cache_kivi_gb300 import build, kivi
    build.build()
    kivi.lib()
    return kivi


def _declared():
    hdr = open(os.path.join(ROOT, "include", "kivi.h")).read()
    hdr = re.sub(r"/\*.*?\*/", "", hdr, flags=re.S)
    return sorted(set(re.findall(r"\b(kivi_[a-z_0-9]+)\s*\(", hdr)))


def test_every_declared_symbol_is_exported(K):
    names = _declared()
    assert "kivi_decode_attention" in names and len(names) >= 12
    lib = C.CDLL(K.LIB_PATH)
    for n in names:
        assert hasattr(lib, n), n


def test_only_abi_symbols_are_exported(K):
    import subprocess
    out = subprocess.run(["nm", "-D", "--defined-only", K.LIB_PATH], capture_output=True,
                         text=True).stdout
    funcs = [l.split()[-1] for l in out.splitlines() if " T " in l]
    ours = [f for f in funcs if f.startswith("kivi_")]
    assert sorted(ours) == _declared()


def cfg(K, **kw):
    d = dict(bits=2, group=32, residual=32, head_dim=128, batch=2, n_kv_heads=4,
             n_q_heads=16, max_tokens=4096)
    d.update(kw)
    return K.kivi_config(**d)


def test_sizes(K):
    """Tiles of 2 G RB + 8 D bytes (key / value code rows of G tokens, key
    scale / zero [D], value scale / zero [G][D/G]) per G tokens, and rings."""
    s = K.kivi_cache_sizes(cfg(K))
    units = 2 * 4
    assert len(s) == 3
    assert s[0] == units * (4096 // 32) * (2 * 32 * 32 + 8 * 128)
    assert s[0] == units * 4096 * 32 * 2 + units * (4096 // 32) * 128 * 2 * 2 + units * 4096 * 4 * 2 * 2
    assert s[1] == s[2] == units * 32 * 128 * 2
    s4 = K.kivi_cache_sizes(cfg(K, bits=4))
    assert s4[0] == units * (4096 // 32) * (2 * 32 * 64 + 8 * 128) and s4[1:] == s[1:]
    s8 = K.kivi_cache_sizes(cfg(K, bits=8))
    assert s8[0] == units * (4096 // 32) * (2 * 32 * 128 + 8 * 128) and s8[1:] == s[1:]
    # outlier-aware keys: a 16-byte index block and 32 fp16 values per channel per tile
    so = K.kivi_cache_sizes(cfg(K, outlier_channels=2))
    assert so[0] == s[0] + units * (4096 // 32) * (16 + 32 * 2 * 2) and so[1:] == s[1:]
    # the shared-window policy keeps up to R + G - 1 fp16 tokens: R + G slots
    ss = K.kivi_cache_sizes(cfg(K, policy=1))
    assert ss[0] == s[0] and ss[1] == ss[2] == units * (32 + 32) * 128 * 2


def test_scale_slot_maps_are_permutations(K):
    """The tile's fp16 scale / zero orders are bijections of the 128 slots,
    and keep each 32-channel quarter in place (the tail split relies on it)."""
    for bits in (2, 3, 4, 8):
        pos = [K.key_scale_pos(c, bits) for c in range(128)]
        assert sorted(pos) == list(range(128))
        assert all(p // 32 == c // 32 for c, p in enumerate(pos))
        # word i of a pair block: channels (P m + i, P m + i + P/2)
        P = {2: 16, 3: 16, 4: 8, 8: 4}[bits]
        assert pos[P + 1] == P + 2 and pos[P + 1 + P // 2] == P + 3
    vpos = [K.value_scale_pos(t, g) for t in range(32) for g in range(4)]
    assert sorted(vpos) == list(range(128))
    assert K.value_scale_pos(9, 2) + 1 == K.value_scale_pos(13, 2)  # pair (9, 13) in one word


@pytest.mark.parametrize("bad,status", [
    (dict(policy=2), 1), (dict(policy=-1), 1), (dict(outlier_channels=5), 1), (dict(outlier_channels=-1), 1),
    (dict(bits=5), 1), (dict(bits=1), 1), (dict(group=16), 1), (dict(head_dim=64), 1),
    (dict(residual=48), 2), (dict(residual=0), 2), (dict(n_q_heads=6), 2),
    (dict(max_tokens=4016, residual=64), 2), (dict(batch=0), 2), (dict(n_kv_heads=0), 2),
    (dict(n_kv_heads=4096, n_q_heads=4096 * 136), 2),  # attention grid y: 4096 x 17 chunks of 8
])
def test_config_validation(K, bad, status):
    with pytest.raises(K.KiviError) as e:
        K.kivi_cache_sizes(cfg(K, **bad))
    assert e.value.status == status


def _fake_buffers(K, base=1 << 20, misalign=None):
    ptrs = [base + i * (1 << 16) for i in range(len(K.BUFFER_NAMES))]
    if misalign is not None:
        ptrs[misalign] += 8
    return K.kivi_buffers(*ptrs)


def test_init_validation_and_host_state(K):
    c = cfg(K)
    with pytest.raises(K.KiviError) as e:
        K.kivi_cache_init(c, K.kivi_buffers(*([None] * len(K.BUFFER_NAMES))))
    assert e.value.status == K.KIVI_EINVAL
    for i in range(len(K.BUFFER_NAMES)):
        with pytest.raises(K.KiviError) as e:
            K.kivi_cache_init(c, _fake_buffers(K, misalign=i))
        assert e.value.status == K.KIVI_EINVAL
    # binding never touches the buffers, so fake device addresses are fine here
    h = K.kivi_cache_init(c, _fake_buffers(K))
    try:
        assert K.kivi_cache_length(h) == 0
        lib = K.lib()
        # checks that come before any launch
        assert lib.kivi_quantize_prefill(h, 16, 16, 7, 10, None) == K.KIVI_EDTYPE
        assert lib.kivi_quantize_prefill(h, 16, 16, K.KIVI_F16, 4097, None) == K.KIVI_ECAPACITY
        assert lib.kivi_quantize_prefill(h, 16, 16, K.KIVI_F16, -1, None) == K.KIVI_ESHAPE
        assert lib.kivi_quantize_prefill(h, 16, 16, K.KIVI_F16, 0, None) == K.KIVI_OK
        assert lib.kivi_quantize_prefill(h, 0, 16, K.KIVI_F16, 5, None) == K.KIVI_EINVAL
        assert lib.kivi_append_decode(h, 16, 16, 9, None) == K.KIVI_EDTYPE
        assert lib.kivi_append_decode(h, 0, 16, K.KIVI_F16, None) == K.KIVI_EINVAL
        assert lib.kivi_append_tokens(h, 16, 16, 9, 3, None) == K.KIVI_EDTYPE
        assert lib.kivi_append_tokens(h, 16, 16, K.KIVI_F16, 0, None) == K.KIVI_EINVAL
        assert lib.kivi_append_tokens(h, 16, 24, K.KIVI_F16, 3, None) == K.KIVI_EINVAL  # misaligned
        assert lib.kivi_append_tokens(h, 16, 16, K.KIVI_F16, 4097, None) == K.KIVI_ECAPACITY
        assert lib.kivi_cache_set_length(h, 4097) == K.KIVI_ECAPACITY
        assert lib.kivi_cache_set_length(h, -1) == K.KIVI_ECAPACITY
        assert lib.kivi_cache_set_length(h, 100) == K.KIVI_OK and K.kivi_cache_length(h) == 100
        assert lib.kivi_cache_set_length(h, 0) == K.KIVI_OK
        ws = K.kivi_attention_workspace_bytes(h)
        assert lib.kivi_decode_attention(h, 16, K.KIVI_F16, 16, 0.0, 16, ws, None) == K.KIVI_ESTATE
        assert lib.kivi_decode_attention(h, 16, 5, 16, 0.0, 16, ws, None) == K.KIVI_EDTYPE
        # the decode step makes every check of both halves before any launch
        # and leaves the length unchanged on a refusal
        step = lib.kivi_decode_step
        assert step(None, 16, 16, 1, 16, 1, 16, 0.0, 16, ws, None) == K.KIVI_EINVAL
        assert step(h, 16, 16, 9, 16, 1, 16, 0.0, 16, ws, None) == K.KIVI_EDTYPE
        assert step(h, 16, 16, 1, 16, 7, 16, 0.0, 16, ws, None) == K.KIVI_EDTYPE
        assert step(h, 0, 16, 1, 16, 1, 16, 0.0, 16, ws, None) == K.KIVI_EINVAL
        assert step(h, 16, 16, 1, 0, 1, 16, 0.0, 16, ws, None) == K.KIVI_EINVAL
        assert step(h, 16, 16, 1, 16, 1, 0, 0.0, 16, ws, None) == K.KIVI_EINVAL
        assert step(h, 16, 16, 1, 16, 1, 16, 0.0, 16, ws - 16, None) == K.KIVI_EWORKSPACE
        assert step(h, 16, 16, 1, 16, 1, 16, 0.0, 24, ws, None) == K.KIVI_EWORKSPACE
        assert step(h, 16, 16, 1, 16, 1, 16, 0.0, 0, ws, None) == K.KIVI_EWORKSPACE
        assert lib.kivi_cache_set_length(h, 4096) == K.KIVI_OK
        assert step(h, 16, 16, 1, 16, 1, 16, 0.0, 16, ws, None) == K.KIVI_ECAPACITY
        assert K.kivi_cache_length(h) == 4096
        assert lib.kivi_cache_set_length(h, 0) == K.KIVI_OK
        assert K.kivi_cache_length(None) == -1
        K.kivi_cache_reset(h)
    finally:
        K.kivi_cache_destroy(h)
    K.kivi_cache_destroy(None)
    assert K.kivi_status_string(K.KIVI_ECAPACITY) == "cache capacity exceeded"


def test_split_plan_and_workspace(K):
    """The first splits take the fp16 tail, 64 tokens each; the packed tiles
    [0, floor32(l - R)) are shared by up to floor(4 * 152 / units) - (tail
    splits) splits of >= 8 tiles, a
    multiple of four tiles each, so the grid fits one wave of four CTAs per
    SM and the four warps of a CTA get equal shares."""
    # Llama-3-8B decode shape: 64 (b, kv-head) units -> up to 8 tile splits;
    # 127 tiles -> 16 tiles per split -> 8 tile splits
    c = cfg(K, batch=8, n_kv_heads=8, n_q_heads=32, max_tokens=4128)
    h = K.kivi_cache_init(c, _fake_buffers(K))
    try:
        assert K.kivi_attention_splits(h, 4097) == 9
        assert K.kivi_attention_splits(h, 100) == 2   # tail + one 64-token split
        assert K.kivi_attention_splits(h, 40) == 1    # everything is tail
        # 64 groups x (9 split partials + 1 merged group) x 8 heads (a chunk)
        # x (128 + 2) floats, one counter per split group and per group, two
        # generation words per group, the status slot
        assert K.kivi_attention_workspace_bytes(h) == 64 * (9 + 1) * 8 * (128 + 2) * 4 + 64 * 4 * 4 + 16
        K.kivi_set_attention_splits(h, 3)
        assert K.kivi_attention_splits(h, 4097) == 3
        K.kivi_set_attention_splits(h, 1000)  # clamped to the workspace bound
        assert K.kivi_attention_splits(h, 4097) == 9
        # overlapped launches: a third of the budget (3) and >= 128 tiles per
        # packed split -> 1 packed split, the one-split tail riding on it;
        # an override is planned the same way with or without the overlap
        K.kivi_set_attention_splits(h, 0)
        K.kivi_set_attention_overlap(h, 1)
        assert K.kivi_attention_splits(h, 4097) == 1
        for n in (2, 7, 9, 1000):
            K.kivi_set_attention_splits(h, n)
            with_ov = K.kivi_attention_splits(h, 4097)
            K.kivi_set_attention_overlap(h, 0)
            assert K.kivi_attention_splits(h, 4097) == with_ov == min(n, 9), n
            K.kivi_set_attention_overlap(h, 1)
    finally:
        K.kivi_cache_destroy(h)
    # long context, R = 128: 8 units -> 76 splits per unit in one wave; the
    # 128 tail tokens take 2, leaving 74 for 4092 tiles -> 56 tiles per split
    # -> 74 tile splits: 608 CTAs, four per SM
    c = cfg(K, batch=1, n_kv_heads=8, n_q_heads=32, residual=128, max_tokens=131072)
    h = K.kivi_cache_init(c, _fake_buffers(K))
    assert K.kivi_attention_splits(h, 131072) == 76
    # overlapped: budget 25 -> 2 tail splits and 23 packed splits of 180 tiles
    K.kivi_set_attention_overlap(h, 1)
    assert K.kivi_attention_splits(h, 131072) == 25
    K.kivi_cache_destroy(h)
    # 320 units: one split per unit fits the wave, so the tail rides on the
    # packed split
    c = cfg(K, batch=80, n_kv_heads=4, n_q_heads=8, residual=128, max_tokens=512)
    h = K.kivi_cache_init(c, _fake_buffers(K))
    assert K.kivi_attention_splits(h, 450) == 1
    K.kivi_set_attention_overlap(h, 1)
    assert K.kivi_attention_splits(h, 450) == 1
    K.kivi_set_attention_overlap(h, 0)
    # an explicit count keeps separate tail splits: the 130 tail tokens take 3,
    # plus at least one packed split
    K.kivi_set_attention_splits(h, 3)
    assert K.kivi_attention_splits(h, 450) == 4
    K.kivi_cache_destroy(h)
    # batch 64, 28 / 4 heads (GQA 7, one chunk of 8 heads): 256 units -> a
    # budget of 2, one tail split beside one packed split; overlapped, the
    # budget of 1 fuses the tail into the packed split
    c = cfg(K, batch=64, n_kv_heads=4, n_q_heads=28, max_tokens=2560)
    h = K.kivi_cache_init(c, _fake_buffers(K))
    assert K.kivi_attention_splits(h, 2560) == 2
    K.kivi_set_attention_overlap(h, 1)
    assert K.kivi_attention_splits(h, 2560) == 1
    K.kivi_cache_destroy(h)
    # GQA 18 -> three chunks of at most eight query heads
    c = cfg(K, batch=1, n_kv_heads=1, n_q_heads=18, max_tokens=1024)
    h = K.kivi_cache_init(c, _fake_buffers(K))
    assert K.kivi_attention_splits(h, 1024) == 5
    K.kivi_cache_destroy(h)


def test_varlen_host_checks(K):
    """Per-sequence lengths: argument checks and bookkeeping, all on the host
    (every call here returns before any launch)."""
    import ctypes as C
    h = K.kivi_cache_init(cfg(K, batch=3), _fake_buffers(K))
    lib = K.lib()
    L = C.c_int * 3
    try:
        assert lib.kivi_quantize_prefill_varlen(h, 16, 16, 1, 100, L(5, 4097, 3), None) == K.KIVI_ECAPACITY
        assert lib.kivi_quantize_prefill_varlen(h, 16, 16, 1, 100, L(5, 101, 3), None) == K.KIVI_ESHAPE
        assert lib.kivi_quantize_prefill_varlen(h, 16, 16, 1, 100, L(-1, 1, 3), None) == K.KIVI_ECAPACITY
        assert lib.kivi_quantize_prefill_varlen(h, 16, 16, 1, 100, None, None) == K.KIVI_EINVAL
        assert lib.kivi_quantize_prefill_varlen(h, 16, 16, 1, 0, L(0, 0, 0), None) == K.KIVI_OK
        K.kivi_cache_set_lengths(h, [5, 0, 4096])
        assert K.kivi_cache_lengths(h, 3) == [5, 0, 4096] and K.kivi_cache_length(h) == -2
        # the longest sequence is full
        assert lib.kivi_append_decode(h, 16, 16, 1, None) == K.KIVI_ECAPACITY
        assert lib.kivi_append_tokens(h, 16, 16, 1, 1, None) == K.KIVI_ECAPACITY
        # an empty sequence: attention is refused
        need = K.kivi_attention_workspace_bytes(h)
        assert lib.kivi_decode_attention(h, 16, 1, 16, 0.0, 1 << 20, need, None) == K.KIVI_ESTATE
        with pytest.raises(K.KiviError) as e:
            K.kivi_cache_set_lengths(h, [1, 4097, 0])
        assert e.value.status == K.KIVI_ECAPACITY
        assert K.kivi_cache_lengths(h, 3) == [5, 0, 4096]  # unchanged by the refused call
        K.kivi_cache_set_lengths(h, [7, 7, 7])
        assert K.kivi_cache_length(h) == 7
        # prefill needs an empty cache
        assert lib.kivi_quantize_prefill_varlen(h, 16, 16, 1, 100, L(1, 2, 3), None) == K.KIVI_ESTATE
        K.kivi_cache_reset(h)
        assert K.kivi_cache_lengths(h, 3) == [0, 0, 0] and K.kivi_cache_length(h) == 0
    finally:
        K.kivi_cache_destroy(h)


def test_varlen_batch_limit(K):
    """Unequal lengths are limited to KIVI_MAX_VARLEN_BATCH sequences; equal
    lengths are not."""
    h = K.kivi_cache_init(cfg(K, batch=1025, n_kv_heads=1, n_q_heads=1), _fake_buffers(K))
    try:
        with pytest.raises(K.KiviError) as e:
            K.kivi_cache_set_lengths(h, [1] * 1024 + [2])
        assert e.value.status == K.KIVI_ESHAPE
        K.kivi_cache_set_lengths(h, [3] * 1025)
        assert K.kivi_cache_length(h) == 3
    finally:
        K.kivi_cache_destroy(h)


def test_bounded_wait_probe_refusals(K):
    """The wait probe checks its status pointer before anything else: null
    and misaligned pointers are refused without a launch (no GPU needed)."""
    lib = K.lib()
    assert lib.kivi_check_bounded_wait(None, None) == K.KIVI_EINVAL
    assert lib.kivi_check_bounded_wait(0x10002, None) == K.KIVI_EINVAL


@pytest.mark.parametrize("batch,n_kv,n_q,R,bits,cap", [
    (1, 1, 4, 32, 2, 4096), (8, 8, 32, 32, 2, 4224), (1, 8, 32, 128, 2, 8192),
    (64, 4, 28, 32, 2, 2592), (200, 8, 32, 64, 4, 1024), (3, 2, 8, 32, 8, 2048),
    (2, 2, 16, 32, 3, 2048), (16, 4, 28, 32, 4, 1024), (8, 1, 18, 32, 2, 1024)])
def test_split_plan_invariants(K, batch, n_kv, n_q, R, bits, cap):
    """At every length up to the capacity: at least one split and at most
    256; no more than one wave of the grid (attn_ctas_per_sm CTAs on each of
    152 SMs over the (batch, kv-head, head chunk) units), except for lengths
    held entirely in the tail, which take their tail splits; and a workspace
    that holds every split's partial."""
    c = cfg(K, batch=batch, n_kv_heads=n_kv, n_q_heads=n_q, residual=R, bits=bits, max_tokens=cap)
    h = K.kivi_cache_init(c, _fake_buffers(K))
    try:
        grp = n_q // n_kv
        units = batch * n_kv * -(-grp // 8)  # chunks of up to 8 query heads
        two_blocks = min(grp, 8) > 4         # two key blocks of 4 heads
        per_sm = 2 if bits == 8 else (3 if bits == 4 and two_blocks else 4)
        budget = max(min(per_sm * 152 // units, 256), 1)
        max_tail = -(-(R + 31) // 64)
        most = 0
        for l in range(1, cap + 1):
            s = K.kivi_attention_splits(h, l)
            assert 1 <= s <= 256, l
            assert s <= max(budget, max_tail), (l, s, budget)
            most = max(most, s)
        assert K.kivi_attention_workspace_bytes(h) >= units * most * 8 * (128 + 2) * 4
    finally:
        K.kivi_cache_destroy(h)


def test_attention_overlap_setting(K):
    """kivi_set_attention_overlap takes 0 or 1 on a live handle (host only)."""
    c = cfg(K, batch=1, n_kv_heads=1, n_q_heads=4, max_tokens=64)
    h = K.kivi_cache_init(c, _fake_buffers(K))
    try:
        K.kivi_set_attention_overlap(h, 1)
        K.kivi_set_attention_overlap(h, 0)
        for bad in (2, -1):
            with pytest.raises(K.KiviError) as e:
                K.kivi_set_attention_overlap(h, bad)
            assert e.value.status == K.KIVI_EINVAL
    finally:
        K.kivi_cache_destroy(h)
    assert K.lib().kivi_set_attention_overlap(None, 1) == K.KIVI_EINVAL
