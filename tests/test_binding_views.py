"""The binding's inspection views read the arrays inside the cache's own
buffers wherever those buffers start: a tile buffer that is a view into a
larger allocation (as when a caller hands the cache part of a pool) gives the
same views as a fresh buffer holding the same bytes.  CPU only: the C handle
is made over host buffers and no kernel runs."""
import pytest
import torch


@pytest.mark.parametrize("bits,n_out", [(2, 0), (3, 0), (4, 2), (8, 0)])
def test_views_of_an_offset_buffer(bits, n_out):
    from bit_kv_cache_kivi_gb300 import kivi as K
    kw = dict(batch=2, n_kv_heads=2, n_q_heads=4, max_tokens=128, bits=bits, outliers=n_out,
              device="cpu")
    fresh, offset = K.KiviCache(**kw), K.KiviCache(**kw)
    gen = torch.Generator().manual_seed(bits)
    for n in K.BUFFER_NAMES:
        src = torch.randint(0, 256, fresh.buffers[n].shape, dtype=torch.uint8, generator=gen)
        fresh.buffers[n].copy_(src)
        pool = torch.zeros(src.numel() + 8192, dtype=torch.uint8)
        offset.buffers[n] = pool[4096:4096 + src.numel()]
        offset.buffers[n].copy_(src)
    a, b = fresh.layout_views(), offset.layout_views()
    assert a.keys() == b.keys()
    for k in a:
        assert torch.equal(a[k], b[k]), k
    la, lb = fresh.logical_state(), offset.logical_state()
    for k in la:
        assert torch.equal(la[k], lb[k]), k


def test_tile_row_bits_to_plain_rows():
    """The binding's description of a tile's code rows is a bijection onto
    the row's bits at every width (plain at 2/4/8-bit keys), and plain_rows
    turns rows packed by that description into plain LSB-first rows."""
    import numpy as np
    from bit_kv_cache_kivi_gb300.kivi import plain_rows, tile_row_bit
    rng = np.random.default_rng(0)
    for bits in (2, 3, 4, 8):
        for value in (False, True):
            m = [tile_row_bit(e, j, bits, value) for e in range(128) for j in range(bits)]
            assert sorted(m) == list(range(128 * bits)), (bits, value)
            if bits != 3 and not value:
                assert m == list(range(128 * bits))
            codes = rng.integers(0, 1 << bits, (3, 128)).astype(np.uint8)
            tile = np.zeros((3, 16 * bits), np.uint8)
            for r in range(3):
                for e in range(128):
                    for j in range(bits):
                        kb = tile_row_bit(e, j, bits, value)
                        tile[r, kb // 8] |= ((codes[r, e] >> j) & 1) << (kb % 8)
            lsb = ((codes[:, :, None] >> np.arange(bits)) & 1).astype(np.uint8).reshape(3, -1)
            want = np.packbits(lsb, axis=1, bitorder="little")
            assert np.array_equal(plain_rows(torch.from_numpy(tile), bits, value).numpy(), want)
