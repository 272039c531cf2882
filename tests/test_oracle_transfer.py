"""Pins for the oracle's block-outer transfer rows (CPU only)."""

import numpy as np

from oracle import layout


def _pools(n_layers, n_pages):
    # every byte names its own place: layer, page and offset (closed form)
    kv, idx = [], []
    for layer in range(n_layers):
        o = np.arange(layout.KV_PAGE_BYTES)
        kv.append(np.stack([((o * 7 + page * 31 + layer * 101) % 251).astype(np.uint8)
                            for page in range(n_pages)]))
        o = np.arange(layout.IDX_PAGE_BYTES)
        idx.append(np.stack([((o * 13 + page * 17 + layer * 59 + 3) % 241).astype(np.uint8)
                             for page in range(n_pages)]))
    return kv, idx


def test_row_bytes_follow_the_formula():
    kv, idx = _pools(3, 5)
    pages = [4, 0, 2]
    rows = layout.pack_rows(kv, idx, pages)
    assert rows.shape == (3, 3 * 90_112)
    assert layout.ROW_LAYER_BYTES == 73_728 + 16_384
    for i, page in enumerate(pages):
        for layer in range(3):
            at = layer * 90_112
            for o in (0, 1, 9_215, 73_727):
                assert rows[i, at + o] == (o * 7 + page * 31 + layer * 101) % 251
            for o in (0, 5, 16_383):
                assert rows[i, at + 73_728 + o] == (o * 13 + page * 17 + layer * 59 + 3) % 241


def test_unpack_inverts_pack_into_other_pages():
    kv, idx = _pools(2, 6)
    rows = layout.pack_rows(kv, idx, [5, 1, 3])
    kv2 = [np.zeros_like(x) for x in kv]
    idx2 = [np.zeros_like(x) for x in idx]
    layout.unpack_rows(rows, kv2, idx2, [0, 2, 4])
    for layer in range(2):
        for src, dst in ((5, 0), (1, 2), (3, 4)):
            assert np.array_equal(kv2[layer][dst], kv[layer][src])
            assert np.array_equal(idx2[layer][dst], idx[layer][src])
        for untouched in (1, 3, 5):
            assert not kv2[layer][untouched].any() and not idx2[layer][untouched].any()
    # and packing the unpacked pages gives the same rows back
    assert np.array_equal(layout.pack_rows(kv2, idx2, [0, 2, 4]), rows)
