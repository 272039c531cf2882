"""GPU parity of the block-outer transfer rows (pack and unpack) against the oracle.

Pools hold seeded random bytes (drawn with torch, not by the library), so
every byte of a row is checked against the oracle's own gather of those bytes.
"""

import numpy as np
import pytest
import torch

from oracle import layout
from nvfp4_kv_block_gb300 import ops

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _random_caches(n_layers, n_pages, seed):
    g = torch.Generator(device=DEV)
    g.manual_seed(seed)
    caches = []
    for _ in range(n_layers):
        c = ops.KVCache(n_pages, 1.0, 1.0, DEV)
        c.kv_pool.copy_(torch.randint(0, 256, c.kv_pool.shape, generator=g, device=DEV, dtype=torch.int32))
        c.idx_pool.copy_(torch.randint(0, 256, c.idx_pool.shape, generator=g, device=DEV, dtype=torch.int32))
        caches.append(c)
    return caches


@pytest.mark.parametrize("n_layers", [1, 3, 20])
def test_pack_and_unpack_match_oracle(n_layers):
    n_pages = 48
    caches = _random_caches(n_layers, n_pages, seed=100 + n_layers)
    rng = np.random.default_rng(n_layers)
    pages = rng.permutation(n_pages)[:17].astype(np.int32)
    rows = ops.pack_blocks(caches, torch.from_numpy(pages).to(DEV))
    torch.cuda.synchronize()
    assert rows.shape == (17, n_layers * 90_112) and ops.block_row_bytes(n_layers) == n_layers * 90_112
    kv = [c.kv_pool.cpu().numpy() for c in caches]
    idx = [c.idx_pool.cpu().numpy() for c in caches]
    want = layout.pack_rows(kv, idx, pages)
    assert np.array_equal(rows.cpu().numpy(), want)
    # unpack into fresh pools at other page ids
    dest = [ops.KVCache(n_pages, 1.0, 1.0, DEV) for _ in range(n_layers)]
    dpages = rng.permutation(n_pages)[:17].astype(np.int32)
    ops.unpack_blocks(dest, rows, torch.from_numpy(dpages).to(DEV))
    torch.cuda.synchronize()
    kv2 = [np.zeros_like(x) for x in kv]
    idx2 = [np.zeros_like(x) for x in idx]
    layout.unpack_rows(want, kv2, idx2, dpages)
    for layer in range(n_layers):
        assert np.array_equal(dest[layer].kv_pool.cpu().numpy(), kv2[layer])
        assert np.array_equal(dest[layer].idx_pool.cpu().numpy(), idx2[layer])
    assert all(c.read_status() == 0 for c in caches + dest)


def test_page_outside_a_pool_is_flagged_and_skipped():
    caches = _random_caches(2, 8, seed=7)
    pages = torch.tensor([3, 8, -1, 0], dtype=torch.int32, device=DEV)
    rows = torch.zeros((4, 2 * 90_112), dtype=torch.uint8, device=DEV)
    ops.pack_blocks(caches, pages, rows)
    torch.cuda.synchronize()
    assert caches[0].read_status() == ops.STATUS_BAD_PAGE
    r = rows.cpu().numpy()
    assert not r[1].any() and not r[2].any()  # untouched
    kv = [c.kv_pool.cpu().numpy() for c in caches]
    idx = [c.idx_pool.cpu().numpy() for c in caches]
    assert np.array_equal(r[[0, 3]], layout.pack_rows(kv, idx, [3, 0]))
