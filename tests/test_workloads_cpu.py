"""The shared input generator: shapes, determinism and the configured workloads."""

import numpy as np
import torch

from nvfp4_kv_block_gb300 import workloads


def test_configs_match_their_descriptions():
    c = [workloads.config(i) for i in range(5)]
    assert c[0].seq_lens == (4096,) and c[0].n_q == (1,) and c[0].max_pages == 32
    assert c[1].n_seqs == 32 and set(c[1].seq_lens) == {32768} and c[1].n_q_total == 32
    assert c[2].n_seqs == 16 and set(c[2].n_q) == {8} and set(c[2].seq_lens) == {131072}
    assert c[3].n_seqs == 4 and set(c[3].seq_lens) == {524288} and c[3].outliers
    assert c[3].index_bytes() == 4 * 4095 * 128 * 128  # 64 MiB of index per sequence (minus the recent page)
    assert c[4].n_seqs == 64 and c[4].permuted
    assert all(30720 <= L <= 215040 for L in c[4].seq_lens)
    assert all(1 <= n <= 8 for n in c[4].n_q)


def test_block_table_is_a_bijection_onto_the_pool():
    wl = workloads.config(4)
    bt = wl.block_table()
    used = np.concatenate([bt[b, :n] for b, n in enumerate(wl.pages_per_seq)])
    assert np.array_equal(np.sort(used), np.arange(wl.total_pages))
    assert (bt[bt >= 0] < wl.total_pages).all()


def test_generation_is_deterministic_and_chunked():
    wl = workloads.custom("t", [20000, 300], [2, 1], seed=3, outliers=True)
    a = wl.tokens(0, 0, 8000, 8400, "cpu")
    b = wl.tokens(0, 0, 8000, 8400, "cpu")
    assert torch.equal(a, b) and a.shape == (400, 4, 128)
    whole = wl.kv_chunk(0, 0, 0, "cpu")
    assert torch.equal(whole[8000 - 0: 8192], wl.tokens(0, 0, 8000, 8192, "cpu"))
    q, qi, w = wl.queries("cpu")
    assert q.shape == (3, 16, 128) and q.dtype == torch.uint8
    assert qi.shape == (3, 8, 128) and w.shape == (3, 8) and (w >= 0).all()
    s = wl.channel_scales(0, "cpu")
    assert (s >= 19).sum() >= 1  # outlier channels x20
    assert wl.query_positions() == [(0, 19998), (0, 19999), (1, 299)]
