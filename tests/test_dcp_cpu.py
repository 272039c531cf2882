"""The context-split indexer's exchange on CPU: two gloo ranks each take half of
the context's blocks, compute the oracle's local candidates, exchange them and
merge; the merge equals the oracle's single selection (blog, "Parallelize index
work across context")."""

import os
import socket
import sys

import numpy as np
import torch
import torch.multiprocessing as mp

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _worker(rank, world, port, q):
    sys.path.insert(0, ROOT)
    from oracle import formats, indexer
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        rng = np.random.default_rng(5)  # same inputs on both ranks
        L, n_q = 128 * 45 + 17, 3
        keys = formats.encode_e4m3(rng.standard_normal((L, 128)))
        qi = formats.encode_e4m3(rng.standard_normal((n_q, 8, 128)))
        w = rng.uniform(0, 1, (n_q, 8)).astype(np.float32)
        ok = True
        for j in range(n_q):
            r = (L - n_q + j) // 128
            s = indexer.block_scores(qi[j], w[j], keys, r)
            half = (r + 1) // 2
            lo, hi = (0, half) if rank == 0 else (half, 1 << 30)
            mine = indexer.range_candidates(s, r, lo, hi)
            parts = [None] * world
            torch.distributed.all_gather_object(parts, mine)
            ok = ok and indexer.merge_candidates(parts, r) == indexer.select(s, r)
        q.put((rank, ok))
    finally:
        torch.distributed.destroy_process_group()


def test_two_gloo_ranks_merge_to_the_global_selection():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_worker, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=120) for _ in procs)
    for p in procs:
        p.join(timeout=60)
        assert p.exitcode == 0
    assert results == [(0, True), (1, True)]
