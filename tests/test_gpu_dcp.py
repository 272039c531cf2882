"""GPU parity of the context-split indexer (blog, "Parallelize index work across
context": each part of the context yields local top-16 candidates, the parts
exchange them, and the merge selects exactly as one scan over everything).

One process runs four range scans and the merge; two spawned processes on the
same GPU each scan two of the four parts and exchange their candidates over
gloo (CPU) before merging.  Merged selections must equal msa_indexer_topk's
bit for bit; each part's candidates must equal the oracle's local top-16 up to
the allowed swaps, with scores within 1e-4.
"""

import os
import socket
import sys

import numpy as np
import pytest
import torch
import torch.multiprocessing as mp

import oracle
from nvfp4_kv_block_gb300 import harness, ops, workloads

from _dcp import decode_keys, shard_bounds
from _parity import OracleSide

pytestmark = pytest.mark.gpu

DEV = "cuda"
ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _workload():
    # short contexts (every block selected), speculative tokens straddling a
    # block boundary, an empty sequence, longer ragged contexts; pages permuted
    return workloads.custom("dcp_mixed", [129, 0, 2053, 9000, 40000, 131, 70001], [1, 0, 8, 3, 5, 2, 4],
                            seed=31, permuted=True)


def _range_keys(st, wl, bounds):
    _, qi, w = wl.queries(DEV)
    out = []
    for lo, hi in bounds:
        cand, _ = ops.indexer_topk_range(st.cache, qi, w, st.block_table, st.seq_lens, st.q_start_loc, lo, hi)
        out.append(cand)
    return torch.stack(out)


def test_four_parts_merge_to_the_single_call_selection_and_match_the_oracle():
    wl = _workload()
    st = harness.build_state(wl, DEV)
    _, qi, w = wl.queries(DEV)
    ref_sel, ref_n, _ = ops.indexer_topk(st.cache, qi, w, st.block_table, st.seq_lens, st.q_start_loc)
    bounds = shard_bounds(wl.max_pages, 4)
    keys = _range_keys(st, wl, bounds)
    sel, n_sel = ops.indexer_merge_candidates(st.cache, keys, st.seq_lens, st.q_start_loc, wl.max_pages)
    torch.cuda.synchronize()
    assert np.array_equal(sel.cpu().numpy(), ref_sel.cpu().numpy())
    assert np.array_equal(n_sel.cpu().numpy(), ref_n.cpu().numpy())
    # every part's candidates against the oracle's local top-16
    side = OracleSide(wl, DEV)
    scores, blocks = decode_keys(keys.cpu().numpy())
    for j in range(wl.n_q_total):
        b, pos, osel, oscores = side.token(j)
        r = pos // 128
        if r == 0:
            assert (blocks[:, j] == -1).all()
            continue
        for si, (lo, hi) in enumerate(bounds):
            want = oracle.indexer.range_candidates(oscores, r, lo, hi)
            got = [(float(sc), int(bl)) for sc, bl in zip(scores[si, j], blocks[si, j]) if bl >= 0]
            assert len(got) == len(want), (j, si)
            gb, wb = {bl for _, bl in got}, {bl for _, bl in want}
            if gb != wb:  # allowed only between blocks within 1e-4 of the part's cut-off
                cut = want[-1][0]
                assert all(abs(oscores[x] - cut) <= 1e-4 * abs(cut) for x in gb ^ wb), (j, si, gb ^ wb)
            for sc, bl in got:
                assert abs(sc - oscores[bl]) <= 1e-4 * max(1e-30, abs(oscores).max()), (j, bl)
            # keys are written best first
            assert [(-sc, bl) for sc, bl in got] == sorted((-sc, bl) for sc, bl in got)
    assert st.cache.read_status() == 0


def _free_port():
    with socket.socket(socket.AF_INET, socket.SOCK_STREAM) as s:
        s.bind(("127.0.0.1", 0))
        return s.getsockname()[1]


def _rank(rank, world, port, q):
    sys.path.insert(0, ROOT)
    sys.path.insert(0, os.path.join(ROOT, "tests"))
    os.environ.update(MASTER_ADDR="127.0.0.1", MASTER_PORT=str(port))
    torch.distributed.init_process_group("gloo", rank=rank, world_size=world)
    try:
        torch.cuda.set_device(0)
        wl = _workload()
        st = harness.build_state(wl, DEV)
        bounds = shard_bounds(wl.max_pages, 4)
        mine = [bnd for i, bnd in enumerate(bounds) if i % world == rank]
        keys = _range_keys(st, wl, mine).cpu()                       # this rank's parts
        gathered = [torch.empty_like(keys) for _ in range(world)]
        torch.distributed.all_gather(gathered, keys)                 # the exchange (CPU, gloo)
        allk = torch.cat(gathered).to(DEV)
        sel, n_sel = ops.indexer_merge_candidates(st.cache, allk, st.seq_lens, st.q_start_loc, wl.max_pages)
        _, qi, w = wl.queries(DEV)
        ref_sel, ref_n, _ = ops.indexer_topk(st.cache, qi, w, st.block_table, st.seq_lens, st.q_start_loc)
        torch.cuda.synchronize()
        ok = bool(torch.equal(sel, ref_sel) and torch.equal(n_sel, ref_n)) and st.cache.read_status() == 0
        q.put((rank, ok))
    finally:
        torch.distributed.destroy_process_group()


def test_two_ranks_exchange_candidates_over_gloo():
    ctx = mp.get_context("spawn")
    q = ctx.Queue()
    port = _free_port()
    procs = [ctx.Process(target=_rank, args=(r, 2, port, q)) for r in range(2)]
    for p in procs:
        p.start()
    results = sorted(q.get(timeout=600) for _ in procs)
    for p in procs:
        p.join(timeout=120)
        assert p.exitcode == 0
    assert results == [(0, True), (1, True)]
