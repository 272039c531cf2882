"""Failure detection without a GPU fault: a bounded wait that runs out.

Test hooks of the library (a few-millisecond wait limit): the indexer's grid
barrier waits for one CTA more than the launch has; the attention kernel's
producer leaves out its first copy.  The indexer's CTAs all run out of
time at the barrier; the call reports MSA_STATUS_TIMEOUT without touching its
outputs, and the barrier word is back at rest, so the next normal call on the
same workspace, and on the allocation-free entry point's static scratch,
selects exactly as before.  The attention's CTAs run out of time waiting for
the missing page, report MSA_STATUS_TIMEOUT and return; the next call is exact.
Nothing here faults, traps or hangs: each wait ends after its limit.
"""

import numpy as np
import pytest
import torch

from nvfp4_kv_block_gb300 import harness, ops, workloads

pytestmark = pytest.mark.gpu

DEV = "cuda"
LIMIT_NS = 5_000_000  # 5 ms


def test_barrier_timeout_is_reported_and_the_next_calls_recover():
    wl = workloads.custom("timeout_mixed", [4096, 300, 9000], [1, 2, 3], seed=7, permuted=True)
    st = harness.build_state(wl, DEV)
    _, qi, w = wl.queries(DEV)
    T = wl.n_q_total
    args = (st.cache, qi, w, st.block_table, st.seq_lens, st.q_start_loc)
    ref_sel, ref_n, ws = ops.indexer_topk(*args)
    torch.cuda.synchronize()
    ref_sel, ref_n = ref_sel.cpu().numpy(), ref_n.cpu().numpy()
    assert st.cache.read_status() == 0
    sel = torch.full((T, 17), -7, dtype=torch.int32, device=DEV)
    n_sel = torch.full((T,), -7, dtype=torch.int32, device=DEV)
    try:
        ops.set_fault_injection(ops.INJECT_BARRIER_TIMEOUT, LIMIT_NS)
        ops.indexer_topk(*args, ws=ws, sel=sel, n_sel=n_sel)
        torch.cuda.synchronize()
        assert st.cache.read_status() == ops.STATUS_TIMEOUT
        # the selection phase was abandoned: outputs untouched
        assert (sel == -7).all() and (n_sel == -7).all()
        # every CTA withdrew its arrival: the barrier word's count is zero
        word = int(ws[:8].view(torch.int64).item())
        assert word & 0xFFFFFFFF == 0
        # the same through the allocation-free entry point (its static scratch)
        st.cache.status.zero_()
        ops.indexer_topk_noalloc(*args, sel=sel, n_sel=n_sel)
        torch.cuda.synchronize()
        assert st.cache.read_status() == ops.STATUS_TIMEOUT
        assert (sel == -7).all()
    finally:
        ops.set_fault_injection(0, 0)
    st.cache.status.zero_()
    # normal calls on the same workspace and on the static scratch, twice each
    for _ in range(2):
        s1, n1, _ = ops.indexer_topk(*args, ws=ws)
        s2, n2 = ops.indexer_topk_noalloc(*args)
        torch.cuda.synchronize()
        assert np.array_equal(s1.cpu().numpy(), ref_sel) and np.array_equal(n1.cpu().numpy(), ref_n)
        assert np.array_equal(s2.cpu().numpy(), ref_sel) and np.array_equal(n2.cpu().numpy(), ref_n)
    assert st.cache.read_status() == 0
    word = int(ws[:8].view(torch.int64).item())
    assert word & 0xFFFFFFFF == 0 and (word >> 32) >= 3  # three completed barriers


def test_attention_timeout_is_reported_and_the_next_call_recovers():
    # every attention CTA leaves out the copy of its first page: the waits for
    # it run out, every role of the CTA gives up, the CTA waits (bounded) for
    # its copies and tensor-core products in flight, frees tensor memory and
    # returns; the next call on the same cache is exact again
    wl = workloads.custom("attn_timeout", [4096, 2000, 9000], [1, 2, 3], seed=9, permuted=True)
    st = harness.build_state(wl, DEV)
    q, qi, w = wl.queries(DEV)
    sel, n_sel, _ = ops.indexer_topk(st.cache, qi, w, st.block_table, st.seq_lens, st.q_start_loc)
    args = (st.cache, q, sel, n_sel, st.block_table, st.seq_lens, st.q_start_loc, 1)
    ref_o, ref_l = ops.sparse_attn_decode(*args)
    torch.cuda.synchronize()
    ref_o, ref_l = ref_o.clone(), ref_l.clone()
    assert st.cache.read_status() == 0
    try:
        ops.set_fault_injection(ops.INJECT_ATTENTION_TIMEOUT, LIMIT_NS)
        ops.sparse_attn_decode(*args)
        torch.cuda.synchronize()
        assert st.cache.read_status() == ops.STATUS_TIMEOUT
    finally:
        ops.set_fault_injection(0, 0)
    st.cache.status.zero_()
    for _ in range(2):
        o, l = ops.sparse_attn_decode(*args)
        torch.cuda.synchronize()
        assert torch.equal(o, ref_o) and torch.equal(l, ref_l)
    assert st.cache.read_status() == 0
