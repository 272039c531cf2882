"""The allocation-free indexer entry point against the regular one.

msa_indexer_topk_noalloc serves callers that cannot allocate device memory
(a host framework owning every allocation, a decode loop where a cudaMalloc
and its possible device synchronisation are not allowed between steps, a
plug-in that only receives its input and output buffers).  It keeps its
scratch in a static array inside the library instead of a caller workspace,
so its selections must equal those of msa_indexer_topk, call after call.

This file is named to be collected last: if it fails, a run that stops at the
first failure has already run every other test.
"""

import numpy as np
import pytest
import torch

from nvfp4_kv_block_gb300 import harness, ops, workloads

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _workloads():
    return [
        workloads.config(0),
        workloads.custom("noalloc_mixed", [1, 127, 0, 128, 129, 2053, 4096, 130, 5000],
                         [1, 1, 0, 2, 8, 8, 3, 8, 5], seed=91, permuted=True),
    ]


@pytest.mark.parametrize("wl", _workloads(), ids=lambda w: w.name)
def test_noalloc_matches_regular_entry_point_twice(wl):
    st = harness.build_state(wl, DEV)
    q, qi, w = wl.queries(DEV)
    ref_sel, ref_n, _ = ops.indexer_topk(st.cache, qi, w, st.block_table, st.seq_lens, st.q_start_loc)
    torch.cuda.synchronize()
    ref_sel, ref_n = ref_sel.cpu().numpy(), ref_n.cpu().numpy()
    for _ in range(2):  # the static scratch keeps the previous call's contents
        sel, n_sel = ops.indexer_topk_noalloc(st.cache, qi, w, st.block_table, st.seq_lens,
                                              st.q_start_loc)
        torch.cuda.synchronize()
        assert np.array_equal(n_sel.cpu().numpy(), ref_n)
        assert np.array_equal(sel.cpu().numpy(), ref_sel)
    assert st.cache.read_status() == 0
