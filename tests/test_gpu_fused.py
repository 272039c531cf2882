"""GPU parity of the single-launch decode (msa_decode_fused) against the oracle,
through the C ABI, on low-concurrency batches: selections exact up to the
allowed swaps, outputs within 2e-3 * max|V^| over the GPU's own selection, and
the same selection as the four-launch path bit for bit."""

import numpy as np
import pytest
import torch

from nvfp4_kv_block_gb300 import harness, ops, workloads

from _parity import OracleSide, block_scores_from_workspace
from test_gpu_parity import _check_tokens, _small_workload

pytestmark = pytest.mark.gpu

DEV = "cuda"


def _fused(wl, st, repeats=2):
    q, qi, w = wl.queries(DEV)
    bufs = ops.FusedBuffers(wl.n_q_total, wl.max_pages, DEV)
    for _ in range(repeats):  # the workspace's barrier words are reused
        out = ops.decode_fused(st.cache, q, qi, w, st.block_table, st.seq_lens, st.q_start_loc, bufs)
    torch.cuda.synchronize()
    S = block_scores_from_workspace(bufs.ws, wl.n_q_total, wl.max_pages)
    return bufs, out.cpu().numpy(), S


def _four_launch(wl, st):
    q, qi, w = wl.queries(DEV)
    bufs = ops.DecodeBuffers(wl.n_q_total, wl.max_pages, ops.choose_splits(wl.n_q_total), DEV)
    out = ops.decode_step(st.cache, q, qi, w, st.block_table, st.seq_lens, st.q_start_loc, bufs)
    torch.cuda.synchronize()
    return bufs, out.cpu().numpy()


@pytest.mark.parametrize("which", ["tiny", "small_mixed", "long_single"])
def test_fused_decode_matches_oracle_and_the_four_launch_path(which):
    if which == "tiny":
        wl = workloads.config(0)
    elif which == "small_mixed":
        wl = _small_workload()
    else:
        wl = workloads.custom("fused_long", [200_003], [3], seed=13, permuted=True)
    st = harness.build_state(wl, DEV)
    side = OracleSide(wl, DEV)
    bufs, out, S = _fused(wl, st)
    _check_tokens(wl, side, bufs, out, S, range(wl.n_q_total))
    ref, ref_out = _four_launch(wl, st)
    assert np.array_equal(bufs.sel.cpu().numpy(), ref.sel.cpu().numpy())
    assert np.array_equal(bufs.n_sel.cpu().numpy(), ref.n_sel.cpu().numpy())
    assert np.max(np.abs(out - ref_out)) <= 1e-3 * np.max(np.abs(ref_out))
    assert st.cache.read_status() == 0


def test_fused_limits_are_checked_on_the_host():
    wl = workloads.custom("fused_many", [300] * 65, [1] * 65, seed=3)
    st = harness.build_state(wl, DEV)
    q, qi, w = wl.queries(DEV)
    bufs = ops.FusedBuffers(wl.n_q_total, wl.max_pages, DEV)
    with pytest.raises(ops.MsaError, match="unsupported shape"):
        ops.decode_fused(st.cache, q, qi, w, st.block_table, st.seq_lens, st.q_start_loc, bufs)
