"""GPU parity: every kernel of libmsa.so against the CPU oracle, through the C ABI.

Rules (the decode path's acceptance rules):
  * quantised bytes and scales bit-exact;
  * selected block sets exact, except swaps whose oracle block scores differ
    from the selection cut-off by < 1e-4 relative;
  * attention output max-abs error <= 2e-3 * max|V^| (fp32 accumulation), with
    max|V^| the largest dequantised |V| among the pages the oracle attends.
"""

import numpy as np
import pytest
import torch

import oracle
from oracle import formats, layout, nvfp4
from nvfp4_kv_block_gb300 import harness, ops, workloads

from _parity import OracleSide, block_scores_from_workspace, selection_ok, softmax_scale

pytestmark = pytest.mark.gpu

DEV = "cuda"
ATOL_REL = 2e-3


def _small_workload():
    # short (r <= 16), exact page multiples, a boundary-straddling speculative
    # batch, an empty sequence, a longer one with top-16 active; pages permuted
    return workloads.custom("small_mixed", [1, 127, 0, 128, 129, 2053, 4096, 130, 5000],
                            [1, 1, 0, 2, 8, 8, 3, 8, 5], seed=77, permuted=True)


@pytest.fixture(scope="module")
def small():
    wl = _small_workload()
    st = harness.build_state(wl, DEV)
    return wl, st, OracleSide(wl, DEV)


@pytest.fixture(scope="module")
def tiny():
    wl = workloads.config(0)
    st = harness.build_state(wl, DEV)
    return wl, st, OracleSide(wl, DEV)


def _decode(wl, st, n_splits=None):
    q, qi, w = wl.queries(DEV)
    T = wl.n_q_total
    n_splits = n_splits or ops.choose_splits(T)
    bufs = ops.DecodeBuffers(T, wl.max_pages, n_splits, DEV)
    out = ops.decode_step(st.cache, q, qi, w, st.block_table, st.seq_lens, st.q_start_loc, bufs)
    torch.cuda.synchronize()
    S = block_scores_from_workspace(bufs.ws, T, wl.max_pages)
    return bufs, out.cpu().numpy(), S


def _check_tokens(wl, side, bufs, out, S, tokens):
    """Per token: block scores (1e-4 relative), the selection (exact up to
    allowed swaps), and the attention output over the selection the GPU made
    (2e-3 * max|V^|): when a swap was allowed, the oracle attends over the
    GPU's blocks, so every checked token's output is compared."""
    sel = bufs.sel.cpu().numpy()
    n_sel = bufs.n_sel.cpu().numpy()
    worst = 0.0
    for j in tokens:
        b, pos, osel, oscores = side.token(j)
        r = pos // 128
        gsel = [int(x) for x in sel[j, : n_sel[j]]]
        # block scores: fp32 sums of exact FP8 products vs exact float64
        if r > 0:
            ref = np.asarray(oscores)
            err = np.max(np.abs(S[j, :r] - ref)) / max(1e-30, np.max(np.abs(ref)))
            assert err < 1e-4, (j, err)
        ok, diff = selection_ok(gsel, osel, oscores)
        assert ok, (j, gsel, osel, diff)
        assert sorted(gsel) == gsel and gsel[-1] == r and len(gsel) == min(16, r) + 1
        assert all(v == -1 for v in sel[j, n_sel[j]:])
        ref_out, _, vmax = side.attend(j, gsel, softmax_scale())
        e = np.max(np.abs(out[j] - ref_out))
        worst = max(worst, e / vmax)
        assert e <= ATOL_REL * vmax, (j, e, vmax, gsel != osel)
    return worst


def test_encode_scale_and_absmax_match_oracle():
    g = torch.Generator(device=DEV).manual_seed(5)
    x = torch.randn(1_000_003, generator=g, device=DEV) * 3.7
    amax = torch.zeros(1, dtype=torch.float32, device=DEV)
    ops.absmax_(x[:500_000], amax)
    ops.absmax_(x[500_000:], amax)
    ref = float(x.abs().max())
    assert float(amax) == ref
    for a in [ref, 1.0, 448.0, 1e-3, 123.456]:
        assert ops.encode_scale(a) == float(nvfp4.tensor_encode_scale(np.float32(a)))


def test_insert_is_bit_exact(small):
    wl, st, side = small
    kv = st.cache.kv_pool.cpu().numpy()
    ip = st.cache.idx_pool.cpu().numpy()
    bt = wl.block_table()
    assert side.s_enc_k == np.float32(st.cache.s_enc_k) and side.s_enc_v == np.float32(st.cache.s_enc_v)
    for b in range(wl.n_seqs):
        for blk in range(wl.pages_per_seq[b]):
            want_kv, want_idx = side.page_bytes(b, blk)
            phys = bt[b, blk]
            assert np.array_equal(kv[phys], want_kv), (b, blk)
            assert np.array_equal(ip[phys], want_idx), (b, blk)
    assert st.cache.read_status() == 0


def test_fp8_dequant_matches_oracle_for_every_scale_byte():
    rng = np.random.default_rng(11)
    pool = np.zeros((2, layout.KV_PAGE_BYTES), dtype=np.uint8)
    kc = rng.integers(0, 16, (128, 4, 128)).astype(np.uint8)
    vc = rng.integers(0, 16, (128, 4, 128)).astype(np.uint8)
    # every one of the 256 scale bytes appears in K and in V
    ks = rng.permutation(np.resize(np.arange(256), 128 * 4 * 8)).reshape(128, 4, 8).astype(np.uint8)
    vs = rng.permutation(np.resize(np.arange(256), 128 * 4 * 8)).reshape(128, 4, 8).astype(np.uint8)
    for t in range(128):
        layout.write_kv_slot(pool, 1, t, kc[t], ks[t], vc[t], vs[t])
    cache = ops.KVCache(2, 1.0, 1.0, DEV)
    cache.kv_pool.copy_(torch.from_numpy(pool))
    k8, v8 = ops.debug_fp8_page(cache, 1)
    k8 = k8.cpu().numpy().transpose(1, 0, 2)  # -> [token, head, ch]
    v8 = v8.cpu().numpy().transpose(1, 0, 2)
    assert np.array_equal(k8, nvfp4.fp8_operand(kc, ks))
    assert np.array_equal(v8, nvfp4.fp8_operand(vc, vs))


def test_fp8_dequant_of_inserted_pages(tiny):
    wl, st, side = tiny
    bt = wl.block_table()
    for blk in (0, 13, 31):
        k8, v8 = ops.debug_fp8_page(st.cache, int(bt[0, blk]))
        d = side.kv_tokens(0, blk * 128, blk * 128 + 128)
        assert np.array_equal(k8.cpu().numpy().transpose(1, 0, 2), d["k8"])
        assert np.array_equal(v8.cpu().numpy().transpose(1, 0, 2), d["v8"])


def test_tiny_decode_matches_oracle(tiny):
    wl, st, side = tiny
    bufs, out, S = _decode(wl, st)
    _check_tokens(wl, side, bufs, out, S, range(wl.n_q_total))
    assert st.cache.read_status() == 0


def test_small_mixed_decode_matches_oracle(small):
    wl, st, side = small
    bufs, out, S = _decode(wl, st)
    _check_tokens(wl, side, bufs, out, S, range(wl.n_q_total))
    assert st.cache.read_status() == 0


@pytest.mark.parametrize("n_splits", [1, 2, 5, 17, 64])
def test_attention_with_oracle_selection_any_split_count(small, n_splits):
    wl, st, side = small
    q, _, _ = wl.queries(DEV)
    T = wl.n_q_total
    sel = np.full((T, 17), -1, dtype=np.int32)
    n_sel = np.zeros(T, dtype=np.int32)
    refs = []
    for j in range(T):
        _, _, osel, _ = side.token(j)
        sel[j, : len(osel)] = osel
        n_sel[j] = len(osel)
        refs.append(side.attend(j, osel, softmax_scale()))
    o_part, lse_part = ops.sparse_attn_decode(st.cache, q, torch.from_numpy(sel).to(DEV),
                                              torch.from_numpy(n_sel).to(DEV), st.block_table,
                                              st.seq_lens, st.q_start_loc, n_splits)
    lse = torch.empty((T, 16), dtype=torch.float32, device=DEV)
    out = ops.merge_splits(o_part, lse_part, lse=lse).cpu().numpy()
    lse = lse.cpu().numpy()
    lse_part = lse_part.cpu().numpy()
    o_part = o_part.cpu().numpy()
    for j, (ref, ref_lse, vmax) in enumerate(refs):
        assert np.max(np.abs(out[j] - ref)) <= ATOL_REL * vmax
        # the merged log-sum-exp of the splits is the whole selection's
        assert np.allclose(lse[j], ref_lse, rtol=1e-5, atol=1e-4), j
        # and every split is the exact attention over its own share of the
        # selection (entries s, s + S, ...): output and log-sum-exp
        _, _, osel, _ = side.token(j)
        for sp in range(min(n_splits, 3)):
            share = osel[sp::n_splits]
            if not share:
                assert np.all(lse_part[j, sp] == -np.inf) and np.all(o_part[j, sp] == 0)
                continue
            s_ref, s_lse, s_vmax = side.attend(j, share, softmax_scale())
            assert np.max(np.abs(o_part[j, sp] - s_ref)) <= ATOL_REL * s_vmax, (j, sp)
            assert np.allclose(lse_part[j, sp], s_lse, rtol=1e-5, atol=1e-4), (j, sp)
    assert st.cache.read_status() == 0


def _sampled_tokens(wl, rng, at_least=32):
    """At least `at_least` query tokens: the first and the last token of a
    sequence for every query-token count present, then random ones."""
    qsl = wl.q_start_loc
    picked = set()
    seen_nq = set()
    for b in range(wl.n_seqs):
        if wl.n_q[b] > 0 and wl.n_q[b] not in seen_nq:
            seen_nq.add(wl.n_q[b])
            picked.update([qsl[b], qsl[b + 1] - 1])
    for b in (0, wl.n_seqs - 1):
        if wl.n_q[b] > 0:
            picked.update([qsl[b], qsl[b + 1] - 1])
    T = wl.n_q_total
    while len(picked) < min(at_least, T):
        picked.add(int(rng.integers(0, T)))
    return sorted(picked)


@pytest.mark.parametrize("cfg", [1, 2, 3, 4])
def test_full_size_config_sampled(cfg):
    wl = workloads.config(cfg)
    st = harness.build_state(wl, DEV)
    side = OracleSide(wl, DEV)
    bufs, out, S = _decode(wl, st)
    T = wl.n_q_total
    rng = np.random.default_rng(1000 + cfg)
    # every token where the oracle is quick (batched, long-context), else at
    # least 32 covering every query-token count and sequence ends
    tokens = range(T) if cfg in (1, 3) else _sampled_tokens(wl, rng)
    _check_tokens(wl, side, bufs, out, S, tokens)
    # every token (checked or not) got a finite, non-empty output
    assert np.isfinite(out).all()
    assert (np.abs(out).reshape(T, -1).max(axis=1) > 0).all()
    # sampled pages bit-exact, including the partial last page of a sequence
    kv = st.cache.kv_pool
    ip = st.cache.idx_pool
    bt = wl.block_table()
    for _ in range(3):
        b = int(rng.integers(0, wl.n_seqs))
        blk = int(rng.integers(0, wl.pages_per_seq[b]))
        for blk_ in (blk, wl.pages_per_seq[b] - 1):
            want_kv, want_idx = side.page_bytes(b, blk_)
            phys = int(bt[b, blk_])
            assert np.array_equal(kv[phys].cpu().numpy(), want_kv)
            assert np.array_equal(ip[phys].cpu().numpy(), want_idx)
    assert st.cache.read_status() == 0


@pytest.mark.parametrize("ctx", [5121 * 128 + 1, 2_200_000])
def test_topk_of_long_rows_matches_oracle(ctx):
    # Rows of 5,120 blocks (the most the top-k holds in registers) and 5,121
    # (staged in shared memory), and of more than 16,384 blocks (read from L2
    # each time): block scores, selection and output against the oracle.
    wl = workloads.custom(f"long_{ctx}", [ctx], [2], seed=91)
    st = harness.build_state(wl, DEV)
    side = OracleSide(wl, DEV)
    bufs, out, S = _decode(wl, st)
    _check_tokens(wl, side, bufs, out, S, range(wl.n_q_total))
    assert np.isfinite(out).all()
    assert st.cache.read_status() == 0



@pytest.mark.parametrize("ctx", [4800 * 128 + 1, 9000 * 128 + 1])
def test_topk_of_long_rows_several_tokens_per_cta(ctx):
    # More query tokens than CTAs (a CTA selects for several tokens in turn,
    # reusing its buffers) with long rows: ~4,800 blocks (keys held in
    # registers) and ~9,000 (staged in shared memory).  Tokens j and
    # j + (number of SMs) share a CTA.
    n_sm = torch.cuda.get_device_properties(0).multi_processor_count
    wl = workloads.custom(f"pairs_{ctx}", [ctx], [n_sm + 8], seed=93)
    st = harness.build_state(wl, DEV)
    side = OracleSide(wl, DEV)
    bufs, out, S = _decode(wl, st)
    _check_tokens(wl, side, bufs, out, S, [0, 1, n_sm, n_sm + 1, n_sm + 7])
    assert np.isfinite(out).all()
    assert st.cache.read_status() == 0

def test_hand_computed_indexer_case_on_the_gpu():
    # The hand-computed case of tests/golden/indexer_tiny.txt through the
    # library: insert its index keys, scan, select.
    from test_oracle_indexer import _golden_indexer_tiny, golden_indexer_inputs
    _, want_scores, want_sel = _golden_indexer_tiny()
    qi, w, k, L = golden_indexer_inputs()
    n_pages = (L + 127) // 128
    cache = ops.KVCache(n_pages, 1.0, 1.0, DEV)
    kv = torch.zeros((L, 4, 128), dtype=torch.float32, device=DEV)
    slots = torch.arange(L, dtype=torch.int64, device=DEV)
    ops.quantize_kv_insert(cache, kv, kv, torch.from_numpy(k).to(DEV), slots)
    bt = torch.arange(n_pages, dtype=torch.int32, device=DEV).view(1, n_pages)
    sl = torch.tensor([L], dtype=torch.int32, device=DEV)
    qsl = torch.tensor([0, 1], dtype=torch.int32, device=DEV)
    sel, n_sel, ws = ops.indexer_topk(cache, torch.from_numpy(qi).view(1, 8, 128).to(DEV),
                                      torch.from_numpy(w).view(1, 8).to(DEV), bt, sl, qsl)
    torch.cuda.synchronize()
    assert sel[0, : int(n_sel[0])].cpu().tolist() == want_sel
    S = block_scores_from_workspace(ws, 1, n_pages)
    assert [float(x) for x in S[0, :18]] == [want_scores[b] for b in range(18)]
    assert cache.read_status() == 0


def test_most_sequences_per_call():
    # 4,096 sequences, the most one call takes (the sequence metadata in shared
    # memory at its largest): short contexts where every block is selected and
    # longer ones where 16 of up to 20 blocks compete
    rng = np.random.default_rng(5)
    lens = [int(x) for x in rng.integers(129, 2600, 4096)]
    wl = workloads.custom("many_seqs", lens, [1] * 4096, seed=55)
    st = harness.build_state(wl, DEV)
    side = OracleSide(wl, DEV)
    bufs, out, S = _decode(wl, st)
    T = wl.n_q_total
    tokens = sorted(set([0, 1, T // 2, T - 1] + [int(x) for x in rng.integers(0, T, 3)]))
    _check_tokens(wl, side, bufs, out, S, tokens)
    assert np.isfinite(out).all()
    assert st.cache.read_status() == 0


@pytest.mark.parametrize("n_seqs", [115, 116, 300])
def test_sequence_lookup_with_empty_sequences(n_seqs):
    # the attention finds each token's sequence by a search of q_start_loc,
    # kept in shared memory for up to 115 sequences (the room its rings leave)
    # and read from global memory beyond; about 40% of the sequences here
    # have no query token, so q_start_loc repeats values (a token belongs to
    # the last sequence whose start is <= it)
    rng = np.random.default_rng(1000 + n_seqs)
    lens = [int(x) for x in rng.integers(1, 3000, n_seqs)]
    n_q = [0 if rng.random() < 0.4 else int(rng.integers(1, 5)) for _ in range(n_seqs)]
    n_q = [min(a, L) for a, L in zip(n_q, lens)]
    n_q[-1] = 0  # an empty sequence at the end as well
    wl = workloads.custom("lookup_%d" % n_seqs, lens, n_q, seed=n_seqs, permuted=True)
    st = harness.build_state(wl, DEV)
    side = OracleSide(wl, DEV)
    bufs, out, S = _decode(wl, st)
    T = wl.n_q_total
    starts = np.asarray(wl.q_start_loc)
    # the first token after each run of empty sequences, and a few at random
    after_empty = [int(starts[b]) for b in range(1, n_seqs) if n_q[b - 1] == 0 and n_q[b] > 0]
    tokens = sorted(set([0, T - 1] + after_empty[:6] + [int(x) for x in rng.integers(0, T, 4)]))
    _check_tokens(wl, side, bufs, out, S, tokens)
    assert st.cache.read_status() == 0



def test_inconsistent_q_start_loc_is_flagged_without_a_wait():
    # with a q_start_loc that leaves a token outside every sequence, or makes
    # two sequences overlap, every token still gets an output (an empty
    # selection where it has no sequence), the status says BAD_SEQ, and no
    # wait runs out
    wl = workloads.custom("qsl_bad", [3000, 5000], [2, 2], seed=21)
    st = harness.build_state(wl, DEV)
    _, qi, w = wl.queries(DEV)
    ref_sel, ref_n, _ = ops.indexer_topk(st.cache, qi, w, st.block_table, st.seq_lens, st.q_start_loc)
    torch.cuda.synchronize()
    ref_sel, ref_n = ref_sel.cpu().numpy(), ref_n.cpu().numpy()
    assert st.cache.read_status() == 0
    # token 3 outside every sequence (q_start_loc ends at 3 of 4 tokens)
    qsl = torch.tensor([0, 2, 3], dtype=torch.int32, device=DEV)
    sel, n_sel, _ = ops.indexer_topk(st.cache, qi, w, st.block_table, st.seq_lens, qsl)
    torch.cuda.synchronize()
    sel, n_sel = sel.cpu().numpy(), n_sel.cpu().numpy()
    assert st.cache.read_status() & ops.STATUS_BAD_SEQ
    assert not st.cache.read_status() & ops.STATUS_TIMEOUT
    assert n_sel[3] == 0 and (sel[3] == -1).all()
    assert np.array_equal(sel[:2], ref_sel[:2]) and np.array_equal(n_sel[:2], ref_n[:2])
    # overlapping sequences (q_start_loc not non-decreasing)
    st.cache.status.zero_()
    qsl = torch.tensor([0, 3, 2], dtype=torch.int32, device=DEV)
    sel, n_sel, _ = ops.indexer_topk(st.cache, qi, w, st.block_table, st.seq_lens, qsl)
    torch.cuda.synchronize()
    assert st.cache.read_status() & ops.STATUS_BAD_SEQ
    assert not st.cache.read_status() & ops.STATUS_TIMEOUT
    assert (n_sel.cpu().numpy() >= 0).all()

def test_host_validation_errors(tiny):
    wl, st, _ = tiny
    q, qi, w = wl.queries(DEV)
    T = wl.n_q_total
    with pytest.raises(ops.MsaError, match="workspace too small"):
        ops.indexer_topk(st.cache, qi, w, st.block_table, st.seq_lens, st.q_start_loc,
                         ws=torch.empty(16, dtype=torch.uint8, device=DEV))
    with pytest.raises(ops.MsaError, match="invalid argument"):
        ops.sparse_attn_decode(st.cache, q, torch.zeros((T, 17), dtype=torch.int32, device=DEV),
                               torch.zeros(T, dtype=torch.int32, device=DEV), st.block_table,
                               st.seq_lens, st.q_start_loc, n_splits=0)
    bad = ops.KVCache(1, 1.0, 1.0, DEV)
    bad.s_enc_k = float("nan")
    with pytest.raises(ops.MsaError, match="invalid argument"):
        ops.quantize_kv_insert(bad, torch.zeros((1, 4, 128), device=DEV), torch.zeros((1, 4, 128), device=DEV),
                               torch.zeros((1, 128), device=DEV), torch.zeros(1, dtype=torch.int64, device=DEV))


def test_device_status_bits_without_faults(tiny):
    wl, st, _ = tiny
    q, qi, w = wl.queries(DEV)
    # a block table entry outside the pool: flagged, skipped, no fault
    bt = st.block_table.clone()
    bt[0, 3] = wl.total_pages + 5
    cache = ops.KVCache(st.cache.n_pages, st.cache.s_enc_k, st.cache.s_enc_v, DEV)
    cache.kv_pool, cache.idx_pool = st.cache.kv_pool, st.cache.idx_pool
    bufs = ops.DecodeBuffers(wl.n_q_total, wl.max_pages, 2, DEV)
    ops.decode_step(cache, q, qi, w, bt, st.seq_lens, st.q_start_loc, bufs)
    assert cache.read_status() & 0x2
    # a slot outside the pool
    cache2 = ops.KVCache(1, 1.0, 1.0, DEV)
    ops.quantize_kv_insert(cache2, torch.ones((2, 4, 128), device=DEV), torch.ones((2, 4, 128), device=DEV),
                           torch.ones((2, 128), device=DEV),
                           torch.tensor([5, 128 * 7], dtype=torch.int64, device=DEV))
    assert cache2.read_status() & 0x1
    # more query tokens than cached tokens
    cache3 = ops.KVCache(st.cache.n_pages, st.cache.s_enc_k, st.cache.s_enc_v, DEV)
    cache3.kv_pool, cache3.idx_pool = st.cache.kv_pool, st.cache.idx_pool
    sl = torch.tensor([0], dtype=torch.int32, device=DEV)
    ops.decode_step(cache3, q, qi, w, st.block_table, sl, st.q_start_loc, bufs)
    assert cache3.read_status() & 0x4
    # selected blocks outside 0..r_j (negative, past the recent block): flagged
    # and skipped; the valid entries still attend
    cache4 = ops.KVCache(st.cache.n_pages, st.cache.s_enc_k, st.cache.s_enc_v, DEV)
    cache4.kv_pool, cache4.idx_pool = st.cache.kv_pool, st.cache.idx_pool
    T = wl.n_q_total
    sel = torch.full((T, 17), -1, dtype=torch.int32, device=DEV)
    sel[:, 0] = 0
    sel[:, 1] = 31
    sel[:, 2] = 32 + 7   # beyond r_j = 31
    sel[:, 3] = -3
    n_sel = torch.full((T,), 4, dtype=torch.int32, device=DEV)
    o_part, _ = ops.sparse_attn_decode(cache4, q, sel, n_sel, st.block_table, st.seq_lens,
                                       st.q_start_loc, 1)
    torch.cuda.synchronize()
    assert cache4.read_status() == ops.STATUS_BAD_SELECTION
    assert torch.isfinite(o_part).all() and (o_part.abs().amax() > 0)
