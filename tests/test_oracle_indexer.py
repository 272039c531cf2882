"""Pins for the oracle's indexer scores and top-16 + recent selection (CPU only)."""

import itertools
from fractions import Fraction

import numpy as np
import pytest

from oracle import formats, indexer


def _fp8(rng, shape, scale=1.0):
    return formats.encode_e4m3(rng.standard_normal(shape) * scale)


def test_scores_equal_exact_rational_arithmetic():
    rng = np.random.default_rng(0)
    q = _fp8(rng, (8, 128))
    keys = _fp8(rng, (6, 128), 3.0)
    w = rng.uniform(0, 1, 8).astype(np.float32)
    got = indexer.token_scores(q, w, keys)
    qv = [[Fraction(float(formats.decode_e4m3(b))) for b in row] for row in q]
    for t in range(keys.shape[0]):
        kv = [Fraction(float(formats.decode_e4m3(b))) for b in keys[t]]
        exact = Fraction(0)
        for h in range(8):
            d = sum(a * b for a, b in zip(qv[h], kv))
            exact += Fraction(float(w[h])) * max(d, Fraction(0))
        # dots are exact; the 8-term weighted sum rounds at most 8 times
        assert abs(Fraction(got[t]) - exact) <= abs(exact) * Fraction(1, 2 ** 50)


def test_hand_example_closed_form():
    # one-hot queries: head 0 reads dim 0 with q=1, head 1 reads dim 1 with q=2, w=(1, 0.5):
    # score(t) = relu(k0) + relu(k1), hand-checkable
    q = np.zeros((2, 128), dtype=np.uint8)
    q[0, 0] = formats.encode_e4m3(1.0)
    q[1, 1] = formats.encode_e4m3(2.0)
    w = np.array([1.0, 0.5], dtype=np.float32)
    k0 = [1.5, -2.0, 0.25, 3.0]
    k1 = [-1.0, 4.0, 0.5, -6.0]
    keys = np.zeros((4, 128), dtype=np.uint8)
    keys[:, 0] = formats.encode_e4m3(np.array(k0))
    keys[:, 1] = formats.encode_e4m3(np.array(k1))
    assert list(indexer.token_scores(q, w, keys)) == [1.5, 4.0, 0.75, 3.0]


def _brute_topk(scores, k):
    n = len(scores)
    winners = []
    for subset in itertools.combinations(range(n), min(k, n)):
        s = set(subset)
        ok = all((scores[b] > scores[o]) or (scores[b] == scores[o] and b < o)
                 for b in s for o in range(n) if o not in s)
        if ok:
            winners.append(sorted(subset))
    assert len(winners) == 1
    return winners[0]


@pytest.mark.parametrize("seed", range(30))
def test_select_equals_brute_force_on_tiny_inputs(seed):
    rng = np.random.default_rng(seed)
    n = int(rng.integers(1, 10))
    scores = rng.integers(0, 4, n).astype(np.float64)  # many ties
    k = int(rng.integers(1, 6))
    assert indexer.select(scores, n, k) == _brute_topk(list(scores), k) + [n]


def test_select_equals_full_sort_and_keeps_recent():
    rng = np.random.default_rng(11)
    for _ in range(50):
        r = int(rng.integers(17, 600))
        s = np.round(rng.uniform(0, 5, r), 2)  # ties
        got = indexer.select(s, r)
        order = np.lexsort((np.arange(r), -s))   # primary -s, secondary index
        assert got == sorted(order[:16].tolist()) + [r]
        assert len(got) == 17 and got[-1] == r


def test_short_context_selects_every_block():
    for r in range(0, 17):
        assert indexer.select(np.ones(r), r) == list(range(r + 1))


def test_split_scan_merge_is_exact():
    # Local top-16 per chunk, then top-16 of the candidates, equals the global
    # top-16 (the exactness of a split scan, blog "Parallelize index work across context").
    rng = np.random.default_rng(12)
    for _ in range(50):
        r = int(rng.integers(17, 2000))
        s = np.round(rng.uniform(0, 3, r), 1)
        chunk = int(rng.integers(1, 300))
        cands = []
        for lo in range(0, r, chunk):
            idx = np.arange(lo, min(lo + chunk, r))
            loc = idx[np.lexsort((idx, -s[idx]))][:16]
            cands.extend(loc.tolist())
        cands = np.array(cands)
        merged = sorted(cands[np.lexsort((cands, -s[cands]))][:16].tolist())
        assert merged + [r] == indexer.select(s, r)


def test_sequence_positions_and_recent_blocks():
    rng = np.random.default_rng(13)
    seq_len, n_q = 128 * 20 + 3, 8          # tokens 2555..2562 straddle block 19/20
    keys = _fp8(rng, (seq_len, 128))
    q = _fp8(rng, (n_q, 8, 128))
    w = rng.uniform(0, 1, (n_q, 8)).astype(np.float32)
    sels, scs = indexer.sequence_topk(q, w, keys, seq_len)
    for j in range(n_q):
        pos = seq_len - n_q + j
        r = pos // 128
        assert sels[j][-1] == r and len(scs[j]) == r
        assert len(sels[j]) == min(16, r) + 1
        # block scores are maxima of the token scores of full blocks
        ts = indexer.token_scores(q[j], w[j], keys[: r * 128]).reshape(r, 128)
        assert np.array_equal(scs[j], ts.max(axis=1))
    assert sels[0][-1] == 19 and sels[-1][-1] == 20


def _golden_indexer_tiny():
    import os
    path = os.path.join(os.path.dirname(__file__), "golden", "indexer_tiny.txt")
    keys, scores, sel = [], {}, None
    with open(path) as f:
        for line in f:
            parts = line.split()
            if not parts or parts[0].startswith("#"):
                continue
            if parts[0] == "key":
                keys.append((int(parts[1]), int(parts[2]), float(parts[3]), float(parts[4])))
            elif parts[0] == "score":
                scores[int(parts[1])] = float(parts[2])
            elif parts[0] == "sel":
                sel = [int(x) for x in parts[1:]]
    return keys, scores, sel


def golden_indexer_inputs():
    """(q_idx uint8 [8,128], w [8], fp32 keys [2309,128], seq_len) of the hand case."""
    keys, _, _ = _golden_indexer_tiny()
    seq_len = 2309
    k = np.zeros((seq_len, 128), dtype=np.float32)
    for blk, off, k0, k1 in keys:
        k[blk * 128 + off, 0] = k0
        k[blk * 128 + off, 1] = k1
    q = np.zeros((8, 128))
    q[0, 0] = 1.0
    q[1, 1] = 2.0
    w = np.array([1.0, 0.5] + [0.3] * 6, dtype=np.float32)
    return formats.encode_e4m3(q), w, k, seq_len


def test_hand_computed_block_scores_and_selection():
    _, want_scores, want_sel = _golden_indexer_tiny()
    q, w, k, seq_len = golden_indexer_inputs()
    keys = formats.encode_e4m3(k.astype(np.float64))
    # every listed key value is exact in E4M3
    assert np.array_equal(formats.decode_e4m3(keys), k.astype(np.float64))
    r = (seq_len - 1) // 128
    assert r == 18
    s = indexer.block_scores(q, w, keys, r)
    assert [float(x) for x in s] == [want_scores[b] for b in range(r)]
    assert indexer.select(s, r) == want_sel
    sels, scs = indexer.sequence_topk(q[None], w[None], keys, seq_len)
    assert sels[0] == want_sel and np.array_equal(scs[0], s)
    # the recent block outscores every competing block, yet is not a competitor
    assert indexer.token_scores(q, w, keys[18 * 128 + 2: 18 * 128 + 3])[0] == 896.0


def test_block_scores_are_independent_of_the_chunking():
    rng = np.random.default_rng(21)
    keys = _fp8(rng, (40 * 128, 128))
    q = _fp8(rng, (8, 128))
    w = rng.uniform(0, 1, 8).astype(np.float32)
    a = indexer.block_scores(q, w, keys, 40)
    for chunk in (1, 3, 7, 40, 4096):
        assert np.array_equal(indexer.block_scores(q, w, keys, 40, chunk_blocks=chunk), a)
    # and equal to the per-block max written out token by token
    ts = indexer.token_scores(q, w, keys)
    assert all(a[b] == max(ts[b * 128:(b + 1) * 128]) for b in range(40))


def test_decode_table_equals_the_bit_field_definition():
    b = np.arange(256, dtype=np.uint8)
    fast = formats.decode_e4m3(b)
    slow = formats.decode_e4m3(b.astype(np.int64))
    assert np.array_equal(np.isnan(fast), np.isnan(slow))
    assert np.array_equal(fast[~np.isnan(fast)], slow[~np.isnan(slow)])


@pytest.mark.parametrize("seed", range(12))
def test_range_candidates_merge_to_the_global_selection(seed):
    # any tiling of the competing blocks into parts: local top-16 of each part,
    # then the merge, selects exactly what one global selection does (blog,
    # "Parallelize index work across context"), ties included
    rng = np.random.default_rng(100 + seed)
    r = int(rng.integers(1, 700))
    s = np.round(rng.uniform(0, 3, r), 1)  # many ties
    cuts = sorted(set(int(x) for x in rng.integers(0, r + 40, int(rng.integers(0, 6)))))
    bounds = [0] + cuts + [r + 40]
    parts = [indexer.range_candidates(s, r, lo, hi) for lo, hi in zip(bounds[:-1], bounds[1:])]
    assert all(len(p) <= 16 for p in parts)
    assert indexer.merge_candidates(parts, r) == indexer.select(s, r)


def test_range_candidates_on_tiny_inputs_equal_brute_force():
    rng = np.random.default_rng(7)
    for _ in range(40):
        r = int(rng.integers(1, 9))
        s = rng.integers(0, 3, r).astype(np.float64)
        lo, hi = sorted(int(x) for x in rng.integers(0, r + 2, 2))
        k = int(rng.integers(1, 5))
        got = [b for _, b in indexer.range_candidates(s, r, lo, hi, topk=k)]
        blocks = list(range(min(lo, min(hi, r)), min(hi, r)))
        want = _brute_topk([s[b] for b in blocks], k) if blocks else []
        assert sorted(got) == [blocks[i] for i in want]
        # best first: scores non-increasing, ties by ascending block
        pairs = [(-s[b], b) for b in got]
        assert pairs == sorted(pairs)
