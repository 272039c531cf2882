"""Oracle: lightweight-indexer scores, per-block max and top-16 + recent selection.

Test infrastructure only (see ``oracle/__init__``).

The pages: the indexer scores the context over 128-token blocks, selects 16
blocks and keeps the most recent block, so main attention sees about 2,048 keys
per query (blog, "Sparse attention still scans an index"); the index holds 128
FP8 bytes per token and layer (same section).  Selection stays exact when the
scan is split (blog, "Parallelize index work across context").

Readings of the pages (where they are silent): the token score is
    score(t) = sum_h w_h * max(0, q_h . k_idx(t))
over the indexer heads h; a block's score is the max over its tokens; token j
of a sequence sits at pos_j = seq_len - n_q + j and its recent block is
r_j = pos_j // 128; blocks 0..r_j-1 compete and the best min(16, r_j) win by
(score descending, block index ascending); the output is the winners in
ascending order followed by r_j.

Arithmetic: FP8 inputs are decoded exactly; every product of two E4M3 values
is a multiple of 2^-18 below 2^18, so a 128-term dot product is exact in
float64.  The weighted sum over heads is float64.

Parity: pinned (tests/test_oracle_indexer.py) by exact rational dot products,
a closed-form one-hot example, a brute-force top-k over all subsets of tiny
inputs, a full-sort cross-check, the "r <= 16 selects everything" case, the
split-scan merge (range_candidates + merge_candidates over any tiling of the
context equal select, also against brute force), and the hand-computed case of tests/golden/indexer_tiny.txt
(19 blocks of sparse one-hot keys: block maxima at the first and the last
token of a block, ReLU of negative dots, a tie at the cut-off, and a recent
block whose score exceeds every other but does not compete).
"""

import numpy as np

from .formats import decode_e4m3

PAGE_TOKENS = 128


def token_scores(q_idx, w, keys):
    """score(t) for every key row.

    q_idx: uint8 E4M3 [H, D]; w: weights [H]; keys: uint8 E4M3 [n, D].
    Returns float64 [n].
    """
    q = decode_e4m3(q_idx)
    k = decode_e4m3(keys)
    dots = k @ q.T                                   # [n, H], exact
    return np.maximum(dots, 0.0) @ np.asarray(w, dtype=np.float64)


def block_scores(q_idx, w, keys, n_blocks, chunk_blocks=4096):
    """Per-block max of token scores for blocks 0..n_blocks-1 (full blocks).

    Token scores are independent of one another, so the blocks are scored
    ``chunk_blocks`` at a time only to bound the memory of the decoded keys.
    """
    out = np.zeros(n_blocks)
    for b0 in range(0, n_blocks, chunk_blocks):
        b1 = min(n_blocks, b0 + chunk_blocks)
        s = token_scores(q_idx, w, keys[b0 * PAGE_TOKENS: b1 * PAGE_TOKENS])
        out[b0:b1] = s.reshape(b1 - b0, PAGE_TOKENS).max(axis=1)
    return out


def select(scores, recent, topk=16):
    """Top-k of blocks 0..recent-1 by (score desc, index asc), ascending, plus recent."""
    scores = np.asarray(scores, dtype=np.float64)[:recent]
    order = sorted(range(recent), key=lambda b: (-scores[b], b))
    chosen = sorted(order[: min(topk, recent)])
    return chosen + [recent]


def range_candidates(scores, recent, lo, hi, topk=16):
    """Local top-k of one part of the context (blog, "Parallelize index work
    across context"): blocks lo .. min(hi, recent)-1 compete by (score desc,
    index asc); returns [(score, block)], best first."""
    e = min(hi, recent)
    lo = min(lo, e)
    order = sorted(range(lo, e), key=lambda b: (-scores[b], b))
    return [(float(scores[b]), b) for b in order[:topk]]


def merge_candidates(parts, recent, topk=16):
    """Top-k of the union of the parts' candidates by (score desc, index asc),
    in ascending order, then the recent block."""
    pool = [c for part in parts for c in part]
    order = sorted(pool, key=lambda c: (-c[0], c[1]))
    return sorted(b for _, b in order[:topk]) + [recent]


def sequence_topk(q_idx, w, keys, seq_len, topk=16):
    """Selections for all query tokens of one sequence.

    q_idx: uint8 [n_q, H, D]; w: [n_q, H]; keys: uint8 [seq_len, D] (logical
    token order).  Returns (selections, block_scores) with one list / one
    float64 array per query token.
    """
    n_q = q_idx.shape[0]
    sels, scs = [], []
    for j in range(n_q):
        pos = seq_len - n_q + j
        r = pos // PAGE_TOKENS
        s = block_scores(q_idx[j], w[j], keys, r)
        sels.append(select(s, r, topk))
        scs.append(s)
    return sels, scs
