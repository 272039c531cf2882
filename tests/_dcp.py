"""Helpers of the context-split indexer tests: the candidate-key format of the
C ABI (include/msa.h, msa_indexer_topk_range) decoded for comparison."""

import numpy as np


def decode_keys(keys):
    """int64 [..., 16] keys -> (scores float32, blocks int64); empty keys -> (nan, -1)."""
    k = np.asarray(keys).astype(np.int64).view(np.uint64)
    hi = (k >> np.uint64(32)).astype(np.uint32)
    lo = (k & np.uint64(0xFFFFFFFF)).astype(np.uint32)
    bits = np.where(hi & np.uint32(0x80000000), hi & np.uint32(0x7FFFFFFF), ~hi).astype(np.uint32)
    scores = bits.view(np.float32).copy()
    blocks = (np.uint32(0xFFFFFFFF) - lo).astype(np.int64)
    empty = k == 0
    scores[empty] = np.nan
    blocks[empty] = -1
    return scores, blocks


def shard_bounds(n_blocks, n_shards):
    step = -(-n_blocks // n_shards)
    return [(i * step, min(n_blocks, (i + 1) * step)) for i in range(n_shards)]
