"""Oracle: exact GQA attention over the selected tokens, two-pass softmax.

Test infrastructure only (see ``oracle/__init__``).

The pages: main attention runs over the selected blocks only, which is not the
same as dense attention (blog, "Sparse attention still scans an index"); FP8
queries meet K/V dequantised from NVFP4 to FP8 before the matmul (ai4snews
article, third paragraph; blog, "Capacity savings must pay for conversion").

Readings of the pages (where they are silent): 16 query heads share 4 KV heads (head h uses
KV head h // 4); logits = (q8 . k8) * softmax_scale / s_enc_K with
softmax_scale = 1/sqrt(128); out = sum_t p_t v8_t / sum_t p_t / s_enc_V; keys
at positions after the query token are not visible.

Arithmetic: float64 throughout, max-subtracted two-pass softmax.

Parity: pinned (tests/test_oracle_attention.py) by a naive per-key loop over
all blocks (dense attention when every block is selected), the one-dominant-key
and identical-keys special cases and the causal mask of speculative tokens.
"""

import math

import numpy as np

from .formats import decode_e4m3

GQA = 4


def attend(q8, k8, v8, softmax_scale, s_enc_k, s_enc_v):
    """Attention of one query token over n visible keys.

    q8: uint8 E4M3 [Hq, D]; k8, v8: uint8 E4M3 FP8 operands [n, Hkv, D].
    Returns (out [Hq, D], lse [Hq]) in float64; lse is the natural-log
    sum of exp of the scaled logits.
    """
    q = decode_e4m3(q8)
    k = decode_e4m3(k8)
    v = decode_e4m3(v8)
    hq = q.shape[0]
    c = float(np.float32(softmax_scale)) / float(np.float32(s_enc_k))
    out = np.zeros((hq, q.shape[1]))
    lse = np.zeros(hq)
    for h in range(hq):
        g = h // GQA
        logits = (k[:, g, :] @ q[h]) * c
        m = logits.max()
        p = np.exp(logits - m)
        l = p.sum()
        out[h] = (p @ v[:, g, :]) / l / float(np.float32(s_enc_v))
        lse[h] = m + math.log(l)
    return out, lse


def visible_positions(selection, pos, page_tokens=128):
    """Token positions of the selected blocks that are at or before pos."""
    idx = []
    for b in selection:
        lo = b * page_tokens
        hi = min(lo + page_tokens, pos + 1)
        idx.extend(range(lo, hi))
    return np.asarray(idx, dtype=np.int64)
