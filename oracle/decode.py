"""Oracle: one decode step of one sequence, from fp32 inputs to attention output.

Test infrastructure only (see ``oracle/__init__``).

Chains the oracle's own steps in the pages' data-flow order (blog, "Keep
capacity, layer, and system results separate": cache representation, kernel
inputs, ...): quantise K/V to NVFP4 and index keys to FP8, score and select
blocks, dequantise the selected K/V to FP8 and attend.  Nothing here is new
arithmetic; see the modules it calls for readings and parity status.
"""

import math

import numpy as np

from . import attention, formats, indexer, nvfp4


def quantize_sequence(k32, v32, idx32, s_enc_k, s_enc_v):
    """NVFP4 K/V ([L, 4, 128] fp32 each) and E4M3 index keys ([L, 128] fp32)."""
    kc, ks = nvfp4.quantize(k32, s_enc_k)
    vc, vs = nvfp4.quantize(v32, s_enc_v)
    return {
        "k_codes": kc, "k_scales": ks, "v_codes": vc, "v_scales": vs,
        "k8": nvfp4.fp8_operand(kc, ks), "v8": nvfp4.fp8_operand(vc, vs),
        "idx": formats.encode_e4m3(np.asarray(idx32, dtype=np.float32).astype(np.float64)),
    }


def decode_sequence(q8, q_idx, w, cache, seq_len, s_enc_k, s_enc_v,
                    softmax_scale=None, topk=16, tokens=None):
    """Selections, block scores, outputs and LSEs for the query tokens of one sequence.

    q8: uint8 [n_q, 16, 128]; q_idx: uint8 [n_q, 8, 128]; w: [n_q, 8];
    cache: output of quantize_sequence over at least seq_len tokens.
    ``tokens`` restricts the work to a subset of query-token indices.
    """
    if softmax_scale is None:
        softmax_scale = np.float32(1.0 / math.sqrt(q8.shape[-1]))
    n_q = q8.shape[0]
    res = []
    for j in (range(n_q) if tokens is None else tokens):
        pos = seq_len - n_q + j
        r = pos // indexer.PAGE_TOKENS
        s = indexer.block_scores(q_idx[j], w[j], cache["idx"], r)
        sel = indexer.select(s, r, topk)
        vis = attention.visible_positions(sel, pos)
        out, lse = attention.attend(q8[j], cache["k8"][vis], cache["v8"][vis],
                                    softmax_scale, s_enc_k, s_enc_v)
        res.append({"j": j, "sel": sel, "scores": s, "out": out, "lse": lse})
    return res
