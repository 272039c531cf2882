"""CPU oracle for block-sparse attention decode over an NVFP4 KV cache.

TEST INFRASTRUCTURE ONLY.  This package is a plain, slow, obviously-correct
NumPy (float64 unless a step is defined in fp32) restatement of what the decode
path computes.  It exists to check the CUDA path; it is not part of it.

Only ``tests/``, ``__graft_entry__.smoke()`` and the ``cpu_baseline`` /
``--impl reference`` legs of ``bench.py`` may import or call it.  The product
package ``nvfp4_kv_block_gb300`` never imports it, and this package imports
nothing from the product package: the two share no code, tables or constants.

Sources (pages on the method):
  * "vLLM Delivers Day-0 Support for MiniMax-M3.1-Flash" (yuxiaoba.github.io
    blog), section "Sparse attention still scans an index": 128-token KV
    blocks, an indexer that selects 16 blocks and keeps the most recent one,
    128 index bytes per token and layer.
  * same page, section "Capacity savings must pay for conversion", and the
    ai4snews article (third paragraph): NVFP4 K/V are dequantised to FP8
    before the matmul because queries stay FP8; 34,560 vs 61,440 bytes/token.
  * kongchang.com article, section "NVFP4 KV Cache and MoE Weights": NVFP4 is a
    4-bit float with block-wise shared scaling factors.
The details the pages leave open (scoring formula, tie-break, GQA 16/4, the
two-level NVFP4 scale, tolerances) are readings of the pages, each stated in
the header of the module that implements it.

Parity status per function is stated in each module header.
"""

from . import formats, nvfp4, layout, indexer, attention, decode, qkv  # noqa: F401
