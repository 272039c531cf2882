"""Oracle: byte layout of one 128-token KV page and one index page.

Test infrastructure only (see ``oracle/__init__``).

The pages fix the sizes: 128-token blocks (blog, "Sparse attention still scans
an index"), 128 index bytes per token and layer (same section), and NVFP4 K+V
at 576 bytes per token and layer for 4 KV heads of dimension 128 (ai4snews
article, first paragraph: 34,560 bytes/token over the model's layers).  The
placement of bytes inside a page is this library's own format, restated here
independently of the CUDA code from its written specification:

KV page, 73,728 bytes = 4 heads x 18,432 bytes; head g starts at g * 18,432:
    +0      K codes   [128 tokens][64 B]: little-endian 32-bit word i holds
            channels 8i..8i+7 (E2M1 code = sign bit s and magnitude m, 3 bits):
            bits 4n..4n+2 = m of channel 8i+n (n = 0..7), bit 8n+7 = s of
            channel 8i+n and bit 8n+3 = s of channel 8i+4+n (n = 0..3); the
            16-byte chunk c of token t's row (channels 32c..32c+31) is stored
            at chunk position c XOR ((t >> 1) mod 4)
    +8,192  K scales  [8 groups][128 tokens]   E4M3, group k = channels 16k..16k+15
    +9,216  V codes   [128 tokens][64 B], chunks placed like the K codes
    +17,408 V scales  [8 groups][128 tokens]
Index page, 16,384 bytes = [128 tokens][128 B] E4M3 index keys, where the
16-byte chunk c of token t's row (dims 16c..16c+15) is stored at chunk
position c XOR (t mod 8).

Parity: pinned by the byte-count invariants of the pages
(tests/test_oracle_nvfp4.py) and by the hand-placed bytes of
tests/golden/layout_bytes.txt.
"""

import numpy as np

PAGE_TOKENS = 128
KV_HEADS = 4
HEAD_DIM = 128
IDX_DIM = 128
HEAD_BYTES = 18_432
KV_PAGE_BYTES = KV_HEADS * HEAD_BYTES          # 73,728
IDX_PAGE_BYTES = PAGE_TOKENS * IDX_DIM        # 16,384
OFF_KC, OFF_KS, OFF_VC, OFF_VS = 0, 8_192, 9_216, 17_408


def pack_codes(codes):
    """Pack E2M1 codes (4-bit: sign << 3 | magnitude; last axis a multiple of 8)
    into 32-bit little-endian words of 8 channels each, as laid out above."""
    c = np.asarray(codes, dtype=np.uint32)
    g = c.reshape(c.shape[:-1] + (c.shape[-1] // 8, 8))
    mag, sign = g & 7, (g >> 3) & 1
    word = np.zeros(g.shape[:-1], dtype=np.uint32)
    for n in range(8):
        word |= mag[..., n] << (4 * n)
    for n in range(4):
        word |= sign[..., n] << (8 * n + 7)
        word |= sign[..., 4 + n] << (8 * n + 3)
    out = np.empty(word.shape + (4,), dtype=np.uint8)
    for b in range(4):
        out[..., b] = (word >> (8 * b)) & 0xFF
    return out.reshape(c.shape[:-1] + (c.shape[-1] // 2,))


def unpack_codes(packed):
    """Inverse of pack_codes."""
    p = np.asarray(packed, dtype=np.uint32)
    b = p.reshape(p.shape[:-1] + (p.shape[-1] // 4, 4))
    word = b[..., 0] | (b[..., 1] << 8) | (b[..., 2] << 16) | (b[..., 3] << 24)
    out = np.empty(word.shape + (8,), dtype=np.uint8)
    for n in range(8):
        out[..., n] = (word >> (4 * n)) & 7
    for n in range(4):
        out[..., n] |= (((word >> (8 * n + 7)) & 1) << 3).astype(np.uint8)
        out[..., 4 + n] |= (((word >> (8 * n + 3)) & 1) << 3).astype(np.uint8)
    return out.reshape(p.shape[:-1] + (p.shape[-1] * 2,))


def code_chunk_position(c, t):
    """Chunk position of the 16-byte code chunk c in token t's 64-byte row."""
    return c ^ ((t >> 1) % 4)


def write_kv_slot(pool, page, t, k_codes, k_scales, v_codes, v_scales):
    """Write one token's NVFP4 K/V (codes [4,128], scales [4,8]) into slot t of a page.

    ``pool`` is a uint8 array [n_pages, 73,728].
    """
    for g in range(KV_HEADS):
        base = g * HEAD_BYTES
        for off_c, off_s, codes, scales in ((OFF_KC, OFF_KS, k_codes, k_scales),
                                            (OFF_VC, OFF_VS, v_codes, v_scales)):
            row = base + off_c + t * 64
            packed = pack_codes(codes[g])
            for c in range(4):
                pos = code_chunk_position(c, t)
                pool[page, row + 16 * pos:row + 16 * pos + 16] = packed[16 * c:16 * c + 16]
            for k in range(8):
                pool[page, base + off_s + k * PAGE_TOKENS + t] = scales[g][k]


def write_index_slot(pool, page, t, key_bytes):
    """Write one token's 128 E4M3 index-key bytes into slot t (chunk-swizzled)."""
    key_bytes = np.asarray(key_bytes, dtype=np.uint8)
    for c in range(8):
        pos = c ^ (t % 8)
        start = t * IDX_DIM + pos * 16
        pool[page, start:start + 16] = key_bytes[c * 16:(c + 1) * 16]


def read_kv_slot(pool, page, t):
    """Inverse of write_kv_slot: (k_codes, k_scales, v_codes, v_scales) of one slot."""
    out = []
    for off_c, off_s in ((OFF_KC, OFF_KS), (OFF_VC, OFF_VS)):
        codes = np.zeros((KV_HEADS, HEAD_DIM), dtype=np.uint8)
        scales = np.zeros((KV_HEADS, 8), dtype=np.uint8)
        for g in range(KV_HEADS):
            base = g * HEAD_BYTES
            row = base + off_c + t * 64
            packed = np.zeros(64, dtype=np.uint8)
            for c in range(4):
                pos = code_chunk_position(c, t)
                packed[16 * c:16 * c + 16] = pool[page, row + 16 * pos:row + 16 * pos + 16]
            codes[g] = unpack_codes(packed)
            for k in range(8):
                scales[g, k] = pool[page, base + off_s + k * PAGE_TOKENS + t]
        out += [codes, scales]
    return tuple(out)


def read_index_slot(pool, page, t):
    key = np.zeros(IDX_DIM, dtype=np.uint8)
    for c in range(8):
        pos = c ^ (t % 8)
        start = t * IDX_DIM + pos * 16
        key[c * 16:(c + 1) * 16] = pool[page, start:start + 16]
    return key


# ---- block-outer transfer rows ------------------------------------------------
# Blog "vLLM Delivers Day-0 Support for MiniMax-M3.1-Flash", section "AMD uses
# different conversion and communication mechanisms": a KV block spread over
# many pages needs many reads; a block-outer layout keeps one block as one
# contiguous row, read at once.  Reading: the row of a block holds, for every
# layer in order, that layer's KV page (73,728 bytes) followed by its index
# page (16,384 bytes) -- the whole decode state of the block -- so a row is
# n_layers x 90,112 bytes; the same physical page id addresses the block in
# every layer's pools.

ROW_LAYER_BYTES = KV_PAGE_BYTES + IDX_PAGE_BYTES   # 90,112


def pack_rows(kv_pools, idx_pools, pages):
    """Rows [len(pages)][n_layers * 90,112] of the listed physical pages.

    kv_pools, idx_pools: per layer, uint8 [n_pages, 73,728] / [n_pages, 16,384].
    """
    n_layers = len(kv_pools)
    rows = np.zeros((len(pages), n_layers * ROW_LAYER_BYTES), dtype=np.uint8)
    for i, page in enumerate(pages):
        for layer in range(n_layers):
            at = layer * ROW_LAYER_BYTES
            rows[i, at:at + KV_PAGE_BYTES] = kv_pools[layer][page]
            rows[i, at + KV_PAGE_BYTES:at + ROW_LAYER_BYTES] = idx_pools[layer][page]
    return rows


def unpack_rows(rows, kv_pools, idx_pools, pages):
    """Inverse of pack_rows: write row i back into page pages[i] of every layer."""
    for i, page in enumerate(pages):
        for layer in range(len(kv_pools)):
            at = layer * ROW_LAYER_BYTES
            kv_pools[layer][page] = rows[i, at:at + KV_PAGE_BYTES]
            idx_pools[layer][page] = rows[i, at + KV_PAGE_BYTES:at + ROW_LAYER_BYTES]
