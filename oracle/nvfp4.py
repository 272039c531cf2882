"""Oracle: NVFP4 two-level quantiser and the FP8 dequantised operand.

Test infrastructure only (see ``oracle/__init__``).

What the pages fix: the K/V cache is NVFP4, a 4-bit float with block-wise
shared scales (kongchang.com article, "NVFP4 KV Cache and MoE Weights");
34,560 vs 61,440 bytes/token, i.e. 4 bits plus one byte of scale per 16
elements (ai4snews article, first paragraph); queries stay FP8 so the cache
is dequantised to FP8 before the matmul (same article, third paragraph; blog
section "Capacity savings must pay for conversion").

Readings (the pages are silent on these):
  * one E4M3 scale per 16 consecutive channels of one token and head, plus an
    fp32 per-tensor encode scale ``s_enc = fp32(448 / amax)`` over the whole
    K (resp. V) tensor, so that a dequantised element (<= 6 x 72) never
    saturates E4M3;
  * block scale ``sb = E4M3(fp32(fp32(a / 6) * s_enc))`` with a = group amax;
  * element code = E2M1 RNE (ties to even, saturating at 6) of
    ``fp32(|x| * s_enc) / sb``, evaluated exactly; code 0 carries no sign;
  * FP8 operand of an element = its code's sign bit on top of
    ``E4M3(|e2m1| * sb)`` (the tensor scale 1/s_enc is applied after the
    contraction, where it factors out).

Every fp32 step is an IEEE fp32 operation (NumPy float32 arithmetic); the
rest is exact float64.

Parity: pinned (tests/test_oracle_nvfp4.py) by hand-computed groups in
tests/golden/nvfp4_groups.txt, the on-grid round trip, the per-element error
bound of E2M1 rounding and the byte-count invariant of the pages.
"""

import numpy as np

from .formats import (E2M1_MIDS, decode_e2m1, decode_e4m3, encode_e4m3,
                      encode_e2m1_magnitude)

GROUP = 16          # elements per block scale
F32 = np.float32


def tensor_encode_scale(amax):
    """fp32 per-tensor encode scale 448 / amax (1.0 for an all-zero tensor)."""
    amax = F32(amax)
    if amax == 0:
        return F32(1.0)
    return F32(F32(448.0) / amax)


def quantize(x, s_enc):
    """Quantise fp32 rows (last axis a multiple of 16) to NVFP4.

    Returns ``(codes, scales)``: ``codes`` uint8 E2M1 codes 0..15, one per
    element (same shape as x); ``scales`` uint8 E4M3 block scales, one per 16
    consecutive elements of the last axis.
    """
    x = np.asarray(x, dtype=F32)
    s_enc = F32(s_enc)
    g = x.reshape(x.shape[:-1] + (x.shape[-1] // GROUP, GROUP))
    a = np.max(np.abs(g), axis=-1)                       # exact
    t = (a / F32(6.0)).astype(F32)                        # fp32 divide
    u = (t * s_enc).astype(F32)                           # fp32 multiply
    sb_byte = encode_e4m3(u.astype(np.float64))
    sb = decode_e4m3(sb_byte)                             # float64, exact
    y = (np.abs(g) * s_enc).astype(F32).astype(np.float64)  # fp32 multiply
    with np.errstate(divide="ignore", invalid="ignore"):
        # r = y / sb is never formed: the midpoint comparisons of
        # encode_e2m1_magnitude are done as y vs mid*sb, both exact in float64.
        mag = np.zeros(y.shape, dtype=np.int64)
        sbb = np.broadcast_to(sb[..., None], y.shape)
        for k, mid in enumerate(E2M1_MIDS):
            thr = mid * sbb
            mag += (y > thr)
            if k % 2 == 1:
                mag += (y == thr)
        mag = np.where(sbb == 0, 0, mag)
    sign = (g < 0) & (mag != 0)
    codes = (mag | np.where(sign, 8, 0)).astype(np.uint8)
    return codes.reshape(x.shape), sb_byte.astype(np.uint8)


def quantize_reference_ratio(x, s_enc):
    """Same codes as ``quantize`` but via the explicit ratio y / sb (for pins)."""
    x = np.asarray(x, dtype=F32)
    s_enc = F32(s_enc)
    g = x.reshape(x.shape[:-1] + (x.shape[-1] // GROUP, GROUP))
    a = np.max(np.abs(g), axis=-1)
    sb = decode_e4m3(encode_e4m3(((a / F32(6.0)).astype(F32) * s_enc).astype(F32)))
    y = (np.abs(g) * s_enc).astype(F32).astype(np.float64)
    with np.errstate(divide="ignore", invalid="ignore"):
        r = np.where(sb[..., None] > 0, y / np.where(sb[..., None] > 0, sb[..., None], 1.0), 0.0)
    mag = encode_e2m1_magnitude(r)
    sign = (g < 0) & (mag != 0)
    return (mag | np.where(sign, 8, 0)).astype(np.uint8).reshape(x.shape)


def dequantize(codes, scales, s_enc):
    """Exact NVFP4 value of each element: e2m1(code) * sb / s_enc (float64)."""
    codes = np.asarray(codes)
    v = decode_e2m1(codes)
    g = v.reshape(v.shape[:-1] + (v.shape[-1] // GROUP, GROUP))
    sb = decode_e4m3(scales)[..., None]
    return (g * sb / np.float64(F32(s_enc))).reshape(v.shape)


def fp8_operand(codes, scales):
    """E4M3 bytes of the FP8 operand: sign(code) | E4M3(|e2m1(code)| * sb).

    The product |e2m1| * sb has at most 5 significant bits, so it is exact in
    float64 and ``encode_e4m3`` applies the only rounding.
    """
    codes = np.asarray(codes).astype(np.int64)
    mag = decode_e2m1(codes & 7)
    g = mag.reshape(mag.shape[:-1] + (mag.shape[-1] // GROUP, GROUP))
    sb = decode_e4m3(scales)[..., None]
    prod = (g * sb).reshape(mag.shape)
    return (encode_e4m3(prod) | ((codes & 8) << 4).astype(np.uint8)).astype(np.uint8)
