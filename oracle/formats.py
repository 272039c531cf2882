"""Oracle: E2M1 (FP4) and E4M3 (FP8) codecs, written from the bit-field definitions.

Test infrastructure only (see ``oracle/__init__``).

E2M1 -- the element type of NVFP4 (kongchang.com article, "NVFP4 KV Cache and
MoE Weights": a 4-bit float with a very narrow exponent and mantissa).  Bit 3
is the sign, bits 2..1 the exponent (bias 1), bit 0 the mantissa; exponent 0 is
subnormal.  Magnitudes by code 0..7: 0, 0.5, 1, 1.5, 2, 3, 4, 6.

E4M3 -- the FP8 type of queries, index keys, block scales and the dequantised
K/V operand (ai4snews article, third paragraph: the cache is dequantised to FP8
for the matrix multiply).  OCP "E4M3FN": bias 7, no infinities, S.1111.111 is
NaN, largest finite 448, smallest normal 2^-6, smallest subnormal 2^-9.

Encoders round to nearest, ties to the even code, and saturate finite values
(and infinities) to +-448; NaN encodes as 0x7F.  ``encode_e4m3`` never emits
negative zero (a result of zero magnitude is 0x00): this is the canonical-zero
reading used for every stored FP8 byte (index keys, block scales).

Parity: pinned (tests/test_oracle_formats.py) against hand tables in
tests/golden/, against torch's float8_e4m3fn cast and, where installed,
ml_dtypes' float4_e2m1fn / float8_e4m3fn casts.
"""

import numpy as np


def decode_e2m1(code):
    """Value of 4-bit E2M1 codes (array of ints 0..15) as float64."""
    c = np.asarray(code, dtype=np.int64)
    sign = np.where((c >> 3) & 1, -1.0, 1.0)
    e = (c >> 1) & 3
    m = c & 1
    mag = np.where(e == 0, 0.5 * m, np.ldexp(1.0 + 0.5 * m, e - 1))
    return sign * mag


def _decode_e4m3_fields(byte):
    b = np.asarray(byte, dtype=np.int64)
    sign = np.where((b >> 7) & 1, -1.0, 1.0)
    e = (b >> 3) & 15
    m = b & 7
    sub = np.ldexp(m / 8.0, -6)
    nrm = np.ldexp(1.0 + m / 8.0, e - 7)
    mag = np.where(e == 0, sub, nrm)
    mag = np.where((e == 15) & (m == 7), np.nan, mag)
    return sign * mag


# Values of all 256 bytes, from the bit fields above; large uint8 arrays are
# decoded by looking their bytes up here (same values, one gather).
_E4M3_ALL = _decode_e4m3_fields(np.arange(256))


def decode_e4m3(byte):
    """Value of E4M3FN bytes (array of ints 0..255) as float64 (NaN for 0x7F/0xFF)."""
    b = np.asarray(byte)
    if b.dtype == np.uint8:
        return _E4M3_ALL[b]
    return _decode_e4m3_fields(b)


# The 127 non-negative finite E4M3 values, indexed by their code 0x00..0x7E.
_E4M3_POS = decode_e4m3(np.arange(127))
assert np.all(np.diff(_E4M3_POS) > 0)


def encode_e4m3(x):
    """Round float64 values to E4M3FN bytes: RNE, ties to even code, satfinite.

    Exact for any float64 input: the two grid neighbours of |x| lie within a
    factor of two of it, so both distances are computed without rounding
    (Sterbenz) and the comparison, ties included, is exact.
    """
    x = np.asarray(x, dtype=np.float64)
    out = np.zeros(x.shape, dtype=np.uint8)
    nan = np.isnan(x)
    a = np.abs(np.where(nan, 0.0, x))
    a = np.minimum(a, 448.0)  # saturate finite (and infinite) magnitudes
    hi = np.searchsorted(_E4M3_POS, a, side="left")  # first grid value >= a
    hi = np.clip(hi, 0, 126)
    lo = np.clip(hi - 1, 0, 126)
    dlo = a - _E4M3_POS[lo]
    dhi = _E4M3_POS[hi] - a
    pick_hi = (dhi < dlo) | ((dhi == dlo) & (hi % 2 == 0))
    code = np.where(pick_hi, hi, lo)
    code = np.where(a == _E4M3_POS[hi], hi, code)
    neg = (x < 0) & (code != 0)
    out[...] = code.astype(np.uint8) | np.where(neg, 0x80, 0).astype(np.uint8)
    out[nan] = 0x7F
    return out


# E2M1 magnitude grid (codes 0..7) and the midpoints between neighbours.
E2M1_MAGS = decode_e2m1(np.arange(8))
E2M1_MIDS = 0.5 * (E2M1_MAGS[:-1] + E2M1_MAGS[1:])  # 0.25 0.75 1.25 1.75 2.5 3.5 5


def encode_e2m1_magnitude(r):
    """E2M1 magnitude code (0..7) of non-negative float64 ratios: RNE, ties to even, sat 6.

    Code c is the number of midpoints strictly below r, moved up by one when r
    sits exactly on a midpoint whose lower neighbour has an odd code.
    """
    r = np.asarray(r, dtype=np.float64)
    c = np.zeros(r.shape, dtype=np.int64)
    for k, mid in enumerate(E2M1_MIDS):
        c += (r > mid)
        if k % 2 == 1:
            c += (r == mid)
    return c
