"""Oracle: QKV projection, per-head RMS norm, RoPE and the cache bytes they feed.

Test infrastructure only (see ``oracle/__init__``).

The pages: a fused path runs the QKV projection, normalisation, RoPE and cache
insertion without writing the intermediate tensor to HBM (blog "vLLM Delivers
Day-0 Support for MiniMax-M3.1-Flash", section "Reduce both data movement and
resource waits").  They fix nothing else about it.

Readings (the pages are silent on these):
  * the projection maps a token's hidden state x [d] to 25 heads of 128:
    16 query heads, 4 key heads, 4 value heads, 1 index-key head (the heads
    the decode path consumes); W is [25 * 128, d] (output rows), z = W x;
  * query, key and index-key heads are RMS-normalised per head, with one
    128-entry gain vector per kind: y = z / sqrt(mean(z^2) + eps) * gamma,
    eps = 1e-6; value heads are not normalised;
  * RoPE after the norm on query, key and index-key heads: channel pairs
    (i, i + 64), i < 64, rotated by the angle pos * base^(-2 i / 128),
    base = 10,000: (a, b) -> (a cos - b sin, b cos + a sin), the cos / sin
    taken from an fp32 table of the angles (computed in float64, rounded);
  * queries leave as E4M3 (RNE, satfinite), keys and values are quantised to
    NVFP4 with the cache's per-tensor scales (oracle.nvfp4), index keys as
    E4M3, all into the decode path's formats.
Arithmetic: float64 from bf16 / fp32 inputs; the cache bytes are formed from
given fp32 rows (where fp32 rounding decides a code, both sides decide from
the same fp32 values).

Parity: pinned (tests/test_oracle_qkv.py) by closed forms -- one-hot hidden
states select a weight row, a constant head normalises to its gain, position
0 is the identity, pair 0 turns by exactly pos radians and pair 32 by pos/100,
rotations keep each pair's norm -- and by re-deriving the cache bytes through
the pinned quantiser and layout.
"""

import numpy as np

from . import formats, nvfp4

Q_HEADS, KV_HEADS = 16, 4
HEADS = Q_HEADS + 2 * KV_HEADS + 1       # 25
K0, V0, IDX = Q_HEADS, Q_HEADS + KV_HEADS, Q_HEADS + 2 * KV_HEADS
DIM = 128
EPS = 1e-6


def rope_table(max_pos, base=10000.0):
    """fp32 [max_pos][128]: cos of the 64 pair angles, then their sin."""
    pos = np.arange(max_pos, dtype=np.float64)[:, None]
    inv = base ** (-2.0 * np.arange(64, dtype=np.float64) / DIM)
    ang = pos * inv[None, :]
    return np.concatenate([np.cos(ang), np.sin(ang)], axis=1).astype(np.float32)


def rms_norm(z, gamma, eps=EPS):
    """Per-row RMS norm of z [..., 128] times gamma [128], float64."""
    z = np.asarray(z, dtype=np.float64)
    r = 1.0 / np.sqrt(np.mean(z * z, axis=-1, keepdims=True) + eps)
    return z * r * np.asarray(gamma, dtype=np.float64)


def rope(y, cos_sin_rows):
    """Rotate the pairs (i, i + 64) of y [..., 128] by the table rows [..., 128]."""
    y = np.asarray(y, dtype=np.float64)
    cs = np.asarray(cos_sin_rows, dtype=np.float64)
    c, s = cs[..., :64], cs[..., 64:]
    a, b = y[..., :64], y[..., 64:]
    return np.concatenate([a * c - b * s, b * c + a * s], axis=-1)


def project(x, w, gamma_q, gamma_k, gamma_idx, positions, table, eps=EPS):
    """y float64 [n, 25, 128]: the rows that go to the queries and the cache.

    x: [n, d] hidden states, w: [25 * 128, d] (bf16 values as floats)."""
    z = (np.asarray(x, dtype=np.float64) @ np.asarray(w, dtype=np.float64).T).reshape(-1, HEADS, DIM)
    y = z.copy()
    cs = np.asarray(table)[np.asarray(positions)][:, None, :]
    for lo, hi, g in ((0, Q_HEADS, gamma_q), (K0, V0, gamma_k), (IDX, IDX + 1, gamma_idx)):
        y[:, lo:hi] = rope(rms_norm(z[:, lo:hi], g, eps), cs)
    return y


def cache_bytes(y32, s_enc_k, s_enc_v):
    """From fp32 rows y32 [n, 25, 128]: E4M3 queries [n, 16, 128], NVFP4 keys and
    values (codes [n, 4, 128], scales [n, 4, 8]) and E4M3 index keys [n, 128]."""
    y32 = np.asarray(y32, dtype=np.float32)
    q8 = formats.encode_e4m3(y32[:, :Q_HEADS].astype(np.float64))
    kc, ks = nvfp4.quantize(y32[:, K0:V0], s_enc_k)
    vc, vs = nvfp4.quantize(y32[:, V0:IDX], s_enc_v)
    idx = formats.encode_e4m3(y32[:, IDX].astype(np.float64))
    return dict(q8=q8, kc=kc, ks=ks, vc=vc, vs=vs, idx=idx)
