"""Pins for the oracle's QKV projection, RMS norm, RoPE and cache bytes (CPU only)."""

import math

import numpy as np

from oracle import formats, layout, nvfp4, qkv


def test_one_hot_states_select_weight_rows():
    rng = np.random.default_rng(0)
    d = 64
    w = rng.integers(-8, 8, (qkv.HEADS * 128, d)).astype(np.float64)
    x = np.zeros((3, d))
    x[0, 5] = 1.0
    x[1, 0] = 2.0
    x[2, 63] = -1.0
    table = qkv.rope_table(4)
    g = np.ones(128)
    y = qkv.project(x, w, g, g, g, [0, 0, 0], table)
    # value heads are not normalised or rotated: exactly the selected column
    assert np.array_equal(y[0, qkv.V0:qkv.IDX].reshape(-1), w[qkv.V0 * 128:qkv.IDX * 128, 5])
    assert np.array_equal(y[1, qkv.V0:qkv.IDX].reshape(-1), 2 * w[qkv.V0 * 128:qkv.IDX * 128, 0])
    assert np.array_equal(y[2, qkv.V0:qkv.IDX].reshape(-1), -w[qkv.V0 * 128:qkv.IDX * 128, 63])


def test_constant_head_normalises_to_its_gain():
    gamma = np.linspace(0.5, 1.5, 128)
    for c in (3.0, -0.25, 1e3):
        y = qkv.rms_norm(np.full(128, c), gamma, eps=0.0)
        assert np.allclose(y, math.copysign(1.0, c) * gamma, rtol=1e-15)
    # eps only matters next to zero: an all-zero head stays zero
    assert not qkv.rms_norm(np.zeros(128), gamma).any()


def test_rope_table_closed_forms():
    t = qkv.rope_table(300)
    # position 0: cos 1, sin 0 (the identity)
    assert np.all(t[0, :64] == 1.0) and np.all(t[0, 64:] == 0.0)
    # pair 0 turns by exactly pos radians, pair 32 by pos / 100 (base 10,000)
    for p in (1, 7, 299):
        assert t[p, 0] == np.float32(math.cos(p)) and t[p, 64] == np.float32(math.sin(p))
        assert t[p, 32] == np.float32(math.cos(p / 100)) and t[p, 96] == np.float32(math.sin(p / 100))
    # every entry is a unit vector up to fp32 rounding
    assert np.allclose(t[:, :64].astype(np.float64) ** 2 + t[:, 64:].astype(np.float64) ** 2, 1.0, atol=1e-6)


def test_rope_keeps_pair_norms_and_position_zero_is_identity():
    rng = np.random.default_rng(1)
    y = rng.standard_normal((5, 128))
    t = qkv.rope_table(1000)
    r = qkv.rope(y, t[[0, 3, 17, 500, 999]])
    assert np.array_equal(r[0], y[0])
    n0 = y[:, :64] ** 2 + y[:, 64:] ** 2
    n1 = r[:, :64] ** 2 + r[:, 64:] ** 2
    assert np.allclose(n0, n1, rtol=1e-6)
    # a quarter turn of pair 0 at position pi/2 ~ 2: (a, b) -> about (-b, a) only when cos 0; check pos 0 pair
    # mapping sign conventions at a hand-picked angle: cos = 0.6, sin = 0.8
    cs = np.zeros(128)
    cs[:64], cs[64:] = 0.6, 0.8
    out = qkv.rope(np.r_[np.full(64, 1.0), np.full(64, 2.0)], cs)
    assert np.allclose(out[:64], 1.0 * 0.6 - 2.0 * 0.8) and np.allclose(out[64:], 2.0 * 0.6 + 1.0 * 0.8)


def test_cache_bytes_follow_the_pinned_codecs():
    rng = np.random.default_rng(2)
    y32 = (rng.standard_normal((6, qkv.HEADS, 128)) * 2).astype(np.float32)
    b = qkv.cache_bytes(y32, 448 / 8, 448 / 9)
    assert np.array_equal(b["q8"], formats.encode_e4m3(y32[:, :16].astype(np.float64)))
    kc, ks = nvfp4.quantize(y32[:, 16:20], 448 / 8)
    assert np.array_equal(b["kc"], kc) and np.array_equal(b["ks"], ks)
    # the codes decode back within the E2M1 spacing
    deq = nvfp4.dequantize(b["vc"], b["vs"], np.float32(448 / 9))
    assert np.max(np.abs(deq - y32[:, 20:24])) <= np.max(np.abs(y32[:, 20:24])) * 0.17 + 1e-6
    # slot bytes as the page layout places them
    pool = np.zeros((1, layout.KV_PAGE_BYTES), dtype=np.uint8)
    layout.write_kv_slot(pool, 0, 5, b["kc"][0], b["ks"][0], b["vc"][0], b["vs"][0])
    got = layout.read_kv_slot(pool, 0, 5)
    assert all(np.array_equal(a, c) for a, c in zip(got, (b["kc"][0], b["ks"][0], b["vc"][0], b["vs"][0])))
