"""Pins for the oracle's NVFP4 quantiser, FP8 operand and page layout (CPU only)."""

import os

import numpy as np
import pytest
import torch

from oracle import formats, layout, nvfp4

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _cases():
    cases, cur = [], None
    with open(os.path.join(GOLDEN, "nvfp4_groups.txt")) as f:
        for line in f:
            t = line.split()
            if not t or t[0].startswith("#"):
                continue
            if t[0] == "case":
                cur = {"name": t[1], "amax": float(t[2].split("=")[1])}
                cases.append(cur)
            elif t[0] == "x":
                cur["x"] = np.array([float(v) for v in t[1:]], dtype=np.float32)
            elif t[0] == "scale":
                cur["scale"] = int(t[1], 16)
            elif t[0] == "codes":
                cur["codes"] = [int(v) for v in t[1:]]
    return cases


@pytest.mark.parametrize("case", _cases(), ids=lambda c: c["name"])
def test_hand_computed_groups(case):
    s_enc = nvfp4.tensor_encode_scale(case["amax"])
    codes, scales = nvfp4.quantize(case["x"], s_enc)
    assert int(scales[0]) == case["scale"]
    assert list(codes) == case["codes"]


def test_page_byte_counts_match_the_pages():
    # 34,560 (NVFP4) vs 61,440 (FP8) bytes/token over the model's layers (ai4snews);
    # 128 index bytes vs 1,024 dense FP8 K/V bytes per token and layer (blog).
    per_token = layout.KV_PAGE_BYTES // layout.PAGE_TOKENS
    assert per_token == 576 and 34_560 % per_token == 0
    fp8_per_token = 2 * layout.KV_HEADS * layout.HEAD_DIM
    assert fp8_per_token == 1024 and 61_440 // fp8_per_token == 34_560 // per_token
    assert 1 - per_token / fp8_per_token == pytest.approx(0.4375)
    assert layout.IDX_PAGE_BYTES // layout.PAGE_TOKENS == 128
    assert 16 * layout.PAGE_TOKENS == 2048


def test_codes_agree_with_explicit_ratio_and_ml_dtypes():
    rng = np.random.default_rng(1)
    x = (rng.standard_normal((2000, 128)) * np.exp(rng.normal(0, 1.5, (2000, 1)))).astype(np.float32)
    s_enc = nvfp4.tensor_encode_scale(np.abs(x).max())
    codes, scales = nvfp4.quantize(x, s_enc)
    assert np.array_equal(codes, nvfp4.quantize_reference_ratio(x, s_enc))
    ml_dtypes = pytest.importorskip("ml_dtypes")
    sb = formats.decode_e4m3(scales)
    y = (np.abs(x) * s_enc).astype(np.float32).astype(np.float64).reshape(2000, 8, 16)
    r = np.where(sb[..., None] > 0, y / np.where(sb > 0, sb, 1)[..., None], 0)
    # only ratios exactly representable in fp32 are comparable with a float32 cast
    exact = (r.astype(np.float32).astype(np.float64) == r)
    ref = r.astype(np.float32).astype(ml_dtypes.float4_e2m1fn).view(np.uint8) & 7
    assert exact.mean() > 0.2
    assert np.array_equal((codes.reshape(2000, 8, 16) & 7)[exact], ref[exact])


def test_scale_never_exceeds_72_and_dequant_never_saturates():
    rng = np.random.default_rng(2)
    x = (rng.standard_normal((500, 128)) * 30).astype(np.float32)
    s_enc = nvfp4.tensor_encode_scale(np.abs(x).max())
    codes, scales = nvfp4.quantize(x, s_enc)
    assert formats.decode_e4m3(scales).max() <= 72
    # the exact product is at most 6 * 72 = 432, which rounds (tie to even) to 448 at most:
    # the FP8 operand is a rounding, never a saturation
    prod = formats.decode_e2m1(codes & 7).reshape(500, 8, 16) * formats.decode_e4m3(scales)[..., None]
    assert prod.max() <= 432
    assert np.abs(formats.decode_e4m3(nvfp4.fp8_operand(codes, scales))).max() <= 448


def test_round_trip_on_grid():
    # x = e2m1 * sb / s_enc with sb <= 72 and a +-6 code in every group re-quantises to itself.
    rng = np.random.default_rng(3)
    amax = np.float32(7.5)
    s_enc = nvfp4.tensor_encode_scale(amax)
    sb_choices = formats.decode_e4m3(np.arange(0x30, 0x6A))    # 0.5 .. 72
    for _ in range(200):
        sb = rng.choice(sb_choices)
        codes = rng.integers(0, 16, 16)
        codes[rng.integers(0, 16)] = rng.choice([7, 15])
        x = (formats.decode_e2m1(codes) * sb / np.float64(s_enc)).astype(np.float32)
        if not np.all(x.astype(np.float64) * np.float64(s_enc) == formats.decode_e2m1(codes) * sb):
            continue  # only groups whose fp32 image is exact
        c2, s2 = nvfp4.quantize(x, s_enc)
        want = np.where((codes & 7) == 0, 0, codes)
        assert int(s2[0]) == int(formats.encode_e4m3(sb)) and np.array_equal(c2, want)


def test_error_bound_of_e2m1_rounding():
    # For |x|*s_enc <= 6*sb the error is at most half the E2M1 spacing at |x|:
    # 0.25 below 2, 0.5 below 4, 1 below 6 (times sb / s_enc).
    rng = np.random.default_rng(4)
    x = (rng.standard_normal((3000, 128)) * np.exp(rng.normal(0, 1, (1, 128)))).astype(np.float32)
    s_enc = nvfp4.tensor_encode_scale(np.abs(x).max())
    codes, scales = nvfp4.quantize(x, s_enc)
    xh = nvfp4.dequantize(codes, scales, s_enc).reshape(3000, 8, 16)
    sb = formats.decode_e4m3(scales)[..., None]
    r = np.abs(x.astype(np.float64)).reshape(3000, 8, 16) * np.float64(s_enc) / np.where(sb > 0, sb, 1)
    half = np.where(r <= 2, 0.25, np.where(r <= 4, 0.5, 1.0))
    inside = (r <= 6) & (sb > 0)
    err = np.abs(x.reshape(3000, 8, 16) - xh) * np.float64(s_enc) / np.where(sb > 0, sb, 1)
    assert np.all(err[inside] <= half[inside] * (1 + 1e-6))


def test_fp8_operand_is_rounded_product():
    rng = np.random.default_rng(5)
    codes = rng.integers(0, 16, (400, 128)).astype(np.uint8)
    scales = rng.integers(0, 0x6A, (400, 8)).astype(np.uint8)
    got = nvfp4.fp8_operand(codes, scales)
    prod = (formats.decode_e2m1(codes & 7).reshape(400, 8, 16) * formats.decode_e4m3(scales)[..., None]).reshape(400, 128)
    ref = torch.from_numpy(prod.astype(np.float32)).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ref = np.where((ref & 0x7F) == 0, 0, ref)  # sign is added separately below
    assert np.array_equal(got & 0x7F, ref)
    assert np.array_equal(got >> 7, (codes >> 3) & 1)
    # a rounding case: 1.5 * 1.125 = 1.6875 -> 1.625 or 1.75 -> ties to even (1.75 = 0x3E? no: 1.625=0x3D, 1.75=0x3E)
    assert nvfp4.fp8_operand(np.array([3] + [0] * 15), np.array([0x39]))[0] == 0x3E


def test_layout_hand_offsets():
    pool = np.zeros((1, layout.KV_PAGE_BYTES), dtype=np.uint8)
    ipool = np.zeros((1, layout.IDX_PAGE_BYTES), dtype=np.uint8)
    kc = np.arange(4 * 128).reshape(4, 128) % 16
    ks = (np.arange(32).reshape(4, 8) + 1).astype(np.uint8)
    vc = (np.arange(4 * 128).reshape(4, 128) * 7) % 16
    vs = (np.arange(32).reshape(4, 8) + 100).astype(np.uint8)
    key = np.arange(128, dtype=np.uint8)
    with open(os.path.join(GOLDEN, "layout_bytes.txt")) as f:
        rows = [l.split() for l in f if l.strip() and not l.startswith("#")]
    for what, head, tok, el, off, *bits in rows:
        tok, el, off = int(tok), int(el), int(off)
        pool[:] = 0
        ipool[:] = 0
        layout.write_kv_slot(pool, 0, tok, kc, ks, vc, vs)
        layout.write_index_slot(ipool, 0, tok, key)
        if what == "idx":
            assert ipool[0, off] == key[el]
            continue
        g = int(head)
        if what in ("kcode", "vcode"):
            c = kc if what == "kcode" else vc
            shift, sign_off, sign_bit = (int(x) for x in bits)
            assert (pool[0, off] >> shift) & 7 == c[g, el] & 7
            assert (pool[0, sign_off] >> sign_bit) & 1 == c[g, el] >> 3
        else:
            s = ks if what == "kscale" else vs
            assert pool[0, off] == s[g, el]
    # read-back inverts the writes
    pool[:] = 0
    layout.write_kv_slot(pool, 0, 77, kc, ks, vc, vs)
    for a, b in zip(layout.read_kv_slot(pool, 0, 77), (kc, ks, vc, vs)):
        assert np.array_equal(a, b)
    layout.write_index_slot(ipool, 0, 77, key)
    assert np.array_equal(layout.read_index_slot(ipool, 0, 77), key)
