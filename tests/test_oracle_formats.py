"""Pins for the oracle's E2M1 / E4M3 codecs (CPU only)."""

import os

import numpy as np
import pytest
import torch

from oracle import formats

GOLDEN = os.path.join(os.path.dirname(__file__), "golden")


def _rows(name):
    with open(os.path.join(GOLDEN, name)) as f:
        return [l.split() for l in f if l.strip() and not l.startswith("#")]


def test_e2m1_table_matches_hand_table():
    for code, val in _rows("e2m1_codes.txt"):
        got = formats.decode_e2m1(int(code))
        assert got == float(val) and np.signbit(got) == val.startswith("-")


def test_e4m3_landmarks_match_hand_table():
    for byte, val in _rows("e4m3_landmarks.txt"):
        got = formats.decode_e4m3(int(byte, 16))
        if val == "nan":
            assert np.isnan(got)
        else:
            assert got == float(val)


def test_e4m3_decode_all_bytes_matches_torch():
    b = torch.arange(256, dtype=torch.uint8)
    ref = b.view(torch.float8_e4m3fn).to(torch.float64).numpy()
    got = formats.decode_e4m3(np.arange(256))
    both_nan = np.isnan(ref) & np.isnan(got)
    assert np.all(both_nan | (ref == got))


def test_e4m3_encode_matches_torch_cast_on_sweep():
    rng = np.random.default_rng(123)
    x = np.concatenate([
        rng.standard_normal(400_000) * 10.0 ** rng.uniform(-4, 2.6, 400_000),
        rng.uniform(-448, 448, 200_000),
        rng.uniform(-0.02, 0.02, 200_000),
    ]).astype(np.float32)
    x = x[np.abs(x) <= 448]  # torch maps overflow to NaN; saturation is pinned separately
    ref = torch.from_numpy(x).to(torch.float8_e4m3fn).view(torch.uint8).numpy()
    ref = np.where((ref & 0x7F) == 0, 0, ref)  # canonical zero: no negative zero
    got = formats.encode_e4m3(x.astype(np.float64))
    assert np.array_equal(got, ref)


def test_e4m3_encode_ties_go_to_even_code():
    pos = formats.decode_e4m3(np.arange(127))
    mids = 0.5 * (pos[:-1] + pos[1:])
    got = formats.encode_e4m3(mids)
    lo = np.arange(126)
    want = np.where(lo % 2 == 0, lo, lo + 1)
    assert np.array_equal(got, want)
    assert np.array_equal(formats.encode_e4m3(-mids), np.where(want == 0, 0, want | 0x80))


def test_e4m3_encode_saturates_and_nan():
    got = formats.encode_e4m3(np.array([448.0, 460.0, 470.0, 1e9, np.inf, -np.inf, -1e9, np.nan]))
    assert list(got) == [0x7E, 0x7E, 0x7E, 0x7E, 0x7E, 0xFE, 0xFE, 0x7F]


def test_e4m3_encode_round_trips_every_finite_byte():
    b = np.array([i for i in range(256) if i not in (0x7F, 0xFF, 0x80)])
    assert np.array_equal(formats.encode_e4m3(formats.decode_e4m3(b)), b)


def test_e2m1_magnitude_midpoints_and_saturation():
    r = np.array([0.0, 0.25, 0.26, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0, 5.01, 6.0, 7.0, 100.0])
    want = [0, 0, 1, 2, 2, 4, 4, 6, 6, 7, 7, 7, 7]
    assert list(formats.encode_e2m1_magnitude(r)) == want


def test_e2m1_magnitude_matches_ml_dtypes():
    ml_dtypes = pytest.importorskip("ml_dtypes")
    rng = np.random.default_rng(7)
    r = np.concatenate([rng.uniform(0, 8, 200_000), formats.E2M1_MIDS, formats.E2M1_MAGS]).astype(np.float32)
    ref = r.astype(ml_dtypes.float4_e2m1fn).view(np.uint8) & 7
    got = formats.encode_e2m1_magnitude(r.astype(np.float64))
    assert np.array_equal(got, ref)


def test_e4m3_encode_matches_ml_dtypes():
    ml_dtypes = pytest.importorskip("ml_dtypes")
    rng = np.random.default_rng(9)
    x = (rng.standard_normal(300_000) * 10.0 ** rng.uniform(-4, 2.6, 300_000)).astype(np.float32)
    x = x[np.abs(x) <= 448]
    ref = x.astype(ml_dtypes.float8_e4m3fn).view(np.uint8)
    ref = np.where((ref & 0x7F) == 0, 0, ref)
    assert np.array_equal(formats.encode_e4m3(x.astype(np.float64)), ref)
