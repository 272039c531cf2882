"""Pins for the oracle's sparse GQA attention (CPU only)."""

import math

import numpy as np

from oracle import attention, decode, formats, indexer, nvfp4


def _naive(q8, k8, v8, scale, s_enc_k, s_enc_v):
    """Per-key Python loop with math.exp: an independent restatement of attention."""
    hq, d = q8.shape
    out = np.zeros((hq, d))
    for h in range(hq):
        g = h // 4
        q = [float(formats.decode_e4m3(b)) for b in q8[h]]
        logits = []
        for t in range(k8.shape[0]):
            k = formats.decode_e4m3(k8[t, g])
            logits.append(sum(a * b for a, b in zip(q, k)) * float(np.float32(scale)) / float(np.float32(s_enc_k)))
        m = max(logits)
        ws = [math.exp(x - m) for x in logits]
        tot = sum(ws)
        for t, wt in enumerate(ws):
            out[h] += wt / tot * formats.decode_e4m3(v8[t, g]) / float(np.float32(s_enc_v))
    return out


def _cache(rng, L):
    k = (rng.standard_normal((L, 4, 128)) * np.exp(rng.normal(0, 0.5, (1, 4, 128)))).astype(np.float32)
    v = (rng.standard_normal((L, 4, 128)) * np.exp(rng.normal(0, 0.5, (1, 4, 128)))).astype(np.float32)
    idx = rng.standard_normal((L, 128)).astype(np.float32)
    sk = nvfp4.tensor_encode_scale(np.abs(k).max())
    sv = nvfp4.tensor_encode_scale(np.abs(v).max())
    return decode.quantize_sequence(k, v, idx, sk, sv), sk, sv


def test_all_blocks_selected_equals_dense_attention():
    rng = np.random.default_rng(0)
    L = 128 * 5 + 17                       # 6 blocks <= 17: every block is selected
    cache, sk, sv = _cache(rng, L)
    q8 = formats.encode_e4m3(rng.standard_normal((1, 16, 128)))
    qi = formats.encode_e4m3(rng.standard_normal((1, 8, 128)))
    w = rng.uniform(0, 1, (1, 8)).astype(np.float32)
    scale = np.float32(1 / math.sqrt(128))
    res = decode.decode_sequence(q8, qi, w, cache, L, sk, sv, scale)[0]
    assert res["sel"] == list(range(6))
    ref = _naive(q8[0], cache["k8"][:L], cache["v8"][:L], scale, sk, sv)
    assert np.max(np.abs(res["out"] - ref)) < 1e-12


def test_one_dominant_key_returns_its_value_row():
    rng = np.random.default_rng(1)
    n = 300
    q8 = formats.encode_e4m3(np.ones((16, 128)))
    k8 = formats.encode_e4m3(rng.uniform(-0.02, 0.02, (n, 4, 128)))
    k8[123] = formats.encode_e4m3(np.full((4, 128), 8.0))  # logit 8*128*scale ~ 90 above the rest
    v8 = formats.encode_e4m3(rng.standard_normal((n, 4, 128)))
    out, _ = attention.attend(q8, k8, v8, np.float32(1 / math.sqrt(128)), 1.0, 2.0)
    for h in range(16):
        assert np.allclose(out[h], formats.decode_e4m3(v8[123, h // 4]) / 2.0, atol=1e-12)


def test_identical_keys_average_the_values():
    rng = np.random.default_rng(2)
    n = 200
    q8 = formats.encode_e4m3(rng.standard_normal((16, 128)))
    k8 = np.repeat(formats.encode_e4m3(rng.standard_normal((1, 4, 128))), n, axis=0)
    v8 = formats.encode_e4m3(rng.standard_normal((n, 4, 128)))
    out, lse = attention.attend(q8, k8, v8, 0.1, 1.0, 1.0)
    mean_v = formats.decode_e4m3(v8).mean(axis=0)
    for h in range(16):
        assert np.allclose(out[h], mean_v[h // 4], atol=1e-12)
        logit = float(formats.decode_e4m3(q8[h]) @ formats.decode_e4m3(k8[0, h // 4])) * float(np.float32(0.1))
        assert math.isclose(lse[h], logit + math.log(n), rel_tol=1e-12, abs_tol=1e-12)


def test_speculative_tokens_ignore_later_keys():
    rng = np.random.default_rng(3)
    L, n_q = 128 * 3 + 40, 8
    cache, sk, sv = _cache(rng, L)
    q8 = formats.encode_e4m3(rng.standard_normal((n_q, 16, 128)))
    qi = formats.encode_e4m3(rng.standard_normal((n_q, 8, 128)))
    w = rng.uniform(0, 1, (n_q, 8)).astype(np.float32)
    base = decode.decode_sequence(q8, qi, w, cache, L, sk, sv)
    # perturb the keys/values after token j's position: its output must not move
    j = 3
    pos = L - n_q + j
    pert = {k: v.copy() for k, v in cache.items()}
    pert["k8"][pos + 1:] ^= 0x15
    pert["v8"][pos + 1:] ^= 0x15
    again = decode.decode_sequence(q8, qi, w, pert, L, sk, sv, tokens=[j])[0]
    assert np.array_equal(again["out"], base[j]["out"])
    assert list(attention.visible_positions([0, 3], pos)) == list(range(128)) + list(range(384, pos + 1))
    # while a later token does see the perturbation
    later = decode.decode_sequence(q8, qi, w, pert, L, sk, sv, tokens=[n_q - 1])[0]
    assert not np.array_equal(later["out"], base[n_q - 1]["out"])
