"""GPU parity of the attention's softmax under logits built to stress its
reference maximum.

The attention kernel keeps, per query head, a reference m and writes
P = 256 * 2^(x - m) as FP8; m moves (with a rescale of the row sums and of the
O accumulator in tensor memory) only when a row exceeds it by more than 0.75
in log2 units.  Random keys move it about twice per 17-page item; here the
keys of each KV head are aligned with its four query heads and scaled per
page, so that:
  * growing:  the logits rise by ~2.9 log2 units per page (a rescale on
    every page of the item),
  * jump:     the last page lies ~160 log2 units above the rest (the earlier
    pages' weight underflows to zero),
  * falling:  the first page holds the maximum (no rescale after it).
Inputs are seeded and synthetic; the expected output is the oracle's exact
attention (float64) over the oracle's own NVFP4 -> FP8 operands of the same
fp32 keys and values; the cache is written by the library's insert, whose
bytes the insert parity test pins to the oracle.
"""

import numpy as np
import pytest
import torch

import oracle
from oracle import formats, nvfp4
from nvfp4_kv_block_gb300 import ops

pytestmark = pytest.mark.gpu

DEV = "cuda"
ATOL_REL = 2e-3
N_BLOCKS = 18  # blocks 0..17; the query token sits at the last position (block 17 is full)
SOFTMAX_SCALE = 1.0 / np.sqrt(128.0)


def _inputs(kind, seed):
    rng = np.random.default_rng(seed)
    T = N_BLOCKS * 128
    q8 = formats.encode_e4m3(rng.standard_normal((16, 128)))
    qd = formats.decode_e4m3(q8)
    page = np.arange(T) // 128
    if kind == "growing":
        a = 0.35 * page
    elif kind == "jump":
        a = np.where(page == N_BLOCKS - 1, 20.0, 0.2)
    else:  # falling
        a = 0.35 * (N_BLOCKS - 1 - page)
    k = 0.3 * rng.standard_normal((T, 4, 128))
    for g in range(4):
        d = qd[4 * g:4 * g + 4].sum(0)
        d = d / np.linalg.norm(d)
        k[:, g, :] += a[:, None] * np.sqrt(128.0) * d[None, :]
    v = rng.standard_normal((T, 4, 128))
    idx = rng.standard_normal((T, 128))
    return q8, k.astype(np.float32), v.astype(np.float32), idx.astype(np.float32)


@pytest.mark.parametrize("kind", ["growing", "jump", "falling"])
@pytest.mark.parametrize("n_splits", [1, 2, 64])
def test_reference_max_softmax_matches_oracle(kind, n_splits):
    q8, k, v, idx = _inputs(kind, seed={"growing": 11, "jump": 12, "falling": 13}[kind])
    T = k.shape[0]
    # per-tensor scales: the oracle's encoding of max|x| (the library's insert
    # uses the same definition; both take the fp32 maximum)
    s_enc_k = nvfp4.tensor_encode_scale(np.float32(np.abs(k).max()))
    s_enc_v = nvfp4.tensor_encode_scale(np.float32(np.abs(v).max()))
    cache = ops.KVCache(N_BLOCKS, float(s_enc_k), float(s_enc_v), DEV)
    ops.quantize_kv_insert(cache, torch.from_numpy(k).to(DEV), torch.from_numpy(v).to(DEV),
                           torch.from_numpy(idx).to(DEV), torch.arange(T, dtype=torch.int64, device=DEV))
    # selection: blocks 1..16, then the recent block 17
    blocks = list(range(1, 17)) + [17]
    sel = torch.full((1, 17), -1, dtype=torch.int32, device=DEV)
    sel[0, :] = torch.tensor(blocks, dtype=torch.int32)
    n_sel = torch.tensor([17], dtype=torch.int32, device=DEV)
    bt = torch.arange(N_BLOCKS, dtype=torch.int32, device=DEV).view(1, N_BLOCKS)
    seq_lens = torch.tensor([T], dtype=torch.int32, device=DEV)
    qsl = torch.tensor([0, 1], dtype=torch.int32, device=DEV)
    q = torch.from_numpy(q8).to(DEV).view(1, 16, 128)
    o_part, lse_part = ops.sparse_attn_decode(cache, q, sel, n_sel, bt, seq_lens, qsl, n_splits,
                                              softmax_scale=SOFTMAX_SCALE)
    lse = torch.empty((1, 16), dtype=torch.float32, device=DEV)
    out = ops.merge_splits(o_part, lse_part, lse=lse)[0].cpu().numpy()
    lse = lse[0].cpu().numpy()
    assert cache.read_status() == 0
    # oracle: exact attention over the FP8 operands of the selected tokens
    toks = np.concatenate([np.arange(b * 128, b * 128 + 128) for b in blocks])
    kc, ks = nvfp4.quantize(k[toks], s_enc_k)
    vc, vs = nvfp4.quantize(v[toks], s_enc_v)
    k8, v8 = nvfp4.fp8_operand(kc, ks), nvfp4.fp8_operand(vc, vs)
    ref, ref_lse = oracle.attention.attend(q8, k8, v8, SOFTMAX_SCALE, s_enc_k, s_enc_v)
    vmax = float(np.max(np.abs(formats.decode_e4m3(v8)))) / float(s_enc_v)
    err = np.max(np.abs(out - ref))
    assert err <= ATOL_REL * vmax, (kind, n_splits, err, vmax)
    assert np.allclose(lse, ref_lse, rtol=1e-5, atol=1e-4), (kind, n_splits, lse - ref_lse)
    if kind == "jump":
        # the last block carries (almost) all the weight
        last = np.arange(17 * 128, 18 * 128)
        kc2, ks2 = nvfp4.quantize(k[last], s_enc_k)
        vc2, vs2 = nvfp4.quantize(v[last], s_enc_v)
        ref_last, _ = oracle.attention.attend(q8, nvfp4.fp8_operand(kc2, ks2), nvfp4.fp8_operand(vc2, vs2),
                                              SOFTMAX_SCALE, s_enc_k, s_enc_v)
        assert np.max(np.abs(out - ref_last)) <= ATOL_REL * vmax
