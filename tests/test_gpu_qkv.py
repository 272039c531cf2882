"""GPU parity of the fused QKV projection -> RMS norm -> RoPE -> FP8 query and
NVFP4 cache insertion (blog, "Reduce both data movement and resource waits")
against the oracle, through the C ABI.

  * the RoPE table equals the oracle's (both computed in float64, rounded to
    fp32) to within one fp32 ulp;
  * the rows before rounding (y_out) lie within a bound derived from the
    arithmetic: fp32 accumulation of d exact bf16 products errs by at most
    d * 2^-24 / (1 - d * 2^-24) * sum_i |x_i w_i| per projected channel, the
    RMS norm scales that by at most (1 + max|z| / rms z) * max|gamma| / rms z,
    and a RoPE pair adds two such errors; plus 1e-5 relative for the fp32
    norm and rotation;
  * the cache bytes and the FP8 queries are bit-exact against the oracle's
    quantisers applied to those same fp32 rows (where fp32 rounding decides a
    code, both sides decide from the same values), and a run without y_out
    writes identical bytes.
"""

import numpy as np
import pytest
import torch

from oracle import layout, qkv
from nvfp4_kv_block_gb300 import ops, workloads

pytestmark = pytest.mark.gpu

DEV = "cuda"
S_ENC_K, S_ENC_V = 448.0 / 8.0, 448.0 / 6.0


def _run(inp, with_y=True):
    cache = ops.KVCache(inp["n_pages"], S_ENC_K, S_ENC_V, DEV)
    table = ops.rope_table(inp["max_pos"], device=DEV)
    n = inp["x"].shape[0]
    y = torch.full((n, 25, 128), float("nan"), dtype=torch.float32, device=DEV) if with_y else None
    q8 = ops.qkv_project_insert(cache, inp["x"], inp["w"], inp["gamma_q"], inp["gamma_k"], inp["gamma_idx"],
                                table, inp["positions"], inp["slots"], y_out=y)
    torch.cuda.synchronize()
    return cache, table, q8, y


def _check_rows(inp, table, y_gpu, q8, cache, tokens):
    x = inp["x"].float().cpu().numpy().astype(np.float64)[tokens]
    w = inp["w"].float().cpu().numpy().astype(np.float64)
    pos = inp["positions"].cpu().numpy()[tokens]
    g = [inp[k].cpu().numpy() for k in ("gamma_q", "gamma_k", "gamma_idx")]
    d = x.shape[1]
    want = qkv.project(x, w, *g, pos, table.cpu().numpy())
    # the bound of the accumulation error per channel, then through norm and rope
    acc = np.abs(x) @ np.abs(w).T * (d * 2.0 ** -24 / (1 - d * 2.0 ** -24))
    acc = acc.reshape(len(tokens), 25, 128)
    z = (x @ w.T).reshape(len(tokens), 25, 128)
    yg = y_gpu[tokens]
    gmax = [np.abs(gg).max() for gg in g]
    for ti in range(len(tokens)):
        for h in range(25):
            ez = acc[ti, h].max()
            if qkv.V0 <= h < qkv.IDX:
                tol = ez
            else:
                rms = np.sqrt(np.mean(z[ti, h] ** 2) + qkv.EPS)
                gm = gmax[0] if h < 16 else gmax[1] if h < 20 else gmax[2]
                tol = 2 * gm / rms * ez * (1 + np.abs(z[ti, h]).max() / rms)
            tol += 1e-5 * np.abs(want[ti, h]).max()
            err = np.abs(yg[ti, h] - want[ti, h]).max()
            assert err <= tol, (tokens[ti], h, err, tol)
    # bytes from the GPU's own fp32 rows
    b = qkv.cache_bytes(yg, np.float32(S_ENC_K), np.float32(S_ENC_V))
    assert np.array_equal(q8[tokens], b["q8"])
    kv = cache.kv_pool.cpu().numpy()
    ip = cache.idx_pool.cpu().numpy()
    slots = inp["slots"].cpu().numpy()[tokens]
    for ti, sl in enumerate(slots):
        page, off = int(sl) // 128, int(sl) % 128
        got = layout.read_kv_slot(kv, page, off)
        for a, c in zip(got, (b["kc"][ti], b["ks"][ti], b["vc"][ti], b["vs"][ti])):
            assert np.array_equal(a, c), (tokens[ti], page, off)
        assert np.array_equal(layout.read_index_slot(ip, page, off), b["idx"][ti])


def test_rope_table_matches_oracle():
    t = ops.rope_table(70000, device=DEV).cpu().numpy()
    want = qkv.rope_table(70000)
    assert np.max(np.abs(t.astype(np.float64) - want)) <= 2.0 ** -24


@pytest.mark.parametrize("n,d", [(300, 256), (129, 64)])
def test_fused_projection_small_matches_oracle(n, d):
    inp = workloads.qkv_inputs(n, d, seed=n + d, device=DEV, max_pos=4096)
    cache, table, q8, y = _run(inp)
    y = y.cpu().numpy()
    assert np.isfinite(y).all()
    _check_rows(inp, table, y, q8.cpu().numpy(), cache, list(range(n)))
    # without the diagnostic rows: the same bytes
    cache2, _, q82, _ = _run(inp, with_y=False)
    assert torch.equal(q8, q82)
    assert torch.equal(cache.kv_pool, cache2.kv_pool) and torch.equal(cache.idx_pool, cache2.idx_pool)
    assert cache.read_status() == 0


def test_fused_projection_full_size_sampled():
    n, d = 8192, 3072
    inp = workloads.qkv_inputs(n, d, seed=7, device=DEV)
    cache, table, q8, y = _run(inp)
    rng = np.random.default_rng(3)
    tokens = sorted(set([0, 1, 127, 128, 4095, 4096, n - 1] + [int(t) for t in rng.integers(0, n, 17)]))
    _check_rows(inp, table, y.cpu().numpy(), q8.cpu().numpy(), cache, tokens)
    assert cache.read_status() == 0


def test_fused_projection_two_heads_per_cta_ragged_tail():
    # 47 token tiles x 13 head pairs: the two-heads-per-CTA tile, with a last
    # tile of 112 tokens (rows past the input read as zeros and are not stored)
    n, d = 6000, 512
    inp = workloads.qkv_inputs(n, d, seed=11, device=DEV)
    cache, table, q8, y = _run(inp)
    rng = np.random.default_rng(5)
    tokens = sorted(set([0, 127, 128, 5887, 5888, 5950, n - 1] + [int(t) for t in rng.integers(0, n, 13)]))
    _check_rows(inp, table, y.cpu().numpy(), q8.cpu().numpy(), cache, tokens)
    assert cache.read_status() == 0

