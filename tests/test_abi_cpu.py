"""C-ABI checks that need no GPU: the library builds, loads and exports every
symbol include/msa.h declares; host-side validation rejects bad arguments
before any CUDA call; host helpers agree with the oracle."""

import ctypes
import os

import numpy as np
import pytest

from nvfp4_kv_block_gb300 import build, ops
from oracle import nvfp4


@pytest.fixture(scope="module")
def lib():
    if not os.path.exists(ops.LIB_PATH):
        build.build()
    return ops.lib()


def test_header_declares_the_boundary():
    names = ops.header_symbols()
    for required in ("msa_quantize_kv_insert", "msa_indexer_topk", "msa_sparse_attn_decode",
                     "msa_merge_splits", "msa_indexer_workspace_bytes"):
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    for name in ops.header_symbols():
        assert hasattr(lib, name), name


def test_encode_scale_matches_oracle(lib):
    rng = np.random.default_rng(0)
    for a in list(rng.uniform(1e-3, 1e3, 500)) + [1.0, 448.0, 3.0, 7.7]:
        assert ops.encode_scale(a) == float(nvfp4.tensor_encode_scale(np.float32(a)))
    assert ops.encode_scale(0.0) == 1.0


def test_workspace_bytes(lib):
    assert ops.indexer_workspace_bytes(32, 256) == 256 + 32 * 256 * 16
    assert ops.indexer_workspace_bytes(3, 5) % 256 == 0 and ops.indexer_workspace_bytes(3, 5) >= 60


def _cache(**kw):
    c = ops._Cache(1, 1, 1, 128, 4, 128, 128, 1.0, 1.0, 0)
    for k, v in kw.items():
        setattr(c, k, v)
    return c


def test_host_validation_needs_no_gpu(lib):
    P = ctypes.c_void_p
    fake = P(16)  # never dereferenced: validation fails first
    assert lib.msa_quantize_kv_insert(None, fake, fake, fake, fake, 1, None) == -1
    bad_shape = _cache(head_dim=64)
    assert lib.msa_quantize_kv_insert(ctypes.byref(bad_shape), fake, fake, fake, fake, 1, None) == -2
    c = _cache()
    assert lib.msa_quantize_kv_insert(ctypes.byref(c), fake, fake, fake, fake, -1, None) == -1
    # 7 indexer heads, topk 8, too many sequences, tiny workspace
    args = [fake, fake, 8, fake, 4, fake, fake, 1, 1, 16, fake, fake, fake, 1 << 20, None]
    a = list(args); a[2] = 7
    assert lib.msa_indexer_topk(ctypes.byref(c), *a) == -2
    a = list(args); a[9] = 8
    assert lib.msa_indexer_topk(ctypes.byref(c), *a) == -2
    a = list(args); a[7] = 5000
    assert lib.msa_indexer_topk(ctypes.byref(c), *a) == -2
    a = list(args); a[13] = 8
    assert lib.msa_indexer_topk(ctypes.byref(c), *a) == -3
    nan_scale = _cache(s_enc_v=float("nan"))
    assert lib.msa_indexer_topk(ctypes.byref(nan_scale), *args) == -1
    attn = [fake, 16, 0.1, fake, fake, fake, 4, fake, fake, 1, 1, 4, fake, fake, None]
    a = list(attn); a[1] = 8
    assert lib.msa_sparse_attn_decode(ctypes.byref(c), *a) == -2
    a = list(attn); a[11] = 0
    assert lib.msa_sparse_attn_decode(ctypes.byref(c), *a) == -1
    a = list(attn); a[11] = 65
    assert lib.msa_sparse_attn_decode(ctypes.byref(c), *a) == -1
    assert lib.msa_merge_splits(fake, fake, 1, 16, 0, fake, None, None) == -1
    assert lib.msa_debug_fp8_page(ctypes.byref(c), 5, fake, fake, None) == -1
    assert lib.msa_status_string(-3) == b"workspace too small"
    assert lib.msa_status_string(0x10) == b"device: a bounded wait timed out; results invalid"
    assert lib.msa_status_string(0x8) == b"device: selected block outside 0..r_j"
    assert lib.msa_merge_splits(fake, fake, 1, 2000, 2, fake, None, None) == -2


def test_block_rows_validation_needs_no_gpu(lib):
    P = ctypes.c_void_p
    fake = P(16)
    c = _cache()
    assert lib.msa_block_row_bytes(20) == 20 * 90_112 and lib.msa_block_row_bytes(0) == 0
    assert lib.msa_pack_blocks(ctypes.byref(c), 0, fake, 1, fake, None) == -1
    assert lib.msa_pack_blocks(ctypes.byref(c), 129, fake, 1, fake, None) == -2
    assert lib.msa_pack_blocks(ctypes.byref(c), 1, fake, 1, P(17), None) == -1  # unaligned rows
    bad = _cache(head_dim=64)
    assert lib.msa_unpack_blocks(ctypes.byref(bad), 1, fake, fake, 1, None) == -2


def test_fault_injection_settings_are_validated_on_the_host(lib):
    assert lib.msa_debug_set_fault_injection(0x100, 0) == -1
    assert lib.msa_debug_set_fault_injection(ops.INJECT_BARRIER_TIMEOUT, 1000) == 0
    assert lib.msa_debug_set_fault_injection(ops.INJECT_ATTENTION_TIMEOUT, 1000) == 0
    assert lib.msa_debug_set_fault_injection(ops.INJECT_BARRIER_TIMEOUT | ops.INJECT_ATTENTION_TIMEOUT, 1000) == 0
    assert lib.msa_debug_set_fault_injection(0x4, 0) == -1
    assert lib.msa_debug_set_fault_injection(0, 0) == 0


def test_noalloc_entry_point_rejects_shapes_beyond_its_scratch(lib):
    # 16 bytes of scratch per (query token, block): 16 tokens x 65,536 blocks needs
    # 16 MiB, beyond the 8 MiB static array; rejected before any CUDA call
    P = ctypes.c_void_p
    fake = P(16)
    c = _cache()
    assert 16 * 65536 * 16 > ops.NOALLOC_SCRATCH_BYTES
    rc = lib.msa_indexer_topk_noalloc(ctypes.byref(c), fake, fake, 8, fake, 65536, fake, fake, 1, 16,
                                      16, fake, fake, None)
    assert rc == -5
    assert lib.msa_status_string(-5) == b"larger than the library's static scratch"
    # the largest shape of the workloads here fits: 297 tokens x 1,680 blocks
    assert ops.indexer_workspace_bytes(297, 1680) <= ops.NOALLOC_SCRATCH_BYTES
