"""Python binding of libmsa.so: argument marshalling only.

Every step of the decode path runs in the library's CUDA kernels; this module
checks tensor dtypes, devices and shapes, passes raw pointers and the current
CUDA stream, and raises on a negative return code.  PyTorch provides device
memory and streams.  There is no fallback: if the library is missing, loading
it raises.
"""

import ctypes
import math
import os
import re

import torch

_HERE = os.path.dirname(os.path.abspath(__file__))
LIB_PATH = os.path.join(_HERE, "_lib", "libmsa.so")
HEADER = os.path.join(os.path.dirname(_HERE), "include", "msa.h")

PAGE_TOKENS = 128
KV_HEADS = 4
HEAD_DIM = 128
IDX_DIM = 128
IDX_HEADS = 8
Q_HEADS = 16
TOPK = 16
KV_PAGE_BYTES = 73_728
NOALLOC_SCRATCH_BYTES = 8 << 20  # MSA_INDEXER_NOALLOC_SCRATCH_BYTES
INJECT_BARRIER_TIMEOUT = 0x1     # MSA_INJECT_BARRIER_TIMEOUT
INJECT_ATTENTION_TIMEOUT = 0x2   # MSA_INJECT_ATTENTION_TIMEOUT
STATUS_BAD_SLOT, STATUS_BAD_PAGE, STATUS_BAD_SEQ, STATUS_BAD_SELECTION, STATUS_TIMEOUT = 0x1, 0x2, 0x4, 0x8, 0x10
IDX_PAGE_BYTES = 16_384

ERRORS = {-1: "invalid argument", -2: "unsupported shape", -3: "workspace too small",
          -4: "kernel launch failed", -5: "larger than the library's static scratch"}


class MsaError(RuntimeError):
    pass


class _Cache(ctypes.Structure):
    _fields_ = [
        ("kv_pool", ctypes.c_void_p),
        ("idx_pool", ctypes.c_void_p),
        ("n_pages", ctypes.c_int64),
        ("page_tokens", ctypes.c_int32),
        ("n_kv_heads", ctypes.c_int32),
        ("head_dim", ctypes.c_int32),
        ("idx_dim", ctypes.c_int32),
        ("s_enc_k", ctypes.c_float),
        ("s_enc_v", ctypes.c_float),
        ("status", ctypes.c_void_p),
    ]


_lib = None
_P = ctypes.c_void_p
_I32 = ctypes.c_int32
_I64 = ctypes.c_int64
_SIGS = {
    "msa_quantize_kv_insert": (ctypes.c_int, [_P, _P, _P, _P, _P, _I32, _P]),
    "msa_indexer_topk": (ctypes.c_int, [_P, _P, _P, _I32, _P, _I32, _P, _P, _I32, _I32, _I32, _P,
                                        _P, _P, ctypes.c_size_t, _P]),
    "msa_indexer_workspace_bytes": (ctypes.c_size_t, [_I32, _I32]),
    "msa_indexer_topk_noalloc": (ctypes.c_int, [_P, _P, _P, _I32, _P, _I32, _P, _P, _I32, _I32, _I32,
                                                _P, _P, _P]),
    "msa_sparse_attn_decode": (ctypes.c_int, [_P, _P, _I32, ctypes.c_float, _P, _P, _P, _I32, _P,
                                              _P, _I32, _I32, _I32, _P, _P, _P]),
    "msa_merge_splits": (ctypes.c_int, [_P, _P, _I32, _I32, _I32, _P, _P, _P]),
    "msa_debug_set_fault_injection": (ctypes.c_int, [_I32, ctypes.c_uint64]),
    "msa_pack_blocks": (ctypes.c_int, [_P, _I32, _P, _I32, _P, _P]),
    "msa_indexer_topk_range": (ctypes.c_int, [_P, _P, _P, _I32, _P, _I32, _P, _P, _I32, _I32, _I32, _I32,
                                              _I32, _P, _P, ctypes.c_size_t, _P]),
    "msa_indexer_merge_candidates": (ctypes.c_int, [_P, _P, _I32, _P, _P, _I32, _I32, _I32, _I32, _P, _P,
                                                    _P]),
    "msa_unpack_blocks": (ctypes.c_int, [_P, _I32, _P, _P, _I32, _P]),
    "msa_block_row_bytes": (ctypes.c_size_t, [_I32]),
    "msa_decode_fused": (ctypes.c_int, [_P, _P, _P, _P, _I32, _I32, ctypes.c_float, _P, _I32, _P, _P, _I32,
                                        _I32, _I32, _P, _P, _P, _P, ctypes.c_size_t, _P]),
    "msa_decode_fused_workspace_bytes": (ctypes.c_size_t, [_I32, _I32]),
    "msa_qkv_project_insert": (ctypes.c_int, [_P, _P, _P, _I32, _I32, _P, _P, _P, _P, _I32, _P, _P,
                                              ctypes.c_float, _P, _P, _P]),
    "msa_rope_table": (ctypes.c_int, [_P, _I32, ctypes.c_double, _P]),
    "msa_absmax": (ctypes.c_int, [_P, _I64, _P, _P]),
    "msa_encode_scale": (ctypes.c_float, [ctypes.c_float]),
    "msa_debug_fp8_page": (ctypes.c_int, [_P, _I64, _P, _P, _P]),
    "msa_read_status": (ctypes.c_int, [_P, _P, _P]),
    "msa_status_string": (ctypes.c_char_p, [ctypes.c_int]),
}


def lib():
    """The loaded libmsa.so (raises if it has not been built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(LIB_PATH):
            raise MsaError(f"{LIB_PATH} is missing: build it with nvfp4_kv_block_gb300.build.build()")
        l = ctypes.CDLL(LIB_PATH)
        for name, (res, args) in _SIGS.items():
            f = getattr(l, name)
            f.restype = res
            f.argtypes = args
        _lib = l
    return _lib


def header_symbols():
    """Names of the functions include/msa.h declares."""
    with open(HEADER) as f:
        text = f.read()
    return sorted(set(re.findall(r"^[A-Za-z_][\w \*]*?\b(msa_\w+)\s*\(", text, re.M)))


def _check(rc):
    if rc != 0:
        raise MsaError(f"libmsa error {rc}: {ERRORS.get(rc, 'unknown')}")


def _stream():
    return ctypes.c_void_p(torch.cuda.current_stream().cuda_stream)


def _ptr(t, dtype, name, dims=None):
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name} must be a torch tensor")
    if t.dtype != dtype:
        raise TypeError(f"{name} must be {dtype}, got {t.dtype}")
    if not t.is_cuda:
        raise ValueError(f"{name} must be a CUDA tensor")
    if not t.is_contiguous():
        raise ValueError(f"{name} must be contiguous")
    if dims is not None and t.dim() != dims:
        raise ValueError(f"{name} must have {dims} dims, got {t.dim()}")
    return ctypes.c_void_p(t.data_ptr())


class KVCache:
    """NVFP4 KV pool + FP8 index pool of n_pages 128-token pages, caller-owned."""

    def __init__(self, n_pages, s_enc_k, s_enc_v, device="cuda"):
        self.n_pages = int(n_pages)
        self.kv_pool = torch.zeros((self.n_pages, KV_PAGE_BYTES), dtype=torch.uint8, device=device)
        self.idx_pool = torch.zeros((self.n_pages, IDX_PAGE_BYTES), dtype=torch.uint8, device=device)
        self.status = torch.zeros(1, dtype=torch.int32, device=device)
        self.s_enc_k = float(s_enc_k)
        self.s_enc_v = float(s_enc_v)

    def struct(self):
        return _Cache(self.kv_pool.data_ptr(), self.idx_pool.data_ptr(), self.n_pages, PAGE_TOKENS,
                      KV_HEADS, HEAD_DIM, IDX_DIM, self.s_enc_k, self.s_enc_v,
                      self.status.data_ptr())

    def read_status(self):
        out = ctypes.c_int32(0)
        c = self.struct()
        _check(lib().msa_read_status(ctypes.byref(c), ctypes.byref(out), _stream()))
        return out.value


def encode_scale(amax):
    return lib().msa_encode_scale(float(amax))


def absmax_(x, amax):
    """Fold max|x| into the device float ``amax`` (shape [1], caller zeroed)."""
    _check(lib().msa_absmax(_ptr(x, torch.float32, "x"), x.numel(), _ptr(amax, torch.float32, "amax"),
                            _stream()))


def quantize_kv_insert(cache, k, v, idx_k, slot_mapping):
    n = k.shape[0]
    if tuple(k.shape) != (n, KV_HEADS, HEAD_DIM) or tuple(v.shape) != (n, KV_HEADS, HEAD_DIM):
        raise ValueError("k, v must be [n, 4, 128]")
    if tuple(idx_k.shape) != (n, IDX_DIM) or tuple(slot_mapping.shape) != (n,):
        raise ValueError("idx_k must be [n, 128] and slot_mapping [n]")
    c = cache.struct()
    _check(lib().msa_quantize_kv_insert(ctypes.byref(c), _ptr(k, torch.float32, "k"),
                                        _ptr(v, torch.float32, "v"), _ptr(idx_k, torch.float32, "idx_k"),
                                        _ptr(slot_mapping, torch.int64, "slot_mapping"), n, _stream()))


def indexer_workspace_bytes(n_q_total, max_pages):
    return lib().msa_indexer_workspace_bytes(int(n_q_total), int(max_pages))


def indexer_topk(cache, q_idx, w, block_table, seq_lens, q_start_loc, ws=None, sel=None,
                 n_sel=None, topk=TOPK):
    """Select blocks for every query token.  Returns (sel [T,17], n_sel [T], ws)."""
    T = q_idx.shape[0]
    if tuple(q_idx.shape) != (T, IDX_HEADS, IDX_DIM) or tuple(w.shape) != (T, IDX_HEADS):
        raise ValueError("q_idx must be [T, 8, 128] uint8 and w [T, 8] float32")
    n_seqs, max_pages = block_table.shape
    if tuple(seq_lens.shape) != (n_seqs,) or tuple(q_start_loc.shape) != (n_seqs + 1,):
        raise ValueError("seq_lens must be [B], q_start_loc [B+1]")
    dev = q_idx.device
    if ws is None:  # zeroed: its first bytes are grid-barrier words
        ws = torch.zeros(indexer_workspace_bytes(T, max_pages), dtype=torch.uint8, device=dev)
    if sel is None:
        sel = torch.empty((T, topk + 1), dtype=torch.int32, device=dev)
    if n_sel is None:
        n_sel = torch.empty((T,), dtype=torch.int32, device=dev)
    c = cache.struct()
    _check(lib().msa_indexer_topk(
        ctypes.byref(c), _ptr(q_idx, torch.uint8, "q_idx"), _ptr(w, torch.float32, "w"), IDX_HEADS,
        _ptr(block_table, torch.int32, "block_table"), max_pages, _ptr(seq_lens, torch.int32, "seq_lens"),
        _ptr(q_start_loc, torch.int32, "q_start_loc"), n_seqs, T, topk, _ptr(sel, torch.int32, "sel"),
        _ptr(n_sel, torch.int32, "n_sel"), _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream()))
    return sel, n_sel, ws


def indexer_topk_range(cache, q_idx, w, block_table, seq_lens, q_start_loc, blk_lo, blk_hi, ws=None,
                       cand=None, topk=TOPK):
    """Local top-16 keys (uint64 stored as int64, [T, 16]) of the blocks
    [blk_lo, blk_hi) of every sequence.  Returns (cand, ws)."""
    T = q_idx.shape[0]
    if tuple(q_idx.shape) != (T, IDX_HEADS, IDX_DIM) or tuple(w.shape) != (T, IDX_HEADS):
        raise ValueError("q_idx must be [T, 8, 128] uint8 and w [T, 8] float32")
    n_seqs, max_pages = block_table.shape
    dev = q_idx.device
    if ws is None:
        ws = torch.zeros(indexer_workspace_bytes(T, max_pages), dtype=torch.uint8, device=dev)
    if cand is None:
        cand = torch.empty((T, topk), dtype=torch.int64, device=dev)
    c = cache.struct()
    _check(lib().msa_indexer_topk_range(
        ctypes.byref(c), _ptr(q_idx, torch.uint8, "q_idx"), _ptr(w, torch.float32, "w"), IDX_HEADS,
        _ptr(block_table, torch.int32, "block_table"), max_pages, _ptr(seq_lens, torch.int32, "seq_lens"),
        _ptr(q_start_loc, torch.int32, "q_start_loc"), n_seqs, T, topk, int(blk_lo), int(blk_hi),
        _ptr(cand, torch.int64, "cand"), _ptr(ws, torch.uint8, "ws"), ws.numel(), _stream()))
    return cand, ws


def indexer_merge_candidates(cache, cand, seq_lens, q_start_loc, max_pages, sel=None, n_sel=None,
                             topk=TOPK):
    """Merge [n_shards, T, 16] candidate keys into (sel [T, 17], n_sel [T])."""
    n_shards, T, _ = cand.shape
    dev = cand.device
    if sel is None:
        sel = torch.empty((T, topk + 1), dtype=torch.int32, device=dev)
    if n_sel is None:
        n_sel = torch.empty((T,), dtype=torch.int32, device=dev)
    c = cache.struct()
    _check(lib().msa_indexer_merge_candidates(
        ctypes.byref(c), _ptr(cand, torch.int64, "cand"), n_shards, _ptr(seq_lens, torch.int32, "seq_lens"),
        _ptr(q_start_loc, torch.int32, "q_start_loc"), seq_lens.shape[0], int(max_pages), T, topk,
        _ptr(sel, torch.int32, "sel"), _ptr(n_sel, torch.int32, "n_sel"), _stream()))
    return sel, n_sel


def indexer_topk_noalloc(cache, q_idx, w, block_table, seq_lens, q_start_loc, sel=None,
                         n_sel=None, topk=TOPK):
    """indexer_topk through the allocation-free entry point (static scratch in the
    library).  Returns (sel [T,17], n_sel [T])."""
    T = q_idx.shape[0]
    if tuple(q_idx.shape) != (T, IDX_HEADS, IDX_DIM) or tuple(w.shape) != (T, IDX_HEADS):
        raise ValueError("q_idx must be [T, 8, 128] uint8 and w [T, 8] float32")
    n_seqs, max_pages = block_table.shape
    if tuple(seq_lens.shape) != (n_seqs,) or tuple(q_start_loc.shape) != (n_seqs + 1,):
        raise ValueError("seq_lens must be [B], q_start_loc [B+1]")
    dev = q_idx.device
    if sel is None:
        sel = torch.empty((T, topk + 1), dtype=torch.int32, device=dev)
    if n_sel is None:
        n_sel = torch.empty((T,), dtype=torch.int32, device=dev)
    c = cache.struct()
    _check(lib().msa_indexer_topk_noalloc(
        ctypes.byref(c), _ptr(q_idx, torch.uint8, "q_idx"), _ptr(w, torch.float32, "w"), IDX_HEADS,
        _ptr(block_table, torch.int32, "block_table"), max_pages, _ptr(seq_lens, torch.int32, "seq_lens"),
        _ptr(q_start_loc, torch.int32, "q_start_loc"), n_seqs, T, topk, _ptr(sel, torch.int32, "sel"),
        _ptr(n_sel, torch.int32, "n_sel"), _stream()))
    return sel, n_sel


def sparse_attn_decode(cache, q, sel, n_sel, block_table, seq_lens, q_start_loc, n_splits,
                       softmax_scale=None, o_part=None, lse_part=None):
    T = q.shape[0]
    if tuple(q.shape) != (T, Q_HEADS, HEAD_DIM):
        raise ValueError("q must be [T, 16, 128] uint8 (E4M3)")
    n_seqs, max_pages = block_table.shape
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(HEAD_DIM)
    dev = q.device
    if o_part is None:
        o_part = torch.empty((T, n_splits, Q_HEADS, HEAD_DIM), dtype=torch.float32, device=dev)
    if lse_part is None:
        lse_part = torch.empty((T, n_splits, Q_HEADS), dtype=torch.float32, device=dev)
    c = cache.struct()
    _check(lib().msa_sparse_attn_decode(
        ctypes.byref(c), _ptr(q, torch.uint8, "q"), Q_HEADS, float(softmax_scale),
        _ptr(sel, torch.int32, "sel"), _ptr(n_sel, torch.int32, "n_sel"),
        _ptr(block_table, torch.int32, "block_table"), max_pages, _ptr(seq_lens, torch.int32, "seq_lens"),
        _ptr(q_start_loc, torch.int32, "q_start_loc"), n_seqs, T, int(n_splits),
        _ptr(o_part, torch.float32, "o_part"), _ptr(lse_part, torch.float32, "lse_part"), _stream()))
    return o_part, lse_part


def merge_splits(o_part, lse_part, out=None, lse=None):
    """LSE merge of the splits: returns out [T, H, 128] (and fills lse [T, H] if given)."""
    T, S, H, D = o_part.shape
    if out is None:
        out = torch.empty((T, H, D), dtype=torch.float32, device=o_part.device)
    lse_p = ctypes.c_void_p(None) if lse is None else _ptr(lse, torch.float32, "lse")
    _check(lib().msa_merge_splits(_ptr(o_part, torch.float32, "o_part"),
                                  _ptr(lse_part, torch.float32, "lse_part"), T, H, S,
                                  _ptr(out, torch.float32, "out"), lse_p, _stream()))
    return out


def block_row_bytes(n_layers):
    return lib().msa_block_row_bytes(int(n_layers))


def _layer_array(caches):
    arr = (_Cache * len(caches))()
    for i, c in enumerate(caches):
        arr[i] = c.struct()
    return arr


def pack_blocks(caches, pages, rows=None):
    """Block-outer rows [n_blocks, n_layers * 90,112] of the physical pages
    ``pages`` (int32 [n_blocks]) from the per-layer caches."""
    n = pages.shape[0]
    if rows is None:
        rows = torch.empty((n, block_row_bytes(len(caches))), dtype=torch.uint8, device=pages.device)
    arr = _layer_array(caches)
    _check(lib().msa_pack_blocks(arr, len(caches), _ptr(pages, torch.int32, "pages", 1), n,
                                 _ptr(rows, torch.uint8, "rows"), _stream()))
    return rows


def unpack_blocks(caches, rows, pages):
    """Write block-outer rows back into pages ``pages`` of every layer's pools."""
    arr = _layer_array(caches)
    _check(lib().msa_unpack_blocks(arr, len(caches), _ptr(rows, torch.uint8, "rows"),
                                   _ptr(pages, torch.int32, "pages", 1), pages.shape[0], _stream()))


QKV_HEADS = 25  # MSA_QKV_HEADS


def rope_table(max_pos, base=10000.0, device="cuda"):
    """fp32 [max_pos, 128] RoPE cos / sin table (msa_rope_table)."""
    t = torch.empty((max_pos, 128), dtype=torch.float32, device=device)
    _check(lib().msa_rope_table(_ptr(t, torch.float32, "cos_sin"), int(max_pos), float(base), _stream()))
    return t


def qkv_project_insert(cache, x, w, gamma_q, gamma_k, gamma_idx, cos_sin, positions, slot_mapping,
                       eps=1e-6, q8=None, y_out=None):
    """Fused projection -> RMS norm -> RoPE -> FP8 queries (returned, [n, 16, 128])
    and NVFP4 / FP8 cache insertion.  ``y_out`` ([n, 25, 128] fp32) receives the
    rows before rounding when given."""
    n, d = x.shape
    if tuple(w.shape) != (QKV_HEADS * HEAD_DIM, d):
        raise ValueError("w must be [25 * 128, d_model] bf16")
    if q8 is None:
        q8 = torch.empty((n, Q_HEADS, HEAD_DIM), dtype=torch.uint8, device=x.device)
    yp = ctypes.c_void_p(None) if y_out is None else _ptr(y_out, torch.float32, "y_out")
    c = cache.struct()
    _check(lib().msa_qkv_project_insert(
        ctypes.byref(c), _ptr(x, torch.bfloat16, "x", 2), _ptr(w, torch.bfloat16, "w", 2), n, d,
        _ptr(gamma_q, torch.float32, "gamma_q"), _ptr(gamma_k, torch.float32, "gamma_k"),
        _ptr(gamma_idx, torch.float32, "gamma_idx"), _ptr(cos_sin, torch.float32, "cos_sin", 2),
        cos_sin.shape[0], _ptr(positions, torch.int32, "positions"), _ptr(slot_mapping, torch.int64, "slot_mapping"),
        float(eps), _ptr(q8, torch.uint8, "q8"), yp, _stream()))
    return q8


def set_fault_injection(flags=0, wait_limit_ns=0):
    """Test hook: wait limit of every later launch (0 = the 2 s default) and
    fault-injection flags (INJECT_BARRIER_TIMEOUT, INJECT_ATTENTION_TIMEOUT); 0, 0 restores
    the defaults."""
    _check(lib().msa_debug_set_fault_injection(int(flags), int(wait_limit_ns)))


def debug_fp8_page(cache, page):
    k8 = torch.empty((KV_HEADS, PAGE_TOKENS, HEAD_DIM), dtype=torch.uint8, device=cache.kv_pool.device)
    v8 = torch.empty_like(k8)
    c = cache.struct()
    _check(lib().msa_debug_fp8_page(ctypes.byref(c), int(page), _ptr(k8, torch.uint8, "k8"),
                                    _ptr(v8, torch.uint8, "v8"), _stream()))
    return k8, v8


def choose_splits(n_q_total, n_sms=152):
    """Splits per query token for the attention kernel.

    The attention kernel runs one persistent CTA per SM; work items are
    (token, KV head, split), dealt round-robin, each with up to
    ceil(17 / splits) pages.  The busiest CTA then streams about
    ceil(items / SMs) x (pages per item + an item overhead of about two pages);
    pick the split count that minimises that, with a small charge per split
    for the partial outputs written and merged, preferring fewer splits on ties.
    At most 4 splits (items of at least 5 pages): with a handful of tokens the
    attention's per-item start-up and the merge launch outweigh the shorter
    items (measured on 4 tokens of 512K context: 2 to 5 splits give the same
    step time, 9 add 2.5 us and 17 add 7 us).
    """
    best, best_cost = 1, None
    for s in range(1, 5):
        items = KV_HEADS * max(1, n_q_total) * s
        cost = math.ceil(items / n_sms) * (math.ceil((TOPK + 1) / s) + 2.0)
        cost *= 1.0 + 0.02 * s
        if best_cost is None or cost < best_cost - 1e-9:
            best, best_cost = s, cost
    return best


class DecodeBuffers:
    """Preallocated outputs and scratch of one decode step (reused across steps)."""

    def __init__(self, n_q_total, max_pages, n_splits, device="cuda"):
        self.T, self.n_splits = n_q_total, n_splits
        self.ws = torch.zeros(indexer_workspace_bytes(n_q_total, max_pages), dtype=torch.uint8, device=device)
        self.sel = torch.empty((n_q_total, TOPK + 1), dtype=torch.int32, device=device)
        self.n_sel = torch.empty((n_q_total,), dtype=torch.int32, device=device)
        self.o_part = torch.empty((n_q_total, n_splits, Q_HEADS, HEAD_DIM), dtype=torch.float32, device=device)
        self.lse_part = torch.empty((n_q_total, n_splits, Q_HEADS), dtype=torch.float32, device=device)
        # one split: its normalised output is already the answer (no merge launch)
        self.out = (self.o_part.view(n_q_total, Q_HEADS, HEAD_DIM) if n_splits == 1 else
                    torch.empty((n_q_total, Q_HEADS, HEAD_DIM), dtype=torch.float32, device=device))


FUSED_MAX_SEQS = 64     # limits of msa_decode_fused (low concurrency)
FUSED_MAX_TOKENS = 64


class FusedBuffers:
    """Outputs and scratch of the single-launch decode step (reused across steps)."""

    def __init__(self, n_q_total, max_pages, device="cuda"):
        self.T = n_q_total
        nbytes = lib().msa_decode_fused_workspace_bytes(int(n_q_total), int(max_pages))
        self.ws = torch.zeros(nbytes, dtype=torch.uint8, device=device)  # zeroed: barrier words
        self.sel = torch.empty((n_q_total, TOPK + 1), dtype=torch.int32, device=device)
        self.n_sel = torch.empty((n_q_total,), dtype=torch.int32, device=device)
        self.out = torch.empty((n_q_total, Q_HEADS, HEAD_DIM), dtype=torch.float32, device=device)


def decode_fused(cache, q, q_idx, w, block_table, seq_lens, q_start_loc, bufs, softmax_scale=None):
    """The decode step in one launch (scan, top-k, attention, merge) for low
    concurrency.  Returns bufs.out [T, 16, 128]; bufs.sel / bufs.n_sel hold the
    selection."""
    T = q.shape[0]
    if tuple(q.shape) != (T, Q_HEADS, HEAD_DIM) or tuple(q_idx.shape) != (T, IDX_HEADS, IDX_DIM):
        raise ValueError("q must be [T, 16, 128] and q_idx [T, 8, 128] uint8 (E4M3)")
    n_seqs, max_pages = block_table.shape
    if softmax_scale is None:
        softmax_scale = 1.0 / math.sqrt(HEAD_DIM)
    c = cache.struct()
    _check(lib().msa_decode_fused(
        ctypes.byref(c), _ptr(q, torch.uint8, "q"), _ptr(q_idx, torch.uint8, "q_idx"), _ptr(w, torch.float32, "w"),
        Q_HEADS, IDX_HEADS, float(softmax_scale), _ptr(block_table, torch.int32, "block_table"), max_pages,
        _ptr(seq_lens, torch.int32, "seq_lens"), _ptr(q_start_loc, torch.int32, "q_start_loc"), n_seqs, T, TOPK,
        _ptr(bufs.sel, torch.int32, "sel"), _ptr(bufs.n_sel, torch.int32, "n_sel"),
        _ptr(bufs.out, torch.float32, "out"), _ptr(bufs.ws, torch.uint8, "ws"), bufs.ws.numel(), _stream()))
    return bufs.out


def decode_step(cache, q, q_idx, w, block_table, seq_lens, q_start_loc, bufs, softmax_scale=None):
    """One decode step: indexer top-k, sparse attention splits, and the LSE merge
    of the splits (3 kernels; 2 with a single split, whose output is final)."""
    indexer_topk(cache, q_idx, w, block_table, seq_lens, q_start_loc, ws=bufs.ws, sel=bufs.sel,
                 n_sel=bufs.n_sel)
    sparse_attn_decode(cache, q, bufs.sel, bufs.n_sel, block_table, seq_lens, q_start_loc,
                       bufs.n_splits, softmax_scale, o_part=bufs.o_part, lse_part=bufs.lse_part)
    if bufs.n_splits > 1:
        merge_splits(bufs.o_part, bufs.lse_part, out=bufs.out)
    return bufs.out
