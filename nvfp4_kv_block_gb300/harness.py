"""Device-side set-up of a workload: fill the NVFP4 cache through the library.

Used by the tests, the benchmark and the smoke check.  Generation (workloads)
and quantisation (libmsa's kernels) run on the GPU chunk by chunk, so the fp32
K/V of a long-context workload never has to be resident at once.
"""

from dataclasses import dataclass

import torch

from . import ops
from .workloads import CHUNK, PAGE_TOKENS


@dataclass
class DeviceState:
    wl: object
    cache: ops.KVCache
    block_table: torch.Tensor  # int32 [B, max_pages]
    seq_lens: torch.Tensor     # int32 [B]
    q_start_loc: torch.Tensor  # int32 [B+1]
    amax_k: float
    amax_v: float


def _slots(bt_row, lo, n, device):
    pos = torch.arange(lo, lo + n, device=device, dtype=torch.int64)
    return bt_row[pos // PAGE_TOKENS].to(torch.int64) * PAGE_TOKENS + pos % PAGE_TOKENS


def build_state(wl, device="cuda"):
    """Quantise and insert every token of the workload; returns the device state."""
    bt = torch.from_numpy(wl.block_table()).to(device)
    amax = torch.zeros(2, dtype=torch.float32, device=device)
    sk = wl.channel_scales(0, device)
    sv = wl.channel_scales(1, device)
    for b in range(wl.n_seqs):
        for c in range(wl.n_chunks(b)):
            ops.absmax_(wl.kv_chunk(0, b, c, device, sk), amax[0:1])
            ops.absmax_(wl.kv_chunk(1, b, c, device, sv), amax[1:2])
    amax_k, amax_v = (float(x) for x in amax.cpu())
    cache = ops.KVCache(wl.total_pages, ops.encode_scale(amax_k), ops.encode_scale(amax_v), device)
    for b in range(wl.n_seqs):
        for c in range(wl.n_chunks(b)):
            k = wl.kv_chunk(0, b, c, device, sk)
            v = wl.kv_chunk(1, b, c, device, sv)
            ik = wl.idx_chunk(b, c, device)
            ops.quantize_kv_insert(cache, k, v, ik, _slots(bt[b], c * CHUNK, k.shape[0], device))
    seq_lens = torch.tensor(wl.seq_lens, dtype=torch.int32, device=device)
    qsl = torch.tensor(wl.q_start_loc, dtype=torch.int32, device=device)
    return DeviceState(wl, cache, bt, seq_lens, qsl, amax_k, amax_v)
