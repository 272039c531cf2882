"""Helpers shared by the GPU parity tests: oracle-side views of a workload.

Inputs come from nvfp4_kv_block_gb300.workloads (the shared seeded generator) or
from torch library routines; every expected value comes from ``oracle``.
"""

import math

import numpy as np
import torch

import oracle
from oracle import formats, layout, nvfp4


def torch_amax(wl, device):
    """Per-tensor max|x| of K and V computed with torch (not with libmsa)."""
    out = []
    for tensor in (0, 1):
        s = wl.channel_scales(tensor, device)
        m = 0.0
        for b in range(wl.n_seqs):
            for c in range(wl.n_chunks(b)):
                m = max(m, float(wl.kv_chunk(tensor, b, c, device, s).abs().max()))
        out.append(m)
    return out


class OracleSide:
    """Oracle quantisation and decode of (parts of) one workload."""

    def __init__(self, wl, device):
        self.wl, self.device = wl, device
        ak, av = torch_amax(wl, device)
        self.s_enc_k = nvfp4.tensor_encode_scale(np.float32(ak))
        self.s_enc_v = nvfp4.tensor_encode_scale(np.float32(av))
        q, qi, w = wl.queries(device)
        self.q = q.cpu().numpy()
        self.qi = qi.cpu().numpy()
        self.w = w.cpu().numpy()
        self._idx = {}

    def idx_bytes(self, b):
        if b not in self._idx:
            if len(self._idx) >= 4:  # long contexts: keep a few sequences only
                self._idx.pop(next(iter(self._idx)))
            L = self.wl.seq_lens[b]
            parts = []
            for lo in range(0, L, 1 << 16):
                x = self.wl.tokens(2, b, lo, min(L, lo + (1 << 16)), self.device).cpu().numpy()
                parts.append(formats.encode_e4m3(x.astype(np.float64)))
            self._idx[b] = np.concatenate(parts) if parts else np.zeros((0, 128), np.uint8)
        return self._idx[b]

    def kv_tokens(self, b, lo, hi):
        """Oracle NVFP4 codes/scales and FP8 operands of tokens [lo, hi) of sequence b."""
        k = self.wl.tokens(0, b, lo, hi, self.device).cpu().numpy()
        v = self.wl.tokens(1, b, lo, hi, self.device).cpu().numpy()
        kc, ks = nvfp4.quantize(k, self.s_enc_k)
        vc, vs = nvfp4.quantize(v, self.s_enc_v)
        return dict(kc=kc, ks=ks, vc=vc, vs=vs, k8=nvfp4.fp8_operand(kc, ks), v8=nvfp4.fp8_operand(vc, vs))

    def page_bytes(self, b, blk):
        """Expected (kv page, index page) bytes of logical block blk of sequence b."""
        L = self.wl.seq_lens[b]
        lo, hi = blk * 128, min(blk * 128 + 128, L)
        d = self.kv_tokens(b, lo, hi)
        idx = self.idx_bytes(b)
        kvp = np.zeros((1, layout.KV_PAGE_BYTES), dtype=np.uint8)
        ip = np.zeros((1, layout.IDX_PAGE_BYTES), dtype=np.uint8)
        for t in range(hi - lo):
            layout.write_kv_slot(kvp, 0, t, d["kc"][t], d["ks"][t], d["vc"][t], d["vs"][t])
            layout.write_index_slot(ip, 0, t, idx[lo + t])
        return kvp[0], ip[0]

    def token(self, j):
        """Oracle selection, block scores, output and max|V^| of query token j."""
        b, pos = self.wl.query_positions()[j]
        r = pos // 128
        scores = oracle.indexer.block_scores(self.qi[j], self.w[j], self.idx_bytes(b), r)
        sel = oracle.indexer.select(scores, r)
        return b, pos, sel, scores

    def attend(self, j, sel, softmax_scale):
        b, pos = self.wl.query_positions()[j]
        k8, v8 = [], []
        for blk in sel:
            lo = blk * 128
            hi = min(lo + 128, pos + 1)
            d = self.kv_tokens(b, lo, hi)
            k8.append(d["k8"])
            v8.append(d["v8"])
        k8 = np.concatenate(k8)
        v8 = np.concatenate(v8)
        out, lse = oracle.attention.attend(self.q[j], k8, v8, softmax_scale, self.s_enc_k, self.s_enc_v)
        vmax = float(np.nanmax(np.abs(formats.decode_e4m3(v8)))) / float(self.s_enc_v)
        return out, lse, vmax


def block_scores_from_workspace(ws, n_q_total, max_pages):
    """Block scores S[T, max_pages] read from an indexer workspace: the
    workspace holds four partial maxima per (token, block) after its first 256
    bytes, and the block score is their max (valid for blocks < r_j)."""
    part = ws[256: 256 + n_q_total * max_pages * 16].view(torch.float32).view(n_q_total, max_pages, 4)
    return part.cpu().numpy().max(axis=-1)


def selection_ok(gpu_sel, ora_sel, ora_scores, rel=1e-4):
    """Sets equal, or every differing block's oracle score within rel of the cut-off."""
    g, o = set(gpu_sel), set(ora_sel)
    if g == o:
        return True, []
    if len(g) != len(o) or max(g) != max(o):
        return False, sorted(g ^ o)
    recent = max(o)
    winners = [b for b in o if b != recent]
    cut = min(ora_scores[b] for b in winners)
    bad = [b for b in (g ^ o) if abs(ora_scores[b] - cut) > rel * abs(cut)]
    return not bad, sorted(g ^ o)


def softmax_scale():
    return np.float32(1.0 / math.sqrt(128))
