"""Seeded synthetic workloads of the decode path (inputs only, no method arithmetic).

This module is the one piece shared by the CUDA path and the CPU oracle: it
draws the fp32 K/V/index-key values, the FP8 queries (torch's own E4M3 cast),
the head weights and the paged metadata.  It quantises nothing and scores
nothing.

Distributions (the pages give none): K and V are N(0, 1) times a per-(KV head,
channel) log-normal scale exp(N(0, 0.5^2)), one scale set per tensor; the
long-context workload multiplies 1% of the (head, channel) pairs by 20.  Index
keys, queries and index queries are N(0, 1); head weights are U(0, 1).

Every chunk of CHUNK tokens of every sequence has its own seed, so any page can
be regenerated alone (on the device that generated it first: CUDA and CPU
random streams differ).
"""

import math
from dataclasses import dataclass, field

import numpy as np
import torch

PAGE_TOKENS = 128
KV_HEADS = 4
HEAD_DIM = 128
IDX_DIM = 128
IDX_HEADS = 8
Q_HEADS = 16
CHUNK = 8192  # tokens per seeded chunk

_K, _V, _IDX, _Q, _QI, _W, _META, _SCALE = range(8)


def _seed(*parts):
    return int(np.random.SeedSequence([int(p) for p in parts]).generate_state(1, np.uint64)[0] >> 1)


def _gen(device, *parts):
    g = torch.Generator(device=device)
    g.manual_seed(_seed(*parts))
    return g


@dataclass(frozen=True)
class Workload:
    name: str
    seq_lens: tuple
    n_q: tuple
    seed: int
    outliers: bool = False
    permuted: bool = False
    description: str = field(default="", compare=False)

    @property
    def n_seqs(self):
        return len(self.seq_lens)

    @property
    def n_q_total(self):
        return int(sum(self.n_q))

    @property
    def pages_per_seq(self):
        return [math.ceil(L / PAGE_TOKENS) for L in self.seq_lens]

    @property
    def max_pages(self):
        return max(self.pages_per_seq)

    @property
    def total_pages(self):
        return int(sum(self.pages_per_seq))

    @property
    def q_start_loc(self):
        return [0] + list(np.cumsum(self.n_q).astype(int))

    def query_positions(self):
        """(seq, position) of every query token, in token order."""
        out = []
        for b, (L, n) in enumerate(zip(self.seq_lens, self.n_q)):
            out += [(b, L - n + j) for j in range(n)]
        return out

    # -- paged metadata -----------------------------------------------------------
    def block_table(self):
        """int32 [n_seqs, max_pages] physical page of every logical block (-1 = none)."""
        bt = np.full((self.n_seqs, self.max_pages), -1, dtype=np.int32)
        pages = np.arange(self.total_pages, dtype=np.int32)
        if self.permuted:
            rng = np.random.default_rng(_seed(self.seed, _META))
            pages = rng.permutation(pages).astype(np.int32)
        at = 0
        for b, n in enumerate(self.pages_per_seq):
            bt[b, :n] = pages[at:at + n]
            at += n
        return bt

    # -- tensors ------------------------------------------------------------------
    def channel_scales(self, tensor, device):
        """fp32 [4, 128] per-(head, channel) scale of K (tensor=0) or V (tensor=1)."""
        g = _gen(device, self.seed, _SCALE, tensor)
        s = torch.exp(0.5 * torch.randn((KV_HEADS, HEAD_DIM), generator=g, device=device))
        if self.outliers:
            n_out = max(1, round(0.01 * KV_HEADS * HEAD_DIM))
            idx = torch.randperm(KV_HEADS * HEAD_DIM, generator=g, device=device)[:n_out]
            s.view(-1)[idx] *= 20.0
        return s

    def n_chunks(self, b):
        return math.ceil(self.seq_lens[b] / CHUNK)

    def kv_chunk(self, tensor, b, c, device, scales=None):
        """fp32 [n, 4, 128] of K (0) or V (1) for tokens [c*CHUNK, ...) of sequence b."""
        n = min(CHUNK, self.seq_lens[b] - c * CHUNK)
        g = _gen(device, self.seed, _K if tensor == 0 else _V, b, c)
        x = torch.randn((n, KV_HEADS, HEAD_DIM), generator=g, device=device)
        if scales is None:
            scales = self.channel_scales(tensor, device)
        return x * scales

    def idx_chunk(self, b, c, device):
        """fp32 [n, 128] index keys for tokens [c*CHUNK, ...) of sequence b."""
        n = min(CHUNK, self.seq_lens[b] - c * CHUNK)
        g = _gen(device, self.seed, _IDX, b, c)
        return torch.randn((n, IDX_DIM), generator=g, device=device)

    def tokens(self, tensor, b, lo, hi, device):
        """fp32 rows of tokens [lo, hi) of sequence b: K (0), V (1) or index keys (2)."""
        out = []
        scales = self.channel_scales(tensor, device) if tensor in (0, 1) else None
        for c in range(lo // CHUNK, (hi - 1) // CHUNK + 1):
            x = self.idx_chunk(b, c, device) if tensor == 2 else self.kv_chunk(tensor, b, c, device, scales)
            s0 = max(lo, c * CHUNK) - c * CHUNK
            s1 = min(hi, (c + 1) * CHUNK) - c * CHUNK
            out.append(x[s0:s1])
        return torch.cat(out)

    def queries(self, device):
        """(q E4M3 [T,16,128] uint8, q_idx E4M3 [T,8,128] uint8, w fp32 [T,8])."""
        T = self.n_q_total
        g = _gen(device, self.seed, _Q)
        q = torch.randn((T, Q_HEADS, HEAD_DIM), generator=g, device=device)
        g = _gen(device, self.seed, _QI)
        qi = torch.randn((T, IDX_HEADS, IDX_DIM), generator=g, device=device)
        g = _gen(device, self.seed, _W)
        w = torch.rand((T, IDX_HEADS), generator=g, device=device)
        f8 = torch.float8_e4m3fn
        return q.to(f8).view(torch.uint8), qi.to(f8).view(torch.uint8), w

    # -- algorithmic bytes of one decode step (indexer + attention) ----------------
    def index_bytes(self):
        """Index pages the scan must read: blocks 0..r_last-1 of every sequence."""
        return sum(((L - 1) // PAGE_TOKENS) * PAGE_TOKENS * IDX_DIM for L in self.seq_lens if L > 0)


def _uniform_ints(seed, lo, hi, n):
    rng = np.random.default_rng(seed)
    return [int(x) for x in rng.integers(lo, hi + 1, n)]


def config(i):
    """The five workloads (index 0..4)."""
    if i == 0:
        return Workload("tiny_b1_ctx4k", (4096,), (1,), seed=0,
                        description="batch 1, 1 query token, context 4,096")
    if i == 1:
        return Workload("batched_b32_ctx32k", (32768,) * 32, (1,) * 32, seed=1,
                        description="batch 32, 1 query token each, context 32,768")
    if i == 2:
        return Workload("specverify_b16_q8_ctx128k", (131072,) * 16, (8,) * 16, seed=2,
                        description="batch 16, 8 causal query tokens each, context 131,072")
    if i == 3:
        return Workload("longctx_b4_ctx512k", (524288,) * 4, (1,) * 4, seed=3, outliers=True,
                        description="batch 4, 1 query token, context 524,288, 1% outlier channels x20")
    if i == 4:
        lens = _uniform_ints(_seed(4, 100), 30720, 215040, 64)
        nq = _uniform_ints(_seed(4, 101), 1, 8, 64)
        return Workload("ragged_64seq_ctx30k_215k", tuple(lens), tuple(nq), seed=4, permuted=True,
                        description="64 sequences, lengths U[30,720, 215,040], 1..8 query tokens, "
                                    "pages at random positions of one pool")
    raise ValueError(i)


def custom(name, seq_lens, n_q, seed, outliers=False, permuted=False):
    return Workload(name, tuple(int(x) for x in seq_lens), tuple(int(x) for x in n_q), seed,
                    outliers, permuted)


# -- fused projection inputs (synthetic weights: no trained checkpoint) -----------
QKV_HEADS = 25  # 16 query, 4 key, 4 value, 1 index-key heads of 128


def qkv_inputs(n_tokens, d_model, seed, device, max_pos=65536, n_pages=None):
    """Seeded inputs of the fused QKV projection: bf16 hidden states x [n, d]
    ~ N(0, 1), bf16 weights w [25 * 128, d] ~ N(0, 1/d), fp32 RMS-norm gains
    ~ 1 + 0.1 N(0, 1) (query, key, index key), int32 positions uniform in
    [0, max_pos), and int64 slots: distinct random slots of a pool of n_pages
    pages (default: just enough pages)."""
    g = _gen(device, seed, _META, 17)
    x = torch.randn((n_tokens, d_model), generator=g, device=device).to(torch.bfloat16)
    w = (torch.randn((QKV_HEADS * HEAD_DIM, d_model), generator=g, device=device) / math.sqrt(d_model)).to(torch.bfloat16)
    gammas = [1.0 + 0.1 * torch.randn(HEAD_DIM, generator=g, device=device) for _ in range(3)]
    positions = torch.randint(0, max_pos, (n_tokens,), generator=g, device=device, dtype=torch.int32)
    if n_pages is None:
        n_pages = max(1, math.ceil(n_tokens / PAGE_TOKENS) + 1)
    slots = torch.randperm(n_pages * PAGE_TOKENS, generator=g, device=device)[:n_tokens].to(torch.int64)
    return dict(x=x, w=w, gamma_q=gammas[0], gamma_k=gammas[1], gamma_idx=gammas[2], positions=positions,
                slots=slots, n_pages=n_pages, max_pos=max_pos)
