"""Benchmark of the NVFP4 block-sparse attention decode step on GB300.

One step = indexer (block scores + top-16/recent selection, one cooperative
launch) + split sparse attention + LSE merge of the splits (skipped when there
is one split: its output is final) over one batch of resident query tokens.  Prints ONE JSON line (rank 0).

  python bench.py [--gpus N] [--steps K] [--warmup W] [--config I] [--impl gb300|reference]

The default workload is the largest single-GPU one (--config 4: 64 ragged
sequences of 30,720-215,040 tokens with 1-8 query tokens each, pages at random
pool positions); --config 0..3 run the tiny, batched, speculative-verify and
512K long-context workloads.

--impl reference times the CPU oracle (the plain float64 restatement of the
method; there is no other reference implementation) on a bounded sample of
the same workload on this host's cores.
Multi-GPU (torchrun): every rank runs an independent replica of the workload
(replicas only: the path has no exchange step); the time is the max over ranks.
"""

import argparse
import dataclasses
import hashlib
import json
import math
import os
import subprocess
import sys
import time

import numpy as np
import torch

ROOT = os.path.dirname(os.path.abspath(__file__))
sys.path.insert(0, ROOT)

from nvfp4_kv_block_gb300 import harness, ops, workloads  # noqa: E402

ROOFLINE_NOMINAL_GBS = 8000.0
L2_FLUSH_BYTES = 512 << 20


def measured_peaks():
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            d = json.load(f)
        return float(d["hbm_gbs"]), "measured"
    return 6800.0, "fallback"


def measured_bf16_peak():
    """Dense bf16 tensor TFLOP/s measured on this machine (burst: a kernel timed alone)."""
    p = os.path.join(ROOT, "MEASURED_PEAKS.json")
    if os.path.exists(p):
        with open(p) as f:
            return float(json.load(f)["bf16_tflops"]), "measured"
    return 1900.0, "fallback"


def kernel_source_hash():
    """Hash of the indexer kernel's sources (its DRAM counters go stale when they change)."""
    h = hashlib.sha256()
    csrc = os.path.join(ROOT, "nvfp4_kv_block_gb300", "csrc")
    for f in ("common.cuh", "indexer.cu"):
        with open(os.path.join(csrc, f), "rb") as fh:
            h.update(f.encode() + fh.read())
    return h.hexdigest()[:16]


def committed_traffic(config_name):
    """DRAM bytes per indexer launch from the committed ncu summary
    (profiles/indexer_traffic.txt: lines "workload source_hash bytes"), if it
    was taken on the current kernel sources (else None)."""
    p = os.path.join(ROOT, "profiles", "indexer_traffic.txt")
    if not os.path.exists(p):
        return None
    with open(p) as f:
        for line in f:
            parts = line.split()
            if len(parts) == 3 and not line.startswith("#") and parts[0] == config_name:
                return float(parts[2]) if parts[1] == kernel_source_hash() else None
    return None


class ClockSampler:
    FIELDS = ("index,clocks.sm,clocks.max.sm,power.draw,clocks_event_reasons.active,"
              "clocks_event_reasons.hw_slowdown,clocks_event_reasons.hw_thermal_slowdown,"
              "clocks_event_reasons.sw_thermal_slowdown,clocks_event_reasons.sw_power_cap")

    def __init__(self, index):
        self.index = index
        self.proc = None
        self.lines = []

    def start(self):
        try:
            self.proc = subprocess.Popen(
                ["nvidia-smi", "-i", str(self.index), f"--query-gpu={self.FIELDS}",
                 "--format=csv,noheader,nounits", "-lms", "200"],
                stdout=subprocess.PIPE, stderr=subprocess.DEVNULL, text=True)
        except (OSError, FileNotFoundError):
            self.proc = None

    def stop(self):
        if self.proc is None:
            return None
        self.proc.terminate()
        try:
            out, _ = self.proc.communicate(timeout=5)
        except subprocess.TimeoutExpired:
            self.proc.kill()
            out, _ = self.proc.communicate()
        rows = [l.split(",") for l in out.strip().splitlines() if l.strip()]
        sm = [float(r[1]) for r in rows if len(r) >= 9 and r[1].strip().replace(".", "").isdigit()]
        mx = [float(r[2]) for r in rows if len(r) >= 9 and r[2].strip().replace(".", "").isdigit()]
        reasons = set()
        names = ["hw_slowdown", "hw_thermal_slowdown", "sw_thermal_slowdown", "sw_power_cap"]
        for r in rows:
            if len(r) < 9:
                continue
            for n, v in zip(names, r[5:9]):
                if "Active" in v and "Not" not in v:
                    reasons.add(n)
        if not sm:
            return None
        return {"sm_mhz": float(np.median(sm)), "sm_max_mhz": max(mx) if mx else None,
                "reasons": sorted(reasons), "samples": len(sm)}


def algorithmic_bytes(wl, sel, n_sel):
    """Bytes the step must move: index pages scanned + KV pages selected by any
    query token of a sequence (576 B per valid token) + queries, weights,
    output and metadata.  Workspace traffic is not counted."""
    idx = wl.index_bytes()
    kv = 0
    qsl = wl.q_start_loc
    for b in range(wl.n_seqs):
        blocks = set()
        for j in range(qsl[b], qsl[b + 1]):
            blocks.update(int(x) for x in sel[j, : n_sel[j]])
        L = wl.seq_lens[b]
        for blk in blocks:
            kv += 576 * min(128, L - 128 * blk)
    T = wl.n_q_total
    small = T * (16 * 128 + 8 * 128 + 8 * 4 + 16 * 128 * 4) + wl.n_seqs * (wl.max_pages * 4 + 8) + 4
    return idx, kv, idx + kv + small


def packed(dev, tensors):
    """One device buffer holding the given tensors at 256-byte-aligned offsets:
    views with the same shapes and dtypes (contents copied), so that a step's
    inputs arrive from the host in a single copy."""
    offs, at = [], 0
    for t in tensors:
        offs.append(at)
        at += (t.numel() * t.element_size() + 255) // 256 * 256
    buf = torch.empty(at, dtype=torch.uint8, device=dev)
    views = []
    for t, o in zip(tensors, offs):
        v = buf[o:o + t.numel() * t.element_size()].view(t.dtype).view(t.shape)
        v.copy_(t)
        views.append(v)
    return buf, views


def run_gpu(args, rank, world, local_rank):
    dev = f"cuda:{local_rank}"
    torch.cuda.set_device(local_rank)
    wl = workloads.config(args.config)
    st = harness.build_state(wl, dev)
    q, qi, w = wl.queries(dev)
    # the step's inputs (queries, index queries, head weights, block table,
    # sequence lengths, query start offsets) live in one device buffer
    in_buf, (q, qi, w, bt, sl, qsl) = packed(dev, [q, qi, w, st.block_table, st.seq_lens, st.q_start_loc])
    st = dataclasses.replace(st, block_table=bt, seq_lens=sl, q_start_loc=qsl)
    T = wl.n_q_total
    n_splits = args.splits or ops.choose_splits(T)
    bufs = ops.DecodeBuffers(T, wl.max_pages, n_splits, dev)
    fbufs = ops.FusedBuffers(T, wl.max_pages, dev) if args.fused else None
    flush = torch.empty(L2_FLUSH_BYTES // 4, dtype=torch.float32, device=dev)
    stream = torch.cuda.current_stream()

    def step():
        if fbufs is not None:
            return ops.decode_fused(st.cache, q, qi, w, st.block_table, st.seq_lens, st.q_start_loc, fbufs)
        return ops.decode_step(st.cache, q, qi, w, st.block_table, st.seq_lens, st.q_start_loc, bufs)

    step()
    torch.cuda.synchronize()
    sel = (fbufs or bufs).sel.cpu().numpy()
    n_sel = (fbufs or bufs).n_sel.cpu().numpy()
    idx_bytes, kv_bytes, alg_bytes = algorithmic_bytes(wl, sel, n_sel)

    # the step as one CUDA graph (indexer, attention and, with several splits, the
    # merge: chained with
    # programmatic dependent launch) so that host launch latency does not gap
    # the kernels; a second graph holds the indexer alone for its own timing
    def run_indexer():
        ops.indexer_topk(st.cache, qi, w, st.block_table, st.seq_lens, st.q_start_loc, ws=bufs.ws,
                         sel=bufs.sel, n_sel=bufs.n_sel)

    def run_attention():
        ops.sparse_attn_decode(st.cache, q, bufs.sel, bufs.n_sel, st.block_table, st.seq_lens,
                               st.q_start_loc, n_splits, o_part=bufs.o_part, lse_part=bufs.lse_part)
        if n_splits > 1:  # a single split's output is final
            ops.merge_splits(bufs.o_part, bufs.lse_part, out=bufs.out)

    def run_step():
        if fbufs is not None:  # the whole step in one launch
            step()
            return
        run_indexer()
        run_attention()

    if args.eager:
        g_step, g_idx = run_step, run_indexer
    else:
        side = torch.cuda.Stream()
        side.wait_stream(stream)
        with torch.cuda.stream(side):
            run_step()
        stream.wait_stream(side)
        graph_s, graph_i = torch.cuda.CUDAGraph(), torch.cuda.CUDAGraph()
        with torch.cuda.graph(graph_s):
            run_step()
        with torch.cuda.graph(graph_i):
            run_indexer()
        g_step, g_idx = graph_s.replay, graph_i.replay
    if fbufs is not None:  # one kernel: the roofline line times the step itself
        g_idx = g_step
    for _ in range(args.warmup):
        flush.fill_(1.0)
        g_step()
        flush.fill_(1.0)
        g_idx()
    torch.cuda.synchronize()

    def timed(fn, n):
        evs = [(torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)) for _ in range(n)]
        for i in range(n):
            flush.fill_(float(i))
            evs[i][0].record(stream)
            fn()
            evs[i][1].record(stream)
        torch.cuda.synchronize()
        return [a.elapsed_time(b) for a, b in evs]

    clocks = ClockSampler(local_rank)
    if world > 1:
        torch.distributed.barrier()
    torch.cuda.synchronize()
    clocks.start()
    time.sleep(0.3)
    torch.cuda.nvtx.range_push("timed")
    step_ms = timed(g_step, args.steps)
    torch.cuda.nvtx.range_pop()
    if world > 1:
        torch.distributed.barrier()
    idx_ms = timed(g_idx, args.steps)
    torch.cuda.synchronize()
    clk = clocks.stop()
    ms = float(np.mean(step_ms))
    t_idx = float(np.mean(idx_ms))

    # end to end through the public API: pinned host inputs -> device (one copy
    # of the packed inputs), step, output -> host
    h_in = in_buf.cpu().pin_memory()
    h_out = torch.empty((T, 16, 128), dtype=torch.float32).pin_memory()
    h2d = h_in.numel()
    d2h = h_out.numel() * 4
    e2e_ms = []
    for i in range(args.warmup + args.steps):
        flush.fill_(float(i))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        in_buf.copy_(h_in, non_blocking=True)
        g_step()
        h_out.copy_((fbufs or bufs).out, non_blocking=True)
        e1.record(stream)
        e1.synchronize()
        if i >= args.warmup:
            e2e_ms.append(e0.elapsed_time(e1))
    e2e = float(np.mean(e2e_ms))

    ins = time_insert(args, flush, stream, dev) if args.insert_tokens > 0 else None
    pack = time_pack(args, flush, stream, dev) if args.pack_blocks > 0 else None
    qkvm = time_qkv(args, flush, stream, dev) if args.qkv_tokens > 0 else None

    if world > 1:
        ms, t_idx, e2e = max_over_ranks([ms, t_idx, e2e], dev)
    return dict(wl=wl, T=T, ms=ms, t_idx=t_idx, e2e=e2e, h2d=h2d, d2h=d2h, n_splits=n_splits,
                idx_bytes=idx_bytes, kv_bytes=kv_bytes, alg_bytes=alg_bytes, clocks=clk,
                roof_bytes=alg_bytes if fbufs is not None else idx_bytes,
                launches=(1 if fbufs is not None else (3 if n_splits > 1 else 2)) * args.steps, insert=ins,
                pack=pack, qkv=qkvm)


# Algorithmic bytes of inserting one token: fp32 K and V (2 x 4 x 128 x 4), the
# fp32 index key (128 x 4) and its int64 slot read; NVFP4 K and V (576 B: codes
# and scales) and the FP8 index key (128 B) written.
INSERT_READ_BYTES = 2 * 4 * 128 * 4 + 128 * 4 + 8
INSERT_WRITE_BYTES = 576 + 128


def time_qkv(args, flush, stream, dev):
    """Fused QKV projection -> RMS norm -> RoPE -> FP8 queries and NVFP4 cache
    insert of a prefill chunk (synthetic bf16 weights), as its own
    sub-measurement; a tensor-core contraction, so its rate is FLOP/s against
    the measured bf16 peak.  The library GEMM of the same shape alone (torch /
    cuBLAS, no epilogue) is timed beside it for context."""
    n, d = args.qkv_tokens, args.qkv_dmodel
    inp = workloads.qkv_inputs(n, d, seed=11, device=dev)
    cache = ops.KVCache(inp["n_pages"], 448.0 / 8.0, 448.0 / 6.0, dev)
    table = ops.rope_table(inp["max_pos"], device=dev)
    q8 = torch.empty((n, 16, 128), dtype=torch.uint8, device=dev)

    def fused():
        ops.qkv_project_insert(cache, inp["x"], inp["w"], inp["gamma_q"], inp["gamma_k"], inp["gamma_idx"], table,
                               inp["positions"], inp["slots"], q8=q8)

    def gemm():
        torch.matmul(inp["x"], inp["w"].t())

    def t(fn):
        for _ in range(args.warmup):
            fn()
        ts = []
        for i in range(args.steps):
            flush.fill_(float(i))
            e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
            e0.record(stream)
            fn()
            e1.record(stream)
            torch.cuda.synchronize()
            ts.append(e0.elapsed_time(e1))
        return float(np.mean(ts))

    ms, ms_gemm = t(fused), t(gemm)
    flops = 2.0 * n * d * workloads.QKV_HEADS * 128
    return {"kernel": "qkv_fused_kernel (msa_qkv_project_insert)", "tokens": n, "d_model": d,
            "heads_out": workloads.QKV_HEADS, "ms_per_launch": ms, "flops_per_launch": flops,
            "achieved_tflops": flops / (ms * 1e-3) / 1e12, "library_gemm_ms": ms_gemm,
            "library_gemm_tflops": flops / (ms_gemm * 1e-3) / 1e12}


def time_pack(args, flush, stream, dev):
    """Block-outer pack of a batch of blocks from several layers' pools into
    contiguous rows (off the decode step; its own sub-measurement).  Algorithmic
    bytes: every row byte read once from the pools and written once."""
    n, layers = args.pack_blocks, args.pack_layers
    caches = [ops.KVCache(n, 1.0, 1.0, dev) for _ in range(layers)]
    g = torch.Generator(device=dev)
    g.manual_seed(777)
    pages = torch.randperm(n, generator=g, device=dev).to(torch.int32)
    rows = torch.empty((n, ops.block_row_bytes(layers)), dtype=torch.uint8, device=dev)
    for _ in range(args.warmup):
        ops.pack_blocks(caches, pages, rows)
    ts = []
    for i in range(args.steps):
        flush.fill_(float(i))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        ops.pack_blocks(caches, pages, rows)
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    ms = float(np.mean(ts))
    byts = 2 * rows.numel()
    return {"kernel": "block_rows_kernel (msa_pack_blocks)", "blocks": n, "layers": layers,
            "row_bytes": int(rows.shape[1]), "ms_per_launch": ms, "algorithmic_bytes_per_launch": byts,
            "achieved_gbs": byts / (ms * 1e-3) / 1e9}


def time_insert(args, flush, stream, dev):
    """Quantise-insert of a batch of new tokens into random slots of a scratch
    pool (off the decode step; reported as its own sub-measurement)."""
    n = args.insert_tokens
    pages = (n + 127) // 128
    g = torch.Generator(device=dev)
    g.manual_seed(12345)
    k = torch.randn((n, 4, 128), generator=g, device=dev)
    v = torch.randn((n, 4, 128), generator=g, device=dev)
    ik = torch.randn((n, 128), generator=g, device=dev)
    slots = torch.randperm(pages * 128, generator=g, device=dev)[:n].to(torch.int64)
    cache = ops.KVCache(pages, 448.0 / 6.0, 448.0 / 6.0, dev)
    for _ in range(args.warmup):
        ops.quantize_kv_insert(cache, k, v, ik, slots)
    ts = []
    for i in range(args.steps):
        flush.fill_(float(i))
        e0, e1 = torch.cuda.Event(enable_timing=True), torch.cuda.Event(enable_timing=True)
        e0.record(stream)
        ops.quantize_kv_insert(cache, k, v, ik, slots)
        e1.record(stream)
        torch.cuda.synchronize()
        ts.append(e0.elapsed_time(e1))
    ms = float(np.mean(ts))
    byts = n * (INSERT_READ_BYTES + INSERT_WRITE_BYTES)
    return {"kernel": "quantize_insert_kernel (msa_quantize_kv_insert)", "tokens": n,
            "slots": "random permutation of the pool", "ms_per_launch": ms,
            "algorithmic_bytes_per_launch": byts, "achieved_gbs": byts / (ms * 1e-3) / 1e9}


def max_over_ranks(values, device):
    """Element-wise max of a list of floats over all ranks of the process group:
    the slowest replica sets each time."""
    t = torch.tensor(values, dtype=torch.float64, device=device)
    torch.distributed.all_reduce(t, op=torch.distributed.ReduceOp.MAX)
    return [float(x) for x in t.cpu()]


def oracle_sample(wl, device, budget_s):
    """Time the CPU oracle (indexer + selection + attention) on query tokens of
    the first sequences, repeated until budget_s seconds of oracle work."""
    import oracle
    from oracle import formats, nvfp4

    q, qi, w = (x.cpu().numpy() for x in wl.queries(device))
    amax = [0.0, 0.0]
    for tensor in (0, 1):
        s = wl.channel_scales(tensor, device)
        for b in range(wl.n_seqs):
            for c in range(wl.n_chunks(b)):
                amax[tensor] = max(amax[tensor], float(wl.kv_chunk(tensor, b, c, device, s).abs().max()))
    s_enc_k = nvfp4.tensor_encode_scale(np.float32(amax[0]))
    s_enc_v = nvfp4.tensor_encode_scale(np.float32(amax[1]))
    scale = np.float32(1 / math.sqrt(128))
    # untimed preparation: oracle quantisation of the sampled sequences
    prep = []
    qsl = wl.q_start_loc
    for b in range(min(2, wl.n_seqs)):
        L = wl.seq_lens[b]
        idx = formats.encode_e4m3(wl.tokens(2, b, 0, L, device).cpu().numpy().astype(np.float64))
        prep.append((b, idx, None))
    pages = {}
    done, t_work = 0, 0.0
    while t_work < budget_s:
        for b, idx, _ in prep:
            for j in range(qsl[b], qsl[b + 1]):
                pos = wl.seq_lens[b] - wl.n_q[b] + (j - qsl[b])
                r = pos // 128
                t0 = time.perf_counter()
                scores = oracle.indexer.block_scores(qi[j], w[j], idx, r)
                sel = oracle.indexer.select(scores, r)
                t_idx = time.perf_counter() - t0
                # the selected pages' FP8 operands are prepared outside the timed region
                ks, vs = [], []
                for blk in sel:
                    lo, hi = blk * 128, min(blk * 128 + 128, pos + 1)
                    if (b, lo, hi) not in pages:
                        kc, kk = nvfp4.quantize(wl.tokens(0, b, lo, hi, device).cpu().numpy(), s_enc_k)
                        vc, vv = nvfp4.quantize(wl.tokens(1, b, lo, hi, device).cpu().numpy(), s_enc_v)
                        pages[(b, lo, hi)] = (nvfp4.fp8_operand(kc, kk), nvfp4.fp8_operand(vc, vv))
                    ks.append(pages[(b, lo, hi)][0])
                    vs.append(pages[(b, lo, hi)][1])
                k8, v8 = np.concatenate(ks), np.concatenate(vs)
                t0 = time.perf_counter()
                oracle.attention.attend(q[j], k8, v8, scale, s_enc_k, s_enc_v)
                t_work += t_idx + time.perf_counter() - t0
                done += 1
    cores = len(os.sched_getaffinity(0))
    seqs = ", ".join(str(b) for b, _, _ in prep)
    return done / t_work, cores, f"{done} query tokens of sequence(s) {seqs} (indexer over the full context + attention), {t_work:.1f} s of oracle work"


def main():
    ap = argparse.ArgumentParser()
    ap.add_argument("--gpus", type=int, default=1)
    ap.add_argument("--steps", type=int, default=20)
    ap.add_argument("--warmup", type=int, default=5)
    # default: the largest single-GPU workload (64 ragged sequences, 30K-215K
    # context, 1-8 query tokens each, 297 in all)
    ap.add_argument("--config", type=int, default=4)
    ap.add_argument("--insert-tokens", type=int, default=262144,
                    help="tokens of the timed quantise-insert sub-measurement (0: skip)")
    ap.add_argument("--pack-blocks", type=int, default=2048,
                    help="blocks of the timed block-outer pack sub-measurement (0: skip)")
    ap.add_argument("--pack-layers", type=int, default=4)
    ap.add_argument("--qkv-tokens", type=int, default=8192,
                    help="tokens of the timed fused QKV projection + insert sub-measurement (0: skip)")
    ap.add_argument("--qkv-dmodel", type=int, default=3072)
    ap.add_argument("--splits", type=int, default=0)
    ap.add_argument("--impl", default="gb300", choices=["gb300", "reference"])
    ap.add_argument("--cpu-budget", type=float, default=12.0)
    ap.add_argument("--no-cpu-baseline", action="store_true")
    ap.add_argument("--eager", action="store_true", help="launch kernels eagerly instead of CUDA graphs")
    ap.add_argument("--fused", action="store_true",
                    help="the whole step as one launch (msa_decode_fused; low concurrency, <= 64 tokens)")
    args = ap.parse_args()
    args.warmup = max(3, args.warmup)

    world = int(os.environ.get("WORLD_SIZE", "1"))
    rank = int(os.environ.get("RANK", "0"))
    local_rank = int(os.environ.get("LOCAL_RANK", "0"))
    wl = workloads.config(args.config)
    config = {"workload": wl.name, "description": wl.description, "n_seqs": wl.n_seqs,
              "query_tokens": wl.n_q_total, "context": list(sorted(set(wl.seq_lens)))[:4],
              "page_tokens": 128, "q_heads": 16, "kv_heads": 4, "head_dim": 128,
              "idx_heads": 8, "topk": 16, "l2": "512 MiB buffer written between timed steps",
              "parallelism": f"replicas x{world}" if world > 1 else "single GPU"}

    if args.impl == "reference":
        if rank != 0:
            return
        dev = "cuda" if torch.cuda.is_available() else "cpu"
        qps, cores, sample = oracle_sample(wl, dev, args.cpu_budget)
        line = {"impl": "reference", "metric": "decode query tokens/s (NVFP4 sparse attention)",
                "value": qps, "unit": "queries/s", "n_gpus": world, "steps": args.steps,
                "warmup": args.warmup, "higher_is_better": True, "scaling": "weak",
                "vs_baseline": None, "dtype": "f64", "data": "synthetic", "config": config,
                "cpu_baseline": {"value": qps, "unit": "queries/s", "cores": cores, "kind": "oracle",
                                 "sample": sample},
                "e2e": {"value": qps, "unit": "queries/s", "h2d_bytes_per_step": 0,
                        "d2h_bytes_per_step": 0}}
        print(json.dumps(line))
        return

    if world > 1:
        torch.distributed.init_process_group("nccl", device_id=torch.device(f"cuda:{local_rank}"))
    r = run_gpu(args, rank, world, local_rank)
    if world > 1:
        torch.distributed.destroy_process_group()
    if rank != 0:
        return
    peak, peak_kind = measured_peaks()
    T = r["T"]
    qps = world * T / (r["ms"] * 1e-3)
    step_gbs = r["alg_bytes"] / (r["ms"] * 1e-3) / 1e9
    idx_gbs = r["roof_bytes"] / (r["t_idx"] * 1e-3) / 1e9
    line = {
        "metric": "decode query tokens/s (NVFP4 sparse attention)", "value": qps, "unit": "queries/s",
        "n_gpus": world, "steps": args.steps, "warmup": args.warmup, "ms_per_step": r["ms"],
        "higher_is_better": True, "scaling": "weak", "vs_baseline": None, "dtype": "e4m3/e2m1 in, f32 accum",
        "data": "synthetic", "config": config,
        "hbm": {"algorithmic_bytes_per_step": r["alg_bytes"], "index_bytes": r["idx_bytes"],
                "kv_bytes": r["kv_bytes"], "achieved_gbs": step_gbs,
                "frac_of_8tbs": step_gbs / ROOFLINE_NOMINAL_GBS,
                f"frac_of_{peak_kind}": step_gbs / peak},
        "roofline": {"kernel": ("decode_fused_kernel (msa_decode_fused: the whole step)" if args.fused else
                               "indexer_scan_kernel (msa_indexer_topk: block scores + selection)"), "bound": "hbm",
                     "achieved": idx_gbs, "peak": peak, "unit": "GB/s", "frac": idx_gbs / peak,
                     "peak_kind": peak_kind, "traffic": committed_traffic(wl.name),
                     "algorithmic_bytes_per_launch": r["roof_bytes"], "ms_per_launch": r["t_idx"]},
        "e2e": {"value": world * T / (r["e2e"] * 1e-3), "unit": "queries/s",
                "h2d_bytes_per_step": r["h2d"], "d2h_bytes_per_step": r["d2h"], "ms_per_step": r["e2e"]},
        "gpu_launches": r["launches"], "n_splits": r["n_splits"], "clocks": r["clocks"],
    }
    if r["insert"] is not None:
        ins = dict(r["insert"])
        ins["frac"] = ins["achieved_gbs"] / peak
        ins["peak_kind"] = peak_kind
        line["quantize_insert"] = ins
    if r["qkv"] is not None:
        qk = dict(r["qkv"])
        tf_peak, tf_kind = measured_bf16_peak()
        qk["peak_tflops"] = tf_peak
        qk["frac"] = qk["achieved_tflops"] / tf_peak
        qk["peak_kind"] = tf_kind
        line["qkv_project_insert"] = qk
    if r["pack"] is not None:
        pk = dict(r["pack"])
        pk["frac"] = pk["achieved_gbs"] / peak
        pk["peak_kind"] = peak_kind
        line["pack_blocks"] = pk
    if not args.no_cpu_baseline:
        qps_cpu, cores, sample = oracle_sample(r["wl"], "cuda", args.cpu_budget)
        line["cpu_baseline"] = {"value": qps_cpu, "unit": "queries/s", "cores": cores, "kind": "oracle",
                                "sample": sample}
    print(json.dumps(line))


if __name__ == "__main__":
    main()
