// Lightweight indexer: FP8 index scan with per-block max, then top-16 + recent.
//
// "vLLM Delivers Day-0 Support for MiniMax-M3.1-Flash" blog, section "Sparse
// attention still scans an index": KV lives in 128-token blocks, the indexer
// scores the context, keeps 16 blocks plus the most recent one, and reads 128
// index bytes per token.  Section "Parallelize index work across context":
// splitting the scan keeps the selection exact (each block score is computed
// once, by one CTA, and the selection runs over all of them).
//
// Scan (hot loop), one persistent CTA per SM.  The pages to scan (blocks
// 0..r_last-1 of every sequence) are flattened and cut into contiguous ranges
// of equal weighted cost, one per CTA.  Warp-specialised pipeline:
//   warp 0      TMA producer: one 16 KB cp.async.bulk per index page into a
//               6-stage shared-memory ring;
//   warps 1-2   MMA issuers, alternate pages: per page, 4 x tcgen05.mma
//               kind::f8f6f4 with M = 128 tokens (the page, A from shared
//               memory), N = 8 heads x query tokens (B: the segment's index
//               queries, one copy per issuer), K = 128 dims, fp32 accumulators
//               in tensor memory (6 buffers); tcgen05.commit frees the stage and
//               hands the accumulator to the epilogue;
//   warps 3-14  epilogue, three sets of four taking every third page:
//               tcgen05.ld of one token row per thread, ReLU, head weights, sum
//               over heads, block max over the 128 rows; one fp32 per (query
//               token, block) and quarter is written.
// The index page is stored pre-swizzled (chunk c of token t at chunk c ^ (t&7)),
// which is exactly the 128-byte-swizzled K-major operand layout, so a plain
// bulk copy lands it ready for the tensor core.
#include "common.cuh"
#include "topk.cuh"

namespace msa {
namespace {

struct ScanParams {
  const uint8_t* idx_pool;
  int64_t n_pages;
  const uint8_t* q_idx;  // [T][8][128]
  const float* w;        // [T][8]
  const int* block_table;
  int max_pages;
  const int* seq_lens;
  const int* q_start_loc;
  int n_seqs;
  int n_q_total;
  float* scores;  // [T][max_pages][4] partial block maxima
  int* sel;       // [T][17]
  int* n_sel;     // [T]
  unsigned long long* sync;  // grid-barrier word (generation << 32 | arrivals)
  int* status;
  unsigned long long wait_ns;  // limit of one bounded wait
  int barrier_extra;           // test hook: arrivals the barrier waits for beyond the grid (0)
  int blk_lo, blk_hi;          // logical blocks scanned and selected from: [blk_lo, blk_hi)
  unsigned long long* cand;    // range mode: [T][16] local top-16 keys instead of sel / n_sel
};

constexpr int kScanThreads = 480;  // 15 warps: producer, 2 MMA issuers, 3 epilogue sets of 4
constexpr int kStages = 6;
constexpr int kNqMax = 8;                       // query tokens per pass
constexpr int kBRows = kNqMax * kIdxHeads;      // 64
constexpr int kBBytes = kBRows * kIdxDim;       // 8 KB
constexpr int kMmaWarps = 2;                    // MMA issuers, pages it with it % 2 == issuer
constexpr int kEpiSets = 3;                     // epilogue sets, pages it with it % 3 == set
constexpr int kAccs = kMmaWarps * kEpiSets;     // 6 accumulators: acc = it % 6 fixes both
constexpr int kTmemCols = 512;                  // 6 x 64 columns, allocated as a power of two
constexpr int kOffStages = 0;
constexpr int kOffB = kStages * kIdxPageBytes;  // 131,072
constexpr int kOffBars = kOffB + 2 * kMmaWarps * kBBytes;  // two B slots per MMA issuer
constexpr int kNumBars = 2 * kStages + 2 * kMmaWarps + 2 * kAccs + kMmaWarps;
constexpr int kOffMisc = kOffBars + kNumBars * 8;
constexpr int kOffPrefix = kOffMisc + 32;  // misc: tmem slot, abort, page range [2] (int64), copies issued

// After kOffPrefix, per sequence: weighted page prefix (int64, n_seqs + 1),
// page prefix (n_seqs + 1), seq_lens (n_seqs), q_start_loc (n_seqs + 1).
size_t scan_smem_bytes(int n_seqs) { return 1024 + kOffPrefix + 20 * (size_t)n_seqs + 16; }

// Cost model of the scan, fitted to per-CTA scan times on the ragged batch
// (152 partitions, contiguous and permuted page layouts agreeing): the cost of
// one page for a pass of n = 1..8 query tokens (flat while the page's bytes
// set the pace, rising once the epilogue's per-token work does), and the cost
// of starting a segment (a sequence's pass: new query tile, pipeline refill),
// about six pages.  Weights in thousandths of a one-token page.
__constant__ int kPassPageCost[kNqMax + 1] = {0, 1000, 1009, 1017, 1022, 1038, 1072, 1094, 1139};
constexpr long long kSegmentCost = 6000;
__device__ __forceinline__ long long page_weight(int n_q) {
  return (long long)(n_q / kNqMax) * kPassPageCost[kNqMax] + kPassPageCost[n_q % kNqMax];
}
// Weight of a sequence: its pages, plus one segment start per pass.
__device__ __forceinline__ long long seq_weight(int pages, int n_q) {
  return pages > 0 ? (long long)((n_q + kNqMax - 1) / kNqMax) * kSegmentCost + pages * page_weight(n_q) : 0;
}

// Blocks a sequence's query tokens compete over: 0..r_last-1, r_last =
// (seq_len-1)/128 (the recent block of its last token); scanned: their part
// in [blk_lo, blk_hi), starting at block scan_first.
__device__ __forceinline__ int r_last_of(const SeqInfo& s) {
  return (s.ok && s.seq_len > 0 && s.n_q > 0) ? (s.seq_len - 1) / kPageTokens : 0;
}
__device__ __forceinline__ int scan_first(const ScanParams& p, const SeqInfo& s) {
  return min(p.blk_lo, r_last_of(s));
}
__device__ __forceinline__ int scan_pages(const ScanParams& p, const SeqInfo& s) {
  return min(p.blk_hi, r_last_of(s)) - scan_first(p, s);
}

// Walks the segments (sequence, query-token group, page range) of the flattened
// page range [pg, pg_end).  Every role of the CTA walks the same sequence.
template <typename F>
__device__ __forceinline__ void for_each_segment(const ScanParams& p, const int* s_prefix, const int* s_sl,
                                                 const int* s_qsl, long long pg, long long pg_end, F&& f) {
  int lo = 0, hi = p.n_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_prefix[mid] <= pg) lo = mid; else hi = mid - 1;
  }
  int b = lo;
  while (pg < pg_end) {
    while (s_prefix[b + 1] <= pg) ++b;
    const SeqInfo s = load_seq(b, s_sl, s_qsl, p.max_pages, p.n_q_total);
    // logical blocks of this piece (the sequence's scanned blocks start at scan_first)
    const int lo_b = scan_first(p, s);
    const int page0 = lo_b + (int)(pg - s_prefix[b]);
    const int page1 = lo_b + (int)(min((long long)s_prefix[b + 1], pg_end) - s_prefix[b]);
    for (int j0 = 0; j0 < s.n_q; j0 += kNqMax) {
      if (!f(b, s, j0, min(kNqMax, s.n_q - j0), page0, page1)) return;
    }
    pg = s_prefix[b] + (page1 - lo_b);
    ++b;
  }
}

__global__ void __launch_bounds__(kScanThreads, 1) indexer_scan_kernel(ScanParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar0 = sbase + kOffBars;
  // barrier addresses
  auto full = [&](int i) { return bar0 + 8 * i; };
  auto empty = [&](int i) { return bar0 + 8 * (kStages + i); };
  auto bempty = [&](int i) { return bar0 + 8 * (2 * kStages + i); };  // B slot i = 2 issuer + slot
  auto tfull = [&](int i) { return bar0 + 8 * (2 * kStages + 2 * kMmaWarps + i); };
  auto tempty = [&](int i) { return bar0 + 8 * (2 * kStages + 2 * kMmaWarps + kAccs + i); };
  auto done_bar = [&](int m) { return bar0 + 8 * (2 * kStages + 2 * kMmaWarps + 2 * kAccs + m); };
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  const WaitCtl wc{s_abort, p.wait_ns};
  int* s_issued = reinterpret_cast<int*>(smem + kOffMisc + 24);
  long long* s_wpre = reinterpret_cast<long long*>(smem + kOffPrefix);
  int* s_prefix = reinterpret_cast<int*>(s_wpre + (p.n_seqs + 1));
  int* s_sl = s_prefix + (p.n_seqs + 1);
  int* s_qsl = s_sl + p.n_seqs;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  pdl_wait();     // inputs may come from the previous kernel in the stream
  pdl_trigger();  // the attention kernel may launch and run its prologue

  // -- sequence metadata in shared memory; exclusive prefixes over sequences of
  //    the pages each one scans and of their weighted cost ----------------------
  for (int b = tid; b <= p.n_seqs; b += kScanThreads) s_qsl[b] = p.q_start_loc[b];
  for (int b = tid; b < p.n_seqs; b += kScanThreads) s_sl[b] = p.seq_lens[b];
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(full(i), 1);
      mbar_init(empty(i), 1);
    }
    for (int i = 0; i < 2 * kMmaWarps; ++i) mbar_init(bempty(i), 1);
    for (int i = 0; i < kAccs; ++i) {
      mbar_init(tfull(i), 1);
      mbar_init(tempty(i), 4);
    }
    for (int m = 0; m < kMmaWarps; ++m) mbar_init(done_bar(m), 1);
    *s_abort = 0;
    *s_issued = 0;
    fence_barrier_init();
  }
  __syncthreads();
  {
    // thread t takes the contiguous run of sequences [b0, b0 + per)
    const int per = (p.n_seqs + kScanThreads - 1) / kScanThreads;
    const int b0 = tid * per, b1 = min(b0 + per, p.n_seqs);
    long long lp = 0, lw = 0;
    for (int b = b0; b < b1; ++b) {
      const SeqInfo s = load_seq(b, s_sl, s_qsl, p.max_pages, p.n_q_total);
      if (!s.ok && blockIdx.x == 0) set_status(p.status, MSA_STATUS_BAD_SEQ);
      const int pages = scan_pages(p, s);
      lp += pages;
      lw += seq_weight(pages, s.n_q);
    }
    // block-wide exclusive scan of (lp, lw): warp scans, then the warp totals
    long long ip = lp, iw = lw;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const long long yp = __shfl_up_sync(0xffffffffu, ip, o);
      const long long yw = __shfl_up_sync(0xffffffffu, iw, o);
      if (lane >= o) {
        ip += yp;
        iw += yw;
      }
    }
    __shared__ long long s_wsum[2][kScanThreads / 32];
    if (lane == 31) {
      s_wsum[0][warp] = ip;
      s_wsum[1][warp] = iw;
    }
    __syncthreads();
    long long rp = ip - lp, rw = iw - lw;
    for (int i = 0; i < warp; ++i) {
      rp += s_wsum[0][i];
      rw += s_wsum[1][i];
    }
    for (int b = b0; b < b1; ++b) {
      s_prefix[b] = (int)rp;
      s_wpre[b] = rw;
      const SeqInfo s = load_seq(b, s_sl, s_qsl, p.max_pages, p.n_q_total);
      const int pages = scan_pages(p, s);
      rp += pages;
      rw += seq_weight(pages, s.n_q);
    }
    if (tid == kScanThreads - 1) {
      s_prefix[p.n_seqs] = (int)rp;
      s_wpre[p.n_seqs] = rw;
    }
  }
  if (warp == 1) tmem_alloc(smem_u32(s_tmem), kTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  // CTA c scans the pages whose weighted cost falls in [c W / G, (c+1) W / G)
  // (each sequence's segment cost placed before its pages)
  const long long w_total = s_wpre[p.n_seqs];
  auto page_at = [&](long long x) -> long long {
    if (x >= w_total) return s_prefix[p.n_seqs];
    int lo = 0, hi = p.n_seqs - 1;  // last b with s_wpre[b] <= x: a sequence with pages
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_wpre[mid] <= x) lo = mid; else hi = mid - 1;
    }
    // the sequence's segment starts come first on the weighted axis
    const SeqInfo s = load_seq(lo, s_sl, s_qsl, p.max_pages, p.n_q_total);
    const long long seg = (long long)((s.n_q + kNqMax - 1) / kNqMax) * kSegmentCost;
    return s_prefix[lo] + max(0ll, x - s_wpre[lo] - seg) / page_weight(s.n_q);
  };
  // one thread computes the range (64-bit divisions are slow in every thread)
  long long* s_range = reinterpret_cast<long long*>(smem + kOffMisc + 8);
  if (tid == 0) {
    s_range[0] = page_at((long long)blockIdx.x * w_total / gridDim.x);
    s_range[1] = page_at((long long)(blockIdx.x + 1) * w_total / gridDim.x);
  }
  __syncthreads();
  const long long pg_begin = s_range[0], pg_end = s_range[1];
  if (warp == 1 + kMmaWarps) {
    // L2 prefetch of what each segment of the range starts with (index
    // queries, head weights, the first block-table entries): after the first,
    // a segment switch no longer waits on DRAM for them
    int sg = 0;
    for_each_segment(p, s_prefix, s_sl, s_qsl, pg_begin, pg_end, [&](int b, const SeqInfo& s, int j0, int nq, int page0, int page1) {
      if ((sg++ & 31) == lane) {
        const uint8_t* qi = p.q_idx + (size_t)(s.q0 + j0) * kIdxHeads * kIdxDim;
        asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(qi), "r"(nq * kIdxHeads * kIdxDim) : "memory");
        asm volatile("prefetch.global.L2 [%0];" ::"l"(p.w + (size_t)(s.q0 + j0) * kIdxHeads));
        asm volatile("prefetch.global.L2 [%0];" ::"l"(p.block_table + (size_t)b * p.max_pages + page0));
      }
      return true;
    });
  }

  if (warp == 0) {
    // ---------------- producer: index pages -----------------------------------
    int it = 0;
    for_each_segment(p, s_prefix, s_sl, s_qsl, pg_begin, pg_end, [&](int b, const SeqInfo& s, int j0, int nq, int page0, int page1) {
      // block-table entries are fetched 32 at a time (one coalesced load per
      // 32 pages, the next batch in flight) so that no dependent global load
      // sits between two page copies
      const int* bt = p.block_table + (size_t)b * p.max_pages;
      int nxt = page0 + lane < page1 ? bt[page0 + lane] : 0;
      for (int base = page0; base < page1; base += 32) {
        const int cur = nxt;
        nxt = base + 32 + lane < page1 ? bt[base + 32 + lane] : 0;
        const int n = min(32, page1 - base);
        for (int k = 0; k < n; ++k, ++it) {
          const int st = it % kStages;
          int phys = __shfl_sync(0xffffffffu, cur, k);
          if (phys < 0 || phys >= p.n_pages) phys = 0;  // flagged by the epilogue
          if (!mbar_wait(empty(st), ((it / kStages) & 1) ^ 1, wc)) return false;
          if (lane == 0) {
            mbar_arrive_expect_tx(full(st), kIdxPageBytes);
            bulk_g2s(sbase + kOffStages + st * kIdxPageBytes, p.idx_pool + (size_t)phys * kIdxPageBytes,
                     kIdxPageBytes, full(st));
          }
          __syncwarp();
        }
      }
      return true;
    });
    if (lane == 0) *s_issued = it;  // copies issued, for the drain after an abort
  } else if (warp <= kMmaWarps) {
    // ---------------- MMA warps: B tile of each segment, then the MMAs ----------
    // issuer m takes the pages with it % 2 == m: one thread issues a
    // tcgen05.mma every ~140 cycles, four per page, so two issuers keep up
    // with the page stream; each builds its own copy of the segment's B tile
    const int mw = warp - 1;
    int it = 0, sg = 0;
    for_each_segment(p, s_prefix, s_sl, s_qsl, pg_begin, pg_end, [&](int b, const SeqInfo& s, int j0, int nq, int page0, int page1) {
      const int slot = 2 * mw + (sg & 1);
      // the MMAs that read this slot two segments ago must be done
      if (!mbar_wait(bempty(slot), ((sg >> 1) & 1) ^ 1, wc)) return false;
      // index queries of tokens j0..j0+nq-1 -> rows (token, head), 128-byte
      // swizzled K-major; rows up to the MMA's N are zero-padded
      const int n_rows = 16 * ((nq + 1) >> 1);
      uint8_t* bt_s = smem + kOffB + slot * kBBytes;
      const uint8_t* qsrc = p.q_idx + (size_t)(s.q0 + j0) * kIdxHeads * kIdxDim;
#pragma unroll
      for (int half = 0; half < 2; ++half) {
        uint4 v[8];
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int e = lane + 32 * (8 * half + u), row = e >> 3, c = e & 7;
          v[u] = (row < nq * kIdxHeads) ? *reinterpret_cast<const uint4*>(qsrc + row * kIdxDim + c * 16)
                                        : make_uint4(0, 0, 0, 0);
        }
#pragma unroll
        for (int u = 0; u < 8; ++u) {
          const int e = lane + 32 * (8 * half + u), row = e >> 3, c = e & 7;
          if (row < n_rows) *reinterpret_cast<uint4*>(bt_s + row * kIdxDim + ((c ^ (row & 7)) << 4)) = v[u];
        }
      }
      fence_proxy_async_smem();
      __syncwarp();
      bool ok = true;
      if (lane == 0) {
        const uint32_t idesc = umma_idesc_e4m3(128, n_rows);
        const uint64_t bdesc = umma_desc_sw128(sbase + kOffB + slot * kBBytes);
        for (int page = page0; page < page1; ++page, ++it) {
          if ((it & 1) != mw) continue;
          const int st = it % kStages, acc = it % kAccs;
          if (!mbar_wait(full(st), (it / kStages) & 1, wc)) { ok = false; break; }
          if (!mbar_wait(tempty(acc), ((it / kAccs) & 1) ^ 1, wc)) { ok = false; break; }
          tc_fence_after();
          const uint64_t adesc = umma_desc_sw128(sbase + kOffStages + st * kIdxPageBytes);
#pragma unroll
          for (int k = 0; k < 4; ++k)  // K = 32 bytes per MMA: +32 B = +2 in the encoded address
            umma_e4m3(tmem + acc * 64, adesc + 2 * k, bdesc + 2 * k, idesc, k > 0);
          umma_commit(empty(st));
          umma_commit(tfull(acc));
        }
        if (ok) umma_commit(bempty(slot));
      }
      ok = __shfl_sync(0xffffffffu, (int)ok, 0) != 0;
      it = __shfl_sync(0xffffffffu, it, 0);
      ++sg;
      return ok;
    });
  } else {
    // ---------------- epilogue: three sets of four warps, set = it % 3 ----------
    // warps 3..6, 7..10, 11..14 -> TMEM lane quadrants 3,0,1,2; each warp
    // writes the max over its 32 token rows, the top-k phase takes the max of
    // the four.
    const int quad = warp & 3, set = (warp - 1 - kMmaWarps) >> 2;
    int it = 0;
    for_each_segment(p, s_prefix, s_sl, s_qsl, pg_begin, pg_end, [&](int b, const SeqInfo& s, int j0, int nq, int page0, int page1) {
      // head weights of the segment's tokens: read per page (L1 hits after the
      // first), not held in registers
      const float4* wseg = reinterpret_cast<const float4*>(p.w + (size_t)(s.q0 + j0) * kIdxHeads);
      const int* bt = p.block_table + (size_t)b * p.max_pages;
      float* srow = p.scores + ((size_t)(s.q0 + j0 + lane) * p.max_pages) * 4 + quad;
      int bt_nxt = page0 + lane < page1 ? bt[page0 + lane] : 0;
      int bt_cur = 0;
      for (int page = page0; page < page1; ++page, ++it) {
        if (((page - page0) & 31) == 0) {  // block-table entries 32 at a time
          bt_cur = bt_nxt;
          bt_nxt = page + 32 + lane < page1 ? bt[page + 32 + lane] : 0;
        }
        const int phys = __shfl_sync(0xffffffffu, bt_cur, (page - page0) & 31);
        if (it % kEpiSets != set) continue;
        const int acc = it % kAccs;
        if (!mbar_wait(tfull(acc), (it / kAccs) & 1, wc)) return false;
        tc_fence_after();
        // the columns of up to four query tokens (8 heads each) per load, the
        // loads of a page back to back, one wait per half; the accumulator is
        // released before the second half's math
        const uint32_t ta = tmem + ((uint32_t)(32 * quad) << 16) + acc * 64;
        uint32_t v0[32], v1[32];
        if (nq <= 2) tmem_ld32x32b_x16(ta, v0);
        else tmem_ld32x32b_x32(ta, v0);
        if (nq > 4) tmem_ld32x32b_x32(ta + 32, v1);
        tmem_wait_ld();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(tempty(acc));
        float mine = -INFINITY;
#pragma unroll
        for (int jj = 0; jj < kNqMax; ++jj) {
          if (jj < nq) {
            const float4 wa = __ldg(wseg + 2 * jj), wb = __ldg(wseg + 2 * jj + 1);
            const float wh[8] = {wa.x, wa.y, wa.z, wa.w, wb.x, wb.y, wb.z, wb.w};
            float sc = 0.f;
#pragma unroll
            for (int h = 0; h < kIdxHeads; ++h)
              sc = fmaf(wh[h], fmaxf(__uint_as_float(jj < 4 ? v0[8 * jj + h] : v1[8 * (jj - 4) + h]), 0.f), sc);
            const float x = warp_max_f32(sc);
            if (lane == jj) mine = x;
          }
        }
        if (lane < nq) {
          const bool bad = phys < 0 || phys >= p.n_pages;
          if (bad && lane == 0 && quad == 0) set_status(p.status, MSA_STATUS_BAD_PAGE);
          srow[(size_t)page * 4] = bad ? -INFINITY : mine;
        }
      }
      return true;
    });
  }

  // ---------------- scan teardown ---------------------------------------------
  tc_fence_before();
  __syncthreads();
  if (*s_abort) {
    // after an abort (bounded waits that ignore the flag): no tcgen05.mma may
    // still run when tensor memory is released, and no bulk copy may still be
    // writing the ring when its shared memory is reused or the CTA exits
    if (warp >= 1 && warp <= kMmaWarps && lane == 0) {
      umma_commit(done_bar(warp - 1));
      mbar_wait_drain(done_bar(warp - 1), 0, p.wait_ns);
    }
    if (warp == 0 && lane == 0) {
      const int n = *s_issued;
      for (int k = max(0, n - kStages); k < n; ++k) mbar_wait_drain(full(k % kStages), (k / kStages) & 1, p.wait_ns);
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }

  // ---------------- every block score written: top-k, tokens spread over CTAs --
  TopkSmem sm;
  sm.sc = reinterpret_cast<float*>(smem + kOffStages);                                 // 64 KB
  sm.cand = reinterpret_cast<unsigned long long*>(smem + kOffStages + 4 * kTopkStage);  // 16 KB
  sm.tmax = reinterpret_cast<unsigned long long*>(smem + kOffB);                       // NT x 8 B
  sm.win = reinterpret_cast<unsigned long long*>(smem + kOffB + 8 * kScanThreads);
  sm.misc = reinterpret_cast<int*>(sm.win + kTopK);
  // every CTA counts itself in, also after an abort of its own, so that the
  // barrier word is back at rest when the launch ends
  if (tid == 0) grid_barrier(p.sync, gridDim.x + p.barrier_extra, wc);
  __syncthreads();
  if (!*s_abort) {
    const TopkArgs ta{p.scores, p.max_pages, p.n_seqs, p.n_q_total, p.sel, p.n_sel, p.status, p.blk_lo,
                      p.blk_hi, p.cand};
    for (int j = blockIdx.x; j < p.n_q_total; j += gridDim.x) {
      select_token<kScanThreads>(ta, j, s_sl, s_qsl, sm);
      __syncthreads();
    }
  }
  if (tid == 0 && *s_abort) set_status(p.status, MSA_STATUS_TIMEOUT);
}

}  // namespace

cudaError_t launch_indexer_topk(const msa_cache* c, const uint8_t* q_idx, const float* w,
                                const int* block_table, int max_pages, const int* seq_lens,
                                const int* q_start_loc, int n_seqs, int n_q_total, int* sel,
                                int* n_sel, void* ws, int blk_lo, int blk_hi,
                                unsigned long long* cand, cudaStream_t stream) {
  if (n_q_total == 0 || n_seqs == 0) return cudaSuccess;
  // per-device launch set-up, done once (not a stream operation, so a later call
  // may be captured into a CUDA graph)
  static DeviceSetup setup;
  int dev = 0, n_sm = 0;
  cudaError_t e = setup.get(&dev, &n_sm, [](int) {
    return cudaFuncSetAttribute(indexer_scan_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)scan_smem_bytes(kMaxSeqs));
  });
  if (e != cudaSuccess) return e;
  const LaunchSettings ls = launch_settings();
  // workspace: [0, 256) grid-barrier words, then the partial block maxima
  unsigned long long* sync = static_cast<unsigned long long*>(ws);
  float* scores = reinterpret_cast<float*>(static_cast<uint8_t*>(ws) + kWsSyncBytes);
  ScanParams sp{static_cast<const uint8_t*>(c->idx_pool), c->n_pages, q_idx, w, block_table,
                max_pages, seq_lens, q_start_loc, n_seqs, n_q_total, scores, sel, n_sel, sync,
                c->status, ls.wait_ns, (ls.inject & kInjectBarrierTimeout) ? 1 : 0, blk_lo, blk_hi,
                cand};
  // one CTA per SM, all co-resident (cooperative launch): the top-k phase
  // waits for every CTA's scan at a grid barrier
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(n_sm);
  cfg.blockDim = dim3(kScanThreads);
  cfg.dynamicSmemBytes = scan_smem_bytes(n_seqs);
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, indexer_scan_kernel, sp);
}

}  // namespace msa

// ---------------------------------------------------------------------------
// Allocation-free variant of the indexer call.  Its scratch (the partial block
// maxima) lives in a file-scope device array instead of a caller workspace.
// Every GPU that loads the library holds this array until the process exits.
static __device__ __align__(256) float g_static_scores[msa::kStaticScratchBytes / sizeof(float)];

namespace msa {
namespace {
std::mutex g_static_mu;
float* g_static_ptr[64] = {nullptr};  // device address of g_static_scores, per device
}  // namespace

cudaError_t launch_indexer_topk_noalloc(const msa_cache* c, const uint8_t* q_idx, const float* w,
                                        const int* block_table, int max_pages, const int* seq_lens,
                                        const int* q_start_loc, int n_seqs, int n_q_total, int* sel,
                                        int* n_sel, cudaStream_t stream) {
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  float* scratch = nullptr;
  {
    // One-time set-up per device, with that device current: the host-side
    // symbol is only a stand-in, the kernels need the device address.
    std::lock_guard<std::mutex> lock(g_static_mu);
    if (!g_static_ptr[dev]) {
      void* ptr = nullptr;
      e = cudaGetSymbolAddress(&ptr, g_static_scores);
      if (e != cudaSuccess) return e;
      g_static_ptr[dev] = static_cast<float*>(ptr);
    }
    scratch = g_static_ptr[dev];
  }
  return launch_indexer_topk(c, q_idx, w, block_table, max_pages, seq_lens, q_start_loc, n_seqs,
                             n_q_total, sel, n_sel, static_cast<void*>(scratch), 0, 0x7FFFFFFF,
                             nullptr, stream);
}

}  // namespace msa
