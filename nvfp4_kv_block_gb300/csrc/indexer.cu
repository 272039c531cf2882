// Lightweight indexer: FP8 index scan with per-block max, then top-16 + recent.
//
// "vLLM Delivers Day-0 Support for MiniMax-M3.1-Flash" blog, section "Sparse
// attention still scans an index": KV lives in 128-token blocks, the indexer
// scores the context, keeps 16 blocks plus the most recent one, and reads 128
// index bytes per token.  Section "Parallelize index work across context":
// splitting the scan keeps the selection exact (each block score is computed
// once, by one warp, and the selection runs over all of them).
//
// Scan (hot loop): the pages to scan (blocks 0..r_last-1 of every sequence)
// are flattened and cut into equal contiguous ranges, one per warp.  A warp
// streams its pages 16 tokens at a time with 128-bit loads straight into
// mma.sync fragments (tokens are the M dimension, the 8 indexer heads the N
// dimension, the 128 dims the K dimension: 4 x m16n8k32 E4M3 MMAs per 16
// tokens and query token), applies ReLU and the head weights on the fp32
// accumulators, sums the heads with two quad shuffles and keeps the block max
// in registers.  Only one fp32 per (query token, block) is written.
//
// Fragment mapping.  A page row (one token) holds 8 chunks of 16 dims,
// chunk c stored at position c ^ (token & 7).  Lane (g = lane/4, t = lane%4)
// loads chunks t and t+4 of tokens g and g+8 of the 16-token tile; word s of
// chunk t (dims 16t+4s..16t+4s+3) is the A fragment of k-step s at k columns
// 4t..4t+3, word s of chunk t+4 the one at columns 16+4t..16+4t+3.  The index
// query uses the same dims -> (k-step, column) map, so the dot product is
// unchanged.
#include "common.cuh"

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
  float* scores;  // [T][max_pages]
  int* status;
};

constexpr int kScanThreads = 128;

// Pages to scan for sequence b: blocks 0..r_last-1, r_last = (seq_len-1)/128.
__device__ __forceinline__ int scan_pages(const SeqInfo& s) {
  return (s.ok && s.seq_len > 0 && s.n_q > 0) ? (s.seq_len - 1) / kPageTokens : 0;
}

template <int NQ>
__global__ void __launch_bounds__(kScanThreads) indexer_scan_kernel(ScanParams p) {
  __shared__ int s_prefix[kMaxSeqs + 1];
  __shared__ int s_warp_sum[kScanThreads / 32];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;

  // -- exclusive prefix over sequences of the pages each one scans ------------
  {
    const int per = (p.n_seqs + kScanThreads - 1) / kScanThreads;
    const int b0 = tid * per;
    int local = 0;
    for (int b = b0; b < b0 + per && b < p.n_seqs; ++b) {
      const SeqInfo s = load_seq(b, p.seq_lens, p.q_start_loc, p.max_pages, p.n_q_total);
      if (!s.ok) set_status(p.status, MSA_STATUS_BAD_SEQ);
      local += scan_pages(s);
    }
    int incl = local;
#pragma unroll
    for (int o = 1; o < 32; o <<= 1) {
      const int y = __shfl_up_sync(0xffffffffu, incl, o);
      if (lane >= o) incl += y;
    }
    if (lane == 31) s_warp_sum[warp] = incl;
    __syncthreads();
    int base = 0;
    for (int i = 0; i < warp; ++i) base += s_warp_sum[i];
    int run = base + incl - local;
    for (int b = b0; b < b0 + per && b < p.n_seqs; ++b) {
      s_prefix[b] = run;
      run += scan_pages(load_seq(b, p.seq_lens, p.q_start_loc, p.max_pages, p.n_q_total));
    }
    if (tid == kScanThreads - 1) s_prefix[p.n_seqs] = base + incl;
    __syncthreads();
  }
  const long long total = s_prefix[p.n_seqs];
  const long long gw = (long long)blockIdx.x * (kScanThreads / 32) + warp;
  const long long nw = (long long)gridDim.x * (kScanThreads / 32);
  long long pg = gw * total / nw;
  const long long pg_end = (gw + 1) * total / nw;
  if (pg >= pg_end) return;

  const int g = lane >> 2, t = lane & 3;
  // byte offsets, inside a 16-token tile, of this lane's four 16-byte loads
  const int off_a0 = g * kIdxDim + ((t ^ g) << 4);        // token g,   chunk t
  const int off_a1 = g * kIdxDim + (((t + 4) ^ g) << 4);  // token g,   chunk t+4
  const int off_a2 = off_a0 + 8 * kIdxDim;                // token g+8, chunk t
  const int off_a3 = off_a1 + 8 * kIdxDim;                // token g+8, chunk t+4

  // sequence holding page pg
  int b = 0;
  {
    int lo = 0, hi = p.n_seqs - 1;
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (s_prefix[mid] <= pg) lo = mid; else hi = mid - 1;
    }
    b = lo;
  }
  while (pg < pg_end) {
    while (s_prefix[b + 1] <= pg) ++b;
    const SeqInfo s = load_seq(b, p.seq_lens, p.q_start_loc, p.max_pages, p.n_q_total);
    const int page0 = (int)(pg - s_prefix[b]);
    const int page1 = (int)(min((long long)s_prefix[b + 1], pg_end) - s_prefix[b]);
    const int* bt = p.block_table + (size_t)b * p.max_pages;
    for (int j0 = 0; j0 < s.n_q; j0 += NQ) {
      const int nq = min(NQ, s.n_q - j0);
      // index-query fragments and head weights of up to NQ query tokens
      uint4 qb0[NQ], qb1[NQ];
      float w0[NQ], w1[NQ];
#pragma unroll
      for (int jj = 0; jj < NQ; ++jj) {
        const int tok = s.q0 + j0 + min(jj, nq - 1);
        const uint8_t* qrow = p.q_idx + ((size_t)tok * kIdxHeads + g) * kIdxDim;
        qb0[jj] = *reinterpret_cast<const uint4*>(qrow + 16 * t);
        qb1[jj] = *reinterpret_cast<const uint4*>(qrow + 64 + 16 * t);
        const float2 wv = *reinterpret_cast<const float2*>(p.w + (size_t)tok * kIdxHeads + 2 * t);
        w0[jj] = wv.x;
        w1[jj] = wv.y;
      }
      // stream tiles: 8 tiles of 16 tokens per page, one tile prefetched ahead
      const int n_tiles = (page1 - page0) * 8;
      auto tile_base = [&](int tile, bool& bad) -> const uint8_t* {
        const int phys = bt[page0 + (tile >> 3)];
        bad = phys < 0 || phys >= p.n_pages;
        const int64_t pp = bad ? 0 : phys;
        return p.idx_pool + pp * kIdxPageBytes + (tile & 7) * (16 * kIdxDim);
      };
      bool bad_cur;
      const uint8_t* src = tile_base(0, bad_cur);
      uint4 cur0 = ld_stream_v4(src + off_a0), cur1 = ld_stream_v4(src + off_a1);
      uint4 cur2 = ld_stream_v4(src + off_a2), cur3 = ld_stream_v4(src + off_a3);
      float bmax[NQ];
#pragma unroll
      for (int jj = 0; jj < NQ; ++jj) bmax[jj] = -INFINITY;
      for (int tile = 0; tile < n_tiles; ++tile) {
        uint4 nxt0 = cur0, nxt1 = cur1, nxt2 = cur2, nxt3 = cur3;
        bool bad_nxt = false;
        if (tile + 1 < n_tiles) {
          const uint8_t* ns = tile_base(tile + 1, bad_nxt);
          nxt0 = ld_stream_v4(ns + off_a0);
          nxt1 = ld_stream_v4(ns + off_a1);
          nxt2 = ld_stream_v4(ns + off_a2);
          nxt3 = ld_stream_v4(ns + off_a3);
        }
        const uint32_t A0[4] = {cur0.x, cur0.y, cur0.z, cur0.w};
        const uint32_t A1[4] = {cur1.x, cur1.y, cur1.z, cur1.w};
        const uint32_t A2[4] = {cur2.x, cur2.y, cur2.z, cur2.w};
        const uint32_t A3[4] = {cur3.x, cur3.y, cur3.z, cur3.w};
#pragma unroll
        for (int jj = 0; jj < NQ; ++jj) {
          if (jj < nq) {
            const uint32_t B0[4] = {qb0[jj].x, qb0[jj].y, qb0[jj].z, qb0[jj].w};
            const uint32_t B1[4] = {qb1[jj].x, qb1[jj].y, qb1[jj].z, qb1[jj].w};
            float acc[4] = {0.f, 0.f, 0.f, 0.f};
            // a0: token g dims of chunk t; a1: token g+8 chunk t; a2: token g chunk t+4; a3: token g+8 chunk t+4
#pragma unroll
            for (int ks = 0; ks < 4; ++ks) mma_e4m3(acc, A0[ks], A2[ks], A1[ks], A3[ks], B0[ks], B1[ks]);
            // rows g, g+8 (tokens); columns 2t, 2t+1 (heads)
            float v0 = fmaf(w1[jj], fmaxf(acc[1], 0.f), w0[jj] * fmaxf(acc[0], 0.f));
            float v1 = fmaf(w1[jj], fmaxf(acc[3], 0.f), w0[jj] * fmaxf(acc[2], 0.f));
            v0 += __shfl_xor_sync(0xffffffffu, v0, 1);
            v1 += __shfl_xor_sync(0xffffffffu, v1, 1);
            v0 += __shfl_xor_sync(0xffffffffu, v0, 2);
            v1 += __shfl_xor_sync(0xffffffffu, v1, 2);
            bmax[jj] = fmaxf(bmax[jj], fmaxf(v0, v1));
          }
        }
        if ((tile & 7) == 7) {
          const int page = page0 + (tile >> 3);
#pragma unroll
          for (int jj = 0; jj < NQ; ++jj) {
            float m = bmax[jj];
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 4));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 8));
            m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, 16));
            if (lane == jj && jj < nq)
              p.scores[(size_t)(s.q0 + j0 + jj) * p.max_pages + page] = bad_cur ? -INFINITY : m;
            bmax[jj] = -INFINITY;
          }
          if (bad_cur && lane == 0) set_status(p.status, MSA_STATUS_BAD_PAGE);
        }
        cur0 = nxt0; cur1 = nxt1; cur2 = nxt2; cur3 = nxt3;
        bad_cur = bad_nxt;
      }
    }
    pg = s_prefix[b] + page1;
    ++b;
  }
}

// ---------------------------------------------------------------------------
// Top-16 + recent per query token.  Keys are (ordered score << 32) | ~block,
// unique, larger = better (higher score, then lower block).  256 threads:
// each takes the max key of its strided blocks; the 16th largest of those 256
// maxima, theta, is a lower bound of the 16th largest key overall (the 16
// largest maxima are 16 distinct keys), so every winner has key >= theta.  The
// few candidates >= theta are ranked exactly by counting.
constexpr int kTopkThreads = 256;
constexpr int kMaxCand = 4096;

struct TopkParams {
  const float* scores;
  int max_pages;
  const int* seq_lens;
  const int* q_start_loc;
  int n_seqs;
  int n_q_total;
  int* sel;
  int* n_sel;
  int* status;
};

__device__ __forceinline__ unsigned long long block_key(const float* row, int blk) {
  return ((unsigned long long)ordered_bits(row[blk]) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)blk);
}

__global__ void __launch_bounds__(kTopkThreads) topk_kernel(TopkParams p) {
  __shared__ unsigned long long s_key[kTopkThreads];
  __shared__ unsigned long long s_cand[kMaxCand];
  __shared__ int s_win[kTopK];
  __shared__ unsigned long long s_theta;
  __shared__ int s_ncand;
  const int j = blockIdx.x, tid = threadIdx.x;
  const int b = find_seq(p.q_start_loc, p.n_seqs, j);
  const SeqInfo s = load_seq(b, p.seq_lens, p.q_start_loc, p.max_pages, p.n_q_total);
  int* out = p.sel + (size_t)j * kSelStride;
  if (!s.ok || j < s.q0 || j >= s.q0 + s.n_q) {
    if (tid == 0) set_status(p.status, MSA_STATUS_BAD_SEQ);
    if (tid < kSelStride) out[tid] = -1;
    if (tid == 0) p.n_sel[j] = 0;
    return;
  }
  const int pos = s.seq_len - s.n_q + (j - s.q0);
  const int r = pos / kPageTokens;
  const float* row = p.scores + (size_t)j * p.max_pages;
  if (r <= kTopK) {
    if (tid < kSelStride) out[tid] = tid <= r ? tid : -1;
    if (tid == 0) p.n_sel[j] = r + 1;
    return;
  }
  unsigned long long mykey = 0;
  for (int blk = tid; blk < r; blk += kTopkThreads) {
    const unsigned long long k = block_key(row, blk);
    mykey = k > mykey ? k : mykey;
  }
  s_key[tid] = mykey;
  if (tid == 0) s_ncand = 0;
  __syncthreads();
  int rank = 0;
  for (int i = 0; i < kTopkThreads; ++i) rank += s_key[i] > mykey;
  if (rank == kTopK - 1) s_theta = mykey;
  __syncthreads();
  const unsigned long long theta = s_theta;
  for (int blk = tid; blk < r; blk += kTopkThreads) {
    const unsigned long long k = block_key(row, blk);
    if (k >= theta) {
      const int slot = atomicAdd(&s_ncand, 1);
      if (slot < kMaxCand) s_cand[slot] = k;
    }
  }
  __syncthreads();
  const int nc = min(s_ncand, kMaxCand);
  for (int c = tid; c < nc; c += kTopkThreads) {
    const unsigned long long k = s_cand[c];
    int rk = 0;
    for (int i = 0; i < nc; ++i) rk += s_cand[i] > k;
    if (rk < kTopK) s_win[rk] = (int)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFu));
  }
  __syncthreads();
  if (tid < kTopK) {
    const int blk = s_win[tid];
    int at = 0;
#pragma unroll
    for (int i = 0; i < kTopK; ++i) at += s_win[i] < blk;
    out[at] = blk;
  }
  if (tid == 0) {
    out[kTopK] = r;
    p.n_sel[j] = kTopK + 1;
  }
}

}  // namespace

cudaError_t launch_indexer_topk(const msa_cache* c, const uint8_t* q_idx, const float* w,
                                const int* block_table, int max_pages, const int* seq_lens,
                                const int* q_start_loc, int n_seqs, int n_q_total, int* sel,
                                int* n_sel, float* scores, cudaStream_t stream) {
  if (n_q_total == 0 || n_seqs == 0) return cudaSuccess;
  ScanParams sp{static_cast<const uint8_t*>(c->idx_pool), c->n_pages, q_idx, w, block_table,
                max_pages, seq_lens, q_start_loc, n_seqs, n_q_total, scores, c->status};
  const int blocks = 152 * 8;
  if (n_q_total == n_seqs)
    indexer_scan_kernel<1><<<blocks, kScanThreads, 0, stream>>>(sp);
  else
    indexer_scan_kernel<8><<<blocks, kScanThreads, 0, stream>>>(sp);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  TopkParams tp{scores, max_pages, seq_lens, q_start_loc, n_seqs, n_q_total, sel, n_sel, c->status};
  topk_kernel<<<n_q_total, kTopkThreads, 0, stream>>>(tp);
  return cudaGetLastError();
}

}  // namespace msa
