// Log-sum-exp merge of the attention splits, and a debug view of the FP8
// operands the attention kernel feeds to the tensor core.
//
// "vLLM Delivers Day-0 Support for MiniMax-M3.1-Flash" blog, section "Sparse
// attention still scans an index": attention is exact over the selected
// blocks; a split-context decode computes it per split as (o_s, lse_s) and
// combines them with softmax weights exp(lse_s - max) -- the same result as
// one softmax over the union of the splits' keys.
#include "common.cuh"

namespace msa {
namespace {

// out[j][h][:] = sum_s exp(lse_s - L) o_s and lse_out[j][h] = L; one CTA per
// (token, head), thread = channel.
__global__ void __launch_bounds__(kHeadDim) merge_kernel(const float* __restrict__ o_part,
                                                         const float* __restrict__ lse_part,
                                                         int n_heads, int n_splits,
                                                         float* __restrict__ out,
                                                         float* __restrict__ lse_out) {
  const int row = blockIdx.x;  // j * n_heads + h
  const int j = row / n_heads, h = row % n_heads;
  const int ch = threadIdx.x;
  pdl_wait();  // partials come from the attention kernel
  float M = -INFINITY;
  for (int sp = 0; sp < n_splits; ++sp)
    M = fmaxf(M, lse_part[((size_t)j * n_splits + sp) * n_heads + h]);
  float num = 0.f, den = 0.f;
  if (M != -INFINITY) {
    for (int sp = 0; sp < n_splits; ++sp) {
      const size_t r = ((size_t)j * n_splits + sp) * n_heads + h;
      const float f = __expf(lse_part[r] - M);
      den += f;
      num += f * o_part[r * kHeadDim + ch];
    }
  }
  out[(size_t)row * kHeadDim + ch] = den > 0.f ? num / den : 0.f;
  if (lse_out && ch == 0) lse_out[row] = den > 0.f ? M + logf(den) : -INFINITY;
}

// Dequantised FP8 operands of one page in logical order, through the same
// table and dequant8 as the attention kernel.  Thread = (head, token, group).
__global__ void __launch_bounds__(256) debug_fp8_page_kernel(const uint8_t* __restrict__ kv_pool,
                                                             int64_t page, uint8_t* k8,
                                                             uint8_t* v8) {
  __shared__ uint2 s_tab[256];
  build_dequant_table(s_tab, threadIdx.x, blockDim.x);
  __syncthreads();
  const int id = blockIdx.x * blockDim.x + threadIdx.x;  // < 2 * 4 * 128 * 8
  if (id >= 2 * kKvHeads * kPageTokens * 8) return;
  const int grp = id & 7, tok = (id >> 3) & 127, head = (id >> 10) & 3, isv = id >> 12;
  const uint8_t* base = kv_pool + (size_t)page * kKvPageBytes + head * kHeadBytes;
  // group grp = 8 code bytes at offset 8 (grp & 1) of code chunk grp >> 1
  const uint8_t* codes = base + (isv ? kOffVc : kOffKc) + tok * 64 +
                         (code_chunk_pos(grp >> 1, tok) << 4) + (grp & 1) * 8;
  const uint8_t sb = base[(isv ? kOffVs : kOffKs) + grp * kPageTokens + tok];
  const uint2 c = *reinterpret_cast<const uint2*>(codes);
  const uint2 d0 = dequant8(c.x, s_tab[sb]), d1 = dequant8(c.y, s_tab[sb]);
  uint8_t* dst = (isv ? v8 : k8) + ((size_t)head * kPageTokens + tok) * kHeadDim + grp * 16;
  *reinterpret_cast<uint4*>(dst) = make_uint4(d0.x, d0.y, d1.x, d1.y);
}

// Merge of the indexer's per-shard candidates (blog, "Parallelize index work
// across context": each GPU scans part of the context, the local candidates
// are exchanged, and a merge gives the final top-16 -- exactly the selection
// of one scan over everything, because every block competes once, with the
// same score, in exactly one shard).  One warp per query token: its
// n_shards x 16 keys are staged in shared memory and ranked by counting (keys
// are unique: the block id is part of the key; zero = empty); the 16 best
// non-empty keys win, output in ascending block order, then the recent block.
constexpr int kMergeWarps = 4;
constexpr int kMaxShards = 64;

__global__ void __launch_bounds__(32 * kMergeWarps) merge_candidates_kernel(
    const unsigned long long* __restrict__ cand, int n_shards, const int* __restrict__ seq_lens,
    const int* __restrict__ q_start_loc, int n_seqs, int max_pages, int n_q_total, int* sel,
    int* n_sel, int* status) {
  __shared__ unsigned long long s_keys[kMergeWarps][kMaxShards * kTopK];
  __shared__ unsigned long long s_win[kMergeWarps][kTopK];
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  const int j = blockIdx.x * kMergeWarps + wid;
  pdl_wait();  // candidates come from the range scans
  if (j >= n_q_total) return;
  unsigned long long* keys = s_keys[wid];
  unsigned long long* win = s_win[wid];
  int* out = sel + (size_t)j * kSelStride;
  const int b = find_seq(q_start_loc, n_seqs, j);
  const SeqInfo s = load_seq(b, seq_lens, q_start_loc, max_pages, n_q_total);
  if (!(s.ok && s.q0 <= j && j < s.q0 + s.n_q)) {
    if (lane == 0) set_status(status, MSA_STATUS_BAD_SEQ);
    if (lane < kSelStride) out[lane] = -1;
    if (lane == 0) n_sel[j] = 0;
    return;
  }
  const int r = (s.seq_len - s.n_q + (j - s.q0)) / kPageTokens;
  const int nk = n_shards * kTopK;
  for (int i = lane; i < nk; i += 32)
    keys[i] = cand[((size_t)(i / kTopK) * n_q_total + j) * kTopK + (i % kTopK)];
  if (lane < kTopK) win[lane] = 0ull;
  __syncwarp();
  for (int i = lane; i < nk; i += 32) {
    const unsigned long long k = keys[i];
    if (k == 0ull) continue;
    int rk = 0;
    for (int t = 0; t < nk; ++t) rk += keys[t] > k;
    if (rk < kTopK) win[rk] = k;
  }
  __syncwarp();
  // winners are ranks 0 .. nw-1 (ranks of distinct non-zero keys are distinct)
  const unsigned long long mine = lane < kTopK ? win[lane] : 0ull;
  const int nw = __popc(__ballot_sync(0xffffffffu, mine != 0ull));
  const int blk = (int)(0xFFFFFFFFu - (uint32_t)(mine & 0xFFFFFFFFu));
  bool bad = false;
  if (mine != 0ull) {
    bad = blk < 0 || blk >= r;
    int at = 0;
    for (int t = 0; t < nw; ++t) {
      const unsigned long long o = win[t];
      at += (int)(0xFFFFFFFFu - (uint32_t)(o & 0xFFFFFFFFu)) < blk;
    }
    out[at] = blk;
  }
  if (__any_sync(0xffffffffu, bad) && lane == 0) set_status(status, MSA_STATUS_BAD_SELECTION);
  if (lane == nw) out[nw] = r;
  if (lane > nw && lane < kSelStride) out[lane] = -1;
  if (lane == 0) n_sel[j] = nw + 1;
}

}  // namespace

cudaError_t launch_merge_candidates(const unsigned long long* cand, int n_shards, const int* seq_lens,
                                    const int* q_start_loc, int n_seqs, int max_pages, int n_q_total,
                                    int* sel, int* n_sel, int* status, cudaStream_t stream) {
  if (n_q_total == 0) return cudaSuccess;
  return launch_pdl(merge_candidates_kernel, dim3((n_q_total + kMergeWarps - 1) / kMergeWarps),
                    dim3(32 * kMergeWarps), 0, stream, cand, n_shards, seq_lens, q_start_loc, n_seqs,
                    max_pages, n_q_total, sel, n_sel, status);
}

cudaError_t launch_merge(const float* o_part, const float* lse_part, int n_q_total, int n_heads,
                         int n_splits, float* out, float* lse_out, cudaStream_t stream) {
  if (n_q_total == 0) return cudaSuccess;
  return launch_pdl(merge_kernel, dim3(n_q_total * n_heads), dim3(kHeadDim), 0, stream, o_part,
                    lse_part, n_heads, n_splits, out, lse_out);
}

cudaError_t launch_debug_fp8_page(const msa_cache* c, int64_t page, uint8_t* k8, uint8_t* v8,
                                  cudaStream_t stream) {
  debug_fp8_page_kernel<<<(2 * kKvHeads * kPageTokens * 8) / 256, 256, 0, stream>>>(
      static_cast<const uint8_t*>(c->kv_pool), page, k8, v8);
  return cudaGetLastError();
}

}  // namespace msa
