// C ABI of libmsa.so: host-side validation and kernel launches.  See
// include/msa.h for the contract of every entry point.
#include <math.h>

#include "common.cuh"

namespace msa {
cudaError_t launch_quantize_insert(const msa_cache*, const float*, const float*, const float*,
                                   const int64_t*, int, cudaStream_t);
cudaError_t launch_absmax(const float*, int64_t, float*, cudaStream_t);
cudaError_t launch_indexer_topk(const msa_cache*, const uint8_t*, const float*, const int*, int,
                                const int*, const int*, int, int, int*, int*, void*, int, int,
                                unsigned long long*, cudaStream_t);
cudaError_t launch_merge_candidates(const unsigned long long*, int, const int*, const int*, int, int,
                                    int, int*, int*, int*, cudaStream_t);
cudaError_t launch_indexer_topk_noalloc(const msa_cache*, const uint8_t*, const float*, const int*,
                                        int, const int*, const int*, int, int, int*, int*,
                                        cudaStream_t);
cudaError_t launch_sparse_attn_tc(const msa_cache*, const uint8_t*, float, const int*, const int*,
                                  const int*, int, const int*, const int*, int, int, int, float*,
                                  float*, cudaStream_t);
cudaError_t launch_merge(const float*, const float*, int, int, int, float*, float*, cudaStream_t);
cudaError_t launch_debug_fp8_page(const msa_cache*, int64_t, uint8_t*, uint8_t*, cudaStream_t);
size_t decode_fused_workspace_bytes(int, int);
int decode_fused_max_seqs();
int decode_fused_max_tokens();
cudaError_t launch_decode_fused(const msa_cache*, const uint8_t*, const uint8_t*, const float*, float,
                                const int*, int, const int*, const int*, int, int, int*, int*, float*,
                                void*, cudaStream_t);
int qkv_heads_out();
cudaError_t launch_rope_table(float*, int, double, cudaStream_t);
cudaError_t launch_qkv_fused(const msa_cache*, const void*, const void*, int, int, const float*, const float*,
                             const float*, const float*, int, const int*, const int64_t*, float, uint8_t*,
                             float*, cudaStream_t);
cudaError_t launch_block_rows(const msa_cache*, int, const int*, int, uint8_t*, bool, cudaStream_t);

namespace {
std::atomic<unsigned long long> g_wait_ns{kDefaultWaitLimitNs};
std::atomic<int> g_inject{0};
}  // namespace

LaunchSettings launch_settings() {
  return LaunchSettings{g_wait_ns.load(std::memory_order_relaxed), g_inject.load(std::memory_order_relaxed)};
}
}  // namespace msa

namespace {

constexpr int32_t kMaxPagesPerSeq = 65536;

int check_cache(const msa_cache* c) {
  if (!c || !c->kv_pool || !c->idx_pool || c->n_pages <= 0) return MSA_ERR_INVALID_ARG;
  if (c->page_tokens != msa::kPageTokens || c->n_kv_heads != msa::kKvHeads ||
      c->head_dim != msa::kHeadDim || c->idx_dim != msa::kIdxDim)
    return MSA_ERR_UNSUPPORTED_SHAPE;
  if (!(c->s_enc_k > 0.f) || !(c->s_enc_v > 0.f) || !isfinite(c->s_enc_k) || !isfinite(c->s_enc_v))
    return MSA_ERR_INVALID_ARG;
  return MSA_OK;
}

int launched(cudaError_t e) { return e == cudaSuccess ? MSA_OK : MSA_ERR_LAUNCH_FAILED; }

}  // namespace

extern "C" {

int msa_quantize_kv_insert(const msa_cache* cache, const float* k, const float* v,
                           const float* idx_k, const int64_t* slot_mapping, int32_t n_tokens,
                           msa_stream_t stream) {
  if (int rc = check_cache(cache)) return rc;
  if (n_tokens < 0) return MSA_ERR_INVALID_ARG;
  if (n_tokens > 0 && (!k || !v || !idx_k || !slot_mapping)) return MSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k) | reinterpret_cast<uintptr_t>(v) |
       reinterpret_cast<uintptr_t>(idx_k)) & 15)
    return MSA_ERR_INVALID_ARG;  // float4 loads
  return launched(msa::launch_quantize_insert(cache, k, v, idx_k, slot_mapping, n_tokens,
                                              reinterpret_cast<cudaStream_t>(stream)));
}

size_t msa_indexer_workspace_bytes(int32_t n_q_total, int32_t max_pages) {
  // 256 bytes of grid-barrier words, then 4 partial maxima per (token, block)
  if (n_q_total <= 0 || max_pages <= 0) return 256;
  const size_t b = (size_t)n_q_total * (size_t)max_pages * 4 * sizeof(float);
  return 256 + (b + 255) / 256 * 256;
}

int msa_indexer_topk(const msa_cache* cache, const uint8_t* q_idx, const float* w,
                     int32_t n_idx_heads, const int32_t* block_table, int32_t max_pages,
                     const int32_t* seq_lens, const int32_t* q_start_loc, int32_t n_seqs,
                     int32_t n_q_total, int32_t topk, int32_t* sel, int32_t* n_sel, void* ws,
                     size_t ws_bytes, msa_stream_t stream) {
  if (int rc = check_cache(cache)) return rc;
  if (n_idx_heads != msa::kIdxHeads || topk != msa::kTopK) return MSA_ERR_UNSUPPORTED_SHAPE;
  if (n_seqs < 0 || n_q_total < 0 || max_pages <= 0) return MSA_ERR_INVALID_ARG;
  if (n_seqs > msa::kMaxSeqs || max_pages > kMaxPagesPerSeq) return MSA_ERR_UNSUPPORTED_SHAPE;
  if (n_q_total > 0 && (!q_idx || !w || !block_table || !seq_lens || !q_start_loc || !sel ||
                        !n_sel || !ws || n_seqs == 0))
    return MSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q_idx) & 15) || (reinterpret_cast<uintptr_t>(w) & 7) ||
      (reinterpret_cast<uintptr_t>(ws) & 15))
    return MSA_ERR_INVALID_ARG;
  if (ws_bytes < msa_indexer_workspace_bytes(n_q_total, max_pages))
    return MSA_ERR_WORKSPACE_TOO_SMALL;
  return launched(msa::launch_indexer_topk(cache, q_idx, w, block_table, max_pages, seq_lens,
                                           q_start_loc, n_seqs, n_q_total, sel, n_sel, ws, 0,
                                           0x7FFFFFFF, nullptr,
                                           reinterpret_cast<cudaStream_t>(stream)));
}

int msa_indexer_topk_range(const msa_cache* cache, const uint8_t* q_idx, const float* w,
                           int32_t n_idx_heads, const int32_t* block_table, int32_t max_pages,
                           const int32_t* seq_lens, const int32_t* q_start_loc, int32_t n_seqs,
                           int32_t n_q_total, int32_t topk, int32_t blk_lo, int32_t blk_hi,
                           uint64_t* cand, void* ws, size_t ws_bytes, msa_stream_t stream) {
  if (int rc = check_cache(cache)) return rc;
  if (n_idx_heads != msa::kIdxHeads || topk != msa::kTopK) return MSA_ERR_UNSUPPORTED_SHAPE;
  if (n_seqs < 0 || n_q_total < 0 || max_pages <= 0 || blk_lo < 0 || blk_hi < blk_lo)
    return MSA_ERR_INVALID_ARG;
  if (n_seqs > msa::kMaxSeqs || max_pages > kMaxPagesPerSeq) return MSA_ERR_UNSUPPORTED_SHAPE;
  if (n_q_total > 0 && (!q_idx || !w || !block_table || !seq_lens || !q_start_loc || !cand ||
                        !ws || n_seqs == 0))
    return MSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q_idx) & 15) || (reinterpret_cast<uintptr_t>(w) & 7) ||
      (reinterpret_cast<uintptr_t>(ws) & 15) || (reinterpret_cast<uintptr_t>(cand) & 7))
    return MSA_ERR_INVALID_ARG;
  if (ws_bytes < msa_indexer_workspace_bytes(n_q_total, max_pages))
    return MSA_ERR_WORKSPACE_TOO_SMALL;
  // sel / n_sel are not written in range mode; the candidates are
  return launched(msa::launch_indexer_topk(cache, q_idx, w, block_table, max_pages, seq_lens,
                                           q_start_loc, n_seqs, n_q_total, nullptr, nullptr, ws,
                                           blk_lo, blk_hi,
                                           reinterpret_cast<unsigned long long*>(cand),
                                           reinterpret_cast<cudaStream_t>(stream)));
}

int msa_indexer_merge_candidates(const msa_cache* cache, const uint64_t* cand, int32_t n_shards,
                                 const int32_t* seq_lens, const int32_t* q_start_loc,
                                 int32_t n_seqs, int32_t max_pages, int32_t n_q_total,
                                 int32_t topk, int32_t* sel, int32_t* n_sel, msa_stream_t stream) {
  if (!cache) return MSA_ERR_INVALID_ARG;
  if (topk != msa::kTopK) return MSA_ERR_UNSUPPORTED_SHAPE;
  if (n_shards < 1 || n_shards > 64 || n_seqs < 0 || n_q_total < 0 || max_pages <= 0)
    return MSA_ERR_INVALID_ARG;
  if (n_seqs > msa::kMaxSeqs || max_pages > kMaxPagesPerSeq) return MSA_ERR_UNSUPPORTED_SHAPE;
  if (n_q_total > 0 && (!cand || !seq_lens || !q_start_loc || !sel || !n_sel || n_seqs == 0))
    return MSA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(cand) & 7) return MSA_ERR_INVALID_ARG;
  return launched(msa::launch_merge_candidates(reinterpret_cast<const unsigned long long*>(cand),
                                               n_shards, seq_lens, q_start_loc, n_seqs, max_pages,
                                               n_q_total, sel, n_sel, cache->status,
                                               reinterpret_cast<cudaStream_t>(stream)));
}

int msa_indexer_topk_noalloc(const msa_cache* cache, const uint8_t* q_idx, const float* w,
                             int32_t n_idx_heads, const int32_t* block_table, int32_t max_pages,
                             const int32_t* seq_lens, const int32_t* q_start_loc, int32_t n_seqs,
                             int32_t n_q_total, int32_t topk, int32_t* sel, int32_t* n_sel,
                             msa_stream_t stream) {
  if (int rc = check_cache(cache)) return rc;
  if (n_idx_heads != msa::kIdxHeads || topk != msa::kTopK) return MSA_ERR_UNSUPPORTED_SHAPE;
  if (n_seqs < 0 || n_q_total < 0 || max_pages <= 0) return MSA_ERR_INVALID_ARG;
  if (n_seqs > msa::kMaxSeqs || max_pages > kMaxPagesPerSeq) return MSA_ERR_UNSUPPORTED_SHAPE;
  if (n_q_total > 0 && (!q_idx || !w || !block_table || !seq_lens || !q_start_loc || !sel ||
                        !n_sel || n_seqs == 0))
    return MSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(q_idx) & 15) || (reinterpret_cast<uintptr_t>(w) & 7))
    return MSA_ERR_INVALID_ARG;
  if (msa_indexer_workspace_bytes(n_q_total, max_pages) > MSA_INDEXER_NOALLOC_SCRATCH_BYTES)
    return MSA_ERR_SCRATCH_CAPACITY;
  return launched(msa::launch_indexer_topk_noalloc(cache, q_idx, w, block_table, max_pages,
                                                   seq_lens, q_start_loc, n_seqs, n_q_total, sel,
                                                   n_sel, reinterpret_cast<cudaStream_t>(stream)));
}

int msa_sparse_attn_decode(const msa_cache* cache, const uint8_t* q, int32_t n_q_heads,
                           float softmax_scale, const int32_t* sel, const int32_t* n_sel,
                           const int32_t* block_table, int32_t max_pages,
                           const int32_t* seq_lens, const int32_t* q_start_loc, int32_t n_seqs,
                           int32_t n_q_total, int32_t n_splits, float* o_part, float* lse_part,
                           msa_stream_t stream) {
  if (int rc = check_cache(cache)) return rc;
  if (n_q_heads != msa::kQHeads) return MSA_ERR_UNSUPPORTED_SHAPE;
  if (n_splits < 1 || n_splits > msa::kMaxSplits || n_q_total < 0 || n_seqs < 0 ||
      max_pages <= 0 || !(softmax_scale > 0.f) || !isfinite(softmax_scale))
    return MSA_ERR_INVALID_ARG;
  if (n_q_total > 65535 || n_seqs > msa::kMaxSeqs) return MSA_ERR_UNSUPPORTED_SHAPE;
  if (n_q_total > 0 && (!q || !sel || !n_sel || !block_table || !seq_lens || !q_start_loc ||
                        !o_part || !lse_part || n_seqs == 0))
    return MSA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(q) & 15) return MSA_ERR_INVALID_ARG;
  return launched(msa::launch_sparse_attn_tc(cache, q, softmax_scale, sel, n_sel, block_table,
                                          max_pages, seq_lens, q_start_loc, n_seqs, n_q_total,
                                          n_splits, o_part, lse_part,
                                          reinterpret_cast<cudaStream_t>(stream)));
}

int msa_merge_splits(const float* o_part, const float* lse_part, int32_t n_q_total,
                     int32_t n_q_heads, int32_t n_splits, float* out, float* lse,
                     msa_stream_t stream) {
  if (n_q_total < 0 || n_q_heads <= 0 || n_splits < 1 || n_splits > msa::kMaxSplits)
    return MSA_ERR_INVALID_ARG;
  if (n_q_heads > 1024 || n_q_total > 65535) return MSA_ERR_UNSUPPORTED_SHAPE;
  if (n_q_total > 0 && (!o_part || !lse_part || !out)) return MSA_ERR_INVALID_ARG;
  return launched(msa::launch_merge(o_part, lse_part, n_q_total, n_q_heads, n_splits, out, lse,
                                    reinterpret_cast<cudaStream_t>(stream)));
}

int msa_absmax(const float* x, int64_t n, float* amax, msa_stream_t stream) {
  if (n < 0 || !amax || (n > 0 && !x)) return MSA_ERR_INVALID_ARG;
  return launched(msa::launch_absmax(x, n, amax, reinterpret_cast<cudaStream_t>(stream)));
}

float msa_encode_scale(float amax) {
  if (!(amax > 0.f) || !isfinite(amax)) return 1.0f;
  volatile float num = 448.0f;  // one IEEE fp32 division, as the quantiser reading states
  return num / amax;
}

int msa_debug_fp8_page(const msa_cache* cache, int64_t page, uint8_t* k8, uint8_t* v8,
                       msa_stream_t stream) {
  if (int rc = check_cache(cache)) return rc;
  if (page < 0 || page >= cache->n_pages || !k8 || !v8) return MSA_ERR_INVALID_ARG;
  if ((reinterpret_cast<uintptr_t>(k8) | reinterpret_cast<uintptr_t>(v8)) & 15)
    return MSA_ERR_INVALID_ARG;
  return launched(
      msa::launch_debug_fp8_page(cache, page, k8, v8, reinterpret_cast<cudaStream_t>(stream)));
}

int msa_read_status(const msa_cache* cache, int32_t* host_out, msa_stream_t stream) {
  if (!cache || !host_out) return MSA_ERR_INVALID_ARG;
  if (!cache->status) {
    *host_out = 0;
    return MSA_OK;
  }
  cudaStream_t s = reinterpret_cast<cudaStream_t>(stream);
  if (cudaMemcpyAsync(host_out, cache->status, sizeof(int32_t), cudaMemcpyDeviceToHost, s) !=
      cudaSuccess)
    return MSA_ERR_LAUNCH_FAILED;
  return cudaStreamSynchronize(s) == cudaSuccess ? MSA_OK : MSA_ERR_LAUNCH_FAILED;
}

size_t msa_decode_fused_workspace_bytes(int32_t n_q_total, int32_t max_pages) {
  if (n_q_total <= 0 || max_pages <= 0) return 256;
  return msa::decode_fused_workspace_bytes(n_q_total, max_pages);
}

int msa_decode_fused(const msa_cache* cache, const uint8_t* q, const uint8_t* q_idx, const float* w,
                     int32_t n_q_heads, int32_t n_idx_heads, float softmax_scale,
                     const int32_t* block_table, int32_t max_pages, const int32_t* seq_lens,
                     const int32_t* q_start_loc, int32_t n_seqs, int32_t n_q_total, int32_t topk,
                     int32_t* sel, int32_t* n_sel, float* out, void* ws, size_t ws_bytes,
                     msa_stream_t stream) {
  if (int rc = check_cache(cache)) return rc;
  if (n_q_heads != msa::kQHeads || n_idx_heads != msa::kIdxHeads || topk != msa::kTopK)
    return MSA_ERR_UNSUPPORTED_SHAPE;
  if (n_seqs < 0 || n_q_total < 0 || max_pages <= 0 || !(softmax_scale > 0.f) || !isfinite(softmax_scale))
    return MSA_ERR_INVALID_ARG;
  if (n_seqs > msa::decode_fused_max_seqs() || n_q_total > msa::decode_fused_max_tokens() ||
      max_pages > kMaxPagesPerSeq)
    return MSA_ERR_UNSUPPORTED_SHAPE;
  if (n_q_total > 0 && (!q || !q_idx || !w || !block_table || !seq_lens || !q_start_loc || !sel ||
                        !n_sel || !out || !ws || n_seqs == 0))
    return MSA_ERR_INVALID_ARG;
  if (((reinterpret_cast<uintptr_t>(q) | reinterpret_cast<uintptr_t>(q_idx)) & 15) ||
      (reinterpret_cast<uintptr_t>(ws) & 15))
    return MSA_ERR_INVALID_ARG;
  if (ws_bytes < msa_decode_fused_workspace_bytes(n_q_total, max_pages)) return MSA_ERR_WORKSPACE_TOO_SMALL;
  return launched(msa::launch_decode_fused(cache, q, q_idx, w, softmax_scale, block_table, max_pages,
                                           seq_lens, q_start_loc, n_seqs, n_q_total, sel, n_sel, out,
                                           ws, reinterpret_cast<cudaStream_t>(stream)));
}

int msa_rope_table(float* cos_sin, int32_t max_pos, double base, msa_stream_t stream) {
  if (max_pos < 0 || (max_pos > 0 && !cos_sin) || !(base > 1.0) || !isfinite(base)) return MSA_ERR_INVALID_ARG;
  return launched(msa::launch_rope_table(cos_sin, max_pos, base, reinterpret_cast<cudaStream_t>(stream)));
}

int msa_qkv_project_insert(const msa_cache* cache, const void* x, const void* w, int32_t n_tokens,
                           int32_t d_model, const float* gamma_q, const float* gamma_k,
                           const float* gamma_idx, const float* cos_sin, int32_t max_pos,
                           const int32_t* positions, const int64_t* slot_mapping, float eps,
                           uint8_t* q8, float* y_out, msa_stream_t stream) {
  if (int rc = check_cache(cache)) return rc;
  if (n_tokens < 0 || max_pos <= 0 || !(eps >= 0.f) || !isfinite(eps)) return MSA_ERR_INVALID_ARG;
  if (d_model < 64 || d_model % 64 != 0 || d_model > 65536) return MSA_ERR_UNSUPPORTED_SHAPE;
  if (n_tokens > 0 && (!x || !w || !gamma_q || !gamma_k || !gamma_idx || !cos_sin || !positions ||
                       !slot_mapping || !q8))
    return MSA_ERR_INVALID_ARG;
  if (((reinterpret_cast<uintptr_t>(x) | reinterpret_cast<uintptr_t>(w) | reinterpret_cast<uintptr_t>(cos_sin) |
        reinterpret_cast<uintptr_t>(q8) | reinterpret_cast<uintptr_t>(y_out)) & 15))
    return MSA_ERR_INVALID_ARG;
  return launched(msa::launch_qkv_fused(cache, x, w, n_tokens, d_model, gamma_q, gamma_k, gamma_idx, cos_sin,
                                        max_pos, positions, slot_mapping, eps, q8, y_out,
                                        reinterpret_cast<cudaStream_t>(stream)));
}

size_t msa_block_row_bytes(int32_t n_layers) {
  return n_layers > 0 ? (size_t)n_layers * (msa::kKvPageBytes + msa::kIdxPageBytes) : 0;
}

static int block_rows(const msa_cache* layers, int32_t n_layers, const int32_t* pages,
                      int32_t n_blocks, uint8_t* rows, bool pack, msa_stream_t stream) {
  if (!layers || n_layers <= 0 || n_blocks < 0) return MSA_ERR_INVALID_ARG;
  if (n_layers > msa::kMaxLayers) return MSA_ERR_UNSUPPORTED_SHAPE;
  for (int l = 0; l < n_layers; ++l) {
    if (int rc = check_cache(&layers[l])) return rc;
    if ((reinterpret_cast<uintptr_t>(layers[l].kv_pool) | reinterpret_cast<uintptr_t>(layers[l].idx_pool)) & 15)
      return MSA_ERR_INVALID_ARG;
  }
  if (n_blocks > 0 && (!pages || !rows)) return MSA_ERR_INVALID_ARG;
  if (reinterpret_cast<uintptr_t>(rows) & 15) return MSA_ERR_INVALID_ARG;
  return launched(msa::launch_block_rows(layers, n_layers, pages, n_blocks, rows, pack,
                                         reinterpret_cast<cudaStream_t>(stream)));
}

int msa_pack_blocks(const msa_cache* layers, int32_t n_layers, const int32_t* pages,
                    int32_t n_blocks, uint8_t* rows, msa_stream_t stream) {
  return block_rows(layers, n_layers, pages, n_blocks, rows, true, stream);
}

int msa_unpack_blocks(const msa_cache* layers, int32_t n_layers, const uint8_t* rows,
                      const int32_t* pages, int32_t n_blocks, msa_stream_t stream) {
  return block_rows(layers, n_layers, pages, n_blocks, const_cast<uint8_t*>(rows), false, stream);
}

int msa_debug_set_fault_injection(int32_t flags, uint64_t wait_limit_ns) {
  if (flags & ~(MSA_INJECT_BARRIER_TIMEOUT | MSA_INJECT_ATTENTION_TIMEOUT)) return MSA_ERR_INVALID_ARG;
  msa::g_wait_ns.store(wait_limit_ns ? (unsigned long long)wait_limit_ns : msa::kDefaultWaitLimitNs,
                       std::memory_order_relaxed);
  msa::g_inject.store(flags, std::memory_order_relaxed);
  return MSA_OK;
}

const char* msa_status_string(int code) {
  switch (code) {
    case MSA_OK: return "ok";
    case MSA_ERR_INVALID_ARG: return "invalid argument";
    case MSA_ERR_UNSUPPORTED_SHAPE: return "unsupported shape";
    case MSA_ERR_WORKSPACE_TOO_SMALL: return "workspace too small";
    case MSA_ERR_LAUNCH_FAILED: return "kernel launch failed";
    case MSA_ERR_SCRATCH_CAPACITY: return "larger than the library's static scratch";
    case MSA_STATUS_BAD_SLOT: return "device: slot outside the pool";
    case MSA_STATUS_BAD_PAGE: return "device: block table entry outside the pool";
    case MSA_STATUS_BAD_SEQ: return "device: inconsistent sequence lengths / query counts";
    case MSA_STATUS_BAD_SELECTION: return "device: selected block outside 0..r_j";
    case MSA_STATUS_TIMEOUT: return "device: a bounded wait timed out; results invalid";
    default: return code > 0 ? "device: several status bits" : "unknown error";
  }
}

}  // extern "C"
