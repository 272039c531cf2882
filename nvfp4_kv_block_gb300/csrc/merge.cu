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

}  // namespace

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
