// NVFP4 quantise-and-insert of new K/V tokens and FP8 index keys.
//
// The KV cache is stored as NVFP4 and the index as 128 FP8 bytes per token
// ("vLLM Delivers Day-0 Support for MiniMax-M3.1-Flash" blog, sections
// "Sparse attention still scans an index" and "Capacity savings must pay for
// conversion").  Two-level scale: one E4M3 scale per 16 channels of a token
// and head, on top of an fp32 per-tensor encode scale s_enc.
//
// Work decomposition: one warp per (token, job), job 0..3 = K heads, 4..7 = V
// heads, 8 = index key; lane l owns channels 4l..4l+3, so a 16-channel group
// is four lanes and its amax is two shuffles away.  Write-bound, off the
// decode path.
#include "common.cuh"

namespace msa {
namespace {

__global__ void __launch_bounds__(256) quantize_insert_kernel(
    uint8_t* __restrict__ kv_pool, uint8_t* __restrict__ idx_pool, int64_t n_pages,
    const float* __restrict__ k, const float* __restrict__ v, const float* __restrict__ idx_k,
    const int64_t* __restrict__ slot_mapping, int n_tokens, float s_enc_k, float s_enc_v,
    int* status) {
  const int lane = threadIdx.x & 31;
  const long long n_jobs = (long long)n_tokens * 9;
  const long long warp0 = ((long long)blockIdx.x * blockDim.x + threadIdx.x) >> 5;
  const long long nwarps = ((long long)gridDim.x * blockDim.x) >> 5;
  for (long long job = warp0; job < n_jobs; job += nwarps) {
    const int t = (int)(job / 9);
    const int kind = (int)(job % 9);
    const int64_t slot = slot_mapping[t];
    if (slot < 0) continue;
    const int64_t page = slot / kPageTokens;
    const int off = (int)(slot % kPageTokens);
    if (page >= n_pages) {
      if (lane == 0) set_status(status, MSA_STATUS_BAD_SLOT);
      continue;
    }
    if (kind == 8) {
      // index key: 128 fp32 -> E4M3, chunk c = lane / 4 lands at chunk c ^ (off & 7)
      const float4 x = reinterpret_cast<const float4*>(idx_k + (size_t)t * kIdxDim)[lane];
      const uint32_t lo = f32x2_to_e4m3x2(x.x, x.y);
      const uint32_t hi = f32x2_to_e4m3x2(x.z, x.w);
      uint32_t word = 0;
      word |= canon_zero(lo & 0xFF);
      word |= canon_zero(lo >> 8) << 8;
      word |= canon_zero(hi & 0xFF) << 16;
      word |= canon_zero(hi >> 8) << 24;
      const int c = lane >> 2;
      uint8_t* dst = idx_pool + (size_t)page * kIdxPageBytes + off * kIdxDim +
                     ((c ^ (off & 7)) << 4) + ((lane & 3) << 2);
      *reinterpret_cast<uint32_t*>(dst) = word;
      continue;
    }
    const bool is_v = kind >= 4;
    const int g = kind & 3;
    const float s_enc = is_v ? s_enc_v : s_enc_k;
    const float* src = (is_v ? v : k) + ((size_t)t * kKvHeads + g) * kHeadDim;
    const float4 x = reinterpret_cast<const float4*>(src)[lane];
    const float ax = fabsf(x.x), ay = fabsf(x.y), az = fabsf(x.z), aw = fabsf(x.w);
    float a = fmaxf(fmaxf(ax, ay), fmaxf(az, aw));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 1));
    a = fmaxf(a, __shfl_xor_sync(0xffffffffu, a, 2));
    // sb = E4M3(fp32(fp32(a / 6) * s_enc)); IEEE divide and multiply, no contraction
    const uint32_t sb_byte = f32_to_e4m3(__fmul_rn(__fdiv_rn(a, 6.0f), s_enc));
    const float sb = e4m3_to_f32(sb_byte);
    uint32_t c0 = e2m1_code(__fmul_rn(ax, s_enc), sb);
    uint32_t c1 = e2m1_code(__fmul_rn(ay, s_enc), sb);
    uint32_t c2 = e2m1_code(__fmul_rn(az, s_enc), sb);
    uint32_t c3 = e2m1_code(__fmul_rn(aw, s_enc), sb);
    c0 |= (x.x < 0.f && c0) ? 8u : 0u;
    c1 |= (x.y < 0.f && c1) ? 8u : 0u;
    c2 |= (x.z < 0.f && c2) ? 8u : 0u;
    c3 |= (x.w < 0.f && c3) ? 8u : 0u;
    // lanes 2i and 2i + 1 make code word i (channels 8i..8i+7) together
    const uint32_t cs[4] = {c0, c1, c2, c3};
    const uint32_t part = code_word_part(cs, lane & 1);
    const uint32_t word = part | __shfl_xor_sync(0xffffffffu, part, 1);
    uint8_t* head = kv_pool + (size_t)page * kKvPageBytes + g * kHeadBytes;
    const int off_c = is_v ? kOffVc : kOffKc;
    const int off_s = is_v ? kOffVs : kOffKs;
    // word i = lane >> 1: offset 4 (i & 3) of code chunk i >> 2
    if ((lane & 1) == 0)
      *reinterpret_cast<uint32_t*>(head + off_c + off * 64 + (code_chunk_pos(lane >> 3, off) << 4) +
                                   (((lane >> 1) & 3) << 2)) = word;
    if ((lane & 3) == 0) head[off_s + (lane >> 2) * kPageTokens + off] = (uint8_t)sb_byte;
  }
}

__global__ void __launch_bounds__(256) absmax_kernel(const float* __restrict__ x, int64_t n,
                                                     float* amax) {
  float m = 0.f;
  const int64_t stride = (int64_t)gridDim.x * blockDim.x;
  int64_t i = (int64_t)blockIdx.x * blockDim.x + threadIdx.x;
  const int64_t n4 = n / 4;
  const float4* x4 = reinterpret_cast<const float4*>(x);
  const bool aligned = (reinterpret_cast<uintptr_t>(x) & 15) == 0;
  if (aligned) {
    for (int64_t e = i; e < n4; e += stride) {
      const float4 v = x4[e];
      m = fmaxf(m, fmaxf(fmaxf(fabsf(v.x), fabsf(v.y)), fmaxf(fabsf(v.z), fabsf(v.w))));
    }
    for (int64_t e = n4 * 4 + i; e < n; e += stride) m = fmaxf(m, fabsf(x[e]));
  } else {
    for (int64_t e = i; e < n; e += stride) m = fmaxf(m, fabsf(x[e]));
  }
#pragma unroll
  for (int o = 16; o; o >>= 1) m = fmaxf(m, __shfl_xor_sync(0xffffffffu, m, o));
  // non-negative floats order like their bit patterns
  if ((threadIdx.x & 31) == 0) atomicMax(reinterpret_cast<int*>(amax), __float_as_int(m));
}

}  // namespace

cudaError_t launch_quantize_insert(const msa_cache* c, const float* k, const float* v,
                                   const float* idx_k, const int64_t* slot_mapping, int n_tokens,
                                   cudaStream_t stream) {
  if (n_tokens == 0) return cudaSuccess;
  const long long warps = (long long)n_tokens * 9;
  long long blocks = (warps + 7) / 8;
  if (blocks > 152 * 32) blocks = 152 * 32;
  quantize_insert_kernel<<<(int)blocks, 256, 0, stream>>>(
      static_cast<uint8_t*>(c->kv_pool), static_cast<uint8_t*>(c->idx_pool), c->n_pages, k, v,
      idx_k, slot_mapping, n_tokens, c->s_enc_k, c->s_enc_v, c->status);
  return cudaGetLastError();
}

cudaError_t launch_absmax(const float* x, int64_t n, float* amax, cudaStream_t stream) {
  if (n == 0) return cudaSuccess;
  long long blocks = (n / 4 + 255) / 256;
  if (blocks > 152 * 8) blocks = 152 * 8;
  if (blocks < 1) blocks = 1;
  absmax_kernel<<<(int)blocks, 256, 0, stream>>>(x, n, amax);
  return cudaGetLastError();
}

}  // namespace msa
