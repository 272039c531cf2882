// Split-context sparse GQA attention over the selected NVFP4 blocks, and the
// log-sum-exp merge of the splits.
//
// "vLLM Delivers Day-0 Support for MiniMax-M3.1-Flash" blog, section "Sparse
// attention still scans an index": exact attention over the selected blocks
// only; section "Capacity savings must pay for conversion" and the ai4snews
// article (third paragraph): queries stay FP8, so NVFP4 K/V are converted to
// FP8 before the matrix multiply.
//
// One CTA = (split, KV head, query token), four warps.  Warp w owns tokens
// 32w..32w+31 of every page the split visits and keeps its own online-softmax
// state; the four states are merged at the end.  Per page and warp:
//   K: 16-byte loads of the NVFP4 codes + 4-byte loads of the group scales
//      -> NVFP4->FP8 through a 256-entry shared-memory table and byte permutes
//      (no FP16 round trip) -> mma.sync A fragments directly in registers;
//   S = K q^T with m16n8k32 E4M3 MMAs (M = 16 tokens, N = 4 query heads
//      duplicated to 8, K = 128 channels), fp32 accumulators;
//   online softmax in the exp2 domain;
//   P = exp scaled by 2^8 split into two E4M3 terms (hi in columns 0..3, the
//      rounding remainder in columns 4..7 -- the duplicated heads);
//   V: 8-byte code loads of 8 consecutive tokens per lane -> FP8 -> 4x4 byte
//      transposes -> A fragments of V^T (M = channels, K = tokens);
//   O^T += V^T P with m16n8k32 E4M3 MMAs.
// Channel and token orders inside the MMAs are permutations chosen so that
// each lane's loads are whole 16-channel scale groups; the contraction is
// unchanged and the output is written back in logical channel order.
#include "common.cuh"

namespace msa {
namespace {

constexpr int kAttnThreads = 128;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct AttnParams {
  const uint8_t* kv_pool;
  int64_t n_pages;
  const uint8_t* q;  // [T][16][128]
  const int* sel;
  const int* n_sel;
  const int* block_table;
  int max_pages;
  const int* seq_lens;
  const int* q_start_loc;
  int n_seqs;
  int n_q_total;
  int n_splits;
  float scale_log2;  // softmax_scale / s_enc_k * log2(e)
  float out_scale;   // 1 / (256 * s_enc_v)
  float* o_part;     // [T][S][16][128]
  float* lse_part;   // [T][S][16]
  int* status;
};

// 4x4 byte transpose: out[n] byte i = in[i] byte n.
__device__ __forceinline__ void transpose4x4(uint32_t r0, uint32_t r1, uint32_t r2, uint32_t r3,
                                             uint32_t& c0, uint32_t& c1, uint32_t& c2, uint32_t& c3) {
  const uint32_t t0 = prmt(r0, r1, 0x5140u);
  const uint32_t t1 = prmt(r0, r1, 0x7362u);
  const uint32_t t2 = prmt(r2, r3, 0x5140u);
  const uint32_t t3 = prmt(r2, r3, 0x7362u);
  c0 = prmt(t0, t2, 0x5410u);
  c1 = prmt(t0, t2, 0x7632u);
  c2 = prmt(t1, t3, 0x5410u);
  c3 = prmt(t1, t3, 0x7632u);
}

__global__ void __launch_bounds__(kAttnThreads, 3) sparse_attn_kernel(AttnParams p) {
  __shared__ uint2 s_tab[256];
  __shared__ float s_m[4][4], s_l[4][4];
  __shared__ float s_o[4][4][kHeadDim];
  __shared__ int s_qsl[kMaxSeqs + 1];
  __shared__ int s_blk[kSelStride], s_phys[kSelStride];
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int g = lane >> 2, t = lane & 3;
  const int split = blockIdx.x, kvh = blockIdx.y, j = blockIdx.z;
  build_dequant_table(s_tab, tid, kAttnThreads);
  for (int i = tid; i <= p.n_seqs; i += kAttnThreads) s_qsl[i] = p.q_start_loc[i];
  __syncthreads();

  const int b = find_seq(s_qsl, p.n_seqs, j);
  const SeqInfo s = load_seq(b, p.seq_lens, s_qsl, p.max_pages, p.n_q_total);
  const bool seq_ok = s.ok && j >= s.q0 && j < s.q0 + s.n_q;
  const int pos = s.seq_len - s.n_q + (j - s.q0);
  const int r_blk = seq_ok ? pos / kPageTokens : -1;
  pdl_wait();     // the selection comes from the top-k kernel
  pdl_trigger();  // the merge kernel may launch and wait
  const int nsel = seq_ok ? min(p.n_sel[j], kSelStride) : 0;
  // this split's block ids and physical pages, fetched once, all in parallel
  if (tid < kSelStride) {
    const int e = split + tid * p.n_splits;
    int blk = -1, phys = -1;
    if (e < nsel) {
      blk = p.sel[(size_t)j * kSelStride + e];
      if (blk < 0 || blk > r_blk) {
        set_status(p.status, MSA_STATUS_BAD_SELECTION);
        blk = -1;
      } else {
        phys = p.block_table[(size_t)b * p.max_pages + blk];
        if (phys < 0 || phys >= p.n_pages) {
          set_status(p.status, MSA_STATUS_BAD_PAGE);
          phys = -1;
        }
      }
    }
    s_blk[tid] = blk;
    s_phys[tid] = phys;
  }

  // query fragments: column n = g holds query head 4*kvh + (g & 3); lane t owns
  // channels 32t..32t+31 -> b0 of k-step s = channels 32t+4s.., b1 = 32t+16+4s..
  const uint8_t* qrow = p.q + ((size_t)j * kQHeads + kvh * kGqa + (g & 3)) * kHeadDim + 32 * t;
  const uint4 qa = *reinterpret_cast<const uint4*>(qrow);
  const uint4 qb = *reinterpret_cast<const uint4*>(qrow + 16);
  const uint32_t QB0[4] = {qa.x, qa.y, qa.z, qa.w};
  const uint32_t QB1[4] = {qb.x, qb.y, qb.z, qb.w};

  float o[8][4];
#pragma unroll
  for (int m = 0; m < 8; ++m) o[m][0] = o[m][1] = o[m][2] = o[m][3] = 0.f;
  float m_run[2] = {-INFINITY, -INFINITY}, l_run[2] = {0.f, 0.f};
  __syncthreads();  // table ready

  const int tok_k = 32 * warp + 4 * g;  // K tokens of this lane: tok_k + i, i < 4
  const int tok_v = 32 * warp + 8 * t;  // V tokens of this lane: tok_v + i, i < 8

  for (int e = split, ei = 0; e < nsel; e += p.n_splits, ++ei) {
    const int blk = s_blk[ei], phys = s_phys[ei];
    if (phys < 0) continue;
    const int valid = blk == r_blk ? (pos % kPageTokens) + 1 : kPageTokens;
    const uint8_t* base = p.kv_pool + (size_t)phys * kKvPageBytes + kvh * kHeadBytes;

    // ---- loads ------------------------------------------------------------
    uint4 kc[4];
#pragma unroll
    for (int i = 0; i < 4; ++i) kc[i] = ld_stream_v4(base + kOffKc + (tok_k + i) * 64 + 16 * t);
    const uint32_t ks0 = ld_stream_u32(base + kOffKs + (2 * t) * kPageTokens + tok_k);
    const uint32_t ks1 = ld_stream_u32(base + kOffKs + (2 * t + 1) * kPageTokens + tok_k);
    uint2 vc[8];
#pragma unroll
    for (int i = 0; i < 8; ++i) vc[i] = ld_stream_v2(base + kOffVc + (tok_v + i) * 64 + 8 * g);
    const uint2 vs = ld_stream_v2(base + kOffVs + g * kPageTokens + tok_v);

    // ---- S = K q^T -----------------------------------------------------------
    // M-tile 0: row g = token tok_k, row g+8 = tok_k+1; M-tile 1: tok_k+2, tok_k+3
    float acc[2][4];
#pragma unroll
    for (int mt = 0; mt < 2; ++mt) {
      acc[mt][0] = acc[mt][1] = acc[mt][2] = acc[mt][3] = 0.f;
      uint32_t lo[2][4], hi[2][4];  // [row][k-step]: group 2t (lo) and 2t+1 (hi)
#pragma unroll
      for (int rr = 0; rr < 2; ++rr) {
        const int i = 2 * mt + rr;
        const uint2 t0 = s_tab[(ks0 >> (8 * i)) & 0xFF];
        const uint2 t1 = s_tab[(ks1 >> (8 * i)) & 0xFF];
        const uint2 d0 = dequant8(kc[i].x, t0), d1 = dequant8(kc[i].y, t0);
        const uint2 d2 = dequant8(kc[i].z, t1), d3 = dequant8(kc[i].w, t1);
        lo[rr][0] = d0.x; lo[rr][1] = d0.y; lo[rr][2] = d1.x; lo[rr][3] = d1.y;
        hi[rr][0] = d2.x; hi[rr][1] = d2.y; hi[rr][2] = d3.x; hi[rr][3] = d3.y;
      }
#pragma unroll
      for (int ks = 0; ks < 4; ++ks)
        mma_e4m3(acc[mt], lo[0][ks], lo[1][ks], hi[0][ks], hi[1][ks], QB0[ks], QB1[ks]);
    }
    // x[i][c]: token tok_k + i, column 2t + c
    float x[4][2];
    x[0][0] = acc[0][0]; x[0][1] = acc[0][1]; x[1][0] = acc[0][2]; x[1][1] = acc[0][3];
    x[2][0] = acc[1][0]; x[2][1] = acc[1][1]; x[3][0] = acc[1][2]; x[3][1] = acc[1][3];

    // ---- online softmax (per column) ------------------------------------------
    float pv[4][2];
    float alpha[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      float mx = -INFINITY;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        x[i][c] = (tok_k + i < valid) ? x[i][c] * p.scale_log2 : -INFINITY;
        mx = fmaxf(mx, x[i][c]);
      }
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 4));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 8));
      mx = fmaxf(mx, __shfl_xor_sync(0xffffffffu, mx, 16));
      const float m_new = fmaxf(m_run[c], mx);
      const bool any = m_new != -INFINITY;
      alpha[c] = any ? exp2f(m_run[c] - m_new) : 1.f;
      float sum = 0.f;
#pragma unroll
      for (int i = 0; i < 4; ++i) {
        pv[i][c] = any ? exp2f(x[i][c] - m_new) : 0.f;
        sum += pv[i][c];
      }
      l_run[c] = l_run[c] * alpha[c] + sum;
      m_run[c] = m_new;
    }
#pragma unroll
    for (int m = 0; m < 8; ++m) {
      o[m][0] *= alpha[0]; o[m][1] *= alpha[1];
      o[m][2] *= alpha[0]; o[m][3] *= alpha[1];
    }

    // ---- P -> E4M3 B fragments ---------------------------------------------------
    // lanes t < 2 (columns 0..3) carry E4M3(256 p); lanes t >= 2 (columns 4..7,
    // the same heads) carry E4M3 of the remainder 256 p - hi.
    uint32_t W[2];
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      uint32_t packed = 0;
#pragma unroll
      for (int i = 0; i < 4; i += 2) {
        const float v0 = pv[i][c] * 256.f, v1 = pv[i + 1][c] * 256.f;
        uint32_t h2 = f32x2_to_e4m3x2(v0, v1);
        if (t >= 2) {
          const float r0 = v0 - e4m3_to_f32(h2 & 0xFF);
          const float r1 = v1 - e4m3_to_f32(h2 >> 8);
          h2 = f32x2_to_e4m3x2(r0, r1);
        }
        packed |= h2 << (8 * i);
      }
      W[c] = packed;
    }
    // B fragment: column n = g, k rows 4t..4t+3 <- tokens 8t..8t+3 (held by lane
    // (g' = 2t, t' = g/2) as W[g&1]); rows 16+4t.. <- tokens 8t+4.. (lane g' = 2t+1)
    const int src0 = 4 * (2 * t) + (g >> 1), src1 = 4 * (2 * t + 1) + (g >> 1);
    const uint32_t u00 = __shfl_sync(0xffffffffu, W[0], src0);
    const uint32_t u01 = __shfl_sync(0xffffffffu, W[1], src0);
    const uint32_t u10 = __shfl_sync(0xffffffffu, W[0], src1);
    const uint32_t u11 = __shfl_sync(0xffffffffu, W[1], src1);
    const uint32_t pb0 = (g & 1) ? u01 : u00;
    const uint32_t pb1 = (g & 1) ? u11 : u10;

    // ---- V: NVFP4 -> FP8, transpose to V^T fragments, O^T += V^T P ----------------
    // lane (g, t): channels 16g..16g+15 (group g), tokens tok_v..tok_v+7.  Row g of
    // M-tile m is channel 16g+2m, row g+8 is channel 16g+2m+1.
    uint32_t X[8][4];
#pragma unroll
    for (int i = 0; i < 8; ++i) {
      const uint32_t sbyte = ((i < 4 ? vs.x : vs.y) >> (8 * (i & 3))) & 0xFF;
      const uint2 tb = s_tab[sbyte];
      const uint2 d0 = dequant8(vc[i].x, tb), d1 = dequant8(vc[i].y, tb);
      X[i][0] = d0.x; X[i][1] = d0.y; X[i][2] = d1.x; X[i][3] = d1.y;
    }
    if (valid < kPageTokens) {
      // masked tokens carry p = 0; their V bytes are zeroed so that stale NaN
      // codes or scales cannot reach the accumulators (0 * NaN = NaN)
#pragma unroll
      for (int i = 0; i < 8; ++i)
        if (tok_v + i >= valid) X[i][0] = X[i][1] = X[i][2] = X[i][3] = 0u;
    }
#pragma unroll
    for (int k = 0; k < 4; ++k) {
      uint32_t a0e, a1e, a0o, a1o, a2e, a3e, a2o, a3o;
      transpose4x4(X[0][k], X[1][k], X[2][k], X[3][k], a0e, a1e, a0o, a1o);
      transpose4x4(X[4][k], X[5][k], X[6][k], X[7][k], a2e, a3e, a2o, a3o);
      mma_e4m3(o[2 * k], a0e, a1e, a2e, a3e, pb0, pb1);
      mma_e4m3(o[2 * k + 1], a0o, a1o, a2o, a3o, pb0, pb1);
    }
  }

  // ---- finish: hi + lo columns, per-warp state to shared memory ---------------------
#pragma unroll
  for (int m = 0; m < 8; ++m)
#pragma unroll
    for (int c = 0; c < 4; ++c) o[m][c] += __shfl_xor_sync(0xffffffffu, o[m][c], 2);
#pragma unroll
  for (int c = 0; c < 2; ++c) {
    float l = l_run[c];
    l += __shfl_xor_sync(0xffffffffu, l, 4);
    l += __shfl_xor_sync(0xffffffffu, l, 8);
    l += __shfl_xor_sync(0xffffffffu, l, 16);
    l_run[c] = l;
  }
  if (t < 2) {
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int h = 2 * t + c;
      if (g == 0) {
        s_m[warp][h] = m_run[c];
        s_l[warp][h] = l_run[c];
      }
#pragma unroll
      for (int m = 0; m < 8; ++m) {
        s_o[warp][h][16 * g + 2 * m] = o[m][c];
        s_o[warp][h][16 * g + 2 * m + 1] = o[m][2 + c];
      }
    }
  }
  __syncthreads();
  // thread tid -> channel tid, all 4 heads of this KV head
  const size_t row0 = ((size_t)j * p.n_splits + split) * kQHeads + kvh * kGqa;
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    float M = -INFINITY;
#pragma unroll
    for (int w = 0; w < 4; ++w) M = fmaxf(M, s_m[w][h]);
    float L = 0.f, acc_o = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int w = 0; w < 4; ++w) {
        const float f = exp2f(s_m[w][h] - M);
        L += f * s_l[w][h];
        acc_o += f * s_o[w][h][tid];
      }
    }
    const bool nonempty = L > 0.f;
    p.o_part[(row0 + h) * kHeadDim + tid] = nonempty ? acc_o / L * p.out_scale : 0.f;
    if (tid == 0) p.lse_part[row0 + h] = nonempty ? (M + log2f(L)) * kLn2 : -INFINITY;
  }
}

// out[j][h][:] = sum_s exp(lse_s - L) o_s; one CTA per (token, head), thread = channel.
__global__ void __launch_bounds__(kHeadDim) merge_kernel(const float* __restrict__ o_part,
                                                         const float* __restrict__ lse_part,
                                                         int n_heads, int n_splits,
                                                         float* __restrict__ out) {
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
  const uint8_t* codes = base + (isv ? kOffVc : kOffKc) + tok * 64 + grp * 8;
  const uint8_t sb = base[(isv ? kOffVs : kOffKs) + grp * kPageTokens + tok];
  const uint2 c = *reinterpret_cast<const uint2*>(codes);
  const uint2 d0 = dequant8(c.x, s_tab[sb]), d1 = dequant8(c.y, s_tab[sb]);
  uint8_t* dst = (isv ? v8 : k8) + ((size_t)head * kPageTokens + tok) * kHeadDim + grp * 16;
  *reinterpret_cast<uint4*>(dst) = make_uint4(d0.x, d0.y, d1.x, d1.y);
}

}  // namespace

cudaError_t launch_sparse_attn(const msa_cache* c, const uint8_t* q, float softmax_scale,
                               const int* sel, const int* n_sel, const int* block_table,
                               int max_pages, const int* seq_lens, const int* q_start_loc,
                               int n_seqs, int n_q_total, int n_splits, float* o_part,
                               float* lse_part, cudaStream_t stream) {
  if (n_q_total == 0) return cudaSuccess;
  AttnParams ap{static_cast<const uint8_t*>(c->kv_pool), c->n_pages, q, sel, n_sel, block_table,
                max_pages, seq_lens, q_start_loc, n_seqs, n_q_total, n_splits,
                softmax_scale / c->s_enc_k * kLog2e, 1.0f / (256.0f * c->s_enc_v), o_part,
                lse_part, c->status};
  dim3 grid(n_splits, kKvHeads, n_q_total);
  return launch_pdl(sparse_attn_kernel, grid, dim3(kAttnThreads), 0, stream, ap);
}

cudaError_t launch_merge(const float* o_part, const float* lse_part, int n_q_total, int n_heads,
                         int n_splits, float* out, cudaStream_t stream) {
  if (n_q_total == 0) return cudaSuccess;
  return launch_pdl(merge_kernel, dim3(n_q_total * n_heads), dim3(kHeadDim), 0, stream, o_part,
                    lse_part, n_heads, n_splits, out);
}

cudaError_t launch_debug_fp8_page(const msa_cache* c, int64_t page, uint8_t* k8, uint8_t* v8,
                                  cudaStream_t stream) {
  debug_fp8_page_kernel<<<(2 * kKvHeads * kPageTokens * 8) / 256, 256, 0, stream>>>(
      static_cast<const uint8_t*>(c->kv_pool), page, k8, v8);
  return cudaGetLastError();
}

}  // namespace msa
