// Split-context sparse GQA attention over the selected NVFP4 blocks on the
// fifth-generation tensor cores (tcgen05, tensor memory).
//
// "vLLM Delivers Day-0 Support for MiniMax-M3.1-Flash" blog, section "Sparse
// attention still scans an index": exact attention over the selected blocks
// only; section "Capacity savings must pay for conversion" and the ai4snews
// article (third paragraph): queries stay FP8, so the NVFP4 K/V are converted
// to FP8 before the matrix multiply.
//
// One CTA = (split, KV head, query token), 128 threads; thread i owns token i
// of the page being processed.  Per selected page:
//   TMA       one 18 KB cp.async.bulk of the (page, head) block (K/V codes and
//             scales), double-buffered so the next page is in flight;
//   dequant   thread i converts its token's 128 K codes to FP8 through a
//             256-entry shared table of scaled E4M3 values and byte permutes,
//             and writes the row into a 128-byte-swizzled tile; same for V;
//   QK^T      tcgen05.mma kind::f8f6f4, M = 128 tokens, N = 16 (4 query heads
//             of this KV head, zero padded), K = 128 channels -> S in TMEM;
//   softmax   thread i reads its token's 4 logits (tcgen05.ld), page max per
//             head (redux), exp2, P scaled by 2^8 as two E4M3 terms (hi +
//             remainder) written as the B operand [8 rows][128 tokens];
//   PV        tcgen05.mma with A = the V tile read MN-major (channels
//             contiguous in each token row: no transpose), B = P, D = O^T
//             [128 channels][16] in TMEM;
//   merge     thread c folds the page's O into its running (m, l, o) state.
// Each CTA writes one normalised partial (O, LSE) per query head; the LSE
// merge kernel combines the splits.
#include "common.cuh"

namespace msa {
namespace {

constexpr int kThreads = 256;  // 2 threads per token: each dequantises 64 channels
constexpr int kRaw = 2;                               // raw (page, head) buffers
constexpr int kOffK8 = 0;                             // [128 tokens][128 B], swizzled
constexpr int kOffV8 = 16384;                         // [128 tokens][128 B], swizzled
constexpr int kOffQP = 32768;                         // [24 rows][128 B]: Q rows 0-3, P rows 8-15
constexpr int kOffRaw = kOffQP + 24 * 128;            // 35,840: 2 x 18,432
constexpr int kOffBars = kOffRaw + kRaw * kHeadBytes;  // rawfull[2], qk, pv, done
constexpr int kOffTmem = kOffBars + 40;
constexpr int kOffSeq = kOffTmem + 4;                 // int: sequence of the token
constexpr int kOffRed = kOffSeq + 12;                 // float [8 warps][4]
constexpr int kOffTab = kOffRed + 128;                // uint2 [256] dequant table (8-aligned)
constexpr int kOffSel = kOffTab + 2048;               // int [17] physical pages, int [17] blocks
constexpr int kSmemBytes = kOffSel + 2 * kSelStride * 4;
constexpr int kSmemAlloc = kSmemBytes + 1024;         // + alignment slack
constexpr uint32_t kTmemCols = 32;                    // S: columns 0-15, O: columns 16-31
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

// Converts half a token row -- 32 code bytes = channels 64*hh..64*hh+63, groups
// 4*hh..4*hh+3 -- to 64 FP8 bytes and stores them into row `row` of a
// 128-byte-swizzled tile (16-byte chunk c at position c ^ (row & 7)).
__device__ __forceinline__ void dequant_half_row(const uint8_t* codes, const uint8_t* scales_col,
                                                 const uint2* tab, uint8_t* tile, int row, int hh,
                                                 bool live) {
#pragma unroll
  for (int cc = 0; cc < 2; ++cc) {
    const int c = 2 * hh + ((cc + (row >> 2)) & 1);  // rotated order: fewer bank conflicts
    const uint4 w = *reinterpret_cast<const uint4*>(codes + 16 * c);
    // 16 code bytes = channels 32c..32c+31 = groups 2c and 2c+1
    const uint2 t0 = tab[scales_col[(2 * c) * kPageTokens]];
    const uint2 t1 = tab[scales_col[(2 * c + 1) * kPageTokens]];
    const uint2 a = dequant8(w.x, t0), b = dequant8(w.y, t0);
    const uint2 d = dequant8(w.z, t1), e = dequant8(w.w, t1);
    uint4 o0 = make_uint4(a.x, a.y, b.x, b.y), o1 = make_uint4(d.x, d.y, e.x, e.y);
    if (!live) o0 = o1 = make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4*>(tile + row * 128 + (((2 * c) ^ (row & 7)) << 4)) = o0;
    *reinterpret_cast<uint4*>(tile + row * 128 + (((2 * c + 1) ^ (row & 7)) << 4)) = o1;
  }
}

__global__ void __launch_bounds__(kThreads, 3) sparse_attn_tc_kernel(AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bar_raw0 = sbase + kOffBars, bar_qk = sbase + kOffBars + 16, bar_pv = sbase + kOffBars + 24;
  const uint32_t bar_done = sbase + kOffBars + 32;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kOffTmem);
  int* s_seq = reinterpret_cast<int*>(smem + kOffSeq);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + kOffSeq + 4);
  float* s_red = reinterpret_cast<float*>(smem + kOffRed);
  uint2* s_tab = reinterpret_cast<uint2*>(smem + kOffTab);
  int* s_phys = reinterpret_cast<int*>(smem + kOffSel);
  int* s_blk = s_phys + kSelStride;
  uint8_t* k8 = smem + kOffK8;
  uint8_t* v8 = smem + kOffV8;
  uint8_t* qp = smem + kOffQP;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int tok = tid & 127, hh = tid >> 7;  // token (= TMEM lane) and channel half
  const int quad = warp & 3;                 // TMEM lane quadrant of this warp
  const int split = blockIdx.x, kvh = blockIdx.y, j = blockIdx.z;

  // ---- prologue that needs no input of the previous kernel -------------------
  build_dequant_table(s_tab, tid, kThreads);
  if (tid == 0) {
    mbar_init(bar_raw0, 1);
    mbar_init(bar_raw0 + 8, 1);
    mbar_init(bar_qk, 1);
    mbar_init(bar_pv, 1);
    mbar_init(bar_done, 1);
    *s_seq = -1;
    *s_abort = 0;
    fence_barrier_init();
  }
  // zero the Q/P tile (rows 4-7 and 16-23 stay zero; Q and P rows are written below)
  for (int i = tid; i < 24 * 128 / 16; i += kThreads) reinterpret_cast<uint4*>(qp)[i] = make_uint4(0, 0, 0, 0);
  if (warp == 0) tmem_alloc(smem_u32(s_tmem), kTmemCols);
  __syncthreads();  // s_seq = -1 is in place before any thread records a match
  // sequence of token j: the b with q_start_loc[b] <= j < q_start_loc[b+1]
  for (int base = 0; base < p.n_seqs; base += kThreads) {
    const int b = base + tid;
    if (b < p.n_seqs && p.q_start_loc[b] <= j && j < p.q_start_loc[b + 1]) *s_seq = b;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const int b = *s_seq;
  SeqInfo s{0, 0, 0, false};
  if (b >= 0) s = load_seq(b, p.seq_lens, p.q_start_loc, p.max_pages, p.n_q_total);
  const bool seq_ok = b >= 0 && s.ok;
  const int pos = s.seq_len - s.n_q + (j - s.q0);
  const int r_blk = seq_ok ? pos / kPageTokens : -1;
  // query rows 0-3: heads 4*kvh .. 4*kvh+3, 128-byte swizzled K-major
  if (tid < 32) {  // query rows 0-3
    const int row = tid >> 3, c = tid & 7;
    const uint4 v = *reinterpret_cast<const uint4*>(p.q + ((size_t)j * kQHeads + kvh * kGqa + row) * kHeadDim + 16 * c);
    *reinterpret_cast<uint4*>(qp + row * 128 + ((c ^ row) << 4)) = v;
  }

  pdl_wait();  // the selection comes from the indexer kernel
  const int nsel = seq_ok ? min(p.n_sel[j], kSelStride) : 0;
  if (tid < kSelStride) {
    const int e = split + tid * p.n_splits;
    int blk = -1, phys = -1;
    if (e < nsel) {
      blk = p.sel[(size_t)j * kSelStride + e];
      if (blk < 0 || blk > r_blk) {
        set_status(p.status, MSA_STATUS_BAD_SELECTION);
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
  if (tid == 0 && !seq_ok) set_status(p.status, MSA_STATUS_BAD_SEQ);
  fence_proxy_async_smem();  // Q rows and zero rows -> visible to the tensor core
  __syncthreads();
  pdl_trigger();
  // compact this split's valid pages (thread 0), then start their copies
  int* s_npg = s_seq + 2;
  if (tid == 0) {
    int n = 0;
    for (int i = 0; i < kSelStride; ++i)
      if (s_phys[i] >= 0) {
        s_phys[n] = s_phys[i];
        s_blk[n] = s_blk[i];
        ++n;
      }
    *s_npg = n;
  }
  __syncthreads();
  const int n_pg = *s_npg;
  auto issue_raw = [&](int e) {
    const uint32_t bar = bar_raw0 + 8 * (e & 1);
    mbar_arrive_expect_tx(bar, kHeadBytes);
    bulk_g2s(sbase + kOffRaw + (e & 1) * kHeadBytes,
             p.kv_pool + (size_t)s_phys[e] * kKvPageBytes + kvh * kHeadBytes, kHeadBytes, bar);
  };
  if (tid == 0) {
    if (n_pg > 0) issue_raw(0);
    if (n_pg > 1) issue_raw(1);
  }

  const uint32_t idesc_qk = umma_idesc_e4m3(128, 16);
  const uint32_t idesc_pv = umma_idesc_e4m3_amn(128, 16);
  float m_run[4], l_run[4], o_run[4];
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    m_run[h] = -INFINITY;
    l_run[h] = 0.f;
    o_run[h] = 0.f;
  }
  // Only thread 0 waits on mbarriers (bounded); a CTA barrier then releases
  // everyone and s_abort, read after it, keeps the control flow uniform.
  // The PV MMA of page e runs while page e+1 is dequantised; its output is
  // folded into the running state once that MMA is known to be done.
  float alpha_prev[4], beta_prev[4];
  auto fold_o = [&]() {  // O of the previous page -> running state (after bar_pv)
    float ov[4];
    // lane = channel tok; half 0 reads the hi columns 16-19, half 1 the remainder 20-23
    tmem_ld4(tmem + ((uint32_t)(32 * quad) << 16) + 16 + 4 * hh, ov);
#pragma unroll
    for (int h = 0; h < 4; ++h) o_run[h] = o_run[h] * alpha_prev[h] + ov[h] * beta_prev[h];
  };
  int n_done = 0;
  for (int e = 0; e < n_pg; ++e) {
    const int valid = s_blk[e] == r_blk ? (pos % kPageTokens) + 1 : kPageTokens;
    const bool live = tok < valid;
    const uint8_t* raw = smem + kOffRaw + (e & 1) * kHeadBytes;
    // every thread waits for the page itself (a timeout only raises s_abort; the
    // next CTA barrier turns it into a uniform exit)
    mbar_wait(bar_raw0 + 8 * (e & 1), (e >> 1) & 1, s_abort);
    // ---- K -> FP8 tile (the previous page's PV MMA only reads V and P) ------------
    dequant_half_row(raw + kOffKc + tok * 64, raw + kOffKs + tok, s_tab, k8, tok, hh, live);
    fence_proxy_async_smem();
    if (tid == 0 && e > 0) mbar_wait(bar_pv, (e - 1) & 1, s_abort);
    tc_fence_before();
    __syncthreads();
    if (*s_abort) break;
    tc_fence_after();
    // ---- S = K8 Q^T on the tensor core --------------------------------------------
    if (tid == 0) {
      const uint64_t adesc = umma_desc_sw128(sbase + kOffK8);
      const uint64_t bdesc = umma_desc_sw128(sbase + kOffQP);
#pragma unroll
      for (int k = 0; k < 4; ++k) umma_e4m3(tmem, adesc + 2 * k, bdesc + 2 * k, idesc_qk, k > 0);
      umma_commit(bar_qk);
    }
    if (e > 0) fold_o();  // the previous page's PV finished before the barrier above
    // ---- V -> FP8 tile (overlaps the QK MMA; the previous PV is done) ----------------
    dequant_half_row(raw + kOffVc + tok * 64, raw + kOffVs + tok, s_tab, v8, tok, hh, live);
    fence_proxy_async_smem();
    mbar_wait(bar_qk, e & 1, s_abort);
    tc_fence_after();
    // ---- softmax over this page -----------------------------------------------------
    float sv[4];
    tmem_ld4(tmem + ((uint32_t)(32 * quad) << 16), sv);
    float x[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      x[h] = live ? sv[h] * p.scale_log2 : -INFINITY;
      const float wm = warp_max(x[h]);
      if (lane == 0) s_red[warp * 4 + h] = wm;
    }
    __syncthreads();  // page maxima complete; raw buffer e&1 no longer read
    if (*s_abort) break;
    if (tid == 0 && e + 2 < n_pg) issue_raw(e + 2);
    uint32_t p_hi = 0, p_lo = 0;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      // both halves of a token computed the same logits: warps 0-3 suffice
      const float mp = fmaxf(fmaxf(s_red[h], s_red[4 + h]), fmaxf(s_red[8 + h], s_red[12 + h]));
      const float m_new = fmaxf(m_run[h], mp);
      // m_new = -inf only while no key so far is visible (then everything is 0)
      alpha_prev[h] = m_new == -INFINITY ? 1.f : fast_exp2(m_run[h] - m_new);
      beta_prev[h] = mp == -INFINITY ? 0.f : fast_exp2(mp - m_new);  // page scale -> running scale
      const float pr = mp == -INFINITY ? 0.f : fast_exp2(x[h] - mp);  // relative to the page max
      l_run[h] = l_run[h] * alpha_prev[h] + (hh == 0 ? pr * beta_prev[h] : 0.f);  // this token
      m_run[h] = m_new;
      const float v256 = pr * 256.f;
      const uint32_t hi = f32_to_e4m3(v256);
      const uint32_t lo = f32_to_e4m3(v256 - e4m3_to_f32(hi));
      p_hi |= hi << (8 * h);
      p_lo |= lo << (8 * h);
    }
    // P rows 8+h (E4M3 of 256 p) and 12+h (E4M3 of the remainder), one byte per
    // token: byte t of row n sits in chunk (t/16) ^ (n & 7)
    // (half 0 writes the hi rows, half 1 the remainder rows)
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const int n = (hh ? 12 : 8) + h;
      qp[n * 128 + (((tok >> 4) ^ (n & 7)) << 4) + (tok & 15)] = (uint8_t)((hh ? p_lo : p_hi) >> (8 * h));
    }
    fence_proxy_async_smem();
    tc_fence_before();
    __syncthreads();
    // ---- O^T[c][n] = sum_t V8[t][c] P[n][t], left running ------------------------------
    if (tid == 0) {
      tc_fence_after();
      const uint64_t bdesc = umma_desc_sw128(sbase + kOffQP + 8 * 128);
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        // A: V tile read MN-major; 32 tokens (4 swizzle atoms of 8 rows) per MMA
        const uint64_t adesc = umma_desc_sw128_lbo_sbo(sbase + kOffV8 + k * 4096, 1024, 1024);
        umma_e4m3(tmem + 16, adesc, bdesc + 2 * k, idesc_pv, k > 0);
      }
      umma_commit(bar_pv);
    }
    ++n_done;
  }
  if (n_done > 0 && !*s_abort) {
    if (tid == 0) mbar_wait(bar_pv, (n_done - 1) & 1, s_abort);
    tc_fence_before();
    __syncthreads();
    tc_fence_after();
    if (!*s_abort) fold_o();
  }
  const bool ok = !*s_abort;

  // ---- finish: l over the tokens, both halves of O, normalised partial output --------
  float* redl = s_red;  // [8 warps][4]
  float* s_o = reinterpret_cast<float*>(smem + kOffK8);  // the K tile is free now: [4][128]
  __syncthreads();
#pragma unroll
  for (int h = 0; h < 4; ++h) {
    float l = l_run[h];
#pragma unroll
    for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
    if (lane == 0) redl[warp * 4 + h] = l;
    if (hh == 1) s_o[h * 128 + tok] = o_run[h];
  }
  __syncthreads();
  const size_t row0 = ((size_t)j * p.n_splits + split) * kQHeads + kvh * kGqa;
  if (hh == 0) {
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      float L = 0.f;
#pragma unroll
      for (int w = 0; w < 4; ++w) L += redl[w * 4 + h];
      const bool nonempty = ok && L > 0.f && m_run[h] != -INFINITY;
      const float o = o_run[h] + s_o[h * 128 + tok];
      p.o_part[(row0 + h) * kHeadDim + tok] = nonempty ? o / L * p.out_scale : 0.f;
      if (tok == 0) p.lse_part[row0 + h] = nonempty ? (m_run[h] + log2f(L)) * kLn2 : -INFINITY;
    }
  }

  // ---- teardown -----------------------------------------------------------------------
  if (*s_abort && tid == 0) {
    set_status(p.status, MSA_STATUS_TIMEOUT);
    // bounded drain: copies still landing, MMAs still running
    volatile int ignore = 0;
    for (int e = n_done; e < min(n_pg, n_done + 2); ++e) mbar_wait(bar_raw0 + 8 * (e & 1), (e >> 1) & 1, &ignore);
    umma_commit(bar_done);  // arrives once every MMA issued so far is complete
    mbar_wait(bar_done, 0, &ignore);
  }
  tc_fence_before();
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kTmemCols);
  }
}

}  // namespace

cudaError_t launch_sparse_attn_tc(const msa_cache* c, const uint8_t* q, float softmax_scale,
                                  const int* sel, const int* n_sel, const int* block_table,
                                  int max_pages, const int* seq_lens, const int* q_start_loc,
                                  int n_seqs, int n_q_total, int n_splits, float* o_part,
                                  float* lse_part, cudaStream_t stream) {
  if (n_q_total == 0) return cudaSuccess;
  static bool s_attr[64] = {false};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  if (!s_attr[dev]) {
    e = cudaFuncSetAttribute(sparse_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemAlloc);
    if (e != cudaSuccess) return e;
    s_attr[dev] = true;
  }
  AttnParams ap{static_cast<const uint8_t*>(c->kv_pool), c->n_pages, q, sel, n_sel, block_table,
                max_pages, seq_lens, q_start_loc, n_seqs, n_q_total, n_splits,
                softmax_scale / c->s_enc_k * kLog2e, 1.0f / (256.0f * c->s_enc_v), o_part,
                lse_part, c->status};
  return launch_pdl(sparse_attn_tc_kernel, dim3(n_splits, kKvHeads, n_q_total), dim3(kThreads),
                    (size_t)kSmemAlloc, stream, ap);
}

}  // namespace msa
