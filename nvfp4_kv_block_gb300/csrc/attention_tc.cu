// Split-context sparse GQA attention over the selected NVFP4 blocks on the
// fifth-generation tensor cores (tcgen05, tensor memory), warp-specialised.
//
// "vLLM Delivers Day-0 Support for MiniMax-M3.1-Flash" blog, section "Sparse
// attention still scans an index": exact attention over the selected blocks
// only; section "Capacity savings must pay for conversion" and the ai4snews
// article (third paragraph): queries stay FP8, so the NVFP4 K/V are converted
// to FP8 before the matrix multiply.
//
// One CTA = (split, KV head, query token); two CTAs per SM.  The split's pages
// flow through a pipeline of warp roles, each hand-off an mbarrier:
//   warp 0      TMA producer: one 18 KB cp.async.bulk per (page, head) block
//               (K/V codes and scales) into a 2-stage ring;
//   warps 6-9   conversion, thread = token: NVFP4 K and V rows -> FP8 through a
//               256-entry shared table of scaled E4M3 values and byte permutes,
//               written as 128-byte-swizzled tiles (K8, V8; two of each);
//   warp 1      MMA issuer: S = K8 Q^T (tcgen05.mma kind::f8f6f4, M = 128
//               tokens, N = 16: the 4 query heads of this KV head, zero padded,
//               K = 128 channels) into one of two TMEM S buffers, and
//               O^T = V8^T P (A = the V tile read MN-major, no transpose) into
//               one of two TMEM O buffers; QK of page e+1 is issued before PV of
//               page e, so the softmax of e+1 overlaps PV(e);
//   warps 2-5   softmax, thread = token row of S: page max per head, P = exp2
//               relative to the page max, scaled by 2^8 and split into two E4M3
//               terms (value + rounding remainder) as the B operand of PV; then
//               thread = channel: the page's O folded into the running
//               (m, l, o) state, O of the split normalised at the end.
// Every wait is bounded; a timeout raises MSA_STATUS_TIMEOUT and the split's
// output is written as empty.  The LSE merge kernel combines the splits.
#include "common.cuh"

namespace msa {
namespace {

constexpr int kThreads = 320;  // 10 warps
constexpr int kTileBytes = 16384;                      // [128 rows][128 B], swizzled
constexpr int kOffK8 = 0;                              // 2 K8 tiles
constexpr int kOffV8 = 2 * kTileBytes;                 // 2 V8 tiles
constexpr int kOffQ = 4 * kTileBytes;                  // [16 rows][128 B]: Q rows 0-3
constexpr int kOffP = kOffQ + 2048;                    // 2 x [16 rows][128 B]: P hi 0-3, lo 4-7
constexpr int kOffRaw = kOffP + 2 * 2048;              // 2 x 18,432 (K/V codes + scales)
constexpr int kOffTab = kOffRaw + 2 * kHeadBytes;      // uint2 [256] dequant table
constexpr int kOffBars = kOffTab + 2048;               // 25 mbarriers
constexpr int kNumBars = 25;
constexpr int kOffMisc = kOffBars + kNumBars * 8;      // tmem slot, seq, abort, n pages, issued
constexpr int kOffRed = kOffMisc + 32;                 // float [2][4 warps][4 heads] page maxima
constexpr int kOffRedL = kOffRed + 128;                // float [4 warps][4 heads] row sums
constexpr int kOffSel = kOffRedL + 64;                 // int [17] phys, [17] valid, [17] block
constexpr int kSmemBytes = kOffSel + 3 * kSelStride * 4;
constexpr int kSmemAlloc = kSmemBytes + 1024;          // + alignment slack
constexpr uint32_t kTmemCols = 64;                     // S: 0, 16; O: 32, 48
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0, "swizzled tiles need 1 KB alignment");
static_assert(kOffRaw % 16 == 0 && kOffTab % 8 == 0 && kOffBars % 8 == 0, "alignment");
static_assert(2 * (kSmemAlloc + 1024) <= 228 * 1024, "two CTAs per SM");

// barrier indices; slot s of each pair is index + s
enum : int {
  kRawFull = 0, kRawEmpty = 2, kK8Full = 4, kK8Empty = 6, kV8Full = 8, kV8Empty = 10,
  kSFull = 12, kSEmpty = 14, kPFull = 16, kPEmpty = 18, kOFull = 20, kOEmpty = 22, kDone = 24
};

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

// OR of a predicate over the threads of a named barrier (all of them wait).
__device__ __forceinline__ bool named_barrier_or(int id, int nthreads, bool pred) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 p, %1, 0;\n bar.red.or.pred q, %2, %3, p;\n"
      " selp.u32 %0, 1, 0, q;\n}"
      : "=r"(r)
      : "r"((uint32_t)pred), "r"(id), "r"(nthreads)
      : "memory");
  return r != 0;
}

// Converts one token row -- 64 code bytes, 8 scale groups -- to 128 FP8 bytes in
// row `row` of a 128-byte-swizzled tile (16-byte chunk j at position j ^ (row & 7)).
// Code chunk c sits at position c ^ ((row >> 1) & 3) of the row, so the 16-byte
// loads of 8 consecutive rows (64 B apart) hit 8 different bank groups; the
// tile stores of 8 consecutive rows do too.
__device__ __forceinline__ void convert_row(const uint8_t* codes, const uint8_t* scales_col,
                                            const uint2* tab, uint8_t* tile, int row, bool live) {
  uint8_t* dst = tile + row * 128;
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    const uint4 w = *reinterpret_cast<const uint4*>(codes + 16 * code_chunk_pos(c, row));
    // 16 code bytes = channels 32c..32c+31 = groups 2c and 2c+1
    const uint2 t0 = tab[scales_col[(2 * c) * kPageTokens]];
    const uint2 t1 = tab[scales_col[(2 * c + 1) * kPageTokens]];
    const uint2 a = dequant8(w.x, t0), b = dequant8(w.y, t0);
    const uint2 d = dequant8(w.z, t1), e = dequant8(w.w, t1);
    uint4 o0 = make_uint4(a.x, a.y, b.x, b.y), o1 = make_uint4(d.x, d.y, e.x, e.y);
    if (!live) o0 = o1 = make_uint4(0, 0, 0, 0);
    *reinterpret_cast<uint4*>(dst + (((2 * c) ^ (row & 7)) << 4)) = o0;
    *reinterpret_cast<uint4*>(dst + (((2 * c + 1) ^ (row & 7)) << 4)) = o1;
  }
}

__global__ void __launch_bounds__(kThreads, 2) sparse_attn_tc_kernel(AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) { return sbase + kOffBars + 8 * i; };
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  int* s_seq = reinterpret_cast<int*>(smem + kOffMisc + 4);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + kOffMisc + 8);
  int* s_npg = reinterpret_cast<int*>(smem + kOffMisc + 12);
  int* s_issued = reinterpret_cast<int*>(smem + kOffMisc + 16);
  float* s_red = reinterpret_cast<float*>(smem + kOffRed);
  float* s_redl = reinterpret_cast<float*>(smem + kOffRedL);
  uint2* s_tab = reinterpret_cast<uint2*>(smem + kOffTab);
  int* s_phys = reinterpret_cast<int*>(smem + kOffSel);
  int* s_valid = s_phys + kSelStride;
  int* s_blk = s_valid + kSelStride;

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int split = blockIdx.x, kvh = blockIdx.y, j = blockIdx.z;

  // ---- prologue that needs no input of the previous kernel -------------------
  build_dequant_table(s_tab, tid, kThreads);
  if (tid == 0) {
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kRawFull + i), 1);
      mbar_init(bar(kRawEmpty + i), 4);
      mbar_init(bar(kK8Full + i), 4);
      mbar_init(bar(kK8Empty + i), 1);
      mbar_init(bar(kV8Full + i), 4);
      mbar_init(bar(kV8Empty + i), 1);
      mbar_init(bar(kSFull + i), 1);
      mbar_init(bar(kSEmpty + i), 4);
      mbar_init(bar(kPFull + i), 4);
      mbar_init(bar(kPEmpty + i), 1);
      mbar_init(bar(kOFull + i), 1);
      mbar_init(bar(kOEmpty + i), 4);
    }
    mbar_init(bar(kDone), 1);
    *s_seq = -1;
    *s_abort = 0;
    *s_issued = 0;
    fence_barrier_init();
  }
  // zero the Q tile and both P tiles (the rows that stay zero pad N to 16)
  for (int i = tid; i < 3 * 2048 / 16; i += kThreads)
    reinterpret_cast<uint4*>(smem + kOffQ)[i] = make_uint4(0, 0, 0, 0);
  if (warp == 1) tmem_alloc(smem_u32(s_tmem), kTmemCols);
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
  if (tid < 32) {  // query rows 0-3: heads 4*kvh .. 4*kvh+3, 128-byte swizzled K-major
    const int row = tid >> 3, c = tid & 7;
    const uint4 v = *reinterpret_cast<const uint4*>(p.q + ((size_t)j * kQHeads + kvh * kGqa + row) * kHeadDim + 16 * c);
    *reinterpret_cast<uint4*>(smem + kOffQ + row * 128 + ((c ^ row) << 4)) = v;
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
  if (tid == 0) {  // compact this split's valid pages; tokens visible in each
    int n = 0;
    for (int i = 0; i < kSelStride; ++i)
      if (s_phys[i] >= 0) {
        s_phys[n] = s_phys[i];
        s_valid[n] = s_blk[i] == r_blk ? (pos % kPageTokens) + 1 : kPageTokens;
        ++n;
      }
    *s_npg = n;
  }
  __syncthreads();
  const int n_pg = *s_npg;

  if (warp == 0) {
    // ---------------- TMA producer ----------------------------------------------
    if (lane == 0) {
      int e = 0;
      for (; e < n_pg; ++e) {
        const int sl = e & 1;
        if (!mbar_wait(bar(kRawEmpty + sl), ((e >> 1) & 1) ^ 1, s_abort)) break;
        mbar_arrive_expect_tx(bar(kRawFull + sl), kHeadBytes);
        bulk_g2s(sbase + kOffRaw + sl * kHeadBytes,
                 p.kv_pool + (size_t)s_phys[e] * kKvPageBytes + kvh * kHeadBytes, kHeadBytes,
                 bar(kRawFull + sl));
      }
      *s_issued = e;
    }
    __syncwarp();
  } else if (warp == 1) {
    // ---------------- MMA issuer --------------------------------------------------
    if (lane == 0) {
      const uint32_t idesc_qk = umma_idesc_e4m3(128, 16);
      const uint32_t idesc_pv = umma_idesc_e4m3_amn(128, 16);
      const uint64_t qdesc = umma_desc_sw128(sbase + kOffQ);
      auto qk = [&](int e) -> bool {
        const int sl = e & 1, ph = (e >> 1) & 1;
        if (!mbar_wait(bar(kK8Full + sl), ph, s_abort)) return false;
        if (!mbar_wait(bar(kSEmpty + sl), ph ^ 1, s_abort)) return false;
        tc_fence_after();
        const uint64_t adesc = umma_desc_sw128(sbase + kOffK8 + sl * kTileBytes);
#pragma unroll
        for (int k = 0; k < 4; ++k)  // K = 32 bytes per MMA: +32 B = +2 in the encoded address
          umma_e4m3(tmem + 16 * sl, adesc + 2 * k, qdesc + 2 * k, idesc_qk, k > 0);
        umma_commit(bar(kK8Empty + sl));
        umma_commit(bar(kSFull + sl));
        return true;
      };
      auto pv = [&](int e) -> bool {
        const int sl = e & 1, ph = (e >> 1) & 1;
        if (!mbar_wait(bar(kV8Full + sl), ph, s_abort)) return false;
        if (!mbar_wait(bar(kPFull + sl), ph, s_abort)) return false;
        if (!mbar_wait(bar(kOEmpty + sl), ph ^ 1, s_abort)) return false;
        tc_fence_after();
        const uint64_t bdesc = umma_desc_sw128(sbase + kOffP + sl * 2048);
#pragma unroll
        for (int k = 0; k < 4; ++k) {
          // A: V tile read MN-major; 32 tokens (4 swizzle atoms of 8 rows) per MMA
          const uint64_t adesc =
              umma_desc_sw128_lbo_sbo(sbase + kOffV8 + sl * kTileBytes + k * 4096, 1024, 1024);
          umma_e4m3(tmem + 32 + 16 * sl, adesc, bdesc + 2 * k, idesc_pv, k > 0);
        }
        umma_commit(bar(kV8Empty + sl));
        umma_commit(bar(kPEmpty + sl));
        umma_commit(bar(kOFull + sl));
        return true;
      };
      bool ok = n_pg == 0 || qk(0);
      for (int e = 0; ok && e < n_pg; ++e) {
        if (e + 1 < n_pg && !qk(e + 1)) break;
        if (!pv(e)) break;
      }
      if (*s_abort) {
        // no tcgen05.mma may still be running when tensor memory is released
        volatile int ignore = 0;
        umma_commit(bar(kDone));
        mbar_wait(bar(kDone), 0, &ignore);
      }
    }
    __syncwarp();
  } else if (warp >= 6) {
    // ---------------- conversion: thread = token --------------------------------
    const int tok = tid - 192;
    for (int e = 0; e < n_pg; ++e) {
      const int sl = e & 1, ph = (e >> 1) & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(kRawFull + sl), ph, s_abort))) break;
      const bool live = tok < s_valid[e];
      const uint8_t* raw = smem + kOffRaw + sl * kHeadBytes;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(kK8Empty + sl), ph ^ 1, s_abort))) break;
      convert_row(raw + kOffKc + tok * 64, raw + kOffKs + tok, s_tab, smem + kOffK8 + sl * kTileBytes, tok, live);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kK8Full + sl));
      if (!__all_sync(0xffffffffu, mbar_wait(bar(kV8Empty + sl), ph ^ 1, s_abort))) break;
      convert_row(raw + kOffVc + tok * 64, raw + kOffVs + tok, s_tab, smem + kOffV8 + sl * kTileBytes, tok, live);
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(kV8Full + sl));
        mbar_arrive(bar(kRawEmpty + sl));
      }
    }
  } else {
    // ---------------- softmax and O folding (warps 2-5) -------------------------
    // warp w reads TMEM lanes 32 (w % 4) ..: row = token of S, channel of O
    const int quad = warp & 3, row = 32 * quad + lane;
    const uint32_t trow = tmem + ((uint32_t)(32 * quad) << 16);
    float m_run[4], l_run[4], o_run[4], a_prev[4], b_prev[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      m_run[h] = -INFINITY;
      l_run[h] = 0.f;
      o_run[h] = 0.f;
      a_prev[h] = 1.f;
      b_prev[h] = 0.f;
    }
    // O of page e (relative to its page max) -> running state
    auto fold = [&](int e) -> bool {
      const int sl = e & 1;
      if (!__all_sync(0xffffffffu, mbar_wait(bar(kOFull + sl), (e >> 1) & 1, s_abort))) return false;
      tc_fence_after();
      float ov[8];
      tmem_ld8(trow + 32 + 16 * sl, ov);  // columns 0-3: hi terms, 4-7: remainders
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kOEmpty + sl));
#pragma unroll
      for (int h = 0; h < 4; ++h) o_run[h] = o_run[h] * a_prev[h] + (ov[h] + ov[4 + h]) * b_prev[h];
      return true;
    };
    bool ok = true;
    for (int e = 0; e < n_pg; ++e) {
      const int sl = e & 1, ph = (e >> 1) & 1;
      bool good = __all_sync(0xffffffffu, mbar_wait(bar(kSFull + sl), ph, s_abort));
      float sv[4] = {0.f, 0.f, 0.f, 0.f};
      if (good) {
        tc_fence_after();
        tmem_ld4(trow + 16 * sl, sv);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kSEmpty + sl));
      }
      const bool live = row < s_valid[e];
      float x[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        x[h] = live ? sv[h] * p.scale_log2 : -INFINITY;
        const float wm = warp_max(x[h]);
        if (lane == 0) s_red[(sl * 4 + quad) * 4 + h] = wm;
      }
      // page maxima complete; the four warps agree on whether to go on
      if (named_barrier_or(1, 128, !good || !ok)) {
        ok = false;
        break;
      }
      uint32_t p_hi = 0, p_lo = 0;
      float a_cur[4], b_cur[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const float* r = s_red + sl * 16 + h;
        const float mp = fmaxf(fmaxf(r[0], r[4]), fmaxf(r[8], r[12]));
        const float m_new = fmaxf(m_run[h], mp);
        // m_new = -inf only while no key so far is visible (then everything is 0)
        a_cur[h] = m_new == -INFINITY ? 1.f : fast_exp2(m_run[h] - m_new);
        b_cur[h] = mp == -INFINITY ? 0.f : fast_exp2(mp - m_new);  // page scale -> running scale
        const float pr = mp == -INFINITY ? 0.f : fast_exp2(x[h] - mp);  // relative to the page max
        l_run[h] = l_run[h] * a_cur[h] + pr * b_cur[h];
        m_run[h] = m_new;
        const float v256 = pr * 256.f;
        const uint32_t hi = f32_to_e4m3(v256);
        const uint32_t lo = f32_to_e4m3(v256 - e4m3_to_f32(hi));
        p_hi |= hi << (8 * h);
        p_lo |= lo << (8 * h);
      }
      // P rows h (E4M3 of 256 p) and 4+h (E4M3 of the remainder), one byte per
      // token: byte t of row n sits in chunk (t/16) ^ (n & 7)
      bool step_ok = __all_sync(0xffffffffu, mbar_wait(bar(kPEmpty + sl), ph ^ 1, s_abort));
      if (step_ok) {
        uint8_t* pt = smem + kOffP + sl * 2048;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          pt[h * 128 + (((row >> 4) ^ h) << 4) + (row & 15)] = (uint8_t)(p_hi >> (8 * h));
          pt[(4 + h) * 128 + (((row >> 4) ^ (4 + h)) << 4) + (row & 15)] = (uint8_t)(p_lo >> (8 * h));
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kPFull + sl));
        if (e > 0) step_ok = fold(e - 1);
      }
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        a_prev[h] = a_cur[h];
        b_prev[h] = b_cur[h];
      }
      ok = ok && step_ok;  // a failure here ends the loop at the next barrier
    }
    if (ok && n_pg > 0) ok = fold(n_pg - 1);
    const bool aborted = named_barrier_or(1, 128, !ok || *s_abort != 0);
    // ---- l over the tokens, normalised partial output (thread = channel) ----------
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      float l = l_run[h];
#pragma unroll
      for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
      if (lane == 0) s_redl[quad * 4 + h] = l;
    }
    named_barrier_sync(1, 128);
    const size_t row0 = ((size_t)j * p.n_splits + split) * kQHeads + kvh * kGqa;
#pragma unroll
    for (int h = 0; h < 4; ++h) {
      const float L = s_redl[h] + s_redl[4 + h] + s_redl[8 + h] + s_redl[12 + h];
      const bool nonempty = !aborted && L > 0.f && m_run[h] != -INFINITY;
      p.o_part[(row0 + h) * kHeadDim + row] = nonempty ? o_run[h] / L * p.out_scale : 0.f;
      if (row == 0) p.lse_part[row0 + h] = nonempty ? (m_run[h] + log2f(L)) * kLn2 : -INFINITY;
    }
  }

  // ---- teardown -----------------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  if (*s_abort && tid == 0) {
    set_status(p.status, MSA_STATUS_TIMEOUT);
    // bounded drain of the copies that may still be landing: the last two issued
    // (each earlier one was consumed before its stage was refilled)
    volatile int ignore = 0;
    const int n_iss = *s_issued;
    for (int e = max(0, n_iss - 2); e < n_iss; ++e)
      mbar_wait(bar(kRawFull + (e & 1)), (e >> 1) & 1, &ignore);
  }
  __syncthreads();
  if (warp == 1) {
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
