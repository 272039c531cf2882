// The whole decode step in one launch, for low concurrency: index scan, top-16
// + recent selection, sparse attention and the log-sum-exp merge.
//
// "vLLM Delivers Day-0 Support for MiniMax-M3.1-Flash" blog, sections "AMD
// uses different conversion and communication mechanisms" (a separate
// single-kernel strategy that reduces launches at low concurrency) and "Keep
// capacity, layer, and system results separate" (fewer launches pay at low
// concurrency, not necessarily at high).  With one or a few query tokens the
// four-launch path is bound by launch and pipeline latency, not by bytes; here
// one cooperative launch runs the four phases with a grid barrier between
// them, every CTA working on one page at a time with all its threads:
//   1. scan: CTA c scores pages c, c + G, ...: the 16 KB index page and the
//      index queries as a 128-byte-swizzled tile pair, 4 x tcgen05.mma
//      kind::f8f6f4 (M = 128 tokens, N = 8 heads x query tokens, K = 128),
//      ReLU . w summed over heads and the block max, written as the four
//      partial maxima the shared top-k reads;
//   2. top-k: CTA c selects for query tokens c, c + G, ... (topk.cuh);
//   3. attention: work item = (token, selected entry e, KV head) = one page:
//      K and V of the page converted NVFP4 -> FP8 (table + byte permutes) into
//      two swizzled tiles, S = K8 Q^T and O^T = V8^T P^T on the tensor core,
//      softmax of the page in between; the page's normalised output and
//      log-sum-exp are split e of the token;
//   4. merge: the CTA that writes the last split of a (token, KV head) -- a
//      counter per pair tells -- merges its splits at once (no fourth phase).
// Short contexts prefetch the KV pages they scan into L2 for the attention.
// Same arithmetic, rounding and layouts as the four-launch path (msa.h).
#include "common.cuh"
#include "topk.cuh"

namespace msa {
namespace {

constexpr int kFThreads = 256;
constexpr int kFNq = 8;            // query tokens per scan pass
constexpr int kFMaxSeqs = 64;      // low-concurrency limits of this path
constexpr int kFMaxTokens = 64;
// Shared memory.  The tiles of the scan and attention phases sit in [0, 42 KB);
// the top-k phase reuses [0, kTopkSmem) (staged scores, candidates, reduction
// scratch); what lives through all phases sits above it.
constexpr int kOffTile0 = 0;       // index page (scan) / K8 tile (attention), 16 KB
constexpr int kOffTile1 = 16384;   // V8 tile, 16 KB
constexpr int kOffB = 32768;       // scan B tile [64 rows][128 B] / attention Q tile [16 rows][128 B]
constexpr int kOffP = 40960;       // P tile [128 tokens][16 B]
constexpr int kTopkSmem = 4 * kTopkStage + 8 * kMaxCand + 8 * kFThreads + 8 * kTopK + 4 * 32;
constexpr int kOffTab = (kTopkSmem + 1023) / 1024 * 1024;  // dequantisation table, uint2 [256]
constexpr int kOffRed = kOffTab + 2048;   // float [64]: maxima and sums across the 4 row warps
constexpr int kOffMisc = kOffRed + 256;   // mbarrier (8), tmem slot, abort flag
constexpr int kOffSeq = kOffMisc + 64;    // s_sl [n_seqs], s_qsl [n_seqs + 1], s_prefix [n_seqs + 1]
constexpr int kFSmem = kOffSeq + 4 * (3 * kFMaxSeqs + 2);
static_assert(kOffP + 2048 <= kTopkSmem, "tiles below the persistent state");
constexpr uint32_t kFTmemCols = 64;
constexpr int kPrefetchPages = 96;  // contexts of at most this many scanned pages prefetch their KV
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;

struct FusedParams {
  const uint8_t* kv_pool;
  const uint8_t* idx_pool;
  int64_t n_pages;
  const uint8_t* q;      // [T][16][128] E4M3
  const uint8_t* q_idx;  // [T][8][128] E4M3
  const float* w;        // [T][8]
  const int* block_table;
  int max_pages;
  const int* seq_lens;
  const int* q_start_loc;
  int n_seqs;
  int n_q_total;
  float scale_log2;  // softmax_scale / s_enc_k * log2(e)
  float out_scale;   // 1 / s_enc_v
  int* sel;          // [T][17]
  int* n_sel;        // [T]
  float* out;        // [T][16][128]
  unsigned long long* sync;  // two grid-barrier words
  float* scores;     // [T][max_pages][4]
  float* o_part;     // [T][17][16][128]
  float* lse_part;   // [T][17][16]
  int* done;         // [T][4] splits written per (token, KV head)
  int* status;
  unsigned long long wait_ns;
};

// One tensor-core pass: thread 0 issues four K = 32 steps and commits; every
// thread waits for the commit (bounded).
__device__ __forceinline__ bool mma4_and_wait(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                              uint32_t bar, uint32_t& phase, const WaitCtl& wc, bool a_step,
                                              uint32_t a_stride16, uint32_t b_stride16) {
  if (threadIdx.x == 0) {
    tc_fence_after();
#pragma unroll
    for (int k = 0; k < 4; ++k)
      umma_e4m3(d_tmem, adesc + (a_step ? a_stride16 * k : 0), bdesc + b_stride16 * k, idesc, k > 0);
    umma_commit(bar);
  }
  const bool ok = mbar_wait(bar, phase, wc);
  phase ^= 1;
  tc_fence_after();
  // the CTA agrees: a wait that ran out in any thread ends the phase for all
  return !__syncthreads_or(!ok);
}

// A CTA has written split e of (token j, KV head g).  It counts the split in;
// the CTA that counts the last of the token's nsel splits merges them:
//   out = sum_e exp(lse_e - M) o_e / sum_e exp(lse_e - M),  M = max_e lse_e,
// per query head of the group (thread = (head, two channels)), then returns
// the counter to zero.  Ends with a barrier of the CTA.
__device__ __forceinline__ void split_done(const FusedParams& p, int j, int g, int nsel, uint8_t* s_flag) {
  __syncthreads();  // the CTA's split is written (CTA scope) before thread 0 counts it
  int* flag = reinterpret_cast<int*>(s_flag);
  if (threadIdx.x == 0) {
    // release: this CTA's writes before the count; acquire: the other CTAs'
    // splits, counted before, visible to the merge below
    int old;
    asm volatile("atom.add.acq_rel.gpu.s32 %0, [%1], 1;" : "=r"(old) : "l"(p.done + j * kKvHeads + g) : "memory");
    *flag = old == nsel - 1;
  }
  __syncthreads();
  if (*flag) {
    const int h = threadIdx.x >> 6, ch = 2 * (threadIdx.x & 63);
    const size_t r0 = (size_t)j * kSelStride * kQHeads + g * kGqa + h;
    // every split's log-sum-exp and output in flight at once, then one pass
    float l[kSelStride];
    float2 o[kSelStride];
#pragma unroll
    for (int e = 0; e < kSelStride; ++e) {
      if (e < nsel) {
        const size_t r = r0 + (size_t)e * kQHeads;
        l[e] = __ldcg(p.lse_part + r);
        o[e] = __ldcg(reinterpret_cast<const float2*>(p.o_part + r * kHeadDim + ch));
      }
    }
    float M = -INFINITY;
#pragma unroll
    for (int e = 0; e < kSelStride; ++e)
      if (e < nsel) M = fmaxf(M, l[e]);
    float den = 0.f, n0 = 0.f, n1 = 0.f;
    if (M != -INFINITY) {
#pragma unroll
      for (int e = 0; e < kSelStride; ++e) {
        if (e < nsel) {
          const float f = __expf(l[e] - M);
          den += f;
          n0 += f * o[e].x;
          n1 += f * o[e].y;
        }
      }
    }
    float2* dst = reinterpret_cast<float2*>(p.out + ((size_t)j * kQHeads + g * kGqa + h) * kHeadDim + ch);
    *dst = den > 0.f ? make_float2(n0 / den, n1 / den) : make_float2(0.f, 0.f);
    if (threadIdx.x == 0) p.done[j * kKvHeads + g] = 0;
  }
  __syncthreads();
}

__global__ void __launch_bounds__(kFThreads, 1) decode_fused_kernel(FusedParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t mbar = sbase + kOffMisc;
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kOffMisc + 8);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + kOffMisc + 12);
  int* s_sl = reinterpret_cast<int*>(smem + kOffSeq);
  int* s_qsl = s_sl + p.n_seqs;
  int* s_prefix = s_qsl + p.n_seqs + 1;
  uint2* s_tab = reinterpret_cast<uint2*>(smem + kOffTab);
  float* red = reinterpret_cast<float*>(smem + kOffRed);
  const WaitCtl wc{s_abort, p.wait_ns};
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = gridDim.x;
  uint32_t phase = 0;

  pdl_wait();
  // ---- prologue: metadata, pages to scan per sequence, table, tensor memory ----
  for (int b = tid; b < p.n_seqs; b += kFThreads) s_sl[b] = p.seq_lens[b];
  for (int b = tid; b <= p.n_seqs; b += kFThreads) s_qsl[b] = p.q_start_loc[b];
  build_dequant_table(s_tab, tid, kFThreads);
  if (tid == 0) {
    mbar_init(mbar, 1);
    *s_abort = 0;
    fence_barrier_init();
  }
  __syncthreads();
  if (tid == 0) {
    int acc = 0;
    for (int b = 0; b < p.n_seqs; ++b) {
      const SeqInfo s = load_seq(b, s_sl, s_qsl, p.max_pages, p.n_q_total);
      if (!s.ok && blockIdx.x == 0) set_status(p.status, MSA_STATUS_BAD_SEQ);
      s_prefix[b] = acc;
      acc += (s.ok && s.seq_len > 0 && s.n_q > 0) ? (s.seq_len - 1) / kPageTokens : 0;
    }
    s_prefix[p.n_seqs] = acc;
  }
  if (warp == 0) tmem_alloc(smem_u32(s_tmem), kFTmemCols);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  const uint32_t tq = tmem + ((uint32_t)(32 * (warp & 3)) << 16);  // this warp's lane quadrant

  // ---- 1. scan ----------------------------------------------------------------
  const int n_scan = s_prefix[p.n_seqs];
  // split counters of phase 3 start at zero (two barriers order this before use)
  for (int i = blockIdx.x * kFThreads + tid; i < p.n_q_total * kKvHeads; i += G * kFThreads) p.done[i] = 0;
  const bool prefetch = n_scan <= kPrefetchPages;
  bool going = true;  // CTA-uniform: false once a wait ran out
  for (int x = blockIdx.x; going && x < n_scan; x += G) {
    int b = 0;
    while (s_prefix[b + 1] <= x) ++b;
    const SeqInfo s = load_seq(b, s_sl, s_qsl, p.max_pages, p.n_q_total);
    const int blk = x - s_prefix[b];
    const int phys = p.block_table[(size_t)b * p.max_pages + blk];
    const bool bad = phys < 0 || phys >= p.n_pages;
    if (bad) {
      if (tid == 0) set_status(p.status, MSA_STATUS_BAD_PAGE);
      for (int j = tid; j < s.n_q; j += kFThreads)
        reinterpret_cast<float4*>(p.scores)[(size_t)(s.q0 + j) * p.max_pages + blk] =
            make_float4(-INFINITY, -INFINITY, -INFINITY, -INFINITY);
      continue;
    }
    if (prefetch && tid < kKvHeads) {
      // short context: most of its KV pages will be selected; warm L2 with
      // this block's (and, at the sequence's last scanned block, the recent
      // block's) KV page while the scan runs
      const uint8_t* kv = p.kv_pool + (size_t)phys * kKvPageBytes + tid * kHeadBytes;
      asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(kv), "r"(kHeadBytes) : "memory");
      if (blk + 1 == s_prefix[b + 1] - s_prefix[b]) {
        const int rp = p.block_table[(size_t)b * p.max_pages + blk + 1];
        if (rp >= 0 && rp < p.n_pages) {
          const uint8_t* kr = p.kv_pool + (size_t)rp * kKvPageBytes + tid * kHeadBytes;
          asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(kr), "r"(kHeadBytes) : "memory");
        }
      }
    }
    // the index page is stored in the swizzled operand layout: a straight copy
    const uint4* src = reinterpret_cast<const uint4*>(p.idx_pool + (size_t)phys * kIdxPageBytes);
#pragma unroll
    for (int u = 0; u < kIdxPageBytes / 16 / kFThreads; ++u)
      reinterpret_cast<uint4*>(smem + kOffTile0)[tid + u * kFThreads] = ld_stream_v4(src + tid + u * kFThreads);
    for (int j0 = 0; j0 < s.n_q; j0 += kFNq) {
      const int nq = min(kFNq, s.n_q - j0);
      const int n_rows = 16 * ((nq + 1) >> 1);
      // index queries (token, head) rows, 128-byte swizzled, zero rows up to N
      const uint8_t* qsrc = p.q_idx + (size_t)(s.q0 + j0) * kIdxHeads * kIdxDim;
      for (int e = tid; e < n_rows * 8; e += kFThreads) {
        const int row = e >> 3, c = e & 7;
        const uint4 v = row < nq * kIdxHeads ? *reinterpret_cast<const uint4*>(qsrc + row * kIdxDim + c * 16)
                                             : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(smem + kOffB + row * kIdxDim + ((c ^ (row & 7)) << 4)) = v;
      }
      fence_proxy_async_smem();
      __syncthreads();
      if (!mma4_and_wait(tmem, umma_desc_sw128(sbase + kOffTile0), umma_desc_sw128(sbase + kOffB),
                         umma_idesc_e4m3(128, n_rows), mbar, phase, wc, true, 2, 2)) {
        going = false;
        break;
      }
      if (warp < 4) {
        // thread = token row of the page: every column in one load, one wait
        uint32_t v[64];
        if (nq <= 2) tmem_ld32x32b_x16(tq, v);
        else if (nq <= 4) tmem_ld32x32b_x32(tq, v);
        else tmem_ld32x32b_x64(tq, v);
        tmem_wait_ld();
#pragma unroll
        for (int jj = 0; jj < kFNq; ++jj) {
          if (jj < nq) {
            const float* wj = p.w + (size_t)(s.q0 + j0 + jj) * kIdxHeads;
            float sc = 0.f;
#pragma unroll
            for (int h = 0; h < kIdxHeads; ++h) sc = fmaf(__ldg(wj + h), fmaxf(__uint_as_float(v[8 * jj + h]), 0.f), sc);
            const float m = warp_max_f32(sc);
            if (lane == 0) red[warp * 8 + jj] = m;
          }
        }
      }
      tc_fence_before();
      __syncthreads();
      if (tid < nq) {
        const float m = fmaxf(fmaxf(red[tid], red[8 + tid]), fmaxf(red[16 + tid], red[24 + tid]));
        reinterpret_cast<float4*>(p.scores)[(size_t)(s.q0 + j0 + tid) * p.max_pages + blk] = make_float4(m, m, m, m);
      }
      __syncthreads();
    }
  }

  // ---- 2. top-16 + recent -----------------------------------------------------
  if (tid == 0) grid_barrier(p.sync, G, wc);
  going = !__syncthreads_or(*s_abort != 0);
  if (going) {
    TopkSmem sm;
    sm.sc = reinterpret_cast<float*>(smem);
    sm.cand = reinterpret_cast<unsigned long long*>(smem + 4 * kTopkStage);
    sm.tmax = reinterpret_cast<unsigned long long*>(smem + 4 * kTopkStage + 8 * kMaxCand);
    sm.win = sm.tmax + kFThreads;
    sm.misc = reinterpret_cast<int*>(sm.win + kTopK);
    const TopkArgs ta{p.scores, p.max_pages, p.n_seqs, p.n_q_total, p.sel, p.n_sel, p.status, 0, 0x7FFFFFFF,
                      nullptr};
    for (int j = blockIdx.x; j < p.n_q_total; j += G) {
      select_token<kFThreads>(ta, j, s_sl, s_qsl, sm);
      __syncthreads();
    }
  }

  // ---- 3. attention, one page (token, entry, KV head) at a time ----------------
  if (tid == 0) grid_barrier(p.sync + 1, G, wc);
  going = !__syncthreads_or(*s_abort != 0);
  // rows 4..15 of the Q tile and bytes 8..15 of every P row pad N to 16
  for (int i = tid; i < (2048 + 2048) / 16; i += kFThreads)
    reinterpret_cast<uint4*>(smem + (i < 128 ? kOffB : kOffP - 2048))[i] = make_uint4(0, 0, 0, 0);
  fence_proxy_async_smem();
  __syncthreads();
  const int n_items = p.n_q_total * kSelStride * kKvHeads;
  for (int item = blockIdx.x; going && item < n_items; item += G) {
    const int j = item / (kSelStride * kKvHeads);
    const int e = (item / kKvHeads) % kSelStride, g = item % kKvHeads;
    const int b = find_seq(s_qsl, p.n_seqs, j);
    const SeqInfo s = load_seq(b, s_sl, s_qsl, p.max_pages, p.n_q_total);
    const bool seq_ok = s.ok && j >= s.q0 && j < s.q0 + s.n_q;  // else flagged in the top-k
    const int nsel = seq_ok ? max(0, min(__ldcg(p.n_sel + j), kSelStride)) : 0;
    if (e >= nsel) {
      if (e == 0)  // nothing to attend: the token's rows are zero
        for (int i = tid; i < kGqa * kHeadDim; i += kFThreads)
          p.out[((size_t)j * kQHeads + g * kGqa) * kHeadDim + i] = 0.f;
      continue;
    }
    const int pos = s.seq_len - s.n_q + (j - s.q0), r = pos / kPageTokens;
    const int blk = __ldcg(p.sel + (size_t)j * kSelStride + e);
    int phys = -1;
    if (blk < 0 || blk > r) {
      if (tid == 0) set_status(p.status, MSA_STATUS_BAD_SELECTION);
    } else {
      phys = p.block_table[(size_t)b * p.max_pages + blk];
      if (phys < 0 || phys >= p.n_pages) {
        if (tid == 0) set_status(p.status, MSA_STATUS_BAD_PAGE);
        phys = -1;
      }
    }
    const size_t row0 = ((size_t)j * kSelStride + e) * kQHeads + g * kGqa;
    if (phys < 0) {  // an empty split
      for (int i = tid; i < kGqa * kHeadDim; i += kFThreads) p.o_part[row0 * kHeadDim + i] = 0.f;
      if (tid < kGqa) p.lse_part[row0 + tid] = -INFINITY;
      split_done(p, j, g, nsel, smem + kOffMisc + 16);
      continue;
    }
    const int valid = blk == r ? pos % kPageTokens + 1 : kPageTokens;
    // K (threads 0..127) and V (128..255) of token t -> FP8, row t of a tile
    {
      const int t = tid & 127;
      const bool is_v = tid >= 128;
      const uint8_t* head = p.kv_pool + (size_t)phys * kKvPageBytes + g * kHeadBytes + (is_v ? kOffVc : kOffKc);
      uint4 chunk[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) chunk[c] = ld_stream_v4(head + t * 64 + 16 * code_chunk_pos(c, t));
      uint32_t sc[8];
#pragma unroll
      for (int k = 0; k < 8; ++k) sc[k] = head[(kOffKs - kOffKc) + k * kPageTokens + t];
      uint8_t* tile = smem + (is_v ? kOffTile1 : kOffTile0) + t * 128;
      const bool live = t < valid;
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint2 t0 = s_tab[sc[2 * c]], t1 = s_tab[sc[2 * c + 1]];
        const uint2 a = dequant8(chunk[c].x, t0), bb = dequant8(chunk[c].y, t0);
        const uint2 d = dequant8(chunk[c].z, t1), ee = dequant8(chunk[c].w, t1);
        const uint4 lo = live ? make_uint4(a.x, a.y, bb.x, bb.y) : make_uint4(0, 0, 0, 0);
        const uint4 hi = live ? make_uint4(d.x, d.y, ee.x, ee.y) : make_uint4(0, 0, 0, 0);
        *reinterpret_cast<uint4*>(tile + (((2 * c) ^ (t & 7)) << 4)) = lo;
        *reinterpret_cast<uint4*>(tile + (((2 * c + 1) ^ (t & 7)) << 4)) = hi;
      }
    }
    if (warp == 0) {  // the 4 query rows of KV head g, 128-byte swizzled
      const int row = lane >> 3, c = lane & 7;
      *reinterpret_cast<uint4*>(smem + kOffB + row * 128 + ((c ^ row) << 4)) = *reinterpret_cast<const uint4*>(
          p.q + ((size_t)j * kQHeads + g * kGqa + row) * kHeadDim + 16 * c);
    }
    fence_proxy_async_smem();
    __syncthreads();
    // S = K8 Q^T: 128 tokens x 16 (4 heads, zero padded), columns 0..15
    if (!mma4_and_wait(tmem, umma_desc_sw128(sbase + kOffTile0), umma_desc_sw128(sbase + kOffB),
                       umma_idesc_e4m3(128, 16), mbar, phase, wc, true, 2, 2)) {
      going = false;
      break;
    }
    float v[4] = {0.f, 0.f, 0.f, 0.f}, x[4];
    if (warp < 4) {
      float sv[4];
      tmem_ld4(tq, sv);
      const bool live = 32 * warp + lane < valid;
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        x[h] = live ? sv[h] * p.scale_log2 : -INFINITY;
        const float m = warp_max_f32(x[h]);
        if (lane == 0) red[warp * 4 + h] = m;
      }
    }
    __syncthreads();
    float mp[4];
#pragma unroll
    for (int h = 0; h < 4; ++h) mp[h] = fmaxf(fmaxf(red[h], red[4 + h]), fmaxf(red[8 + h], red[12 + h]));
    if (warp < 4) {
      // 256 p relative to the page max, as two E4M3 terms (hi, remainder)
#pragma unroll
      for (int h = 0; h < 4; ++h) v[h] = fast_exp2(x[h] - mp[h] + 8.f);
      const uint32_t hi01 = cvt_e4m3x2_f32(v[1], v[0]), hi23 = cvt_e4m3x2_f32(v[3], v[2]);
      const uint32_t lo01 = cvt_e4m3x2_f16x2(hsub2_u32(cvt_f16x2_f32(v[1], v[0]), cvt_f16x2_e4m3x2(hi01)));
      const uint32_t lo23 = cvt_e4m3x2_f16x2(hsub2_u32(cvt_f16x2_f32(v[3], v[2]), cvt_f16x2_e4m3x2(hi23)));
      *reinterpret_cast<uint2*>(smem + kOffP + 16 * (32 * warp + lane)) =
          make_uint2(prmt(hi01, hi23, 0x5410u), prmt(lo01, lo23, 0x5410u));
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        float l = v[h];
#pragma unroll
        for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) red[32 + warp * 4 + h] = l;
      }
    }
    tc_fence_before();
    fence_proxy_async_smem();
    __syncthreads();
    // O^T = V8^T P^T: 128 channels x 16, columns 16..31
    if (!mma4_and_wait(tmem + 16, umma_desc_sw128_lbo_sbo(sbase + kOffTile1, 1024, 1024),
                       umma_desc_noswz_lbo_sbo(sbase + kOffP, 128, 128), umma_idesc_e4m3_amn_bmn(128, 16), mbar,
                       phase, wc, true, 4096 >> 4, 512 >> 4)) {
      going = false;
      break;
    }
    if (warp < 4) {  // thread = channel
      float ov[8];
      tmem_ld8(tq + 16, ov);
      const int ch = 32 * warp + lane;
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        const float L = red[32 + h] + red[36 + h] + red[40 + h] + red[44 + h];
        p.o_part[(row0 + h) * kHeadDim + ch] = (ov[h] + ov[4 + h]) / L * p.out_scale;
        if (ch == 0) p.lse_part[row0 + h] = (mp[h] + log2f(L) - 8.f) * kLn2;
      }
    }
    tc_fence_before();
    split_done(p, j, g, nsel, smem + kOffMisc + 16);
  }

  // ---- teardown ----------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  if (*s_abort && tid == 0) {
    // a wait ran out: the last commit must have landed before tensor memory goes
    umma_commit(mbar);
    mbar_wait_drain(mbar, phase, p.wait_ns);
  }
  __syncthreads();
  if (warp == 0) {
    tc_fence_after();
    tmem_dealloc(tmem, kFTmemCols);
  }
  if (tid == 0 && *s_abort) set_status(p.status, MSA_STATUS_TIMEOUT);
}

}  // namespace

size_t decode_fused_workspace_bytes(int n_q_total, int max_pages) {
  const size_t scores = (size_t)n_q_total * max_pages * 16;
  const size_t o = (size_t)n_q_total * kSelStride * kQHeads * kHeadDim * 4;
  const size_t lse = (size_t)n_q_total * kSelStride * kQHeads * 4;
  const size_t done = (size_t)n_q_total * kKvHeads * 4;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  return 256 + up(scores) + up(o) + up(lse) + up(done);
}

int decode_fused_max_seqs() { return kFMaxSeqs; }
int decode_fused_max_tokens() { return kFMaxTokens; }

cudaError_t launch_decode_fused(const msa_cache* c, const uint8_t* q, const uint8_t* q_idx, const float* w,
                                float softmax_scale, const int* block_table, int max_pages,
                                const int* seq_lens, const int* q_start_loc, int n_seqs, int n_q_total,
                                int* sel, int* n_sel, float* out, void* ws, cudaStream_t stream) {
  if (n_q_total == 0 || n_seqs == 0) return cudaSuccess;
  static DeviceSetup setup;
  int dev = 0, n_sm = 0;
  cudaError_t e = setup.get(&dev, &n_sm, [](int) {
    return cudaFuncSetAttribute(decode_fused_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kFSmem + 1024);
  });
  if (e != cudaSuccess) return e;
  auto up = [](size_t x) { return (x + 255) / 256 * 256; };
  uint8_t* base = static_cast<uint8_t*>(ws);
  float* scores = reinterpret_cast<float*>(base + 256);
  float* o_part = reinterpret_cast<float*>(base + 256 + up((size_t)n_q_total * max_pages * 16));
  float* lse_part = reinterpret_cast<float*>(reinterpret_cast<uint8_t*>(o_part) +
                                             up((size_t)n_q_total * kSelStride * kQHeads * kHeadDim * 4));
  int* done = reinterpret_cast<int*>(reinterpret_cast<uint8_t*>(lse_part) +
                                     up((size_t)n_q_total * kSelStride * kQHeads * 4));
  FusedParams fp{static_cast<const uint8_t*>(c->kv_pool), static_cast<const uint8_t*>(c->idx_pool), c->n_pages,
                 q, q_idx, w, block_table, max_pages, seq_lens, q_start_loc, n_seqs, n_q_total,
                 softmax_scale / c->s_enc_k * kLog2e, 1.0f / c->s_enc_v, sel, n_sel, out,
                 static_cast<unsigned long long*>(ws), scores, o_part, lse_part, done, c->status,
                 launch_settings().wait_ns};
  // one CTA per SM at most, as many as the largest phase has pages
  long long work = (long long)n_q_total * kSelStride * kKvHeads;
  const int grid = (int)(work < n_sm ? work : n_sm);
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(grid);
  cfg.blockDim = dim3(kFThreads);
  cfg.dynamicSmemBytes = kFSmem + 1024;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeCooperative;
  attr[0].val.cooperative = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, decode_fused_kernel, fp);
}

}  // namespace msa
