// Split-context sparse GQA attention over the selected NVFP4 blocks on the
// fifth-generation tensor cores (tcgen05, tensor memory): one persistent,
// warp-specialised CTA per SM.
//
// "vLLM Delivers Day-0 Support for MiniMax-M3.1-Flash" blog, section "Sparse
// attention still scans an index": exact attention over the selected blocks
// only; section "Capacity savings must pay for conversion" and the ai4snews
// article (third paragraph): queries stay FP8, so the NVFP4 K/V are converted
// to FP8 before the matrix multiply.
//
// Work item = (query token j, KV head, split): the split's share of j's
// selected pages (entries split, split + S, ... of its selection).  CTA c
// takes items c, c + G, c + 2G, ...; its pages (numbered e = 0, 1, ... across
// its items) flow through warp roles, every hand-off an mbarrier and every
// wait bounded:
//   warp 0       scheduler and TMA producer: per item, the sequence of j
//                (a 32-way search of q_start_loc, copied to shared memory when
//                it fits beside the rings: up to 115 sequences), the selected
//                blocks, their physical pages and the tokens visible in each,
//                and the 4 query rows as a swizzled tile, into a ring of kRecs
//                item records;
//                then one 18,432-byte cp.async.bulk copy per page of the item
//                (the KV head's K and V codes and scales) into a ring of stages;
//   warps 1-2    QK issuers, warp 1 + s for the pages of set s (e % 2 == s):
//                S = K8 Q^T (kind::f8f6f4, M = 128 tokens, N = 16: the 4 query
//                heads, zero padded, K = 128, A from tensor memory);
//   warps 3-4    PV issuers, warp 3 + s for set s: O_s^T += V8^T P (A = the V
//                tile read MN-major, no transpose, B = P), accumulated in tensor
//                memory over the item's pages, one buffer per set and item
//                parity; the commit per page frees the page's V tile and P tile;
//   warps 5-12   softmax, two sets of 4 warps; set s takes the pages with
//                e % 2 == s, thread = token row of S: P = 256 * 2^(x - m) for a
//                reference m per head that changes only when a row of the page
//                exceeds it by more than kGrowth (then m = page max + kHeadroom,
//                and the set's row sums and O accumulator are rescaled); P is
//                written as two E4M3 terms (value + rounding remainder), the B
//                operand of PV.  At the item's end set 1 hands its (m, row sum)
//                to set 0, which reads both O accumulators (thread = channel)
//                and writes the normalised partial (O, LSE); the LSE merge
//                kernel combines the splits;
//   warps 13 ..  kGroups conversion warpgroups; group g converts the pages with
//                e % kGroups == g, thread = token: NVFP4 -> FP8 through a
//                256-entry shared table of scaled E4M3 values and byte
//                permutes, K written with tcgen05.st straight into tensor memory
//                (the A operand of QK), V into a 128-byte-swizzled shared tile.
#include "common.cuh"

namespace msa {
namespace {

constexpr int kInjectAttentionTimeout = 2;  // test hook: the producer leaves out its first copy
constexpr int kGroups = 3;      // conversion warpgroups
constexpr int kSets = 2;        // softmax sets (set = e % 2, also the S slot)
constexpr int kWarpSmax0 = 1 + 2 * kSets;  // warp 0 scheduler and producer, then a QK and a PV issuer per set
constexpr int kWarpConv0 = kWarpSmax0 + 4 * kSets;
constexpr int kThreads = 32 * (kWarpConv0 + 4 * kGroups);
constexpr int kStages = 6;     // raw page ring
constexpr int kRecs = 3;       // item records in flight
constexpr int kSlots = 6;      // K8 buffers (tensor memory), V8 tiles and P tiles: slot = e % kSlots
// A group waits only for its own pages' slots and stages; for a parity wait
// never to see a phase two behind, the same group must own every page of a
// slot (and of a stage): kGroups divides both ring sizes.
static_assert(kSlots % kGroups == 0 && kStages % kGroups == 0, "groups own whole slots and stages");
// Likewise a softmax set reuses the P tile (and waits on the PV commit) of its
// own page e - kSlots: kSets divides kSlots.
static_assert(kSlots % kSets == 0, "sets own whole P tiles");
constexpr int kTileBytes = 16384;                      // [128 rows][128 B], swizzled
constexpr int kOffV8 = 0;                              // kSlots V8 tiles
constexpr int kOffQ = kSlots * kTileBytes;             // kRecs x [16 rows][128 B]
constexpr int kOffP = kOffQ + kRecs * 2048;            // kSlots x [128 tokens][16 B]
constexpr int kOffRaw = kOffP + kSlots * 2048;         // kStages x 18,432
constexpr int kOffTab = kOffRaw + kStages * kHeadBytes;  // uint2 [256]
constexpr int kOffRec = kOffTab + 2048;                // kRecs x 256 B
constexpr int kOffRed = kOffRec + kRecs * 256;         // float [set][4 warps][4 heads] page maxima
constexpr int kOffRedL = kOffRed + 64 * kSets;         // float [set][4 warps][4 heads] row sums
constexpr int kOffMerge = kOffRedL + 64 * kSets;       // float [item parity][m 4, L 4] of set 1
constexpr int kOffBars = kOffMerge + 64;
// barrier indices
constexpr int kRawFull = 0, kRawEmpty = kStages, kK8Full = 2 * kStages, kK8Empty = kK8Full + kSlots,
              kSFull = kK8Empty + kSlots, kSEmpty = kSFull + 2, kV8Full = kSEmpty + 2,
              kPFull = kV8Full + kSlots, kPVDone = kPFull + kSlots, kOFree = kPVDone + kSlots,
              kMergeFull = kOFree + 2, kMergeEmpty = kMergeFull + 2,
              kRecFull = kMergeEmpty + 2, kRecEmpty = kRecFull + kRecs, kDone = kRecEmpty + kRecs,
              kNumBars = kDone + 1;  // kDone: every MMA of the CTA is done (one commit per issuer)
constexpr int kOffMisc = kOffBars + ((kNumBars * 8 + 15) / 16) * 16;  // tmem, abort, issued pages
constexpr int kOffQsl = kOffMisc + 16;  // int [n_seqs + 1] copy of q_start_loc
constexpr uint32_t kTmS = 32 * kSlots;  // TMEM columns: K8 slot i at 32 i, S slot s at kTmS + 16 s,
constexpr uint32_t kTmO = kTmS + 32;    // O of set s for item parity b at kTmO + 16 (2 b + s)
constexpr uint32_t kTmemCols = 512;
static_assert(kTmO + 64 <= kTmemCols, "tensor memory columns");
static_assert(kSets == 2, "S slots, O buffers and the merge are laid out for two sets");
// producer, QK issuers (a commit: the Q tile), PV issuers, the softmax warps, the conversion warps
constexpr int kRecEmptyCount = 1 + 2 * kSets + 4 * kSets + 4 * kGroups;
// P = 256 * 2^(x - m) must stay below the largest finite E4M3 value (448):
// a row more than kGrowth above m (256 * 2^0.75 = 430.5) moves m to the page
// max + kHeadroom, so that later pages rarely move it again.
constexpr float kGrowth = 0.75f;
constexpr float kHeadroom = 1.0f;
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0, "swizzled tiles need 1 KB alignment");
static_assert(kOffRaw % 16 == 0 && kHeadBytes % 16 == 0, "bulk copy alignment");
static_assert(kOffVs - kOffVc == kOffKs - kOffKc, "K and V halves share one layout");

constexpr int kSmemOptin = 232448;  // largest dynamic shared memory of one CTA (227 KB)
constexpr int kQslShared = (kSmemOptin - 1024 - kOffQsl) / 4;  // q_start_loc entries that fit beside the rings
static_assert(kQslShared >= 2, "shared memory");
bool qsl_fits(int n_seqs) { return n_seqs + 1 <= kQslShared; }
size_t attn_smem_bytes(int n_seqs) { return 1024 + kOffQsl + (qsl_fits(n_seqs) ? 4 * (size_t)(n_seqs + 1) : 0); }

// One item record (256 bytes of shared memory).
struct ItemRec {
  int n_pg;                // pages of the item after dropping invalid entries
  int j, kvh, split;
  int phys[kSelStride];    // physical page of each
  int valid[kSelStride];   // tokens of the page visible to j (128 except the recent block)
};
static_assert(sizeof(ItemRec) <= 256, "record slot");

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
  int n_items;       // T * 4 * n_splits
  float scale_log2;  // softmax_scale / s_enc_k * log2(e)
  float out_scale;   // 1 / s_enc_v (O and L both carry the factor 256 of P)
  float* o_part;     // [T][S][16][128]
  float* lse_part;   // [T][S][16]
  int* status;
  unsigned long long wait_ns;  // limit of one bounded wait
  int qsl_shared;              // q_start_loc copied to shared memory (else read from global)
  int skip_first_copy;         // test hook: the producer leaves out page 0's copy (its waits run out)
};

// 16 registers per thread -> 32 TMEM lanes x 16 columns (thread = lane).
__device__ __forceinline__ void tmem_st16(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x16.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16};"
      ::"r"(taddr), "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]),
      "r"(r[8]), "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15])
      : "memory");
}

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

// Every lane of the warp waits; the result is the same for all of them.
__device__ __forceinline__ bool warp_wait(uint32_t bar, uint32_t parity, const WaitCtl& w) {
  return __all_sync(0xffffffffu, mbar_wait(bar, parity, w));
}

// One 32-channel code chunk of a token: 16 code bytes at `codes` and the two
// group scales at sc[0] and sc[kPageTokens] -> 32 FP8 bytes in o[0..7].
__device__ __forceinline__ void convert_chunk(const uint8_t* codes, const uint8_t* sc, const uint2* tab,
                                              uint32_t* o) {
  const uint4 w = *reinterpret_cast<const uint4*>(codes);
  const uint2 t0 = tab[sc[0]];
  const uint2 t1 = tab[sc[kPageTokens]];
  const uint2 a = dequant8(w.x, t0), b = dequant8(w.y, t0);
  const uint2 d = dequant8(w.z, t1), e = dequant8(w.w, t1);
  o[0] = a.x; o[1] = a.y; o[2] = b.x; o[3] = b.y;
  o[4] = d.x; o[5] = d.y; o[6] = e.x; o[7] = e.y;
}

__global__ void __launch_bounds__(kThreads, 1) sparse_attn_tc_kernel(AttnParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  auto bar = [&](int i) { return sbase + kOffBars + 8 * i; };
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  const WaitCtl wc{s_abort, p.wait_ns};
  int* s_issued = reinterpret_cast<int*>(smem + kOffMisc + 8);
  uint2* s_tab = reinterpret_cast<uint2*>(smem + kOffTab);
  int* s_qsl = reinterpret_cast<int*>(smem + kOffQsl);
  auto rec = [&](int slot) { return reinterpret_cast<ItemRec*>(smem + kOffRec + 256 * slot); };

  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int G = gridDim.x;
  // items of this CTA: blockIdx.x + k * G for k < n_mine
  const int n_mine = p.n_items > (int)blockIdx.x ? (p.n_items - 1 - (int)blockIdx.x) / G + 1 : 0;

  // ---- prologue ------------------------------------------------------------------
  build_dequant_table(s_tab, tid, kThreads);
  if (tid == 0) {
    for (int i = 0; i < kStages; ++i) {
      mbar_init(bar(kRawFull + i), 1);
      mbar_init(bar(kRawEmpty + i), 4);  // the 4 warps of the converting group
    }
    for (int i = 0; i < kSlots; ++i) {
      mbar_init(bar(kK8Full + i), 4);
      mbar_init(bar(kK8Empty + i), 1);
      mbar_init(bar(kV8Full + i), 4);
      mbar_init(bar(kPFull + i), 4);
      mbar_init(bar(kPVDone + i), 1);
    }
    for (int i = 0; i < 2; ++i) {
      mbar_init(bar(kSFull + i), 1);
      mbar_init(bar(kSEmpty + i), 4);
      mbar_init(bar(kOFree + i), 4);       // set 0 has read both O buffers of this parity
      mbar_init(bar(kMergeFull + i), 4);   // set 1's (m, L) written
      mbar_init(bar(kMergeEmpty + i), 4);  // set 0 has read them
    }
    for (int i = 0; i < kRecs; ++i) {
      mbar_init(bar(kRecFull + i), 1);
      mbar_init(bar(kRecEmpty + i), kRecEmptyCount);
    }
    mbar_init(bar(kDone), 2 * kSets);
    *s_abort = 0;
    *s_issued = 0;
    fence_barrier_init();
  }
  // zero the Q tiles and the P tiles (rows that stay zero pad N to 16)
  for (int i = tid; i < (kRecs + kSlots) * 2048 / 16; i += kThreads)
    reinterpret_cast<uint4*>(smem + kOffQ)[i] = make_uint4(0, 0, 0, 0);
  // q_start_loc does not come from the previous kernel
  if (p.qsl_shared)
    for (int i = tid; i <= p.n_seqs; i += kThreads) s_qsl[i] = p.q_start_loc[i];
  if (warp == 2) tmem_alloc(smem_u32(s_tmem), kTmemCols);
  fence_proxy_async_smem();
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;
  pdl_wait();  // the selection comes from the indexer kernel
  pdl_trigger();

  if (warp == 0) {
    // ---------------- scheduler and TMA producer ---------------------------------------------
    // per item: the record (all lanes), then lane 0 streams the item's pages
    const int* qsl = p.qsl_shared ? s_qsl : p.q_start_loc;
    int e = 0;
    bool ok = true;
    for (int k = 0; ok && k < n_mine; ++k) {
      const int slot = k % kRecs;
      if (!warp_wait(bar(kRecEmpty + slot), ((k / kRecs) & 1) ^ 1, wc)) break;
      const int item = blockIdx.x + k * G;
      const int split = item % p.n_splits, kvh = (item / p.n_splits) % kKvHeads;
      const int j = item / (p.n_splits * kKvHeads);
      // sequence b of token j: the last b with q_start_loc[b] <= j.  32-ary
      // search, each round one sample per lane over the remaining range; a
      // malformed q_start_loc still gives an index in range, rejected below
      int lo = 0, span = p.n_seqs;
      while (span > 1) {
        const int step = (span + 31) >> 5, idx = lo + lane * step;
        const bool le = idx < lo + span && qsl[idx] <= j;
        const int cnt = max(__popc(__ballot_sync(0xffffffffu, le)), 1);
        const int nlo = lo + (cnt - 1) * step;
        span = min(step, lo + span - nlo);
        lo = nlo;
      }
      const int b = p.n_seqs > 0 ? lo : -1;
      // first round of loads, all independent: sequence length, selection, query rows
      const int seq_len = b >= 0 ? p.seq_lens[b] : 0;
      const int nsel_raw = p.n_sel[j];
      const int e_sel = split + lane * p.n_splits;
      const int blk_raw = lane < kSelStride && e_sel < kSelStride ? p.sel[(size_t)j * kSelStride + e_sel] : -1;
      const uint4 qv = *reinterpret_cast<const uint4*>(
          p.q + ((size_t)j * kQHeads + kvh * kGqa + (lane >> 3)) * kHeadDim + 16 * (lane & 7));
      const int q0 = b >= 0 ? qsl[b] : 0, n_q = b >= 0 ? qsl[b + 1] - q0 : 0;
      const bool seq_ok = b >= 0 && q0 <= j && j < q0 + n_q && q0 >= 0 && q0 + n_q <= p.n_q_total &&
                          seq_len >= n_q && seq_len <= p.max_pages * kPageTokens;
      const int pos = seq_len - n_q + (j - q0);
      const int r_blk = seq_ok ? pos / kPageTokens : -1;
      const int nsel = seq_ok ? min(nsel_raw, kSelStride) : 0;
      int phys = -1;
      if (lane < kSelStride && e_sel < nsel) {
        if (blk_raw < 0 || blk_raw > r_blk) {
          set_status(p.status, MSA_STATUS_BAD_SELECTION);
        } else {
          phys = p.block_table[(size_t)b * p.max_pages + blk_raw];  // second round
          if (phys < 0 || phys >= p.n_pages) {
            set_status(p.status, MSA_STATUS_BAD_PAGE);
            phys = -1;
          }
        }
      }
      if (lane == 0 && !seq_ok) set_status(p.status, MSA_STATUS_BAD_SEQ);
      // compact the valid entries (order kept)
      const unsigned okmask = __ballot_sync(0xffffffffu, phys >= 0);
      ItemRec* r = rec(slot);
      if (phys >= 0) {
        const int at = __popc(okmask & ((1u << lane) - 1));
        r->phys[at] = phys;
        r->valid[at] = blk_raw == r_blk ? (pos % kPageTokens) + 1 : kPageTokens;
      }
      const int n = __popc(okmask);
      if (lane == 0) {
        r->n_pg = n;
        r->j = j;
        r->kvh = kvh;
        r->split = split;
      }
      // query rows 0-3 (heads 4 kvh .. 4 kvh + 3), 128-byte swizzled K-major
      {
        const int row = lane >> 3, c = lane & 7;
        *reinterpret_cast<uint4*>(smem + kOffQ + slot * 2048 + row * 128 + ((c ^ row) << 4)) = qv;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) {
        mbar_arrive(bar(kRecFull + slot));
        // one copy per page: the KV head's K and V codes and scales
        const uint8_t* head = p.kv_pool + (size_t)kvh * kHeadBytes;
        for (int i = 0; i < n; ++i, ++e) {
          const int st = e % kStages;
          if (!mbar_wait(bar(kRawEmpty + st), ((e / kStages) & 1) ^ 1, wc)) { ok = false; break; }
          if (e == 0 && p.skip_first_copy) continue;  // nothing will complete stage 0
          mbar_arrive_expect_tx(bar(kRawFull + st), kHeadBytes);
          bulk_g2s(sbase + kOffRaw + st * kHeadBytes, head + (size_t)r->phys[i] * kKvPageBytes, kHeadBytes,
                   bar(kRawFull + st));
          *s_issued = e + 1;
        }
        if (ok) mbar_arrive(bar(kRecEmpty + slot));
      }
      ok = __shfl_sync(0xffffffffu, ok, 0);
    }
  } else if (warp < 1 + kSets) {
    // ---------------- QK issuers: warp 1 + s takes the pages of set s (e % 2 == s) ---------------
    if (lane == 0) {
      const int s = warp - 1;
      const uint32_t idesc = umma_idesc_e4m3(128, 16);
      int e0 = 0;
      bool ok = true;
      for (int k = 0; ok && k < n_mine; ++k) {
        const int slot = k % kRecs;
        if (!mbar_wait(bar(kRecFull + slot), (k / kRecs) & 1, wc)) break;
        const int n = rec(slot)->n_pg;
        const uint64_t bdesc = umma_desc_sw128(sbase + kOffQ + slot * 2048);
        bool issued = false;
        for (int i = (s - e0) & 1; i < n; i += kSets) {
          const int e = e0 + i, ks = e % kSlots, kph = (e / kSlots) & 1, sph = (e >> 1) & 1;
          if (!mbar_wait(bar(kK8Full + ks), kph, wc) || !mbar_wait(bar(kSEmpty + s), sph ^ 1, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // K = 32 per MMA: 8 TMEM columns of A, +32 B (+2) of B
            umma_e4m3_ts(tmem + kTmS + 16 * s, tmem + 32 * ks + 8 * kk, bdesc + 2 * kk, idesc, kk > 0);
          umma_commit(bar(kK8Empty + ks));
          umma_commit(bar(kSFull + s));
          issued = true;
        }
        if (!ok) break;
        // the record's Q tile is free once these MMAs are done
        if (issued) umma_commit(bar(kRecEmpty + slot));
        else mbar_arrive(bar(kRecEmpty + slot));
        e0 += n;
      }
      umma_commit(bar(kDone));  // arrives when every MMA of this thread is done
    }
    __syncwarp();
  } else if (warp < 1 + 2 * kSets) {
    // ---------------- PV issuers: warp 1 + kSets + s takes the pages of set s -------------------
    if (lane == 0) {
      const int s = warp - 1 - kSets;
      const uint32_t idesc = umma_idesc_e4m3_amn_bmn(128, 16);
      int e0 = 0, ni = 0;  // ni: items with pages so far (O buffer parity ni & 1)
      bool ok = true;
      for (int k = 0; ok && k < n_mine; ++k) {
        const int slot = k % kRecs;
        if (!mbar_wait(bar(kRecFull + slot), (k / kRecs) & 1, wc)) break;
        const int n = rec(slot)->n_pg;
        mbar_arrive(bar(kRecEmpty + slot));  // nothing else of the record is needed
        const int ob = ni & 1, i0 = (s - e0) & 1;
        // O buffers of parity ob are free once set 0 has read item ni - 2's output from them
        if (n > i0 && ni >= 2 && !mbar_wait(bar(kOFree + ob), ((ni >> 1) - 1) & 1, wc)) break;
        for (int i = i0; i < n; i += kSets) {
          const int e = e0 + i, v = e % kSlots, vph = (e / kSlots) & 1;
          if (!mbar_wait(bar(kV8Full + v), vph, wc) || !mbar_wait(bar(kPFull + v), vph, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk) {
            // A: V tile read MN-major; 32 tokens (4 swizzle atoms of 8 rows) per MMA.
            // B: P tile, MN-major without swizzle: token t's 16 bytes at 16 t, so
            // a core matrix (8 tokens x 16 bytes) is 128 contiguous bytes and the
            // 32 tokens of one MMA are 512 bytes
            const uint64_t adesc =
                umma_desc_sw128_lbo_sbo(sbase + kOffV8 + v * kTileBytes + kk * 4096, 1024, 1024);
            const uint64_t bdesc = umma_desc_noswz_lbo_sbo(sbase + kOffP + v * 2048 + kk * 512, 128, 128);
            // set s's accumulator; its first page of the item (i < 2) overwrites it
            umma_e4m3(tmem + kTmO + 16 * (2 * ob + s), adesc, bdesc, idesc, (i >= 2 || kk > 0) ? 1u : 0u);
          }
          // page e's V tile and P tile are free (and O holds page e) once this is done
          umma_commit(bar(kPVDone + v));
        }
        if (n > 0) ++ni;
        e0 += n;
      }
      umma_commit(bar(kDone));
    }
    __syncwarp();
  } else if (warp >= kWarpConv0) {
    // ---------------- conversion: group g converts pages e % kGroups == g ------------------
    const int g = (warp - kWarpConv0) >> 2, quad = warp & 3;
    const int tok = 32 * quad + lane;  // K rows land in TMEM lanes 32 quad .. (warp % 4 rule)
    // Per-thread offsets, fixed for the whole kernel: code chunk c of token tok
    // sits at position c ^ ((tok >> 1) & 3) of its 64-byte row (8 consecutive
    // tokens hit 8 bank groups), its two group scales at [2c][tok] and
    // [2c + 1][tok] after the codes; in the V tile 16-byte chunk j of row tok
    // sits at position j ^ (tok & 7).
    uint32_t code_off[4], sc_off[4], v_off[4][2];
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      code_off[c] = tok * 64 + 16 * code_chunk_pos(c, tok);
      sc_off[c] = (kOffKs - kOffKc) + 2 * c * kPageTokens + tok;
      v_off[c][0] = tok * 128 + (((2 * c) ^ (tok & 7)) << 4);
      v_off[c][1] = tok * 128 + (((2 * c + 1) ^ (tok & 7)) << 4);
    }
    const uint32_t trow = tmem + ((uint32_t)(32 * quad) << 16);
    int e = 0;
    bool ok = true;
    for (int k = 0; ok && k < n_mine; ++k) {
      const int slot = k % kRecs;
      if (!warp_wait(bar(kRecFull + slot), (k / kRecs) & 1, wc)) break;
      const ItemRec* r = rec(slot);
      const int n = r->n_pg;
      for (int i = 0; i < n; ++i, ++e) {
        if (e % kGroups != g) continue;
        const int st = e % kStages, sl = e % kSlots;
        const uint32_t sph = (e / kSlots) & 1;
        // the raw page, and K8 slot sl (free once QK of page e - kSlots is done)
        if (!warp_wait(bar(kRawFull + st), (e / kStages) & 1, wc) || !warp_wait(bar(kK8Empty + sl), sph ^ 1, wc)) {
          ok = false;
          break;
        }
        const uint8_t* raw = smem + kOffRaw + st * kHeadBytes;
        // K: row tok of A in TMEM, columns 32 sl + 8c .. + 7 = channels 32c .. 32c + 31
        // (rows past the query position stay as converted: the softmax masks them)
#pragma unroll
        for (int hc = 0; hc < 2; ++hc) {
          uint32_t o[16];
          convert_chunk(raw + kOffKc + code_off[2 * hc], raw + kOffKc + sc_off[2 * hc], s_tab, o);
          convert_chunk(raw + kOffKc + code_off[2 * hc + 1], raw + kOffKc + sc_off[2 * hc + 1], s_tab, o + 8);
          tmem_st16(trow + 32 * sl + 16 * hc, o);
        }
        tmem_wait_st();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kK8Full + sl));
        // V tile sl is free once PV of page e - kSlots is done
        if (e >= kSlots && !warp_wait(bar(kPVDone + sl), sph ^ 1, wc)) {
          ok = false;
          break;
        }
        // tokens after the query position (only in the recent block) become zeros
        const int valid = r->valid[i];
        const bool full = valid >= 32 * quad + 32;  // warp-uniform
        const bool live = tok < valid;
        uint8_t* dst = smem + kOffV8 + sl * kTileBytes;
#pragma unroll
        for (int c = 0; c < 4; ++c) {
          uint32_t oc[8];
          convert_chunk(raw + kOffVc + code_off[c], raw + kOffVc + sc_off[c], s_tab, oc);
          if (!full) {
#pragma unroll
            for (int x = 0; x < 8; ++x) oc[x] = live ? oc[x] : 0u;
          }
          *reinterpret_cast<uint4*>(dst + v_off[c][0]) = make_uint4(oc[0], oc[1], oc[2], oc[3]);
          *reinterpret_cast<uint4*>(dst + v_off[c][1]) = make_uint4(oc[4], oc[5], oc[6], oc[7]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(bar(kV8Full + sl));
          mbar_arrive(bar(kRawEmpty + st));
        }
      }
      if (ok && lane == 0) mbar_arrive(bar(kRecEmpty + slot));
    }
  } else if (warp >= kWarpSmax0) {
    // ---------------- softmax: set s = warps 5 + 4 s .. 8 + 4 s --------------------------------
    // set s takes the pages with e % 2 == s (S slot s); warp w reads TMEM lanes
    // 32 (w % 4) ..: row = token of S, channel of O
    const int set = (warp - kWarpSmax0) >> 2, quad = warp & 3, row = 32 * quad + lane;
    const uint32_t trow = tmem + ((uint32_t)(32 * quad) << 16);
    const int nb = 1 + set;  // named barrier of the set's four warps
    float* red = reinterpret_cast<float*>(smem + kOffRed) + 16 * set;    // [4 warps][4 heads]
    float* redl = reinterpret_cast<float*>(smem + kOffRedL) + 16 * set;  // [4 warps][4 heads]
    int e0 = 0, ni = 0;  // the item's first page; items with pages so far
    bool ok = true;
    for (int k = 0; ok && k < n_mine; ++k) {
      const int slot = k % kRecs;
      if (named_barrier_or(nb, 128, !warp_wait(bar(kRecFull + slot), (k / kRecs) & 1, wc))) break;
      const ItemRec* r = rec(slot);
      const int n = r->n_pg;
      const int ob = ni & 1;
      const uint32_t t_o = trow + kTmO + 16 * (2 * ob + set);  // this set's O accumulator
      const int i0 = (set - e0) & 1;  // the set's first page of the item
      float m_ref[4], l_run[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        m_ref[h] = -INFINITY;
        l_run[h] = 0.f;
      }
      for (int i = i0; i < n; i += kSets) {
        const int e = e0 + i;
        bool good = warp_wait(bar(kSFull + set), (e >> 1) & 1, wc);
        float sv[4] = {0.f, 0.f, 0.f, 0.f};
        if (good) {
          tc_fence_after();
          tmem_ld4(trow + kTmS + 16 * set, sv);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kSEmpty + set));
        }
        const bool live = row < r->valid[i];
        float x[4];
        bool over = false;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          x[h] = live ? sv[h] * p.scale_log2 : -INFINITY;
          over = over || x[h] > m_ref[h] + kGrowth;
        }
        bool step_ok = true;
        // a row above the reference (always on the set's first page), or an abort
        if (named_barrier_or(nb, 128, over || !good || !ok)) {
          if (named_barrier_or(nb, 128, !good || !ok)) {
            ok = false;
            break;
          }
          // exact page max per head over the 128 rows
          float wm[4];
#pragma unroll
          for (int h = 0; h < 4; ++h) wm[h] = warp_max_f32(x[h]);
          if (lane == 0) reinterpret_cast<float4*>(red)[quad] = make_float4(wm[0], wm[1], wm[2], wm[3]);
          named_barrier_sync(nb, 128);
          const float4 r0 = reinterpret_cast<const float4*>(red)[0], r1 = reinterpret_cast<const float4*>(red)[1];
          const float4 r2 = reinterpret_cast<const float4*>(red)[2], r3 = reinterpret_cast<const float4*>(red)[3];
          const float mps[4] = {fmaxf(fmaxf(r0.x, r1.x), fmaxf(r2.x, r3.x)), fmaxf(fmaxf(r0.y, r1.y), fmaxf(r2.y, r3.y)),
                                fmaxf(fmaxf(r0.z, r1.z), fmaxf(r2.z, r3.z)), fmaxf(fmaxf(r0.w, r1.w), fmaxf(r2.w, r3.w))};
          float f[4];
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            // only heads whose page max outgrew the reference move it
            const float m_new = mps[h] > m_ref[h] + kGrowth ? mps[h] + kHeadroom : m_ref[h];
            f[h] = m_ref[h] == -INFINITY ? 0.f : fast_exp2(m_ref[h] - m_new);
            l_run[h] *= f[h];
            m_ref[h] = m_new;
          }
          if (i >= kSets) {
            // O holds the set's earlier pages of the item relative to the old
            // reference: once their PVs are done (PV of page e - 2), rescale it
            const int pv = (e - kSets) % kSlots;
            step_ok = warp_wait(bar(kPVDone + pv), ((e - kSets) / kSlots) & 1, wc);
            if (step_ok) {
              tc_fence_after();
              float ov[8];
              tmem_ld8(t_o, ov);  // thread = channel: hi terms, then remainders
              uint32_t ou[8];
#pragma unroll
              for (int h = 0; h < 4; ++h) {
                ou[h] = __float_as_uint(ov[h] * f[h]);
                ou[4 + h] = __float_as_uint(ov[4 + h] * f[h]);
              }
              tmem_st8(t_o, ou);
              tmem_wait_st();
              tc_fence_before();
            }
          }
        }
        float v[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          // 256 p relative to the reference (<= 256 * 2^kGrowth < 448)
          v[h] = x[h] == -INFINITY ? 0.f : fast_exp2(x[h] - m_ref[h] + 8.f);
          l_run[h] += v[h];
        }
        // 256 p as two E4M3 terms: hi = E4M3(256 p), lo = E4M3(f16(256 p) - hi)
        // (the f16 difference is exact: hi is within a factor of two of 256 p)
        const uint32_t hi01 = cvt_e4m3x2_f32(v[1], v[0]), hi23 = cvt_e4m3x2_f32(v[3], v[2]);
        const uint32_t lo01 = cvt_e4m3x2_f16x2(hsub2_u32(cvt_f16x2_f32(v[1], v[0]), cvt_f16x2_e4m3x2(hi01)));
        const uint32_t lo23 = cvt_e4m3x2_f16x2(hsub2_u32(cvt_f16x2_f32(v[3], v[2]), cvt_f16x2_e4m3x2(hi23)));
        // P tile row = token: bytes 0-3 hi terms of heads 0-3, 4-7 the remainders
        // (bytes 8-15 stay zero: they pad N to 16); tile e % kSlots is free once
        // PV of page e - kSlots (this set's) is done
        const int po = e % kSlots;
        if (step_ok && e >= kSlots) step_ok = warp_wait(bar(kPVDone + po), ((e / kSlots) & 1) ^ 1, wc);
        if (step_ok) {
          *reinterpret_cast<uint2*>(smem + kOffP + po * 2048 + 16 * row) =
              make_uint2(prmt(hi01, hi23, 0x5410u), prmt(lo01, lo23, 0x5410u));
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kPFull + po));
        }
        ok = ok && step_ok;  // a failure here ends the loop at the next barrier
      }
      const bool aborted = named_barrier_or(nb, 128, !ok || *s_abort != 0);
      // ---- this set's sum of p over the 128 rows, per head ----------------------------------------
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        float l = l_run[h];
#pragma unroll
        for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) redl[quad * 4 + h] = l;
      }
      named_barrier_sync(nb, 128);
      float L[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) L[h] = aborted ? 0.f : redl[h] + redl[4 + h] + redl[8 + h] + redl[12 + h];
      // ---- set 1 hands (m, L) over; set 0 merges and writes ---------------------------------------
      float* mg = reinterpret_cast<float*>(smem + kOffMerge) + 8 * (k & 1);
      const uint32_t mph = (k >> 1) & 1;
      bool step_ok = !aborted;
      // the item's last page of each set (page e0 + i with (e0 + i) % 2 == set)
      const int el = e0 + n - 1, e_last = (el & 1) == set ? el : el - 1;
      const bool has_pages = e_last >= e0;
      if (set == 1) {
        // this set's PVs are issued by their own thread, in order: once the last
        // one is done, set 1's accumulator is final (every earlier PV of this
        // set was seen complete by the P tile waits, so the parity wait sees its
        // own phase); the hand-off below tells set 0
        if (step_ok && has_pages)
          step_ok = warp_wait(bar(kPVDone + e_last % kSlots), (e_last / kSlots) & 1, wc);
        tc_fence_before();
        if (step_ok) step_ok = warp_wait(bar(kMergeEmpty + (k & 1)), mph ^ 1, wc);
        if (step_ok) {
          if (row == 0) {
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              mg[h] = m_ref[h];
              mg[4 + h] = L[h];
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kMergeFull + (k & 1)));
        }
      } else {
        // both accumulators, once the item's last PV is done (thread = channel)
        float o0[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f}, o1[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
        const bool has0 = has_pages, has1 = n > ((1 - e0) & 1);  // each set had a page of the item
        // set 0's own accumulator once its last PV is done (its PVs come from one
        // thread, in order); set 1's once set 1 has handed over, which it does
        // only after its own last PV
        if (step_ok && has0) step_ok = warp_wait(bar(kPVDone + e_last % kSlots), (e_last / kSlots) & 1, wc);
        if (step_ok) step_ok = warp_wait(bar(kMergeFull + (k & 1)), mph, wc);
        if (step_ok && n > 0) {
          tc_fence_after();
          if (has0) tmem_ld8(trow + kTmO + 16 * (2 * ob), o0);
          if (has1) tmem_ld8(trow + kTmO + 16 * (2 * ob + 1), o1);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kOFree + ob));  // PVs of item ni + 2 may overwrite them
        }
        const size_t row0 = ((size_t)r->j * p.n_splits + r->split) * kQHeads + r->kvh * kGqa;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          const float m1 = step_ok ? mg[h] : -INFINITY, L1 = step_ok ? mg[4 + h] : 0.f;
          const float m = fmaxf(m_ref[h], m1);
          const float w0 = (m_ref[h] == -INFINITY || L[h] == 0.f) ? 0.f : fast_exp2(m_ref[h] - m);
          const float w1 = (m1 == -INFINITY || L1 == 0.f) ? 0.f : fast_exp2(m1 - m);
          const float Lm = L[h] * w0 + L1 * w1;
          // a set without pages has weight 0 and an unread accumulator (stays 0)
          const float om = (w0 > 0.f ? (o0[h] + o0[4 + h]) * w0 : 0.f) + (w1 > 0.f ? (o1[h] + o1[4 + h]) * w1 : 0.f);
          const bool nonempty = step_ok && n > 0 && Lm > 0.f;
          p.o_part[(row0 + h) * kHeadDim + row] = nonempty ? om / Lm * p.out_scale : 0.f;
          if (row == 0) p.lse_part[row0 + h] = nonempty ? (m + log2f(Lm) - 8.f) * kLn2 : -INFINITY;
        }
        __syncwarp();
        if (lane == 0 && step_ok) mbar_arrive(bar(kMergeEmpty + (k & 1)));
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kRecEmpty + slot));
      if (n > 0) ++ni;
      e0 += n;
      ok = step_ok;
    }
  }

  // ---- teardown -------------------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {
    // every tcgen05.mma is done (both issuers committed after their last one)
    mbar_wait_drain(bar(kDone), 0, p.wait_ns);
    if (*s_abort) {
      set_status(p.status, MSA_STATUS_TIMEOUT);
      // bounded drain of the copies that may still be landing: the last
      // kStages issued (every earlier one was consumed before its stage was
      // refilled)
      const int ni = *s_issued;
      for (int e = max(0, ni - kStages); e < ni; ++e)
        mbar_wait_drain(bar(kRawFull + e % kStages), (e / kStages) & 1, p.wait_ns);
    }
  }
  __syncthreads();
  if (warp == 2) {
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
  static DeviceSetup setup;
  int dev = 0, n_sm = 0;
  cudaError_t e = setup.get(&dev, &n_sm, [](int) {
    return cudaFuncSetAttribute(sparse_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize, kSmemOptin);
  });
  if (e != cudaSuccess) return e;
  const int n_items = n_q_total * kKvHeads * n_splits;
  AttnParams ap{static_cast<const uint8_t*>(c->kv_pool), c->n_pages, q, sel, n_sel, block_table,
                max_pages, seq_lens, q_start_loc, n_seqs, n_q_total, n_splits, n_items,
                softmax_scale / c->s_enc_k * kLog2e, 1.0f / c->s_enc_v, o_part,
                lse_part, c->status, launch_settings().wait_ns, qsl_fits(n_seqs) ? 1 : 0,
                (launch_settings().inject & kInjectAttentionTimeout) ? 1 : 0};
  const int grid = n_items < n_sm ? n_items : n_sm;
  return launch_pdl(sparse_attn_tc_kernel, dim3(grid), dim3(kThreads), attn_smem_bytes(n_seqs), stream, ap);
}

}  // namespace msa
