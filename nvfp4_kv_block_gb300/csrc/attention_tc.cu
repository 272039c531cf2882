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
//   warp 0       scheduler: per item, the sequence of j (shared-memory copy of
//                q_start_loc), the selected blocks, their physical pages and the
//                tokens visible in each, and the 4 query rows as a swizzled
//                tile, into a 4-deep ring of item records;
//   warp 1       TMA producer: per page two 9 KB cp.async.bulk copies, the K
//                half (codes + scales) and the V half, into two 6-stage rings;
//   warp 2       QK issuer: S = K8 Q^T (kind::f8f6f4, M = 128 tokens, N = 16: the
//                4 query heads, zero padded, K = 128, A from tensor memory);
//   warp 3       PV issuer: O^T = V8^T P (A = the V tile read MN-major, no
//                transpose, B = P), one of 4 TMEM O buffers per page; its one
//                commit per page completes the page's O barrier, which also
//                frees the page's V tile and P tile;
//   warps 4 ..   softmax, kSets sets of 4 warps; set s takes the pages with
//                e % kSets == s and keeps its own running (m, l, o): thread = token
//                row of S: page max per head, P = exp2 relative to the page max,
//                scaled by 2^8 and split into two E4M3 terms (value + rounding
//                remainder) as the B operand of PV; thread = channel: the page's
//                O folded into the running state.  At the item's end sets
//                1 .. kSets - 1 hand their states to set 0, which merges them and
//                writes the normalised partial (O, LSE).  The LSE merge kernel
//                combines the splits;
//   next 4 x kConvSets warps: K conversion, thread = (token, part of the row):
//                NVFP4 -> FP8 through a 256-entry shared table of scaled E4M3
//                values and byte permutes, written with tcgen05.st straight into
//                tensor memory (the A operand);
//   last 4 x kConvSets warps: V conversion, the same into a 128-byte-swizzled
//                shared-memory tile (3 tiles).
#include "common.cuh"

namespace msa {
namespace {

constexpr int kConvSets = 2;   // warps per token row of K (and of V): each converts 4 / kConvSets chunks
constexpr int kSets = 2;       // softmax sets of 4 warps; set s takes the pages with e % kSets == s
constexpr int kWarpConv0 = 4 + 4 * kSets;  // first conversion warp
constexpr int kThreads = 32 * (kWarpConv0 + 8 * kConvSets);
constexpr int kStages = 6;     // raw K and raw V ring depth
constexpr int kRecs = 4;       // item records in flight
constexpr int kK8Slots = 4;    // K8 buffers in tensor memory (a power of two: slot = e & 3)
constexpr int kV8Tiles = 4;    // V8 tiles in shared memory (a power of two)
constexpr int kPO = 4;         // P tiles and O buffers
// a V tile is reused only after the PV of page e - kV8Tiles completes the O
// barrier of that page; with kV8Tiles <= kPO no later phase of that barrier can
// complete before the V warps have seen it (that would need page e's V tile)
static_assert(kV8Tiles <= kPO, "V tile reuse waits on the O barrier of page e - kV8Tiles");
static_assert(kV8Tiles == kPO, "a V tile and the O buffer of its page share the slot index");
constexpr int kHalfBytes = kHeadBytes / 2;  // 9,216: codes + scales of K (or V)
constexpr int kTileBytes = 16384;           // [128 rows][128 B], swizzled
constexpr int kOffV8 = 0;                                   // kV8Tiles V8 tiles
constexpr int kOffQ = kV8Tiles * kTileBytes;                // kRecs x [16 rows][128 B]
constexpr int kOffP = kOffQ + kRecs * 2048;                 // kPO x [128 tokens][16 B]
constexpr int kOffKRaw = kOffP + kPO * 2048;                // kStages x 9,216
constexpr int kOffVRaw = kOffKRaw + kStages * kHalfBytes;   // kStages x 9,216
constexpr int kOffTab = kOffVRaw + kStages * kHalfBytes;    // uint2 [256]
constexpr int kOffRec = kOffTab + 2048;                     // kRecs x 256 B
constexpr int kOffMerge = kOffRec + kRecs * 256;            // [kSets - 1][2] x (o [4][128], m [4], L [4]) floats
constexpr int kMergeBytes = (4 * 128 + 8) * 4;
constexpr int kMergeBufs = 2 * (kSets - 1);                 // per helper set, per item parity
constexpr int kOffBars = kOffMerge + kMergeBufs * kMergeBytes;
// barrier indices
constexpr int kKrFull = 0, kKrEmpty = kStages, kVrFull = 2 * kStages, kVrEmpty = 3 * kStages;
constexpr int kK8Full = 4 * kStages, kK8Empty = kK8Full + kK8Slots, kSFull = kK8Empty + kK8Slots,
              kSEmpty = kSFull + kSets, kV8Full = kSEmpty + kSets, kPFull = kV8Full + kV8Tiles,
              kOFull = kPFull + kPO,
              kOEmpty = kOFull + kPO, kRecFull = kOEmpty + kPO, kRecEmpty = kRecFull + kRecs,
              kMergeFull = kRecEmpty + kRecs, kMergeEmpty = kMergeFull + kMergeBufs,
              kDone = kMergeEmpty + kMergeBufs,
              kNumBars = kDone + 2;  // kDone: QK issuer, kDone + 1: PV issuer
constexpr int kOffMisc = kOffBars + ((kNumBars * 8 + 15) / 16) * 16;  // tmem, abort, issued K/V
constexpr int kOffRed = kOffMisc + 16;        // float [kSets][2][4 warps][4 heads] page maxima
constexpr int kOffRedL = kOffRed + 128 * kSets;  // float [kSets][4 warps][4 heads] row sums
constexpr int kOffQsl = kOffRedL + 64 * kSets;   // int [n_seqs + 1] copy of q_start_loc
constexpr uint32_t kTmS = 32 * kK8Slots;      // TMEM columns: K8 slot i at 32 i, S slot s at kTmS + 16 s,
constexpr uint32_t kTmO = kTmS + 16 * kSets;  // O buffers at kTmO + 16 i
constexpr uint32_t kTmemCols = 256;
static_assert(kTmO + 16 * kPO <= kTmemCols, "tensor memory columns");
constexpr int kRecEmptyCount = 1 + 8 * kConvSets + 1 + 1 + 4 * kSets;  // producer, K and V, QK, PV, softmax
static_assert(kPO > kSets, "a set writes P of page e before it folds page e - kSets");
constexpr float kLog2e = 1.4426950408889634f;
constexpr float kLn2 = 0.6931471805599453f;
static_assert(kOffQ % 1024 == 0 && kOffP % 1024 == 0, "swizzled tiles need 1 KB alignment");
static_assert(kOffKRaw % 16 == 0 && kOffVRaw % 16 == 0 && kHalfBytes % 16 == 0, "bulk copy alignment");
static_assert(kOffMerge % 16 == 0, "alignment");

size_t attn_smem_bytes(int n_seqs) { return 1024 + kOffQsl + 4 * (size_t)(n_seqs + 1); }

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
  int* s_issued_k = reinterpret_cast<int*>(smem + kOffMisc + 8);
  int* s_issued_v = reinterpret_cast<int*>(smem + kOffMisc + 12);
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
      mbar_init(bar(kKrFull + i), 1);
      mbar_init(bar(kKrEmpty + i), 4 * kConvSets);
      mbar_init(bar(kVrFull + i), 1);
      mbar_init(bar(kVrEmpty + i), 4 * kConvSets);
    }
    for (int i = 0; i < kK8Slots; ++i) {
      mbar_init(bar(kK8Full + i), 4 * kConvSets);
      mbar_init(bar(kK8Empty + i), 1);
    }
    for (int i = 0; i < kSets; ++i) {
      mbar_init(bar(kSFull + i), 1);
      mbar_init(bar(kSEmpty + i), 4);
    }
    for (int i = 0; i < kMergeBufs; ++i) {
      mbar_init(bar(kMergeFull + i), 4);
      mbar_init(bar(kMergeEmpty + i), 4);
    }
    for (int i = 0; i < kV8Tiles; ++i) mbar_init(bar(kV8Full + i), 4 * kConvSets);
    for (int i = 0; i < kPO; ++i) {
      mbar_init(bar(kPFull + i), 4);
      mbar_init(bar(kOFull + i), 1);
      mbar_init(bar(kOEmpty + i), 4);
    }
    for (int i = 0; i < kRecs; ++i) {
      mbar_init(bar(kRecFull + i), 1);
      mbar_init(bar(kRecEmpty + i), kRecEmptyCount);
    }
    mbar_init(bar(kDone), 1);
    mbar_init(bar(kDone + 1), 1);
    *s_abort = 0;
    *s_issued_k = 0;
    *s_issued_v = 0;
    fence_barrier_init();
  }
  // zero the Q tiles and the P tiles (rows that stay zero pad N to 16)
  for (int i = tid; i < (kRecs + kPO) * 2048 / 16; i += kThreads)
    reinterpret_cast<uint4*>(smem + kOffQ)[i] = make_uint4(0, 0, 0, 0);
  // q_start_loc does not come from the previous kernel
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
    // ---------------- scheduler: item records ------------------------------------------
    for (int k = 0; k < n_mine; ++k) {
      const int slot = k % kRecs;
      if (!warp_wait(bar(kRecEmpty + slot), ((k / kRecs) & 1) ^ 1, wc)) break;
      const int item = blockIdx.x + k * G;
      const int split = item % p.n_splits, kvh = (item / p.n_splits) % kKvHeads;
      const int j = item / (p.n_splits * kKvHeads);
      // sequence b of token j: the last b with q_start_loc[b] <= j (binary search)
      int lo = 0, hi = p.n_seqs - 1;
      while (lo < hi) {
        const int mid = (lo + hi + 1) >> 1;
        if (s_qsl[mid] <= j) lo = mid; else hi = mid - 1;
      }
      const int b = p.n_seqs > 0 ? lo : -1;
      // first round of loads, all independent: sequence length, selection, query rows
      const int seq_len = b >= 0 ? p.seq_lens[b] : 0;
      const int nsel_raw = p.n_sel[j];
      const int e_sel = split + lane * p.n_splits;
      const int blk_raw = lane < kSelStride && e_sel < kSelStride ? p.sel[(size_t)j * kSelStride + e_sel] : -1;
      const uint4 qv = *reinterpret_cast<const uint4*>(
          p.q + ((size_t)j * kQHeads + kvh * kGqa + (lane >> 3)) * kHeadDim + 16 * (lane & 7));
      const int q0 = b >= 0 ? s_qsl[b] : 0, n_q = b >= 0 ? s_qsl[b + 1] - q0 : 0;
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
      if (lane == 0) {
        r->n_pg = __popc(okmask);
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
      if (lane == 0) mbar_arrive(bar(kRecFull + slot));
    }
  } else if (warp == 1) {
    // ---------------- TMA producer: K and V halves of every page -------------------------
    if (lane == 0) {
      int e = 0, st = 0;
      uint32_t ph = 0;  // ring stage of page e and its phase parity
      bool ok = true;
      for (int k = 0; ok && k < n_mine; ++k) {
        const int slot = k % kRecs;
        if (!mbar_wait(bar(kRecFull + slot), (k / kRecs) & 1, wc)) break;
        const ItemRec* r = rec(slot);
        const int n = r->n_pg;
        const uint8_t* head = p.kv_pool + (size_t)r->kvh * kHeadBytes;
        for (int i = 0; i < n; ++i, ++e) {
          const uint8_t* src = head + (size_t)r->phys[i] * kKvPageBytes;
          if (!mbar_wait(bar(kKrEmpty + st), ph ^ 1, wc)) { ok = false; break; }
          mbar_arrive_expect_tx(bar(kKrFull + st), kHalfBytes);
          bulk_g2s(sbase + kOffKRaw + st * kHalfBytes, src, kHalfBytes, bar(kKrFull + st));
          *s_issued_k = e + 1;
          if (!mbar_wait(bar(kVrEmpty + st), ph ^ 1, wc)) { ok = false; break; }
          mbar_arrive_expect_tx(bar(kVrFull + st), kHalfBytes);
          bulk_g2s(sbase + kOffVRaw + st * kHalfBytes, src + kHalfBytes, kHalfBytes, bar(kVrFull + st));
          *s_issued_v = e + 1;
          if (++st == kStages) {
            st = 0;
            ph ^= 1;
          }
        }
        if (ok) mbar_arrive(bar(kRecEmpty + slot));
      }
    }
    __syncwarp();
  }
  else if (warp == 2) {
    // ---------------- QK issuer ---------------------------------------------------------------
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_e4m3(128, 16);
      int e = 0;
      bool ok = true;
      for (int k = 0; ok && k < n_mine; ++k) {
        const int slot = k % kRecs;
        if (!mbar_wait(bar(kRecFull + slot), (k / kRecs) & 1, wc)) break;
        const int n = rec(slot)->n_pg;
        const uint64_t bdesc = umma_desc_sw128(sbase + kOffQ + slot * 2048);
        for (int i = 0; i < n; ++i, ++e) {
          const unsigned ue = e;
          const int sl = ue % kSets, ph = (ue / kSets) & 1, ks = ue % kK8Slots, kph = (ue / kK8Slots) & 1;
          if (!mbar_wait(bar(kK8Full + ks), kph, wc) || !mbar_wait(bar(kSEmpty + sl), ph ^ 1, wc)) {
            ok = false;
            break;
          }
          tc_fence_after();
#pragma unroll
          for (int kk = 0; kk < 4; ++kk)  // K = 32 per MMA: 8 TMEM columns of A, +32 B (+2) of B
            umma_e4m3_ts(tmem + kTmS + 16 * sl, tmem + 32 * ks + 8 * kk, bdesc + 2 * kk, idesc, kk > 0);
          umma_commit(bar(kK8Empty + ks));
          umma_commit(bar(kSFull + sl));
        }
        if (!ok) break;
        // the record's Q tile is free once these MMAs are done
        if (n > 0) umma_commit(bar(kRecEmpty + slot));
        else mbar_arrive(bar(kRecEmpty + slot));
      }
      umma_commit(bar(kDone));  // arrives when every MMA of this thread is done
    }
    __syncwarp();
  } else if (warp == 3) {
    // ---------------- PV issuer ---------------------------------------------------------------
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_e4m3_amn_bmn(128, 16);
      int e = 0;
      bool ok = true;
      for (int k = 0; ok && k < n_mine; ++k) {
        const int slot = k % kRecs;
        if (!mbar_wait(bar(kRecFull + slot), (k / kRecs) & 1, wc)) break;
        const int n = rec(slot)->n_pg;
        mbar_arrive(bar(kRecEmpty + slot));  // nothing else of the record is needed
        for (int i = 0; i < n; ++i, ++e) {
          const unsigned ue = e;
          const int v = ue % kV8Tiles, vph = (ue / kV8Tiles) & 1, po = ue % kPO, pph = (ue / kPO) & 1;
          if (!mbar_wait(bar(kV8Full + v), vph, wc) || !mbar_wait(bar(kPFull + po), pph, wc) ||
              !mbar_wait(bar(kOEmpty + po), pph ^ 1, wc)) {
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
            const uint64_t bdesc = umma_desc_noswz_lbo_sbo(sbase + kOffP + po * 2048 + kk * 512, 128, 128);
            umma_e4m3(tmem + kTmO + 16 * po, adesc, bdesc, idesc, kk > 0);
          }
          // one commit: page e's O is ready, and its V tile and P tile are free
          umma_commit(bar(kOFull + po));
        }
      }
      umma_commit(bar(kDone + 1));
    }
    __syncwarp();
  } else if (warp >= kWarpConv0) {
    // ---------------- conversion: K (warps 12 ..) or V (the next 4 kConvSets) --------
    // thread = token; the kConvSets warps of a token row take its 16-byte code
    // chunks c = cs * kCh .. cs * kCh + kCh - 1
    const bool is_k = warp < kWarpConv0 + 4 * kConvSets;
    constexpr int kCh = 4 / kConvSets;
    const int cs = ((warp - kWarpConv0) >> 2) % kConvSets;
    // K warps write TMEM lanes 32 (warp % 4) ..; V warps any order
    const int tok = 32 * (warp & 3) + lane;
    const int full0 = is_k ? kKrFull : kVrFull, empty0 = is_k ? kKrEmpty : kVrEmpty;
    const uint32_t raw0 = is_k ? kOffKRaw : kOffVRaw;
    // Per-thread offsets of this thread's chunks, fixed for the whole kernel:
    // code chunk c of token tok sits at position c ^ ((tok >> 1) & 3) of its
    // 64-byte row (8 consecutive tokens hit 8 bank groups), its two group
    // scales at [2c][tok] and [2c + 1][tok] after the codes; in the V tile
    // 16-byte chunk j of row tok sits at position j ^ (tok & 7).
    uint32_t code_off[kCh], sc_off[kCh], v_off[kCh][2];
#pragma unroll
    for (int ci = 0; ci < kCh; ++ci) {
      const int c = cs * kCh + ci;
      code_off[ci] = tok * 64 + 16 * code_chunk_pos(c, tok);
      sc_off[ci] = kOffKs + 2 * c * kPageTokens + tok;
      v_off[ci][0] = tok * 128 + (((2 * c) ^ (tok & 7)) << 4);
      v_off[ci][1] = tok * 128 + (((2 * c + 1) ^ (tok & 7)) << 4);
    }
    int e = 0, st = 0;
    uint32_t rph = 0;  // raw ring stage of page e and its phase parity
    bool ok = true;
    for (int k = 0; ok && k < n_mine; ++k) {
      const int slot = k % kRecs;
      if (!warp_wait(bar(kRecFull + slot), (k / kRecs) & 1, wc)) break;
      const ItemRec* r = rec(slot);
      const int n = r->n_pg;
      for (int i = 0; i < n; ++i, ++e) {
        // output slot: the K8 buffer e % kK8Slots (freed by its previous QK) or
        // the V8 tile e % kV8Tiles (freed by the PV of page e - kV8Tiles, whose
        // commit completes the O barrier of that page: O buffer e % kPO, the
        // same index since kV8Tiles == kPO)
        const unsigned ue = e;
        const int os = is_k ? ue % kK8Slots : ue % kV8Tiles;
        const uint32_t oph = is_k ? (ue / kK8Slots) & 1 : (ue / kV8Tiles) & 1;
        bool got = warp_wait(bar(full0 + st), rph, wc);
        if (got) {
          if (is_k) got = warp_wait(bar(kK8Empty + os), oph ^ 1, wc);
          else if (e >= kV8Tiles) got = warp_wait(bar(kOFull + os), oph ^ 1, wc);
        }
        if (!got) {
          ok = false;
          break;
        }
        // tokens after the query position (only in the recent block) become zeros
        const int valid = r->valid[i];
        const bool full = valid >= 32 * (warp & 3) + 32;  // warp-uniform
        const bool live = tok < valid;
        const uint8_t* raw = smem + raw0 + st * kHalfBytes;
        // K: row tok of A in TMEM, columns 32 os + 8c .. + 7 = channels 32c .. 32c + 31
        const uint32_t ta = tmem + ((uint32_t)(32 * (warp & 3)) << 16) + 32 * os;
        uint8_t* dst = smem + kOffV8 + os * kTileBytes;
#pragma unroll
        for (int ci = 0; ci < kCh; ++ci) {
          uint32_t o[8];
          convert_chunk(raw + code_off[ci], raw + sc_off[ci], s_tab, o);
          if (!full) {
#pragma unroll
            for (int x = 0; x < 8; ++x) o[x] = live ? o[x] : 0u;
          }
          if (is_k) {
            tmem_st8(ta + 8 * (cs * kCh + ci), o);
          } else {
            *reinterpret_cast<uint4*>(dst + v_off[ci][0]) = make_uint4(o[0], o[1], o[2], o[3]);
            *reinterpret_cast<uint4*>(dst + v_off[ci][1]) = make_uint4(o[4], o[5], o[6], o[7]);
          }
        }
        if (is_k) {
          tmem_wait_st();
          tc_fence_before();
        } else {
          fence_proxy_async_smem();
        }
        __syncwarp();
        if (lane == 0) {
          if (is_k) mbar_arrive(bar(kK8Full + os));
          else mbar_arrive(bar(kV8Full + os));
          mbar_arrive(bar(empty0 + st));
        }
        if (++st == kStages) {
          st = 0;
          rph ^= 1;
        }
      }
      if (ok && lane == 0) mbar_arrive(bar(kRecEmpty + slot));
    }
  }
  else if (warp >= 4) {
    // ---------------- softmax: set s = warps 4 + 4 s .. 7 + 4 s ------------------------
    // set s takes the pages with e % kSets == s; warp w reads TMEM lanes 32 (w % 4) ..:
    // row = token of S, channel of O
    const int set = (warp - 4) >> 2, quad = warp & 3, row = 32 * quad + lane;
    const uint32_t trow = tmem + ((uint32_t)(32 * quad) << 16);
    const int nb = 1 + set;  // named barrier of the set
    float* red = reinterpret_cast<float*>(smem + kOffRed) + set * 32;   // [2][4 warps][4 heads]
    float* redl = reinterpret_cast<float*>(smem + kOffRedL) + set * 16;  // [4 warps][4 heads]
    int e0 = 0;  // page number of the item's first page
    bool ok = true;
    for (int k = 0; ok && k < n_mine; ++k) {
      const int slot = k % kRecs;
      if (named_barrier_or(nb, 128, !warp_wait(bar(kRecFull + slot), (k / kRecs) & 1, wc))) break;
      const ItemRec* r = rec(slot);
      const int n = r->n_pg;
      float m_run[4], l_run[4], o_run[4], a_prev[4], b_prev[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        m_run[h] = -INFINITY;
        l_run[h] = 0.f;
        o_run[h] = 0.f;
        a_prev[h] = 1.f;
        b_prev[h] = 0.f;
      }
      // O of page ef (relative to its page max) -> running state
      auto fold = [&](int ef) -> bool {
        const int po = (unsigned)ef % kPO;
        if (!warp_wait(bar(kOFull + po), ((unsigned)ef / kPO) & 1, wc)) return false;
        tc_fence_after();
        float ov[8];
        tmem_ld8(trow + kTmO + 16 * po, ov);  // columns 0-3: hi terms, 4-7: remainders
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(bar(kOEmpty + po));
#pragma unroll
        for (int h = 0; h < 4; ++h) o_run[h] = o_run[h] * a_prev[h] + (ov[h] + ov[4 + h]) * b_prev[h];
        return true;
      };
      int e_prev = -1;
      for (int e = e0 + (set - e0 % kSets + kSets) % kSets; e < e0 + n; e += kSets) {
        const int ph = ((unsigned)e / kSets) & 1;
        bool good = warp_wait(bar(kSFull + set), ph, wc);
        float sv[4] = {0.f, 0.f, 0.f, 0.f};
        if (good) {
          tc_fence_after();
          tmem_ld4(trow + kTmS + 16 * set, sv);
          tc_fence_before();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kSEmpty + set));
        }
        const bool live = row < r->valid[e - e0];
        float* rd = red + ph * 16;
        float x[4], wm[4];
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          x[h] = live ? sv[h] * p.scale_log2 : -INFINITY;
          wm[h] = warp_max_f32(x[h]);
        }
        if (lane == 0) reinterpret_cast<float4*>(rd)[quad] = make_float4(wm[0], wm[1], wm[2], wm[3]);
        // page maxima complete; the set's four warps agree on whether to go on
        if (named_barrier_or(nb, 128, !good || !ok)) {
          ok = false;
          break;
        }
        float a_cur[4], b_cur[4], v[4];
        {
          const float4 r0 = reinterpret_cast<const float4*>(rd)[0], r1 = reinterpret_cast<const float4*>(rd)[1];
          const float4 r2 = reinterpret_cast<const float4*>(rd)[2], r3 = reinterpret_cast<const float4*>(rd)[3];
          const float mps[4] = {fmaxf(fmaxf(r0.x, r1.x), fmaxf(r2.x, r3.x)), fmaxf(fmaxf(r0.y, r1.y), fmaxf(r2.y, r3.y)),
                                fmaxf(fmaxf(r0.z, r1.z), fmaxf(r2.z, r3.z)), fmaxf(fmaxf(r0.w, r1.w), fmaxf(r2.w, r3.w))};
#pragma unroll
          for (int h = 0; h < 4; ++h) {
            const float mp = mps[h];
            // one of the two rescale factors is 1: the running state (a) moves
            // to the page max when it grows, else the page (b) to the running max
            const bool grow = mp > m_run[h];
            const float f = fast_exp2(grow ? m_run[h] - mp : mp - m_run[h]);
            a_cur[h] = grow ? f : 1.f;
            b_cur[h] = grow ? 1.f : (mp == -INFINITY ? 0.f : f);
            m_run[h] = fmaxf(m_run[h], mp);
            // 256 p relative to the page max (<= 256: exact range of E4M3)
            v[h] = mp == -INFINITY ? 0.f : fast_exp2(x[h] - mp + 8.f);
            l_run[h] = l_run[h] * a_cur[h] + v[h] * b_cur[h];
          }
        }
        // 256 p as two E4M3 terms: hi = E4M3(256 p), lo = E4M3(f16(256 p) - hi)
        // (the f16 difference is exact: hi is within a factor of two of 256 p)
        const uint32_t hi01 = cvt_e4m3x2_f32(v[1], v[0]), hi23 = cvt_e4m3x2_f32(v[3], v[2]);
        const uint32_t lo01 = cvt_e4m3x2_f16x2(hsub2_u32(cvt_f16x2_f32(v[1], v[0]), cvt_f16x2_e4m3x2(hi01)));
        const uint32_t lo23 = cvt_e4m3x2_f16x2(hsub2_u32(cvt_f16x2_f32(v[3], v[2]), cvt_f16x2_e4m3x2(hi23)));
        // P tile row = token: bytes 0-3 hi terms of heads 0-3, 4-7 the remainders
        // (bytes 8-15 stay zero: they pad N to 16)
        const int po = (unsigned)e % kPO;
        // P tile po is free once the PV of page e - kPO is done (its O barrier)
        bool step_ok = warp_wait(bar(kOFull + po), (((unsigned)e / kPO) & 1) ^ 1, wc);
        if (step_ok) {
          *reinterpret_cast<uint2*>(smem + kOffP + po * 2048 + 16 * row) =
              make_uint2(prmt(hi01, hi23, 0x5410u), prmt(lo01, lo23, 0x5410u));
          fence_proxy_async_smem();
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kPFull + po));
          if (e_prev >= 0) step_ok = fold(e_prev);
        }
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          a_prev[h] = a_cur[h];
          b_prev[h] = b_cur[h];
        }
        e_prev = e;
        ok = ok && step_ok;  // a failure here ends the loop at the next barrier
      }
      if (ok && e_prev >= 0) ok = fold(e_prev);
      const bool aborted = named_barrier_or(nb, 128, !ok || *s_abort != 0);
      // ---- this set's sum of p over its tokens -------------------------------------------
      float L[4];
#pragma unroll
      for (int h = 0; h < 4; ++h) {
        float l = l_run[h];
#pragma unroll
        for (int o = 16; o; o >>= 1) l += __shfl_xor_sync(0xffffffffu, l, o);
        if (lane == 0) redl[quad * 4 + h] = l;
      }
      named_barrier_sync(nb, 128);
#pragma unroll
      for (int h = 0; h < 4; ++h) L[h] = aborted ? 0.f : redl[h] + redl[4 + h] + redl[8 + h] + redl[12 + h];
      // ---- merge the sets' states: sets 1 .. kSets - 1 hand over, set 0 writes ------------
      const int mph = (k >> 1) & 1;
      auto merge_buf = [&](int helper) {  // o [4][128], m [4], L [4]
        return reinterpret_cast<float*>(smem + kOffMerge + (2 * (helper - 1) + (k & 1)) * kMergeBytes);
      };
      if (set > 0) {
        const int mb = 2 * (set - 1) + (k & 1);
        float* mo = merge_buf(set);
        if (warp_wait(bar(kMergeEmpty + mb), mph ^ 1, wc)) {
#pragma unroll
          for (int h = 0; h < 4; ++h) mo[h * 128 + row] = o_run[h];
          if (row == 0) {
#pragma unroll
            for (int h = 0; h < 4; ++h) {
              mo[512 + h] = m_run[h];
              mo[516 + h] = L[h];
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(bar(kMergeFull + mb));
        }
      } else {
        bool got = true;
#pragma unroll
        for (int hs = 1; hs < kSets; ++hs)
          got = warp_wait(bar(kMergeFull + 2 * (hs - 1) + (k & 1)), mph, wc) && got;
        const size_t row0 = ((size_t)r->j * p.n_splits + r->split) * kQHeads + r->kvh * kGqa;
#pragma unroll
        for (int h = 0; h < 4; ++h) {
          float m = m_run[h];
#pragma unroll
          for (int hs = 1; hs < kSets; ++hs) m = fmaxf(m, got ? merge_buf(hs)[512 + h] : -INFINITY);
          const float w0 = (m_run[h] == -INFINITY || L[h] == 0.f) ? 0.f : fast_exp2(m_run[h] - m);
          float Lm = L[h] * w0, om = o_run[h] * w0;
#pragma unroll
          for (int hs = 1; hs < kSets; ++hs) {
            const float* mo = merge_buf(hs);
            const float m1 = got ? mo[512 + h] : -INFINITY, L1 = got ? mo[516 + h] : 0.f;
            const float w1 = (m1 == -INFINITY || L1 == 0.f) ? 0.f : fast_exp2(m1 - m);
            Lm += L1 * w1;
            om += (got ? mo[h * 128 + row] : 0.f) * w1;
          }
          const bool nonempty = !aborted && got && Lm > 0.f;
          p.o_part[(row0 + h) * kHeadDim + row] = nonempty ? om / Lm * p.out_scale : 0.f;
          if (row == 0) p.lse_part[row0 + h] = nonempty ? (m + log2f(Lm) - 8.f) * kLn2 : -INFINITY;
        }
        __syncwarp();
        if (lane == 0 && got) {
#pragma unroll
          for (int hs = 1; hs < kSets; ++hs) mbar_arrive(bar(kMergeEmpty + 2 * (hs - 1) + (k & 1)));
        }
      }
      __syncwarp();
      if (lane == 0) mbar_arrive(bar(kRecEmpty + slot));
      e0 += n;
      ok = !aborted;
    }
  }

  // ---- teardown -------------------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  if (tid == 0) {
    // every tcgen05.mma is done (both issuers committed after their last one)
    mbar_wait_drain(bar(kDone), 0, p.wait_ns);
    mbar_wait_drain(bar(kDone + 1), 0, p.wait_ns);
    if (*s_abort) {
      set_status(p.status, MSA_STATUS_TIMEOUT);
      // bounded drain of the copies that may still be landing: the last kStages
      // issued on each ring (every earlier one was consumed before its stage was
      // refilled)
      const int nk = *s_issued_k, nv = *s_issued_v;
      for (int e = max(0, nk - kStages); e < nk; ++e)
        mbar_wait_drain(bar(kKrFull + e % kStages), (e / kStages) & 1, p.wait_ns);
      for (int e = max(0, nv - kStages); e < nv; ++e)
        mbar_wait_drain(bar(kVrFull + e % kStages), (e / kStages) & 1, p.wait_ns);
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
    return cudaFuncSetAttribute(sparse_attn_tc_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                (int)attn_smem_bytes(kMaxSeqs));
  });
  if (e != cudaSuccess) return e;
  const int n_items = n_q_total * kKvHeads * n_splits;
  AttnParams ap{static_cast<const uint8_t*>(c->kv_pool), c->n_pages, q, sel, n_sel, block_table,
                max_pages, seq_lens, q_start_loc, n_seqs, n_q_total, n_splits, n_items,
                softmax_scale / c->s_enc_k * kLog2e, 1.0f / c->s_enc_v, o_part,
                lse_part, c->status, launch_settings().wait_ns};
  const int grid = n_items < n_sm ? n_items : n_sm;
  return launch_pdl(sparse_attn_tc_kernel, dim3(grid), dim3(kThreads), attn_smem_bytes(n_seqs), stream, ap);
}

}  // namespace msa
