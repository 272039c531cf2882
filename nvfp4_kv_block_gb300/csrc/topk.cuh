// Top-16 + recent selection of one query token over its block scores, shared
// by the indexer scan kernel and the fused low-concurrency decode kernel.
//
// "vLLM Delivers Day-0 Support for MiniMax-M3.1-Flash" blog, section "Sparse
// attention still scans an index": of the blocks before a query token's own
// (most recent) block, the 16 with the highest block scores are kept (ties to
// the lower block), plus the most recent block.
#pragma once

#include "common.cuh"

namespace msa {

// What select_token reads and writes.
struct TopkArgs {
  const float* scores;        // [T][max_pages][4] partial block maxima (block score = their max)
  int max_pages;
  int n_seqs;
  int n_q_total;
  int* sel;                   // [T][17]
  int* n_sel;                 // [T]
  int* status;
  int blk_lo, blk_hi;         // competing blocks: [blk_lo, blk_hi) within [0, r_j)
  unsigned long long* cand;   // range mode: [T][16] keys instead of sel / n_sel
};

// ---------------------------------------------------------------------------
// Top-16 + recent per query token, run by the scan kernel's CTAs after a grid
// barrier (every block score is then written).  Keys are
// (ordered score << 32) | ~block: unique, larger = better (higher score, then
// lower block).  The token's block scores are staged in shared memory by one
// coalesced pass, a lower bound theta of the 16th largest key prunes them to a
// few candidates, which are ranked exactly by counting.
constexpr int kMaxCand = 2048;
constexpr int kTopkStage = 16384;  // block scores staged in shared memory up to this many blocks
constexpr int kWsSyncBytes = 256;  // grid-barrier words at the start of the indexer workspace

__device__ __forceinline__ unsigned long long umax64(unsigned long long a, unsigned long long b) {
  return a > b ? a : b;
}

struct TopkSmem {
  float* sc;                 // [kTopkStage]
  unsigned long long* cand;  // [kMaxCand]
  unsigned long long* tmax;  // [NT] per-warp survivors, theta, reduction scratch
  unsigned long long* win;   // [16] winning keys by rank
  int* misc;                 // [0] n_cand, [1..] per-warp counts
};

// Sequence of query token j (-1 if none): the b with q_start_loc[b] <= j <
// q_start_loc[b+1], by binary search in the shared-memory copy of q_start_loc
// (non-decreasing for valid input; anything else ends as -1 or a sequence that
// fails its checks).
__device__ __forceinline__ int token_sequence(const int* s_qsl, int n_seqs, int j) {
  if (n_seqs <= 0) return -1;
  int lo = 0, hi = n_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (s_qsl[mid] <= j) lo = mid; else hi = mid - 1;
  }
  return (s_qsl[lo] <= j && j < s_qsl[lo + 1]) ? lo : -1;
}

__device__ __forceinline__ unsigned long long make_key(float sc, int blk) {
  return ((unsigned long long)ordered_bits(sc) << 32) | (unsigned long long)(0xFFFFFFFFu - (uint32_t)blk);
}
__device__ __forceinline__ int key_block(unsigned long long k) {
  return (int)(0xFFFFFFFFu - (uint32_t)(k & 0xFFFFFFFFu));
}

// Top-16 of query token j over its competing blocks [lo, e), e = min(blk_hi,
// r_j), lo = min(blk_lo, e).  Final mode (p.cand == nullptr; the whole range
// [0, r_j)): sel = the winners ascending, then r_j.  Range mode: the winners'
// keys in rank order (best first), zero-padded, into p.cand[j][0..15].
template <int NT>
__device__ void select_token(const TopkArgs& p, int j, const int* s_sl, const int* s_qsl,
                             const TopkSmem& sm) {
  const int tid = threadIdx.x, lane = tid & 31;
  const bool range_mode = p.cand != nullptr;
  const int b = token_sequence(s_qsl, p.n_seqs, j);
  SeqInfo s{0, 0, 0, false};
  if (b >= 0) s = load_seq(b, s_sl, s_qsl, p.max_pages, p.n_q_total);
  int* out = p.sel + (size_t)j * kSelStride;
  unsigned long long* kout = range_mode ? p.cand + (size_t)j * kTopK : nullptr;
  if (b < 0 || !s.ok) {
    if (tid == 0) set_status(p.status, MSA_STATUS_BAD_SEQ);
    if (range_mode) {
      if (tid < kTopK) kout[tid] = 0ull;
    } else {
      if (tid < kSelStride) out[tid] = -1;
      if (tid == 0) p.n_sel[j] = 0;
    }
    return;
  }
  const int pos = s.seq_len - s.n_q + (j - s.q0);
  const int r = pos / kPageTokens;
  const int e = min(p.blk_hi, r), lo = min(p.blk_lo, e);
  const int n = e - lo;  // competing blocks lo .. e-1
  // block score = max of the four partial maxima (written by other CTAs: read
  // through L2)
  const float4* row = reinterpret_cast<const float4*>(p.scores + (size_t)j * p.max_pages * 4) + lo;
  if (n <= kTopK) {
    if (range_mode) {
      // every block of the range wins; warp 0 ranks their keys, best first
      if (tid < 32) {
        unsigned long long k = 0ull;
        if (tid < n) {
          const float4 v = __ldcg(row + tid);
          k = make_key(fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)), lo + tid);
        }
        int rk = 0;
#pragma unroll
        for (int t = 0; t < kTopK; ++t) rk += __shfl_sync(0xffffffffu, k, t) > k;
        if (tid < n) kout[rk] = k;
        else if (tid < kTopK) kout[tid] = 0ull;
      }
    } else {
      if (tid < kSelStride) out[tid] = tid <= r ? tid : -1;
      if (tid == 0) p.n_sel[j] = r + 1;
    }
    return;
  }
  if (n <= 64) {
    // short rows: warp 0 alone, two keys per lane (blocks lo + lane and
    // lo + 32 + lane), each ranked by counting over all 64 with shuffles
    if (tid < 32) {
      unsigned long long k0 = 0ull, k1 = 0ull;
      if (lane < n) {
        const float4 v = __ldcg(row + lane);
        k0 = make_key(fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)), lo + lane);
      }
      if (32 + lane < n) {
        const float4 v = __ldcg(row + 32 + lane);
        k1 = make_key(fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w)), lo + 32 + lane);
      }
      int r0 = 0, r1 = 0;
#pragma unroll 8
      for (int t = 0; t < 32; ++t) {
        const unsigned long long a = __shfl_sync(0xffffffffu, k0, t), c = __shfl_sync(0xffffffffu, k1, t);
        r0 += (a > k0) + (c > k0);
        r1 += (a > k1) + (c > k1);
      }
      const bool w0 = k0 != 0ull && r0 < kTopK, w1 = k1 != 0ull && r1 < kTopK;
      if (range_mode) {
        if (w0) kout[r0] = k0;
        if (w1) kout[r1] = k1;
      } else {
        // winners ascending: blocks grow with the lane, first the lo + lane set
        const unsigned b0 = __ballot_sync(0xffffffffu, w0), b1 = __ballot_sync(0xffffffffu, w1);
        const unsigned lt = (1u << lane) - 1u;
        if (w0) out[__popc(b0 & lt)] = lo + lane;
        if (w1) out[__popc(b0) + __popc(b1 & lt)] = lo + 32 + lane;
        if (lane == 0) {
          out[kTopK] = r;
          p.n_sel[j] = kTopK + 1;
        }
      }
    }
    return;
  }
  // Up to kRegKeys blocks per thread the keys live in registers (all loads in
  // flight at once, no shared-memory staging); longer rows are staged in
  // shared memory, or read from L2 each time beyond kTopkStage.
  constexpr int kRegKeys = 16;
  const bool in_regs = n <= kRegKeys * NT;
  const bool staged = !in_regs && n <= kTopkStage;
  auto score = [&](int i) -> float {
    if (staged) return sm.sc[i];
    const float4 v = __ldcg(row + i);
    return fmaxf(fmaxf(v.x, v.y), fmaxf(v.z, v.w));
  };
  auto key = [&](int i) -> unsigned long long { return make_key(score(i), lo + i); };
  unsigned long long kr[kRegKeys];  // block lo + tid + u NT; 0 = no block (every real key is > 0)
  if (in_regs) {
    float4 v4[kRegKeys];
#pragma unroll
    for (int u = 0; u < kRegKeys; ++u) {
      const int i = tid + u * NT;
      v4[u] = i < n ? __ldcg(row + i) : make_float4(0.f, 0.f, 0.f, 0.f);
    }
#pragma unroll
    for (int u = 0; u < kRegKeys; ++u) {
      const int i = tid + u * NT;
      kr[u] = i < n ? make_key(fmaxf(fmaxf(v4[u].x, v4[u].y), fmaxf(v4[u].z, v4[u].w)), lo + i) : 0ull;
    }
  } else if (staged) {
    // batches of 8 loads in flight per thread, then the stores
    for (int base = tid; base < n; base += 8 * NT) {
      float4 v[8];
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = base + u * NT;
        v[u] = i < n ? __ldcg(row + i) : make_float4(0.f, 0.f, 0.f, 0.f);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = base + u * NT;
        if (i < n) sm.sc[i] = fmaxf(fmaxf(v[u].x, v[u].y), fmaxf(v[u].z, v[u].w));
      }
    }
  }
  if (tid == 0) sm.misc[0] = 0;
  __syncthreads();
  // theta: thread t owns blocks t, t + NT, ...  Each warp sorts the score parts
  // of its 32 thread maxima (bitonic, by shuffles), so lane i holds the warp's
  // (i+1)-th largest.  For m in {2, 4, 8, 16}: if 16/m warps each have m keys
  // at or above x, then x <= the 16th largest key; so the (16/m)-th largest of
  // the warps' m-th largest maxima (as a key with the block bits clear) is a
  // lower bound of the 16th largest key, and theta is the largest of these four
  // bounds.  Every winner is then a candidate.  (n > 16 here; real keys are
  // distinct and > 0, a missing key counts as 0.)
  constexpr int kNW = NT / 32;
  unsigned long long vmax = 0;
  if (in_regs) {
#pragma unroll
    for (int u = 0; u < kRegKeys; ++u) vmax = umax64(vmax, kr[u]);
  } else {
    for (int i = tid; i < n; i += NT) vmax = umax64(vmax, key(i));
  }
  uint32_t v = (uint32_t)(vmax >> 32);
#pragma unroll
  for (int k = 2; k <= 32; k <<= 1) {
#pragma unroll
    for (int jj = k >> 1; jj > 0; jj >>= 1) {
      const uint32_t o = __shfl_xor_sync(0xffffffffu, v, jj);
      // descending overall: the lower lane of a pair keeps the larger value in
      // blocks whose bit k is clear, the smaller one where it is set
      const bool lower = (lane & jj) == 0, asc = (lane & k) == 0;
      v = (lower == asc) ? max(v, o) : min(v, o);
    }
  }
  // tmax[4w + s] = warp w's (2 << s)-th largest maximum; tmax[4 kNW] = theta
  if (lane == 1 || lane == 3 || lane == 7 || lane == 15)
    sm.tmax[(tid >> 5) * 4 + (31 - __clz(lane + 1)) - 1] = (unsigned long long)v << 32;
  if (tid == 0) sm.tmax[4 * kNW] = 0ull;
  __syncthreads();
  if (tid < 4 * kNW) {
    const int set = tid & 3;
    const unsigned long long x = sm.tmax[tid];
    int rk = 0;
#pragma unroll
    for (int w = 0; w < kNW; ++w) rk += sm.tmax[4 * w + set] > x;
    if (rk == (8 >> set) - 1) atomicMax(&sm.tmax[4 * kNW], x);
  }
  __syncthreads();
  const unsigned long long theta = sm.tmax[4 * kNW];
  // candidates: keys >= theta, written without atomics: per-thread counts, a
  // scan over lanes and warps, then each thread writes its own
  int cnt = 0;
  if (in_regs) {
#pragma unroll
    for (int u = 0; u < kRegKeys; ++u) cnt += kr[u] >= theta;
  } else {
    for (int i = tid; i < n; i += NT) cnt += key(i) >= theta;
  }
  int incl = cnt;
#pragma unroll
  for (int o = 1; o < 32; o <<= 1) {
    const int y = __shfl_up_sync(0xffffffffu, incl, o);
    if (lane >= o) incl += y;
  }
  if (lane == 31) sm.misc[1 + (tid >> 5)] = incl;
  __syncthreads();
  int at = incl - cnt, nc_all = 0;
#pragma unroll
  for (int w = 0; w < kNW; ++w) {
    const int c = sm.misc[1 + w];
    at += w < (tid >> 5) ? c : 0;
    nc_all += c;
  }
  if (cnt) {
    if (in_regs) {
#pragma unroll
      for (int u = 0; u < kRegKeys; ++u) {
        if (kr[u] >= theta) {
          if (at < kMaxCand) sm.cand[at] = kr[u];
          ++at;
        }
      }
    } else {
      for (int i = tid; i < n; i += NT) {
        const unsigned long long k = key(i);
        if (k >= theta) {
          if (at < kMaxCand) sm.cand[at] = k;
          ++at;
        }
      }
    }
  }
  if (tid == 0) sm.misc[0] = nc_all;
  __syncthreads();
  const int nc = sm.misc[0];
  if (nc <= kMaxCand) {
    // exact rank of each candidate by counting; pairs of keys per load (a zero
    // pad never counts: every key is > 0)
    if (tid == 0 && (nc & 1) && nc < kMaxCand) sm.cand[nc] = 0ull;
    __syncthreads();
    const ulonglong2* c2 = reinterpret_cast<const ulonglong2*>(sm.cand);
    for (int c = tid; c < nc; c += NT) {
      const unsigned long long k = sm.cand[c];
      int rk = 0;
      for (int i = 0; i < (nc + 1) / 2; ++i) {
        const ulonglong2 v = c2[i];
        rk += (v.x > k) + (v.y > k);
      }
      if (rk < kTopK) sm.win[rk] = k;
    }
  } else {
    // too many candidates for the buffer (adversarial score layouts): 16 rounds
    // of CTA-wide argmax, each over the keys below the previous winner
    unsigned long long bound = ~0ull;
    for (int k = 0; k < kTopK; ++k) {
      unsigned long long best = 0;
      if (in_regs) {
#pragma unroll
        for (int u = 0; u < kRegKeys; ++u)
          if (kr[u] < bound) best = umax64(best, kr[u]);
      } else {
        for (int i = tid; i < n; i += NT) {
          const unsigned long long kk = key(i);
          if (kk < bound) best = umax64(best, kk);
        }
      }
      sm.tmax[tid] = best;
      __syncthreads();
      if (tid == 0) {
        for (int i = 1; i < NT; ++i) best = umax64(best, sm.tmax[i]);
        sm.tmax[0] = best;
        sm.win[k] = best;
      }
      __syncthreads();
      bound = sm.tmax[0];
      __syncthreads();
    }
  }
  __syncthreads();
  if (range_mode) {
    if (tid < kTopK) kout[tid] = sm.win[tid];
    return;
  }
  if (tid < kTopK) {
    const int blk = key_block(sm.win[tid]);
    int at = 0;
#pragma unroll
    for (int i = 0; i < kTopK; ++i) at += key_block(sm.win[i]) < blk;
    out[at] = blk;
  }
  if (tid == 0) {
    out[kTopK] = r;
    p.n_sel[j] = kTopK + 1;
  }
}


}  // namespace msa
