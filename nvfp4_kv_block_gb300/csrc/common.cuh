// Shared device helpers of the NVFP4 sparse-attention decode kernels (sm_103a).
//
// Page formats and shapes follow include/msa.h.  The FP8 (E4M3) and FP4
// (E2M1) conversions use the hardware round-to-nearest-even converters through
// CUDA's cuda_fp8.h intrinsics.
#pragma once

#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include <atomic>
#include <mutex>

#include "../../include/msa.h"

namespace msa {

constexpr int kPageTokens = 128;
constexpr int kKvHeads = 4;
constexpr int kHeadDim = 128;
constexpr int kIdxDim = 128;
constexpr int kIdxHeads = 8;
constexpr int kQHeads = 16;
constexpr int kGqa = kQHeads / kKvHeads;
constexpr int kTopK = 16;
constexpr int kSelStride = kTopK + 1;
constexpr int kHeadBytes = 18432;
constexpr int kKvPageBytes = kKvHeads * kHeadBytes;  // 73,728
constexpr int kIdxPageBytes = kPageTokens * kIdxDim;  // 16,384
constexpr int kOffKc = 0, kOffKs = 8192, kOffVc = 9216, kOffVs = 17408;
// The 16-byte code chunk c (channels 32c..32c+31) of token t sits at chunk
// position c ^ ((t >> 1) & 3) of the token's 64-byte code row: one thread per
// token can then read chunk c of 32 consecutive rows (64 B apart) without
// shared-memory bank conflicts.
__host__ __device__ __forceinline__ int code_chunk_pos(int c, int t) { return c ^ ((t >> 1) & 3); }
constexpr int kMaxSeqs = 4096;
constexpr int kMaxSplits = 64;
constexpr int kMaxLayers = 128;  // layers one block-outer row may hold
// Capacity of the file-scope scratch of msa_indexer_topk_noalloc.
constexpr size_t kStaticScratchBytes = MSA_INDEXER_NOALLOC_SCRATCH_BYTES;

__device__ __forceinline__ void set_status(int* status, int bits) {
  if (status) atomicOr(status, bits);
}

// ---- loads -----------------------------------------------------------------
// Streaming loads of read-only cache data: not kept in L1.
__device__ __forceinline__ uint4 ld_stream_v4(const void* p) {
  uint4 v;
  asm("ld.global.nc.L1::no_allocate.v4.u32 {%0,%1,%2,%3}, [%4];"
      : "=r"(v.x), "=r"(v.y), "=r"(v.z), "=r"(v.w)
      : "l"(p));
  return v;
}
__device__ __forceinline__ uint2 ld_stream_v2(const void* p) {
  uint2 v;
  asm("ld.global.nc.L1::no_allocate.v2.u32 {%0,%1}, [%2];" : "=r"(v.x), "=r"(v.y) : "l"(p));
  return v;
}
__device__ __forceinline__ uint32_t ld_stream_u32(const void* p) {
  uint32_t v;
  asm("ld.global.nc.L1::no_allocate.u32 %0, [%1];" : "=r"(v) : "l"(p));
  return v;
}

// ---- byte permute ----------------------------------------------------------
// PTX prmt.b32 (default mode): output byte n is byte (c >> 4n) & 7 of {b:a};
// if bit 3 of that selector nibble is set, the selected byte's sign bit is
// replicated over the output byte instead.
__device__ __forceinline__ uint32_t prmt(uint32_t a, uint32_t b, uint32_t c) {
  uint32_t d;
  asm("prmt.b32 %0, %1, %2, %3;" : "=r"(d) : "r"(a), "r"(b), "r"(c));
  return d;
}

// ---- E4M3 helpers -----------------------------------------------------------
__device__ __forceinline__ uint32_t f32_to_e4m3(float x) {
  return (uint32_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}
// Two floats -> two E4M3 bytes, x in the low byte.
__device__ __forceinline__ uint32_t f32x2_to_e4m3x2(float x, float y) {
  return (uint32_t)__nv_cvt_float2_to_fp8x2(make_float2(x, y), __NV_SATFINITE, __NV_E4M3);
}
__device__ __forceinline__ float e4m3_to_f32(uint32_t byte) {
  __half_raw h = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)(byte & 0xFF), __NV_E4M3);
  return __half2float(__half(h));
}
// Canonical zero: an E4M3 byte of zero magnitude becomes 0x00.
__device__ __forceinline__ uint32_t canon_zero(uint32_t byte) {
  return (byte & 0x7F) ? byte : 0u;
}

// Order-preserving map of an fp32 value to uint32 (larger float -> larger int).
__device__ __forceinline__ uint32_t ordered_bits(float f) {
  uint32_t u = __float_as_uint(f);
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}
__device__ __forceinline__ float from_ordered_bits(uint32_t u) {
  return __uint_as_float((u & 0x80000000u) ? (u & 0x7FFFFFFFu) : ~u);
}
// Warp-wide max of a float with one redux.sync on its order-preserving bits.
__device__ __forceinline__ float warp_max(float x) {
  return from_ordered_bits(__reduce_max_sync(0xffffffffu, ordered_bits(x)));
}
// Warp-wide max of a float (one redux.sync; -inf allowed, no NaN inputs).
__device__ __forceinline__ float warp_max_f32(float x) {
  float y;
  asm("redux.sync.max.f32 %0, %1, 0xffffffff;" : "=f"(y) : "f"(x));
  return y;
}
// Packed conversions: two fp32 -> two E4M3 (RNE, satfinite; hi -> byte 1,
// lo -> byte 0), two E4M3 -> f16x2 (exact), f16x2 -> two E4M3, two fp32 ->
// f16x2 (hi -> upper half), and an f16x2 difference.
__device__ __forceinline__ uint32_t cvt_e4m3x2_f32(float hi, float lo) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f32 %0, %1, %2;" : "=h"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ uint32_t cvt_f16x2_e4m3x2(uint32_t x) {
  uint32_t d;
  asm("cvt.rn.f16x2.e4m3x2 %0, %1;" : "=r"(d) : "h"((uint16_t)x));
  return d;
}
__device__ __forceinline__ uint32_t cvt_e4m3x2_f16x2(uint32_t x) {
  uint16_t d;
  asm("cvt.rn.satfinite.e4m3x2.f16x2 %0, %1;" : "=h"(d) : "r"(x));
  return d;
}
__device__ __forceinline__ uint32_t cvt_f16x2_f32(float hi, float lo) {
  uint32_t d;
  asm("cvt.rn.f16x2.f32 %0, %1, %2;" : "=r"(d) : "f"(hi), "f"(lo));
  return d;
}
__device__ __forceinline__ uint32_t hsub2_u32(uint32_t a, uint32_t b) {
  uint32_t d;
  asm("sub.rn.f16x2 %0, %1, %2;" : "=r"(d) : "r"(a), "r"(b));
  return d;
}
// 2^x with the hardware approximation (relative error about 2^-22; 2^-inf = 0).
__device__ __forceinline__ float fast_exp2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

// ---- NVFP4 quantisation ------------------------------------------------------
// E2M1 magnitude code of y / sb, round to nearest, ties to the even code,
// saturating at 6.  Each comparison is y against midpoint * sb, which is
// exact in fp32 (at most 7 significant bits), so the ratio is never rounded.
__device__ __forceinline__ uint32_t e2m1_code(float y, float sb) {
  uint32_t c = 0;
  c += y > 0.25f * sb;   // 0   | 0.5  tie -> 0
  c += y >= 0.75f * sb;  // 0.5 | 1    tie -> 1
  c += y > 1.25f * sb;   // 1   | 1.5  tie -> 1
  c += y >= 1.75f * sb;  // 1.5 | 2    tie -> 2
  c += y > 2.5f * sb;    // 2   | 3    tie -> 2
  c += y >= 3.5f * sb;   // 3   | 4    tie -> 4
  c += y > 5.0f * sb;    // 4   | 6    tie -> 4
  return sb > 0.f ? c : 0u;
}

// ---- NVFP4 -> FP8 dequantisation --------------------------------------------
// Table entry for scale byte sb: 8 E4M3 bytes, entry m = E4M3_RNE(|e2m1(m)| * sb),
// magnitudes m = 0..7 -> 0, 0.5, 1, 1.5, 2, 3, 4, 6.  The product has at most
// five significant bits, so it is exact in fp32 and the conversion is the only
// rounding.  A zero result is stored as 0x00.
__device__ __forceinline__ void build_dequant_table(uint2* tab, int tid, int nthreads) {
  const float mags[8] = {0.f, 0.5f, 1.f, 1.5f, 2.f, 3.f, 4.f, 6.f};
  for (int sb = tid; sb < 256; sb += nthreads) {
    const float s = e4m3_to_f32((uint32_t)sb);
    uint32_t lo = 0, hi = 0;
#pragma unroll
    for (int m = 0; m < 4; ++m) {
      lo |= canon_zero(f32_to_e4m3(mags[m] * s)) << (8 * m);
      hi |= canon_zero(f32_to_e4m3(mags[m + 4] * s)) << (8 * m);
    }
    tab[sb] = make_uint2(lo, hi);
  }
}

// Code word: little-endian 32-bit word i of a token's code row holds channels
// 8i..8i+7, each an E2M1 code (sign << 3 | 3-bit magnitude): the magnitude of
// channel n at bits 4n..4n+2 (n = 0..7), the sign of channel n at bit 8n+7 and
// that of channel 4 + n at bit 8n+3 (n = 0..3).  The magnitudes are then the
// byte-permute selectors of dequant8 as they stand, and each sign bit sits at,
// or 4 bits below, bit 7 of its output byte.
// Bits of channels 4h..4h+3 (h = 0 or 1) of a word, codes c[0..3].
__host__ __device__ __forceinline__ uint32_t code_word_part(const uint32_t (&c)[4], int h) {
  uint32_t w = 0;
#pragma unroll
  for (int n = 0; n < 4; ++n) {
    w |= (c[n] & 7u) << (16 * h + 4 * n);
    w |= ((c[n] >> 3) & 1u) << (8 * n + (h ? 3 : 7));
  }
  return w;
}

// One code word -> eight FP8 operand bytes (x: channels 0..3, y: 4..7), each
// sign(code) | table[magnitude]: two byte permutes of the scaled table by the
// magnitudes (sign bits masked out: a set selector bit 3 would switch the
// permute to sign replication), the sign bits merged in place (x) or after a
// 4-bit shift (y).  7 integer instructions per 8 elements.
__device__ __forceinline__ uint2 dequant8(uint32_t w, uint2 t) {
  const uint32_t m = w & 0x77777777u;
  const uint32_t mag0 = prmt(t.x, t.y, m);
  const uint32_t mag1 = prmt(t.x, t.y, m >> 16);
  return make_uint2(mag0 | (w & 0x80808080u), mag1 | ((w << 4) & 0x80808080u));
}

// ---- mbarrier / TMA bulk copy / tcgen05 (inline PTX) --------------------------
// Every wait is bounded: after kSpinLimit polls or WaitCtl::limit_ns nanoseconds
// the caller gets false and must abandon its loop (the kernel then reports
// MSA_STATUS_TIMEOUT).  The limit is a kernel parameter (2 s unless the host
// lowers it, see msa_debug_set_fault_injection).
constexpr uint32_t kSpinLimit = 1u << 25;
constexpr unsigned long long kDefaultWaitLimitNs = 2000000000ull;  // 2 s

// Bounded-wait control of one CTA: the shared-memory flag its roles raise when
// a wait gives up (the other roles then stop waiting too), and the time limit.
struct WaitCtl {
  volatile int* abort;
  unsigned long long limit_ns;
};

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return (uint32_t)__cvta_generic_to_shared(p);
}
__device__ __forceinline__ unsigned long long globaltimer_ns() {
  unsigned long long t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count));
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes)
               : "memory");
}
// One poll.  The suspend-time hint (20 us) lets the hardware park the thread
// until the phase completes instead of re-issuing the poll.
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2, 20000;\n"
      " selp.u32 %0, 1, 0, p;\n}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}
// Waits for the phase with the given parity; false on timeout or when another
// role has already raised the abort flag (the flag is then raised too).
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, const WaitCtl& w) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t i = 1; i < kSpinLimit; ++i) {
    __nanosleep(32);  // a short back-off: waiting warps leave issue slots to the others
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 15) == 0 && (*w.abort || globaltimer_ns() - t0 > w.limit_ns)) break;
  }
  *w.abort = 1;
  return false;
}
// The same wait for teardown after an abort: it ignores the abort flag (the
// CTA must still see its in-flight copies and MMAs land before it releases
// shared or tensor memory) and is bounded by time and polls only.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, unsigned long long limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t i = 1; i < kSpinLimit; ++i) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((i & 15) == 0 && globaltimer_ns() - t0 > limit_ns) break;
  }
  return false;
}

// Grid-wide barrier of a launch whose CTAs are all co-resident (cooperative
// launch), on one 64-bit word of global memory: generation in the high half,
// arrival count in the low half.  Called by one thread per CTA; every CTA must
// call it exactly once per barrier, also after an abort of its own (so the
// count always reaches `target`).  The CTA that brings the count to `target`
// returns the count to zero and advances the generation in one atomic, which
// releases the others.  A waiter that times out withdraws its arrival (only
// while the generation is unchanged and the count is below `target`, i.e. the
// barrier cannot complete any more without it), raises *abort and returns
// false; so the word is back at rest after every barrier, completed or not,
// and later launches on the same word need no clearing.  `target` is the
// number of CTAs (the fault-injection test passes one more, so that the wait
// runs out).
__device__ __forceinline__ bool grid_barrier(unsigned long long* word, uint32_t target, const WaitCtl& w) {
  __threadfence();
  const unsigned long long old = atomicAdd(word, 1ull);
  const uint32_t gen = (uint32_t)(old >> 32);
  if ((uint32_t)old + 1u == target) {
    atomicAdd(word, (1ull << 32) - target);
    __threadfence();
    return true;
  }
  volatile unsigned long long* vw = word;
  const unsigned long long t0 = globaltimer_ns();
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if ((uint32_t)(*vw >> 32) != gen) {
      __threadfence();
      return true;
    }
    if ((i & 63) == 63 && globaltimer_ns() - t0 > w.limit_ns) break;
  }
  unsigned long long cur = *vw;
  while ((uint32_t)(cur >> 32) == gen && (uint32_t)cur < target) {
    const unsigned long long prev = atomicCAS(word, cur, cur - 1);
    if (prev == cur) {
      *w.abort = 1;
      return false;
    }
    cur = prev;
  }
  // completed while this CTA was giving up: wait (bounded) for the release
  for (uint32_t i = 0; i < kSpinLimit; ++i) {
    if ((uint32_t)(*vw >> 32) != gen) {
      __threadfence();
      return true;
    }
    if ((i & 63) == 63 && globaltimer_ns() - t0 > 2 * w.limit_ns) break;
  }
  *w.abort = 1;
  return false;
}
__device__ __forceinline__ void fence_barrier_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
// Generic-proxy shared-memory writes -> visible to the async proxy (TMA, tensor core).
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}
// 1D bulk copy global -> shared, completion signalled on an mbarrier (tx bytes).
__device__ __forceinline__ void bulk_g2s(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];" ::"r"(dst),
      "l"(src), "r"(bytes), "r"(bar)
      : "memory");
}

__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// Shared-memory matrix descriptor: K-major operand with 128-byte swizzle, rows
// grouped by 8 (1,024 bytes apart); the start address must sit in a
// 1,024-byte-aligned swizzle atom.
__device__ __forceinline__ uint64_t umma_desc_sw128(uint32_t saddr) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4)   // start address
         | ((uint64_t)1 << 16)                 // leading byte offset (unused for swizzled K-major)
         | ((uint64_t)(1024 >> 4) << 32)       // stride byte offset: 8 rows x 128 B
         | ((uint64_t)1 << 46)                 // descriptor version
         | ((uint64_t)2 << 61);                // 128-byte swizzle
}
// Instruction descriptor, kind::f8f6f4: D fp32, A and B E4M3, both K-major, M x N.
__device__ __forceinline__ uint32_t umma_idesc_e4m3(uint32_t M, uint32_t N) {
  return (1u << 4) | ((N >> 3) << 17) | ((M >> 4) << 24);
}
__device__ __forceinline__ void umma_e4m3(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc,
                                          uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// Arrive on an mbarrier once every tcgen05.mma issued so far by this thread is done.
__device__ __forceinline__ void umma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar)
               : "memory");
}
__device__ __forceinline__ void tmem_alloc(uint32_t dst_slot, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_slot),
               "r"(ncols)
               : "memory");
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols)
               : "memory");
}
// 32 TMEM lanes x 16 columns of 32-bit words -> 16 registers per thread.
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, float (&v)[16]) {
  uint32_t r[16];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, "
      "[%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
        "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]),
        "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 16; ++i) v[i] = __uint_as_float(r[i]);
}

// 32 TMEM lanes x N columns of 32-bit words -> N registers per thread, without
// waiting: several loads can be in flight, then one tmem_wait_ld().
__device__ __forceinline__ void tmem_ld32x32b_x16(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld32x32b_x32(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_ld32x32b_x64(uint32_t taddr, uint32_t* r) {
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x64.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32,%33,%34,%35,%36,%37,%38,%39,%40,%41,%42,%43,%44,%45,%46,%47,%48,%49,%50,%51,%52,%53,%54,%55,%56,%57,%58,%59,%60,%61,%62,%63}, [%64];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31]), "=r"(r[32]), "=r"(r[33]), "=r"(r[34]), "=r"(r[35]), "=r"(r[36]), "=r"(r[37]), "=r"(r[38]), "=r"(r[39]), "=r"(r[40]), "=r"(r[41]), "=r"(r[42]), "=r"(r[43]), "=r"(r[44]), "=r"(r[45]), "=r"(r[46]), "=r"(r[47]), "=r"(r[48]), "=r"(r[49]), "=r"(r[50]), "=r"(r[51]), "=r"(r[52]), "=r"(r[53]), "=r"(r[54]), "=r"(r[55]), "=r"(r[56]), "=r"(r[57]), "=r"(r[58]), "=r"(r[59]), "=r"(r[60]), "=r"(r[61]), "=r"(r[62]), "=r"(r[63])
               : "r"(taddr));
}
__device__ __forceinline__ void tmem_wait_ld() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }

// Instruction descriptor, kind::f8f6f4, A MN-major (a_major bit), B K-major.
__device__ __forceinline__ uint32_t umma_idesc_e4m3_amn(uint32_t M, uint32_t N) {
  return umma_idesc_e4m3(M, N) | (1u << 15);
}
// Instruction descriptor, kind::f8f6f4, A and B both MN-major (a_major, b_major bits).
__device__ __forceinline__ uint32_t umma_idesc_e4m3_amn_bmn(uint32_t M, uint32_t N) {
  return umma_idesc_e4m3(M, N) | (1u << 15) | (1u << 16);
}
// Shared-memory descriptor without swizzle (core matrices of 8 rows x 16 bytes,
// 128 contiguous bytes each), with explicit byte offsets between core matrices.
__device__ __forceinline__ uint64_t umma_desc_noswz_lbo_sbo(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) |
         ((uint64_t)(sbo >> 4) << 32) | ((uint64_t)1 << 46);
}
// Shared-memory descriptor with explicit byte offsets (128-byte swizzle).
__device__ __forceinline__ uint64_t umma_desc_sw128_lbo_sbo(uint32_t saddr, uint32_t lbo, uint32_t sbo) {
  return (uint64_t)((saddr & 0x3FFFFu) >> 4) | ((uint64_t)(lbo >> 4) << 16) |
         ((uint64_t)(sbo >> 4) << 32) | ((uint64_t)1 << 46) | ((uint64_t)2 << 61);
}
// 32 TMEM lanes x 8 columns -> 8 registers per thread.
__device__ __forceinline__ void tmem_ld8(uint32_t taddr, float (&v)[8]) {
  uint32_t r[8];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x8.b32 {%0,%1,%2,%3,%4,%5,%6,%7}, [%8];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]),
                 "=r"(r[7])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 8; ++i) v[i] = __uint_as_float(r[i]);
}
// 32 TMEM lanes x 4 columns -> 4 registers per thread.
__device__ __forceinline__ void tmem_ld4(uint32_t taddr, float (&v)[4]) {
  uint32_t r[4];
  asm volatile("tcgen05.ld.sync.aligned.32x32b.x4.b32 {%0,%1,%2,%3}, [%4];"
               : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3])
               : "r"(taddr));
  asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory");
#pragma unroll
  for (int i = 0; i < 4; ++i) v[i] = __uint_as_float(r[i]);
}

// 8 registers per thread -> 32 TMEM lanes x 8 columns (thread = lane).
__device__ __forceinline__ void tmem_st8(uint32_t taddr, const uint32_t* r) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8};" ::"r"(taddr),
               "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7])
               : "memory");
}
// 32 registers per thread -> 32 TMEM lanes x 32 columns (thread = lane).
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t* r) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])
      : "memory");
}
__device__ __forceinline__ void tmem_wait_st() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }
// D (TMEM) = A (TMEM: row m in lane m, K packed four 8-bit elements per column)
// x B (shared-memory descriptor), kind::f8f6f4.
__device__ __forceinline__ void umma_e4m3_ts(uint32_t d_tmem, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                             uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], [%1], %2, %3, p;\n}" ::"r"(d_tmem),
      "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}

__device__ __forceinline__ void named_barrier_sync(int id, int nthreads) {
  asm volatile("bar.sync %0, %1;" ::"r"(id), "r"(nthreads) : "memory");
}


// ---- programmatic dependent launch ------------------------------------------
// Kernels of the decode chain are launched with programmatic stream
// serialisation: a kernel may start while its predecessor finishes, runs its
// input-independent prologue, then waits here for the predecessor's completion
// (and memory) before touching data a previous kernel wrote.
__device__ __forceinline__ void pdl_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
// Lets the next kernel in the stream begin launching (it still waits in pdl_wait).
__device__ __forceinline__ void pdl_trigger() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

template <typename... KArgs, typename... Args>
inline cudaError_t launch_pdl(void (*kernel)(KArgs...), dim3 grid, dim3 block, size_t smem,
                              cudaStream_t stream, Args... args) {
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = grid;
  cfg.blockDim = block;
  cfg.dynamicSmemBytes = smem;
  cfg.stream = stream;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  return cudaLaunchKernelEx(&cfg, kernel, args...);
}

// ---- host-side launch settings ----------------------------------------------------
// Library-wide settings every launch reads (msa_debug_set_fault_injection):
// the limit of one bounded wait, and test-only fault-injection flags.
constexpr int kInjectBarrierTimeout = 1;  // the indexer's grid barrier waits for one CTA more than exist
struct LaunchSettings {
  unsigned long long wait_ns;
  int inject;
};
LaunchSettings launch_settings();  // defined in msa_abi.cu

// One-time per-device launch set-up (SM count, shared-memory opt-in) of one
// kernel.  The set-up runs under a mutex, so first calls from several host
// threads do not race, and the SM count is published only after it succeeded.
struct DeviceSetup {
  std::mutex mu;
  std::atomic<int> n_sm[64] = {};

  // The current device's SM count, running setup(dev) first if this is the
  // first call on the device.
  template <typename F>
  cudaError_t get(int* dev_out, int* n_sm_out, F&& setup) {
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    int n = n_sm[dev].load(std::memory_order_acquire);
    if (n == 0) {
      std::lock_guard<std::mutex> lock(mu);
      n = n_sm[dev].load(std::memory_order_relaxed);
      if (n == 0) {
        e = cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev);
        if (e != cudaSuccess) return e;
        e = setup(dev);
        if (e != cudaSuccess) return e;
        n_sm[dev].store(n, std::memory_order_release);
      }
    }
    *dev_out = dev;
    *n_sm_out = n;
    return cudaSuccess;
  }
};

// ---- sequence metadata --------------------------------------------------------
struct SeqInfo {
  int seq_len;
  int n_q;
  int q0;
  bool ok;
};

// Sequence b's metadata; ok is false (and the sequence must be skipped) when
// its query tokens fall outside [0, n_q_total), n_q < 0, n_q > seq_len or the
// context exceeds the block table row.
__device__ __forceinline__ SeqInfo load_seq(int b, const int* seq_lens, const int* q_start_loc,
                                            int max_pages, int n_q_total) {
  SeqInfo s;
  s.seq_len = seq_lens[b];
  s.q0 = q_start_loc[b];
  s.n_q = q_start_loc[b + 1] - s.q0;
  s.ok = s.n_q >= 0 && s.q0 >= 0 && s.q0 + s.n_q <= n_q_total && s.seq_len >= s.n_q &&
         s.seq_len <= max_pages * kPageTokens;
  return s;
}

// Largest b in [0, n_seqs) with q_start_loc[b] <= j (q_start_loc non-decreasing).
__device__ __forceinline__ int find_seq(const int* q_start_loc, int n_seqs, int j) {
  int lo = 0, hi = n_seqs - 1;
  while (lo < hi) {
    const int mid = (lo + hi + 1) >> 1;
    if (q_start_loc[mid] <= j) lo = mid; else hi = mid - 1;
  }
  return lo;
}

}  // namespace msa
