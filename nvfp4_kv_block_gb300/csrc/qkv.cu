// Fused QKV projection -> RMS norm -> RoPE -> FP8 queries and NVFP4 cache
// insertion, in one kernel.
//
// "vLLM Delivers Day-0 Support for MiniMax-M3.1-Flash" blog, section "Reduce
// both data movement and resource waits": fusing the QKV projection with the
// normalisation, RoPE and cache insertion avoids writing the full intermediate
// tensor to HBM and reading it back.  Here the projection's accumulators never
// leave the SM: each CTA computes one tile of 128 tokens x two heads (256
// output columns) on the tensor core and its epilogue finishes both heads.
//
// Output heads of the projection (columns of W, 128 each): 16 query heads,
// 4 key heads, 4 value heads, 1 index-key head.  Per token and head:
//   query / key / index key:  y = RMSNorm(x W_head) * gamma, then RoPE;
//   value:                    y = x W_head;
// then queries -> E4M3 bytes (the attention's FP8 query), keys and values ->
// NVFP4 into their cache slot (the quantiser of msa_quantize_kv_insert),
// index keys -> E4M3 into the index page.
//
// Tile pipeline (one CTA per tile, two per SM):
//   warp 0      TMA producer: per 64-column K chunk, a 128 x 64 bf16 tile of x
//               and two of W (the two heads; cp.async.bulk.tensor, 128-byte
//               swizzle) into a 2-stage ring;
//   warp 1      MMA issuer: 4 x tcgen05.mma kind::f16 (bf16 in, fp32 out;
//               M = 128 tokens, N = 256 columns, K = 16) per chunk, the
//               accumulator in tensor memory.  One tcgen05.mma costs its
//               issuing thread about 200 cycles whatever its N, so the widest N
//               does the most work per instruction;
//   warps 2-5   epilogue: thread = token row, one head's 128 columns at a time
//               in registers: RMS norm and RoPE are thread-local, so is the
//               NVFP4 quantiser (a 16-channel group lives in one thread).
#include <cuda.h>
#include <cudaTypedefs.h>

#include "common.cuh"

namespace msa {
namespace {

constexpr int kQkvThreads = 192;
constexpr int kChunk = 64;                    // bf16 elements of K per stage (128 bytes)
constexpr int kTileBytes = 128 * kChunk * 2;  // 16 KB per 128-row operand tile
// Tile of H heads per CTA (N = 128 H): the widest N does the most work per
// tcgen05.mma, one head per CTA makes twice the CTAs for short inputs.  The
// ring is sized so that two CTAs fit per SM.
template <int H>
struct QkvTile {
  static constexpr int kStages = H == 2 ? 2 : 3;
  static constexpr int kOffA = 0;                                      // kStages x 16 KB of x
  static constexpr int kOffB = kStages * kTileBytes;                   // kStages x H x 16 KB of W
  static constexpr int kOffGamma = kOffB + kStages * H * kTileBytes;   // 3 x 128 floats
  static constexpr int kOffBarQ = kOffGamma + 3 * 128 * 4;
  static constexpr int kSmem = kOffBarQ + 8 * (2 * kStages + 1) + 16;  // + tmem slot, abort, copies issued
};
constexpr int kHeadsOut = kQHeads + 2 * kKvHeads + 1;  // 25

struct QkvParams {
  CUtensorMap tmap_x;  // x [n_tokens][d_model] bf16, box 64 x 128, 128-byte swizzle
  CUtensorMap tmap_w;  // W [25 * 128][d_model] bf16, same box
  int n_tokens;
  int d_model;
  const float* gamma_q;    // [128]
  const float* gamma_k;    // [128]
  const float* gamma_idx;  // [128]
  const float* cos_sin;    // [max_pos][128]: cos of the 64 pair angles, then their sin
  int max_pos;
  const int* positions;    // [n_tokens]
  const int64_t* slot_mapping;  // [n_tokens]
  uint8_t* kv_pool;
  uint8_t* idx_pool;
  int64_t n_pages;
  float s_enc_k, s_enc_v;
  float eps;
  uint8_t* q8;   // [n_tokens][16][128]
  float* y_out;  // optional [n_tokens][25][128]: the rows before rounding
  int* status;
  unsigned long long wait_ns;
};

__device__ __forceinline__ void tma_load_2d(uint32_t dst, const CUtensorMap* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], "
      "[%4];" ::"r"(dst),
      "l"(reinterpret_cast<uint64_t>(map)), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
// kind::f16 instruction descriptor: D fp32, A and B bf16, both K-major, M x N.
__device__ __forceinline__ uint32_t umma_idesc_bf16(uint32_t M, uint32_t N) {
  return (1u << 4) | (1u << 7) | (1u << 10) | ((N >> 3) << 17) | ((M >> 4) << 24);
}
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t a, uint64_t b, uint32_t idesc, uint32_t acc) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}" ::"r"(d_tmem),
      "l"(a), "l"(b), "r"(idesc), "r"(acc)
      : "memory");
}

// NVFP4 of one 128-channel row held by this thread, written into its slot:
// per 16-channel group the E4M3 scale sb = E4M3(fp32(fp32(a / 6) * s_enc)) and
// the E2M1 codes of fp32(|y| * s_enc) / sb (exact midpoint comparisons), the
// chunk placement of the page format (msa.h).
__device__ __forceinline__ void store_nvfp4_row(const float (&y)[128], float s_enc, uint8_t* head, int off_c,
                                                int off_s, int t) {
  uint32_t words[16];
#pragma unroll
  for (int gq = 0; gq < 8; ++gq) {
    float a = 0.f;
#pragma unroll
    for (int i = 0; i < 16; ++i) a = fmaxf(a, fabsf(y[16 * gq + i]));
    const uint32_t sb_byte = f32_to_e4m3(__fmul_rn(__fdiv_rn(a, 6.0f), s_enc));
    const float sb = e4m3_to_f32(sb_byte);
    head[off_s + gq * kPageTokens + t] = (uint8_t)sb_byte;
#pragma unroll
    for (int w2 = 0; w2 < 2; ++w2) {
      uint32_t word = 0;
#pragma unroll
      for (int h = 0; h < 2; ++h) {
        uint32_t c[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          const float v = y[16 * gq + 8 * w2 + 4 * h + i];
          c[i] = e2m1_code(__fmul_rn(fabsf(v), s_enc), sb);
          c[i] |= (v < 0.f && c[i]) ? 8u : 0u;
        }
        word |= code_word_part(c, h);
      }
      words[2 * gq + w2] = word;
    }
  }
  uint8_t* row = head + off_c + t * 64;
#pragma unroll
  for (int c = 0; c < 4; ++c)
    *reinterpret_cast<uint4*>(row + 16 * code_chunk_pos(c, t)) =
        make_uint4(words[4 * c], words[4 * c + 1], words[4 * c + 2], words[4 * c + 3]);
}

template <int kHeadsPerCta>
__global__ void __launch_bounds__(kQkvThreads, 2) qkv_fused_kernel(const __grid_constant__ QkvParams p) {
  using Tl = QkvTile<kHeadsPerCta>;
  constexpr int kQkvStages = Tl::kStages;
  constexpr int kOffA = Tl::kOffA, kOffB = Tl::kOffB, kOffGamma = Tl::kOffGamma, kOffBarQ = Tl::kOffBarQ;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  auto full = [&](int i) { return sbase + kOffBarQ + 8 * i; };
  auto empty = [&](int i) { return sbase + kOffBarQ + 8 * (kQkvStages + i); };
  const uint32_t done = sbase + kOffBarQ + 8 * (2 * kQkvStages);
  uint32_t* s_tmem = reinterpret_cast<uint32_t*>(smem + kOffBarQ + 8 * (2 * kQkvStages + 1));
  volatile int* s_abort = reinterpret_cast<volatile int*>(smem + kOffBarQ + 8 * (2 * kQkvStages + 1) + 4);
  int* s_issued = reinterpret_cast<int*>(smem + kOffBarQ + 8 * (2 * kQkvStages + 1) + 8);
  float* s_gamma = reinterpret_cast<float*>(smem + kOffGamma);
  const WaitCtl wc{s_abort, p.wait_ns};
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const int mt = blockIdx.x, hd0 = kHeadsPerCta * blockIdx.y;  // 128-token tile, first output head
  const int n_chunks = p.d_model / kChunk;

  if (tid == 0) {
    for (int i = 0; i < kQkvStages; ++i) {
      mbar_init(full(i), 1);
      mbar_init(empty(i), 1);
    }
    mbar_init(done, 1);
    *s_abort = 0;
    *s_issued = 0;
    fence_barrier_init();
  }
  if (tid < 128) {
    s_gamma[tid] = p.gamma_q[tid];
    s_gamma[128 + tid] = p.gamma_k[tid];
    s_gamma[256 + tid] = p.gamma_idx[tid];
  }
  if (warp == 1) tmem_alloc(smem_u32(s_tmem), 128 * kHeadsPerCta);
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *s_tmem;

  if (warp == 0) {
    if (lane == 0) {
      for (int kc = 0; kc < n_chunks; ++kc) {
        const int st = kc % kQkvStages;
        if (!mbar_wait(empty(st), ((kc / kQkvStages) & 1) ^ 1, wc)) break;
        // (rows past either matrix, the token tail or the 26th head, read as zeros)
        mbar_arrive_expect_tx(full(st), (1 + kHeadsPerCta) * kTileBytes);
        tma_load_2d(sbase + kOffA + st * kTileBytes, &p.tmap_x, kc * kChunk, mt * 128, full(st));
#pragma unroll
        for (int h = 0; h < kHeadsPerCta; ++h)
          tma_load_2d(sbase + kOffB + (st * kHeadsPerCta + h) * kTileBytes, &p.tmap_w, kc * kChunk,
                      (hd0 + h) * 128, full(st));
        *s_issued = kc + 1;
      }
    }
    __syncwarp();
  } else if (warp == 1) {
    if (lane == 0) {
      const uint32_t idesc = umma_idesc_bf16(128, 128 * kHeadsPerCta);
      for (int kc = 0; kc < n_chunks; ++kc) {
        const int st = kc % kQkvStages;
        if (!mbar_wait(full(st), (kc / kQkvStages) & 1, wc)) break;
        tc_fence_after();
        const uint64_t a = umma_desc_sw128(sbase + kOffA + st * kTileBytes);
        // the two heads' W tiles are consecutive: one K-major operand of 256 rows
        const uint64_t b = umma_desc_sw128(sbase + kOffB + st * kHeadsPerCta * kTileBytes);
#pragma unroll
        for (int k = 0; k < 4; ++k)  // K = 16 bf16 = 32 bytes per MMA: +2 in the encoded address
          umma_bf16(tmem, a + 2 * k, b + 2 * k, idesc, (kc | k) != 0);
        umma_commit(empty(st));
      }
      umma_commit(done);  // arrives once every MMA of the tile is complete
    }
    __syncwarp();
  } else {
    // ---- epilogue: thread = token row of the tile ------------------------------
    const int quad = warp & 3, row = 32 * quad + lane;
    const int token = mt * 128 + row;
    const bool ok = mbar_wait(done, 0, wc);
    tc_fence_after();
    // the CTA's heads one after the other (128 accumulator columns each)
    for (int h = 0; h < kHeadsPerCta; ++h) {
      const int hd = hd0 + h;
      if (hd >= kHeadsOut) break;
      float y[128];
      if (ok) {
        uint32_t v[128];
        const uint32_t ta = tmem + ((uint32_t)(32 * quad) << 16) + 128 * h;
        tmem_ld32x32b_x32(ta, v);
        tmem_ld32x32b_x32(ta + 32, v + 32);
        tmem_ld32x32b_x32(ta + 64, v + 64);
        tmem_ld32x32b_x32(ta + 96, v + 96);
        tmem_wait_ld();
#pragma unroll
        for (int i = 0; i < 128; ++i) y[i] = __uint_as_float(v[i]);
      }
      const bool is_q = hd < kQHeads, is_k = hd >= kQHeads && hd < kQHeads + kKvHeads;
      const bool is_v = hd >= kQHeads + kKvHeads && hd < kQHeads + 2 * kKvHeads, is_idx = hd == kHeadsOut - 1;
      if (ok && token < p.n_tokens) {
        if (!is_v) {
          // RMS norm over the head's 128 channels, times the head type's gamma
          float ss = 0.f;
#pragma unroll
          for (int i = 0; i < 128; ++i) ss = fmaf(y[i], y[i], ss);
          const float rn = 1.0f / sqrtf(ss / 128.0f + p.eps);
          const float* gm = s_gamma + (is_q ? 0 : is_k ? 128 : 256);
#pragma unroll
          for (int i = 0; i < 128; ++i) y[i] = y[i] * rn * gm[i];
          // RoPE, channel pairs (i, i + 64) rotated by the angle of pair i at the
          // token's position
          const int pos = p.positions[token];
          if (pos >= 0 && pos < p.max_pos) {
            const float4* cs = reinterpret_cast<const float4*>(p.cos_sin + (size_t)pos * 128);
#pragma unroll
            for (int i4 = 0; i4 < 16; ++i4) {
              const float4 c = __ldg(cs + i4), s = __ldg(cs + 16 + i4);
              const float cc[4] = {c.x, c.y, c.z, c.w}, sn[4] = {s.x, s.y, s.z, s.w};
#pragma unroll
              for (int u = 0; u < 4; ++u) {
                const int i = 4 * i4 + u;
                const float a = y[i], b = y[i + 64];
                y[i] = a * cc[u] - b * sn[u];
                y[i + 64] = b * cc[u] + a * sn[u];
              }
            }
          } else if (lane == 0) {
            set_status(p.status, MSA_STATUS_BAD_SEQ);
          }
        }
        if (p.y_out) {
          float4* dst = reinterpret_cast<float4*>(p.y_out + ((size_t)token * kHeadsOut + hd) * 128);
#pragma unroll
          for (int i = 0; i < 32; ++i) dst[i] = make_float4(y[4 * i], y[4 * i + 1], y[4 * i + 2], y[4 * i + 3]);
        }
        if (is_q) {
          uint8_t* dst = p.q8 + ((size_t)token * kQHeads + hd) * 128;
#pragma unroll
          for (int c = 0; c < 8; ++c) {
            uint32_t w[4];
#pragma unroll
            for (int u = 0; u < 4; ++u) {
              const uint32_t lo = f32x2_to_e4m3x2(y[16 * c + 4 * u], y[16 * c + 4 * u + 1]);
              const uint32_t hi = f32x2_to_e4m3x2(y[16 * c + 4 * u + 2], y[16 * c + 4 * u + 3]);
              w[u] = canon_zero(lo & 0xFF) | (canon_zero(lo >> 8) << 8) | (canon_zero(hi & 0xFF) << 16) |
                     (canon_zero(hi >> 8) << 24);
            }
            *reinterpret_cast<uint4*>(dst + 16 * c) = make_uint4(w[0], w[1], w[2], w[3]);
          }
        } else {
          const int64_t slot = p.slot_mapping[token];
          const int64_t page = slot >= 0 ? slot / kPageTokens : -1;
          const int off = slot >= 0 ? (int)(slot % kPageTokens) : 0;
          if (slot >= 0 && page >= p.n_pages) {
            set_status(p.status, MSA_STATUS_BAD_SLOT);
          } else if (slot >= 0) {
            if (is_idx) {
              uint8_t* dst = p.idx_pool + (size_t)page * kIdxPageBytes + off * kIdxDim;
#pragma unroll
              for (int c = 0; c < 8; ++c) {
                uint32_t w[4];
#pragma unroll
                for (int u = 0; u < 4; ++u) {
                  const uint32_t lo = f32x2_to_e4m3x2(y[16 * c + 4 * u], y[16 * c + 4 * u + 1]);
                  const uint32_t hi = f32x2_to_e4m3x2(y[16 * c + 4 * u + 2], y[16 * c + 4 * u + 3]);
                  w[u] = canon_zero(lo & 0xFF) | (canon_zero(lo >> 8) << 8) | (canon_zero(hi & 0xFF) << 16) |
                         (canon_zero(hi >> 8) << 24);
                }
                *reinterpret_cast<uint4*>(dst + ((c ^ (off & 7)) << 4)) = make_uint4(w[0], w[1], w[2], w[3]);
              }
            } else {
              const int g = hd - (is_k ? kQHeads : kQHeads + kKvHeads);
              uint8_t* head = p.kv_pool + (size_t)page * kKvPageBytes + g * kHeadBytes;
              store_nvfp4_row(y, is_k ? p.s_enc_k : p.s_enc_v, head, is_k ? kOffKc : kOffVc,
                              is_k ? kOffKs : kOffVs, off);
            }
          }
        }
      }
    }
    tc_fence_before();
  }

  // ---- teardown ------------------------------------------------------------------
  tc_fence_before();
  __syncthreads();
  if (*s_abort) {
    if (tid == 0) set_status(p.status, MSA_STATUS_TIMEOUT);
    if (tid == 32) {  // the MMA issuer: its last commit before tensor memory goes
      umma_commit(done);
      mbar_wait_drain(done, 1, p.wait_ns);
    }
    if (tid == 0) {  // the producer: its copies in flight
      const int n = *s_issued;
      for (int kc = max(0, n - kQkvStages); kc < n; ++kc)
        mbar_wait_drain(full(kc % kQkvStages), (kc / kQkvStages) & 1, p.wait_ns);
    }
    __syncthreads();
  }
  if (warp == 1) {
    tc_fence_after();
    tmem_dealloc(tmem, 128 * kHeadsPerCta);
  }
}

PFN_cuTensorMapEncodeTiled_v12000 encode_fn() {
  static PFN_cuTensorMapEncodeTiled_v12000 fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* f = nullptr;
    cudaDriverEntryPointQueryResult q;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &f, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<PFN_cuTensorMapEncodeTiled_v12000>(f);
  });
  return fn;
}

// 2D tensor map of a row-major bf16 matrix [rows][cols], box 64 columns x 128 rows,
// 128-byte swizzle; rows beyond the matrix read as zeros.
bool make_map(CUtensorMap* m, const void* base, int rows, int cols) {
  PFN_cuTensorMapEncodeTiled_v12000 fn = encode_fn();
  if (!fn) return false;
  cuuint64_t dims[2] = {(cuuint64_t)cols, (cuuint64_t)rows};
  cuuint64_t strides[1] = {(cuuint64_t)cols * 2};
  cuuint32_t box[2] = {(cuuint32_t)kChunk, 128};
  cuuint32_t estr[2] = {1, 1};
  return fn(m, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, const_cast<void*>(base), dims, strides, box, estr,
            CU_TENSOR_MAP_INTERLEAVE_NONE, CU_TENSOR_MAP_SWIZZLE_128B, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
            CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE) == CUDA_SUCCESS;
}

// cos / sin table of the RoPE angles, in double precision, rounded to fp32:
// angle(pos, i) = pos * base^(-2 i / 128), i < 64.
__global__ void rope_table_kernel(float* table, int max_pos, double base) {
  const long long id = (long long)blockIdx.x * blockDim.x + threadIdx.x;
  if (id >= (long long)max_pos * 64) return;
  const int pos = (int)(id / 64), i = (int)(id % 64);
  const double ang = (double)pos * pow(base, -2.0 * i / 128.0);
  table[(size_t)pos * 128 + i] = (float)cos(ang);
  table[(size_t)pos * 128 + 64 + i] = (float)sin(ang);
}

}  // namespace

int qkv_heads_out() { return kHeadsOut; }

cudaError_t launch_rope_table(float* table, int max_pos, double base, cudaStream_t stream) {
  if (max_pos == 0) return cudaSuccess;
  const long long n = (long long)max_pos * 64;
  rope_table_kernel<<<(unsigned)((n + 255) / 256), 256, 0, stream>>>(table, max_pos, base);
  return cudaGetLastError();
}

cudaError_t launch_qkv_fused(const msa_cache* c, const void* x, const void* w, int n_tokens, int d_model,
                             const float* gamma_q, const float* gamma_k, const float* gamma_idx,
                             const float* cos_sin, int max_pos, const int* positions,
                             const int64_t* slot_mapping, float eps, uint8_t* q8, float* y_out,
                             cudaStream_t stream) {
  if (n_tokens == 0) return cudaSuccess;
  static DeviceSetup setup;
  int dev = 0, n_sm = 0;
  cudaError_t e = setup.get(&dev, &n_sm, [](int) {
    cudaError_t r = cudaFuncSetAttribute(qkv_fused_kernel<1>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         QkvTile<1>::kSmem + 1024);
    if (r != cudaSuccess) return r;
    return cudaFuncSetAttribute(qkv_fused_kernel<2>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                QkvTile<2>::kSmem + 1024);
  });
  if (e != cudaSuccess) return e;
  QkvParams qp{};
  if (!make_map(&qp.tmap_x, x, n_tokens, d_model) || !make_map(&qp.tmap_w, w, kHeadsOut * 128, d_model))
    return cudaErrorInvalidValue;
  qp.n_tokens = n_tokens;
  qp.d_model = d_model;
  qp.gamma_q = gamma_q;
  qp.gamma_k = gamma_k;
  qp.gamma_idx = gamma_idx;
  qp.cos_sin = cos_sin;
  qp.max_pos = max_pos;
  qp.positions = positions;
  qp.slot_mapping = slot_mapping;
  qp.kv_pool = static_cast<uint8_t*>(c->kv_pool);
  qp.idx_pool = static_cast<uint8_t*>(c->idx_pool);
  qp.n_pages = c->n_pages;
  qp.s_enc_k = c->s_enc_k;
  qp.s_enc_v = c->s_enc_v;
  qp.eps = eps;
  qp.q8 = q8;
  qp.y_out = y_out;
  qp.status = c->status;
  qp.wait_ns = launch_settings().wait_ns;
  // two heads per CTA once that still fills two full waves of two CTAs per SM
  const int tiles = (n_tokens + 127) / 128;
  if ((long long)tiles * ((kHeadsOut + 1) / 2) >= 4ll * n_sm) {
    const dim3 grid(tiles, (kHeadsOut + 1) / 2);
    qkv_fused_kernel<2><<<grid, kQkvThreads, QkvTile<2>::kSmem + 1024, stream>>>(qp);
  } else {
    const dim3 grid(tiles, kHeadsOut);
    qkv_fused_kernel<1><<<grid, kQkvThreads, QkvTile<1>::kSmem + 1024, stream>>>(qp);
  }
  return cudaGetLastError();
}

}  // namespace msa
