// Block-outer transfer rows: pack the pages of a list of blocks, from every
// layer's pools, into one contiguous row per block, and unpack rows back.
//
// "vLLM Delivers Day-0 Support for MiniMax-M3.1-Flash" blog, section "AMD
// uses different conversion and communication mechanisms": a KV block split
// over many pages needs many reads to move; a block-outer layout stores the
// block as one contiguous row, moved in one read.  A row here holds, layer by
// layer, the block's KV page (73,728 bytes) and index page (16,384 bytes):
// n_layers x 90,112 bytes.
//
// Pure data movement, bound by HBM: unit = one (block, layer) = 90,112 bytes
// read and 90,112 written.  A persistent grid of CTAs takes units in turn;
// each thread moves 16-byte chunks, eight loads in flight before their
// stores, streaming past L1 on the way in and marked evict-first on the way
// out (the rows are consumed by a transfer, not by this GPU's next kernel).
#include "common.cuh"

namespace msa {
namespace {

constexpr int kRowLayerBytes = kKvPageBytes + kIdxPageBytes;  // 90,112
constexpr int kChunks = kRowLayerBytes / 16;                  // 5,632
constexpr int kKvChunks = kKvPageBytes / 16;                  // 4,608
constexpr int kXferThreads = 256;
constexpr int kInFlight = 8;

struct XferParams {
  uint8_t* kv[kMaxLayers];
  uint8_t* idx[kMaxLayers];
  int64_t n_pages[kMaxLayers];
  int n_layers;
  const int* pages;  // [n_blocks] physical page of each block (every layer)
  int n_blocks;
  uint8_t* rows;     // [n_blocks][n_layers][90,112]
  int* status;
};

__device__ __forceinline__ void st_stream_v4(void* p, uint4 v) {
  asm volatile("st.global.cs.v4.u32 [%0], {%1,%2,%3,%4};" ::"l"(p), "r"(v.x), "r"(v.y), "r"(v.z), "r"(v.w)
               : "memory");
}

// Chunk c of the layer part of a row: KV page bytes first, then the index page.
__device__ __forceinline__ uint8_t* page_chunk(const XferParams& p, int layer, int64_t page, int c) {
  return c < kKvChunks ? p.kv[layer] + page * kKvPageBytes + 16 * c
                       : p.idx[layer] + page * kIdxPageBytes + 16 * (c - kKvChunks);
}

template <bool kPack>
__global__ void __launch_bounds__(kXferThreads) block_rows_kernel(XferParams p) {
  const long long n_units = (long long)p.n_blocks * p.n_layers;
  for (long long u = blockIdx.x; u < n_units; u += gridDim.x) {
    const int blk = (int)(u / p.n_layers), layer = (int)(u % p.n_layers);
    const int64_t page = p.pages[blk];
    if (page < 0 || page >= p.n_pages[layer]) {
      if (threadIdx.x == 0) set_status(p.status, MSA_STATUS_BAD_PAGE);
      continue;
    }
    uint8_t* row = p.rows + (size_t)u * kRowLayerBytes;
    for (int c0 = threadIdx.x; c0 < kChunks; c0 += kInFlight * kXferThreads) {
      uint4 v[kInFlight];
#pragma unroll
      for (int k = 0; k < kInFlight; ++k) {
        const int c = c0 + k * kXferThreads;
        if (c < kChunks) v[k] = ld_stream_v4(kPack ? page_chunk(p, layer, page, c) : row + 16 * c);
      }
#pragma unroll
      for (int k = 0; k < kInFlight; ++k) {
        const int c = c0 + k * kXferThreads;
        if (c < kChunks) {
          if (kPack) st_stream_v4(row + 16 * c, v[k]);
          else *reinterpret_cast<uint4*>(page_chunk(p, layer, page, c)) = v[k];
        }
      }
    }
  }
}

}  // namespace

cudaError_t launch_block_rows(const msa_cache* layers, int n_layers, const int* pages, int n_blocks,
                              uint8_t* rows, bool pack, cudaStream_t stream) {
  if (n_blocks == 0) return cudaSuccess;
  static DeviceSetup setup;
  int dev = 0, n_sm = 0;
  cudaError_t e = setup.get(&dev, &n_sm, [](int) { return cudaSuccess; });
  if (e != cudaSuccess) return e;
  XferParams xp{};
  for (int l = 0; l < n_layers; ++l) {
    xp.kv[l] = static_cast<uint8_t*>(layers[l].kv_pool);
    xp.idx[l] = static_cast<uint8_t*>(layers[l].idx_pool);
    xp.n_pages[l] = layers[l].n_pages;
  }
  xp.n_layers = n_layers;
  xp.pages = pages;
  xp.n_blocks = n_blocks;
  xp.rows = rows;
  xp.status = layers[0].status;
  // four CTAs of 256 threads per SM: 1,024 threads x 8 chunks of 16 bytes in flight
  const long long units = (long long)n_blocks * n_layers;
  const int grid = (int)(units < 4LL * n_sm ? units : 4LL * n_sm);
  if (pack) block_rows_kernel<true><<<grid, kXferThreads, 0, stream>>>(xp);
  else block_rows_kernel<false><<<grid, kXferThreads, 0, stream>>>(xp);
  return cudaGetLastError();
}

}  // namespace msa
