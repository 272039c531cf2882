/*
 * msa.h -- C ABI of the block-sparse attention decode path over an NVFP4 KV cache
 * (library libmsa.so, built for sm_103a).
 *
 * What the path computes (sources: "vLLM Delivers Day-0 Support for
 * MiniMax-M3.1-Flash", yuxiaoba.github.io, sections "Sparse attention still
 * scans an index" and "Capacity savings must pay for conversion"; ai4snews
 * article on MiniMax-M3.1-Flash in vLLM, first and third paragraphs;
 * kongchang.com article, "NVFP4 KV Cache and MoE Weights"):
 *   - the KV cache lives in 128-token blocks (pages), K and V stored as NVFP4:
 *     E2M1 values with one E4M3 scale per 16 channels and an fp32 per-tensor
 *     encode scale;
 *   - a lightweight indexer scores every cached token from FP8 index keys
 *     (128 bytes per token), score(t) = sum_h w_h * ReLU(q_h . k_idx(t)),
 *     takes the max per block, keeps the top-16 blocks (ties to the lower block
 *     index) and always the most recent block;
 *   - exact GQA attention (16 query heads over 4 KV heads, head dim 128) runs
 *     over the selected tokens only, FP8 E4M3 queries against K/V dequantised
 *     from NVFP4 to FP8, with an fp32 online softmax split over the context and
 *     merged by log-sum-exp.
 *
 * Conventions shared by every entry point:
 *   - Pointers are DEVICE pointers unless a parameter says "host".  The library
 *     never allocates, frees or synchronises (msa_read_status excepted); all
 *     work is enqueued on `stream` (a cudaStream_t; NULL = legacy stream).
 *   - Return value: MSA_OK (0) when the work was enqueued, or a negative
 *     MSA_ERR_* code when host-side validation failed (nothing is enqueued).
 *   - Data errors that only the device can see (a physical page id outside the
 *     pool, a sequence with more query tokens than cached tokens, ...) OR a
 *     MSA_STATUS_* bit into the cache's device status word; the offending item
 *     is skipped.  No kernel traps, asserts or waits without a bound.
 *   - Supported shape: 128-token pages, 4 KV heads, head dim 128, index dim
 *     128, 8 indexer heads, 16 query heads (GQA group 4).  Anything else is
 *     MSA_ERR_UNSUPPORTED_SHAPE.
 *
 * Page formats (one physical page id p addresses both pools):
 *   KV page p at kv_pool + p * 73,728 bytes = 4 heads x 18,432 bytes; head g
 *   at offset g * 18,432:
 *     +0       K codes  [128 tokens][64 B]: little-endian 32-bit word i of a
 *              row holds channels 8i..8i+7 as E2M1 codes (sign s, magnitude m):
 *              m of channel 8i+n at bits 4n..4n+2 (n = 0..7), s of channel 8i+n
 *              at bit 8n+7 and s of channel 8i+4+n at bit 8n+3 (n = 0..3); the
 *              16-byte chunk c (channels 32c..32c+31) of token t is stored at
 *              chunk position c XOR ((t >> 1) mod 4) of its row
 *     +8,192   K scales [8 groups][128 tokens]: E4M3 scale of channels 16k..16k+15
 *     +9,216   V codes  [128 tokens][64 B], chunks placed like the K codes
 *     +17,408  V scales [8 groups][128 tokens]
 *   (576 bytes per token and layer: the 34,560 bytes/token of the ai4snews
 *   article over the model's layers.)
 *   Index page p at idx_pool + p * 16,384 bytes = [128 tokens][128 B] E4M3
 *   index keys; the 16-byte chunk c of token t's row (dims 16c..16c+15) is
 *   stored at chunk position c XOR (t mod 8).
 *
 * Sequences and query tokens: sequence b has seq_lens[b] cached tokens (the
 * new query tokens already inserted) and q_start_loc[b+1] - q_start_loc[b]
 * query tokens; query token j of b sits at position
 * pos_j = seq_lens[b] - n_q + j, sees keys at positions <= pos_j, and its
 * recent block is r_j = pos_j / 128.  block_table[b * max_pages + i] is the
 * physical page of logical block i of sequence b.
 */
#ifndef MSA_H
#define MSA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef struct CUstream_st* msa_stream_t; /* same type as cudaStream_t */

/* Host-side return codes. */
#define MSA_OK 0
#define MSA_ERR_INVALID_ARG (-1)      /* null pointer, negative size, ... */
#define MSA_ERR_UNSUPPORTED_SHAPE (-2)
#define MSA_ERR_WORKSPACE_TOO_SMALL (-3)
#define MSA_ERR_LAUNCH_FAILED (-4)    /* a kernel launch returned an error */
#define MSA_ERR_SCRATCH_CAPACITY (-5) /* msa_indexer_topk_noalloc: shape beyond its static scratch */

/* Bytes of the static scratch behind msa_indexer_topk_noalloc. */
#define MSA_INDEXER_NOALLOC_SCRATCH_BYTES ((size_t)8 << 20)

/* Sticky device status bits (OR-ed into *msa_cache.status). */
#define MSA_STATUS_BAD_SLOT 0x1       /* slot_mapping points outside the pool */
#define MSA_STATUS_BAD_PAGE 0x2       /* block_table entry outside the pool */
#define MSA_STATUS_BAD_SEQ 0x4        /* n_q < 0, n_q > seq_len or seq_len > max_pages*128 */
#define MSA_STATUS_BAD_SELECTION 0x8  /* a selected block id outside 0..r_j */
#define MSA_STATUS_TIMEOUT 0x10       /* a bounded on-chip wait gave up (results invalid) */
/* Every on-chip wait is bounded (2 s by default): a wait that runs out sets
 * MSA_STATUS_TIMEOUT, the kernel abandons its work, waits (bounded) for its own
 * copies and tensor-core operations in flight, releases tensor memory and
 * returns.  The context stays usable. */

/* The KV cache and its metadata.  Caller-owned; the library only reads it. */
typedef struct msa_cache {
  void* kv_pool;        /* device, n_pages * 73,728 bytes (format above) */
  void* idx_pool;       /* device, n_pages * 16,384 bytes (format above) */
  int64_t n_pages;      /* physical pages in both pools */
  int32_t page_tokens;  /* must be 128 */
  int32_t n_kv_heads;   /* must be 4 */
  int32_t head_dim;     /* must be 128 */
  int32_t idx_dim;      /* must be 128 */
  float s_enc_k;        /* host value: fp32 per-tensor encode scale of K, > 0 */
  float s_enc_v;        /* host value: fp32 per-tensor encode scale of V, > 0 */
  int32_t* status;      /* device int32, sticky MSA_STATUS_* bits; may be NULL */
} msa_cache;

/*
 * Quantise new tokens to NVFP4 / FP8 and write them into their cache slots.
 * (NVFP4 KV cache: ai4snews article, first and third paragraphs; index keys of
 * 128 FP8 bytes per token: blog, "Sparse attention still scans an index".)
 *
 *   k, v         fp32 [n_tokens][4][128], row-major, contiguous.
 *   idx_k        fp32 [n_tokens][128] index keys.
 *   slot_mapping int64 [n_tokens]: page * 128 + offset; a negative entry skips
 *                the token.  A page >= n_pages sets MSA_STATUS_BAD_SLOT.
 * Per (token, head, 16-channel group) with s = s_enc_k (K) or s_enc_v (V):
 *   a = max|x|, sb = E4M3_RNE_satfinite(fp32(fp32(a / 6) * s)),
 *   code = E2M1 round-to-nearest-even (ties to the even code, saturating at 6)
 *          of fp32(|x| * s) / sb evaluated exactly, sign on non-zero codes only,
 *          all codes 0 when sb == 0.
 * Index keys: E4M3_RNE_satfinite(x); a zero result is stored as 0x00.
 * Slots written by one call must be distinct.
 */
int msa_quantize_kv_insert(const msa_cache* cache, const float* k, const float* v,
                           const float* idx_k, const int64_t* slot_mapping,
                           int32_t n_tokens, msa_stream_t stream);

/*
 * Indexer scan and top-k selection (blog, "Sparse attention still scans an
 * index": 16 blocks plus the most recent one; "Parallelize index work across
 * context": the split scan keeps the selection exact).
 *
 *   q_idx       E4M3 [n_q_total][n_idx_heads = 8][128] index queries.
 *   w           fp32 [n_q_total][8] head weights (>= 0 for the ReLU reading).
 *   block_table int32 [n_seqs][max_pages]; seq_lens int32 [n_seqs];
 *   q_start_loc int32 [n_seqs + 1], non-decreasing, q_start_loc[0] = 0,
 *               q_start_loc[n_seqs] = n_q_total.
 *   topk        must be 16.
 *   sel         int32 [n_q_total][topk + 1] out: min(topk, r_j) selected block
 *               ids of blocks 0..r_j-1 (highest block score first wins, ties to
 *               the lower id) in ascending order, then r_j; padded with -1.
 *   n_sel       int32 [n_q_total] out: min(topk, r_j) + 1.
 *   ws, ws_bytes scratch of at least msa_indexer_workspace_bytes(...) bytes,
 *               16-byte aligned, ZEROED before its first use.  Its first 256
 *               bytes hold grid-barrier words; every call, also one whose
 *               barrier timed out, leaves them at rest (a generation count
 *               apart), so later calls need no clearing.  From
 *               byte 256, after the stream reaches the end of this call, it holds
 *               for every query token j and block i < r_j four fp32 partial
 *               maxima P[j][i][0..3] (row stride 4 * max_pages floats): the maxima
 *               over the block's token quarters; the block score is their max.
 *               Other entries are unspecified.  Calls sharing a workspace must
 *               not overlap on the GPU.
 * Block score S[j][i] = max over the 128 tokens t of block i of
 *   sum_h w[j][h] * max(0, q_idx[j][h] . key(t)), computed with fp32 sums of
 *   exact FP8 products.
 * n_seqs <= 4096.
 */
int msa_indexer_topk(const msa_cache* cache, const uint8_t* q_idx, const float* w,
                     int32_t n_idx_heads, const int32_t* block_table, int32_t max_pages,
                     const int32_t* seq_lens, const int32_t* q_start_loc, int32_t n_seqs,
                     int32_t n_q_total, int32_t topk, int32_t* sel, int32_t* n_sel,
                     void* ws, size_t ws_bytes, msa_stream_t stream);

/*
 * Context-split indexer (blog, "Parallelize index work across context": each
 * GPU scans a part of the context, the local candidates are exchanged, and
 * merging them gives the final top-16 exactly: every block competes once,
 * with the same score, in one part).  The two calls below let a caller run
 * each part where its index pages live and merge anywhere.
 *
 * msa_indexer_topk_range: msa_indexer_topk restricted to the logical blocks
 * [blk_lo, blk_hi) (0 <= blk_lo <= blk_hi) of every sequence: for query token
 * j, only blocks i with blk_lo <= i < min(blk_hi, r_j) are scanned and
 * compete; instead of sel / n_sel it writes
 *   cand  uint64 [n_q_total][16] out: the local top-16 as keys, best first,
 *         zero-padded (fewer than 16 blocks in the range: all of them).
 *         key = (ordered(S) << 32) | (0xFFFFFFFF - block), where ordered(x)
 *         is the fp32 bit pattern of x with the sign bit set for x >= +0 and
 *         all bits inverted for x < 0; a larger key is a higher score, then
 *         a lower block; 0 = no block.
 * Only the block-table entries of the range are read.  Workspace and every
 * other argument as msa_indexer_topk (its scores are written for the blocks
 * of the range only).
 *
 * msa_indexer_merge_candidates: cand holds n_shards (1..64) such arrays,
 * [n_shards][n_q_total][16], whose block ranges are disjoint; per query token
 * the 16 largest non-zero keys win and sel / n_sel are written exactly as
 * msa_indexer_topk writes them (winners ascending, then r_j, -1 padding;
 * n_sel = winners + 1).  When the ranges tile [0, r_j) of every token, the
 * result equals msa_indexer_topk's.  Status bits go to cache->status (the
 * cache's pools are not read): MSA_STATUS_BAD_SEQ for an inconsistent
 * sequence, MSA_STATUS_BAD_SELECTION for a key whose block is not below r_j.
 * Launched as a programmatic dependent of the previous kernel in the stream.
 */
int msa_indexer_topk_range(const msa_cache* cache, const uint8_t* q_idx, const float* w,
                           int32_t n_idx_heads, const int32_t* block_table, int32_t max_pages,
                           const int32_t* seq_lens, const int32_t* q_start_loc, int32_t n_seqs,
                           int32_t n_q_total, int32_t topk, int32_t blk_lo, int32_t blk_hi,
                           uint64_t* cand, void* ws, size_t ws_bytes, msa_stream_t stream);
int msa_indexer_merge_candidates(const msa_cache* cache, const uint64_t* cand, int32_t n_shards,
                                 const int32_t* seq_lens, const int32_t* q_start_loc,
                                 int32_t n_seqs, int32_t max_pages, int32_t n_q_total,
                                 int32_t topk, int32_t* sel, int32_t* n_sel, msa_stream_t stream);

/* Bytes of scratch msa_indexer_topk needs (a multiple of 256). */
size_t msa_indexer_workspace_bytes(int32_t n_q_total, int32_t max_pages);

/*
 * msa_indexer_topk without a workspace argument, for callers that cannot
 * allocate device memory: code that runs inside a host framework which owns
 * every device allocation, real-time decode loops where a cudaMalloc (which
 * may synchronise the device) is not allowed between steps, or plug-ins that
 * receive only their input and output buffers.  The pages have no counterpart
 * of this call; it is a deployment convenience.
 *
 * Same arguments, results and errors as msa_indexer_topk minus ws/ws_bytes.
 * The scratch is a file-scope device array of MSA_INDEXER_NOALLOC_SCRATCH_BYTES
 * (8 MiB) inside the library; every GPU that loads the library keeps it until
 * the process exits.  Shapes that need more, i.e.
 * msa_indexer_workspace_bytes(n_q_total, max_pages) > that capacity, return
 * MSA_ERR_SCRATCH_CAPACITY and enqueue nothing.  Nothing in the array needs
 * clearing by the caller: every score entry a call reads was written earlier
 * by that same call.
 * The array is shared by all calls on a device and keeps the last call's
 * contents, so calls whose kernels overlap on the GPU (e.g. on two streams
 * without ordering) race and must not be issued.  The first call on each
 * device looks up the array's device address (with that device current);
 * make that first call before any stream capture.  No cudaMalloc, cudaFree
 * or allocating routine is called.  (The array starts zeroed when the library
 * is loaded; its grid-barrier words return to rest after every call, also
 * after one that timed out.)
 */
int msa_indexer_topk_noalloc(const msa_cache* cache, const uint8_t* q_idx, const float* w,
                             int32_t n_idx_heads, const int32_t* block_table, int32_t max_pages,
                             const int32_t* seq_lens, const int32_t* q_start_loc, int32_t n_seqs,
                             int32_t n_q_total, int32_t topk, int32_t* sel, int32_t* n_sel,
                             msa_stream_t stream);


/*
 * Split-context sparse GQA attention over the selected blocks (blog, "Sparse
 * attention still scans an index": exact attention over the selected blocks;
 * ai4snews article, third paragraph: FP8 queries, NVFP4 K/V dequantised to FP8
 * before the matmul).
 *
 *   q           E4M3 [n_q_total][n_q_heads = 16][128] queries.
 *   sel, n_sel  as written by msa_indexer_topk (any ascending or unordered
 *               list of distinct block ids <= r_j is accepted).
 *   n_splits    1..64: the selected blocks of each query token are dealt
 *               round-robin to n_splits partial attentions.
 *   o_part      fp32 [n_q_total][n_splits][16][128] out: each split's
 *               normalised output (zero for an empty split).
 *   lse_part    fp32 [n_q_total][n_splits][16] out: natural-log sum of exp of
 *               the split's logits (-inf for an empty split).
 * Per element the FP8 operand is sign(code) | E4M3_RNE(|e2m1(code)| * sb);
 * logits = (q . k8) * softmax_scale / s_enc_k; the value contraction is
 * divided by s_enc_v.  Keys after pos_j are masked.  Limits: n_seqs <= 4096,
 * n_q_total <= 65535 (else MSA_ERR_UNSUPPORTED_SHAPE).
 * Launched as a programmatic dependent of the previous kernel in the stream
 * (msa_indexer_topk lets it start early): it waits for that kernel before it
 * reads sel and n_sel, but copies q_start_loc before the wait, so the kernel
 * just before it must not write q_start_loc.
 */
int msa_sparse_attn_decode(const msa_cache* cache, const uint8_t* q, int32_t n_q_heads,
                           float softmax_scale, const int32_t* sel, const int32_t* n_sel,
                           const int32_t* block_table, int32_t max_pages,
                           const int32_t* seq_lens, const int32_t* q_start_loc,
                           int32_t n_seqs, int32_t n_q_total, int32_t n_splits,
                           float* o_part, float* lse_part, msa_stream_t stream);

/*
 * Log-sum-exp merge of the split partials (blog, "Sparse attention still scans
 * an index": attention over the selected blocks is exact; a split computes it
 * over part of them, and the parts combine by their softmax normalisers):
 *   out[j][h] = sum_s exp(lse[j][s][h] - L) * o_part[j][s][h],
 *   L = log sum_s exp(lse[j][s][h]).
 *   out  fp32 [n_q_total][n_q_heads][128].  A row whose splits are all empty
 *        is written as zeros.
 *   lse  fp32 [n_q_total][n_q_heads] out, or NULL: the merged L (-inf for a
 *        row whose splits are all empty), so that merged results can be merged
 *        again.
 * Limits: n_q_heads <= 1024, n_q_total <= 65535 (else MSA_ERR_UNSUPPORTED_SHAPE).
 */
int msa_merge_splits(const float* o_part, const float* lse_part, int32_t n_q_total,
                     int32_t n_q_heads, int32_t n_splits, float* out, float* lse,
                     msa_stream_t stream);

/*
 * The whole decode step in ONE launch, for low concurrency (blog, "AMD uses
 * different conversion and communication mechanisms": a separate
 * single-kernel strategy reduces launches at low concurrency; "Keep capacity,
 * layer, and system results separate": that advantage need not hold at high
 * concurrency, where msa_indexer_topk + msa_sparse_attn_decode +
 * msa_merge_splits stay the faster path).  Computes exactly what those three
 * calls compute, with the same rounding: the selection into sel / n_sel (as
 * msa_indexer_topk) and the merged output
 *   out fp32 [n_q_total][16][128].
 * One cooperative launch of at most one CTA per SM runs the scan, the top-k,
 * the attention (one page per work item, each selected block a split) and the
 * merge, with a bounded grid barrier between phases.
 *   ws, ws_bytes  scratch of at least msa_decode_fused_workspace_bytes(n_q_total,
 *                 max_pages) bytes, 16-byte aligned, ZEROED before its first use
 *                 (its first 256 bytes hold grid-barrier words that every call,
 *                 also one that timed out, leaves at rest).  Calls sharing a
 *                 workspace must not overlap on the GPU.
 * Other arguments as msa_indexer_topk and msa_sparse_attn_decode.  Limits:
 * n_seqs <= 64, n_q_total <= 64 (else MSA_ERR_UNSUPPORTED_SHAPE).
 */
int msa_decode_fused(const msa_cache* cache, const uint8_t* q, const uint8_t* q_idx, const float* w,
                     int32_t n_q_heads, int32_t n_idx_heads, float softmax_scale,
                     const int32_t* block_table, int32_t max_pages, const int32_t* seq_lens,
                     const int32_t* q_start_loc, int32_t n_seqs, int32_t n_q_total, int32_t topk,
                     int32_t* sel, int32_t* n_sel, float* out, void* ws, size_t ws_bytes,
                     msa_stream_t stream);
size_t msa_decode_fused_workspace_bytes(int32_t n_q_total, int32_t max_pages);

/*
 * Fused QKV projection -> RMS norm -> RoPE -> FP8 queries and cache insertion
 * (blog, "Reduce both data movement and resource waits": fusing the projection
 * with normalisation, RoPE and cache insertion avoids writing the intermediate
 * tensor to HBM and reading it back).  The projection's accumulators stay on
 * the SM; nothing but the outputs below is written.
 *
 *   x          bf16 [n_tokens][d_model] hidden states, row-major, 16-byte aligned;
 *              d_model a multiple of 64 (64 .. 65,536).
 *   w          bf16 [25 * 128][d_model] projection (row = output channel),
 *              16-byte aligned: heads 0-15 queries, 16-19 keys, 20-23 values,
 *              24 the index key (MSA_QKV_HEADS = 25 heads of 128).
 *   gamma_q, gamma_k, gamma_idx  fp32 [128] RMS-norm gains of each head kind.
 *   cos_sin    fp32 [max_pos][128]: cos of the 64 pair angles, then their sin
 *              (msa_rope_table writes it); positions int32 [n_tokens] index it
 *              (a position outside [0, max_pos) leaves the head unrotated and
 *              sets MSA_STATUS_BAD_SEQ).
 *   slot_mapping int64 [n_tokens] as msa_quantize_kv_insert (negative: skip).
 *   q8         uint8 [n_tokens][16][128] out: E4M3 queries (RNE, satfinite).
 *   y_out      fp32 [n_tokens][25][128] out, or NULL: every head's row just
 *              before rounding (diagnostic).
 * Per token: z = W x (fp32 accumulation of bf16 products); query, key and
 * index-key heads y = RoPE(z / sqrt(mean(z^2) + eps) * gamma), channel pairs
 * (i, i + 64) turned by the table's angle i: (a, b) -> (a cos - b sin,
 * b cos + a sin); value heads y = z.  Queries -> q8; keys and values -> NVFP4
 * in the slot, exactly the quantiser of msa_quantize_kv_insert with the
 * cache's s_enc_k / s_enc_v; index keys -> E4M3 in the index page.
 */
#define MSA_QKV_HEADS 25
int msa_qkv_project_insert(const msa_cache* cache, const void* x, const void* w, int32_t n_tokens,
                           int32_t d_model, const float* gamma_q, const float* gamma_k,
                           const float* gamma_idx, const float* cos_sin, int32_t max_pos,
                           const int32_t* positions, const int64_t* slot_mapping, float eps,
                           uint8_t* q8, float* y_out, msa_stream_t stream);
/* RoPE table for msa_qkv_project_insert: cos_sin[pos][i] = cos(pos * base^(-2i/128))
 * and cos_sin[pos][64 + i] = the sin, i < 64, computed in double precision and
 * rounded to fp32 (base > 1, e.g. 10,000). */
int msa_rope_table(float* cos_sin, int32_t max_pos, double base, msa_stream_t stream);

/*
 * Block-outer transfer rows (blog, "AMD uses different conversion and
 * communication mechanisms": a KV block kept as one contiguous row is moved in
 * one read instead of one read per page).  The row of a block holds, for every
 * layer l = 0 .. n_layers-1 in order, that layer's KV page (73,728 bytes, the
 * format above) followed by its index page (16,384 bytes): 90,112 bytes per
 * layer, msa_block_row_bytes(n_layers) per row.
 *
 *   layers   HOST array of n_layers caches (1 <= n_layers <= 128), one per
 *            model layer; block i lives at the same physical page pages[i] in
 *            every layer's pools.
 *   pages    int32 [n_blocks] physical page of each block.  A page outside a
 *            layer's pool sets MSA_STATUS_BAD_PAGE in layers[0].status and that
 *            (block, layer) part of the row is left untouched.
 *   rows     uint8 [n_blocks][msa_block_row_bytes(n_layers)], 16-byte aligned.
 * msa_pack_blocks copies pages -> rows; msa_unpack_blocks copies rows -> pages
 * (so a receiver may place a block at different page ids).  Rows and pages
 * must not overlap; the pages listed in one unpack call must be distinct.
 */
int msa_pack_blocks(const msa_cache* layers, int32_t n_layers, const int32_t* pages,
                    int32_t n_blocks, uint8_t* rows, msa_stream_t stream);
int msa_unpack_blocks(const msa_cache* layers, int32_t n_layers, const uint8_t* rows,
                      const int32_t* pages, int32_t n_blocks, msa_stream_t stream);
/* Bytes of one block-outer row: n_layers * 90,112 (0 for n_layers <= 0). */
size_t msa_block_row_bytes(int32_t n_layers);

/*
 * Helpers for the per-tensor scale.  msa_absmax folds max|x[i]| over n fp32
 * values into *amax (device float, caller-initialised to 0): call it on every
 * chunk of a tensor, then msa_encode_scale(amax) returns the fp32 encode scale
 * 448 / amax (1 for amax == 0).
 */
int msa_absmax(const float* x, int64_t n, float* amax, msa_stream_t stream);
float msa_encode_scale(float amax);

/*
 * Diagnostic: the FP8 operands the attention kernel multiplies, for one page.
 * k8, v8: uint8 [4 heads][128 tokens][128 channels] out, E4M3 bytes in
 * logical channel order, produced by the same device dequantiser as
 * msa_sparse_attn_decode.
 */
int msa_debug_fp8_page(const msa_cache* cache, int64_t page, uint8_t* k8, uint8_t* v8,
                       msa_stream_t stream);

/*
 * Test hook for the failure paths (the pages have no counterpart).  Sets, for
 * every later launch of the library in this process, the time limit of one
 * bounded on-chip wait (wait_limit_ns; 0 restores the default of 2 s) and the
 * fault-injection flags (0 = none):
 *   MSA_INJECT_BARRIER_TIMEOUT  the indexer's grid barrier waits for one CTA
 *                               more than the launch has, so every CTA's wait
 *                               runs out after wait_limit_ns: the call sets
 *                               MSA_STATUS_TIMEOUT, leaves sel/n_sel unwritten
 *                               and its workspace barrier word at rest;
 *   MSA_INJECT_ATTENTION_TIMEOUT  every CTA of the attention kernel leaves out
 *                               the copy of its first page, so the waits for it
 *                               run out after wait_limit_ns: the call sets
 *                               MSA_STATUS_TIMEOUT, its CTAs release tensor
 *                               memory only after their copies and tensor-core
 *                               products in flight are done, and return.
 * Launches already captured into a CUDA graph keep the settings they were
 * captured with.  Unknown flags return MSA_ERR_INVALID_ARG.
 */
#define MSA_INJECT_BARRIER_TIMEOUT 0x1
#define MSA_INJECT_ATTENTION_TIMEOUT 0x2
int msa_debug_set_fault_injection(int32_t flags, uint64_t wait_limit_ns);

/* Copies the device status word to *host_out (synchronous on the stream). */
int msa_read_status(const msa_cache* cache, int32_t* host_out, msa_stream_t stream);

/* Static description of a return code or status bit set. */
const char* msa_status_string(int code);

#ifdef __cplusplus
}
#endif

#endif /* MSA_H */
