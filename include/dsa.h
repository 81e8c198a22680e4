/*
 * dsa.h — C ABI of libdsa.so, the GB300 (sm_103a) DSA decode hot path.
 *
 * DSA ("DeepSeek-style sparse attention") as described in the vLLM Day-0
 * post for Kimi K3.1 Pro, section "K3.1 Pro 中的稀疏注意力" (sparse attention in
 * K3.1 Pro): a small lightning indexer scores every prior token with 32 light
 * heads over a 132-byte FP8 key (128 E4M3 codes + fp32 scale), the 2,048
 * best tokens are kept, and exact MLA attention then runs only over those
 * tokens' 576-byte FP8 latents (or 352-byte NVFP4 latents, see
 * dsa_latent_format_t).  The indexer score is DeepSeek-V3.2's
 *     s[t] = sum_h w[h] * max(0, scale_t * (q_h . k_t))
 * (32 heads x 128 dims, fp32 accumulation and a weighted reduction across
 * heads — same post, AMD section "量化：原生 MXFP4 索引器").
 *
 * The cache is paged and packed ([same post, section "为三类状态服务的 KV 缓存"]):
 * a pool of block rows, each holding one layer's latent page and index-key
 * page for 64 tokens; a block table maps (sequence, logical block) to a row,
 * and the library translates it to page addresses itself on every call.
 *
 * Entry points
 *   dsa_translate_pages      block table -> page addresses
 *   dsa_index_scores(_bf16)  indexer scores (FP8 or MXFP4 keys; fp32 or bf16 out)
 *   dsa_topk(_bf16, _noalloc) top-k per row, ties to the lower index
 *   dsa_topk_paged           the step's top-k, with the selected tokens' physical KV rows
 *   sparse_mla_decode        exact sparse MLA over the selected tokens
 *   dsa_decode_step(_bf16)   the three stages fused on one stream
 *   dsa_cache_append, dsa_quantize_index_query   the step's front end
 *   dsa_index_frontend       the fused indexer front end (norm, projection,
 *                            FP8 query, new tokens into the cache)
 *   dsa_decode_step_frontend the front end and the fused step, one call
 *   dsa_dcp_topk, dsa_dcp_sparse_mla   decode context parallelism (top-k
 *                            merge, partial attention + LSE combine) of W
 *                            token shards, emulated on one GPU
 *   dsa_batch_invariant, dsa_topk_force_multipass   process-wide switches
 *
 * Conventions for every entry point
 *   - All pointers to tensors are DEVICE pointers unless stated otherwise;
 *     the caller owns every buffer, the workspace and the stream.  The
 *     library never allocates, frees or synchronises on the hot path.
 *   - `stream` is a cudaStream_t passed as void* (NULL = legacy default
 *     stream).  Work is enqueued asynchronously, in stream order.
 *   - Host-checkable errors (NULL pointers, misalignment, unsupported sizes,
 *     workspace too small) are returned synchronously and launch nothing.
 *   - Device-detected errors (a block-table entry or token index outside the
 *     cache, a bounded wait that ran out) are written to *dev_status (device
 *     int32) with compare-and-swap from DSA_OK, so the first error wins;
 *     the caller zeroes it and reads it after synchronising.  Outputs of a
 *     call that raised a device error are unspecified.
 *   - A launch failure returns DSA_ERR_CUDA (cudaGetLastError is consumed).
 *   - Row r = b * queries_per_seq + j is query j of sequence b.  With nq
 *     queries per sequence (speculative-verify draft rows) and context L,
 *     row j sees the first L - (nq - 1) + j tokens (causal within the draft).
 */
#ifndef DSA_H_
#define DSA_H_

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

#define DSA_API_VERSION 4
#define DSA_BLOCK_SIZE 64        /* tokens per page */
#define DSA_INDEX_HEADS 32       /* light indexer heads */
#define DSA_INDEX_DIM 128        /* indexer head dim */
#define DSA_MLA_HEADS 96         /* attention heads */
#define DSA_LATENT_DIM 576       /* latent width: keys use all 576 columns */
#define DSA_VALUE_DIM 512        /* values are the first 512 latent columns */
#define DSA_MAX_TOPK 2048        /* top-k of the model; also the largest k accepted */
#define DSA_MAX_QUERIES_PER_SEQ 2048 /* draft rows (1..4) or a prefill chunk (a multiple of 4) */
#define DSA_TOPK_NOALLOC_MAX_ROWS 64  /* row limit of dsa_topk_noalloc */
#define DSA_DCP_MAX_SHARDS 8          /* shards of dsa_dcp_topk and dsa_dcp_sparse_mla */
#define DSA_DCP_MAX_SHARD_TOKENS 65536 /* tokens of one row a shard may hold (16-bit local position) */

typedef enum dsa_status {
  DSA_OK = 0,
  DSA_ERR_INVALID_ARG = 1,   /* NULL pointer, bad size or misaligned buffer */
  DSA_ERR_UNSUPPORTED = 2,   /* valid request this build does not handle */
  DSA_ERR_BOUNDS = 3,        /* block-table entry or token index outside the cache (device) */
  DSA_ERR_TIMEOUT = 4,       /* a bounded in-kernel wait ran out (device) */
  DSA_ERR_CUDA = 5,          /* CUDA launch or runtime error */
  DSA_ERR_WORKSPACE = 6      /* workspace NULL or smaller than the *_workspace_size query */
} dsa_status_t;

typedef enum dsa_key_format {
  DSA_KEY_FP8_E4M3 = 0,      /* 132 B/token: page = 64 x 128 B E4M3 codes, then 64 fp32 scales */
  DSA_KEY_MXFP4 = 1,         /* 68 B/token: page = 64 x 64 B packed E2M1 (element 2i in the low
                                nibble of byte i), then 64 x 4 E8M0 scales (one per 32 elements);
                                no per-token fp32 scale (AMD section: 132 B -> 68 B); the query
                                is E4M3 as for FP8 keys */
  DSA_KEY_MXFP4_NATIVE = 2   /* the MXFP4 page of DSA_KEY_MXFP4 scored against an MXFP4 query by
                                the FP4 x FP4 block-scaled MMA (AMD section: scoring uses native
                                FP4 matrix instructions; fused-decode section: the front end
                                quantises the query to FP8 or MXFP4).  q_index then holds the
                                query's packed E2M1 codes [rows][32][64] followed by its E8M0
                                scales [rows][32][4] (one per 32 dims); head_w is used as given */
} dsa_key_format_t;

typedef enum dsa_latent_format {
  DSA_LATENT_FP8_E4M3 = 0,   /* 576 B/token: page = 64 records of 576 E4M3 codes */
  DSA_LATENT_NVFP4 = 1       /* 352 B/token (packed-cache section: NVFP4 latents): page = 64 records of
                                256 B packed E2M1 for dims 0..511 (element 2i in the low nibble of
                                byte i), 32 E4M3 block scales (one per 16 dims of 0..511), and 64
                                E4M3 codes for dims 512..575 */
} dsa_latent_format_t;

/* One layer's view of the packed paged cache. */
typedef struct dsa_paged_cache {
  void* base;              /* device address of block row 0; 128-byte aligned */
  int64_t row_stride;      /* bytes between block rows; multiple of 128 */
  int64_t latent_off;      /* byte offset of the latent page in a row (64 records); multiple of 128 */
  int64_t index_off;       /* byte offset of the index-key page in a row; multiple of 128 */
  int32_t block_size;      /* tokens per page; must be DSA_BLOCK_SIZE */
  int32_t num_blocks;      /* block rows in the pool (valid table entries are 0..num_blocks-1) */
  int32_t key_format;      /* dsa_key_format_t */
  float latent_scale;      /* per-layer dequantisation scale of the latents: value = latent_scale *
                              e4m3(code), or for NVFP4 dims 0..511 latent_scale * e4m3(block scale)
                              * e2m1(code) */
  int32_t latent_format;   /* dsa_latent_format_t (0 = FP8, the zero-initialised default) */
} dsa_paged_cache_t;

/* The batch of one decode step. */
typedef struct dsa_batch {
  const int32_t* block_table;  /* device int32 [batch][max_blocks_per_seq]; entries past a
                                  sequence's last block are never read */
  const int32_t* seq_lens;     /* device int32 [batch]: context length incl. the current token(s) */
  int32_t max_blocks_per_seq;
  int32_t batch;
  int32_t queries_per_seq;     /* nq: 1 (plain decode), 2..4 (speculative-verify draft rows) or,
                                  for a chunked prefill, a multiple of 4 up to
                                  DSA_MAX_QUERIES_PER_SEQ; row j of a sequence sees its first
                                  seq_len - (nq - 1) + j tokens (causal) */
  int32_t max_seq_len;         /* host-known upper bound of seq_lens; sizes grids and scores */
} dsa_batch_t;

/* Library and status helpers (host only; never fail). */
int32_t dsa_api_version(void);
const char* dsa_status_string(int32_t status);
/* Text of the last CUDA error this thread's calls into the library saw
 * (the reason behind a DSA_ERR_CUDA), or "" if none. */
const char* dsa_last_cuda_error(void);
/* Kernels the library has launched in this process so far (all threads and
 * devices; a memset is not a kernel).  Subtracting two readings around a call
 * gives the kernels that call launched. */
uint64_t dsa_kernel_launches(void);

/*
 * Page translation (Day-0 post, packed-cache section: before every step the
 * block table and cache slots are turned into kernel page addresses).
 * Writes, for every sequence b and logical block j < ceil(seq_len_b / 64),
 * the device byte addresses of its latent page and its index-key page:
 *   latent_pages[b * max_blocks_per_seq + j] = base + row * row_stride + latent_off
 * (likewise index_pages); entries past a sequence's blocks are set to 0.
 * Either output may be NULL.  A table entry outside 0..num_blocks-1 raises
 * DSA_ERR_BOUNDS in *dev_status and yields address 0.  The other entry points
 * translate on the fly and do not need this call.
 */
dsa_status_t dsa_translate_pages(const dsa_paged_cache_t* cache, const dsa_batch_t* batch,
                                 int64_t* latent_pages, int64_t* index_pages,
                                 int32_t* dev_status, void* stream);

/*
 * Lightning-indexer scores (stage 1).
 *   q_index  device E4M3 codes [rows][32][128] (16-byte aligned)
 *   head_w   device fp32 [rows][32]; any query scale is assumed folded into w
 *   scores   device fp32 [rows][ld_scores]; scores[r][t] is written for every
 *            visible t of row r and nothing else is touched
 *   ld_scores >= batch->max_seq_len, multiple of 4
 * FP8 keys: s[t] = sum_h w[h] * max(0, scale_t * (q_h . k_t)).
 * MXFP4 keys: q_h . k_t = sum_{blk<4} 2^(E[t,blk]-127) * sum_{d in blk} q_hd * e2m1(k_td),
 * and scale_t = 1.  Tensor-core accumulation is fp32.
 * rows = batch * queries_per_seq.  MXFP4 keys take one row per sequence, and
 * more than 4 rows per sequence must be a multiple of 4; otherwise, and when
 * batch exceeds 4096 sequences, DSA_ERR_UNSUPPORTED.  Up to 4 rows per
 * sequence share each key read in the decode kernel; a prefill chunk (more
 * than 4 rows, FP8 keys) runs as a dense contraction of 8-row query groups
 * against 512-key blocks (prefill section: the indexer scores every query row
 * of the chunk against the whole context).
 */
dsa_status_t dsa_index_scores(const dsa_paged_cache_t* cache, const dsa_batch_t* batch,
                              const uint8_t* q_index, const float* head_w,
                              float* scores, int64_t ld_scores,
                              int32_t* dev_status, void* stream);

/*
 * Top-k selection (stage 2): for each row r, the min(k, row_lens[r]) tokens
 * with the highest scores among t < row_lens[r]; equal scores go to the
 * lower token index; -0.0 equals +0.0; NaN ranks below every number.
 * idx_out (device int32 [rows][k]) lists them in ascending token order,
 * followed by -1 padding.  The result is unique, hence bit-exact.
 *   scores    device fp32 [rows][ld_scores]
 *   row_lens  device int32 [rows], each <= max_row_len <= ld_scores
 *   k         1 .. DSA_MAX_TOPK
 *   workspace device, >= dsa_topk_workspace_size(rows, max_row_len, k) bytes, 256-B aligned;
 *             that size is 0 (and NULL is accepted) when max_row_len <= k or the rows fit
 *             the on-chip path (max_row_len <= 245,760)
 */
size_t dsa_topk_workspace_size(int32_t rows, int32_t max_row_len, int32_t k);
dsa_status_t dsa_topk(const float* scores, int64_t ld_scores, const int32_t* row_lens,
                      int32_t rows, int32_t max_row_len, int32_t k, int32_t* idx_out,
                      void* workspace, size_t workspace_bytes,
                      int32_t* dev_status, void* stream);

/*
 * Which top-k kernels serve rows longer than 245,760 tokens.  By default
 * (on = 0), in dsa_topk, dsa_topk_paged and the decode steps with fp32
 * scores, such rows take two levels of the cluster kernel over the
 * workspace: the top-k of every segment of at most 163,840 tokens, then the
 * top-k of the row's candidates (two launches).  dsa_topk_noalloc takes one launch of a
 * streaming cluster per row (16 CTAs, or 8 where the device cannot schedule
 * 16); where neither cluster can be scheduled, four kernels over the
 * workspace do the selection.  on != 0 selects the four-kernel path for every
 * later call in this process (all threads and devices), for testing it or for
 * a device shared with work that clusters would contend with.  All paths give
 * the same indices.  Returns the previous setting; never fails.
 */
int32_t dsa_topk_force_multipass(int32_t on);

/*
 * dsa_topk without a workspace argument and without any allocation.  (The
 * source pages have no counterpart; this is a convenience of this library.)
 * Same inputs, outputs, ordering rules and errors as dsa_topk.  It is meant
 * for callers that cannot call cudaMalloc: a host framework that owns the
 * device memory pool and forbids allocations from outside it, or a loop where
 * cudaMalloc/cudaFree must be avoided because they can block or synchronise
 * the device.  The scratch is a 5.5 MiB array of device memory built into the
 * library; every GPU that loads the library holds it until the process ends.
 *   rows <= DSA_TOPK_NOALLOC_MAX_ROWS (64), otherwise DSA_ERR_UNSUPPORTED is
 *   returned and nothing is launched; any row length; k <= DSA_MAX_TOPK.
 * The first call on a device looks up the array's device address (a runtime
 * query, no allocation); make that first call before any stream capture.
 * All calls on a device share the one array: each call clears the parts that
 * must start at zero, but calls whose work overlaps on the GPU (different
 * streams, or concurrent host threads) race and must be serialised.
 */
dsa_status_t dsa_topk_noalloc(const float* scores, int64_t ld_scores, const int32_t* row_lens,
                              int32_t rows, int32_t max_row_len, int32_t k, int32_t* idx_out,
                              int32_t* dev_status, void* stream);

/*
 * Decode context parallelism, the exact top-k merge (Day-0 post,
 * decode-context-parallelism section), emulated on one GPU with `shards` = W
 * token shards: shard r holds the tokens t with t mod W = r.
 *   1. Each shard sends its best ceil(1.5 k / W) tokens, ranked on
 *      bf16-rounded scores, as 32-bit words (the 16-bit order key of the bf16
 *      score above the 16-bit local position t div W).
 *   2. The global top-k is selected from the gathered words by (bf16 key
 *      descending, global token index ascending).
 *   3. A shard whose words were all taken, and which has not sent its full
 *      local top-k, resends its full local top-k, and the selection runs again.
 * The result is the top-k of the bf16-rounded scores (NaN below every number,
 * -0 = +0, ties to the lower index), in ascending token order with -1
 * padding, as from dsa_topk; it differs from dsa_topk's fp32 selection only
 * where scores tie after rounding to bf16.
 *   scores, ld_scores, row_lens, rows, max_row_len, k as for dsa_topk (scores
 *             4-byte aligned; ld_scores >= max_row_len)
 *   shards    1 .. DSA_DCP_MAX_SHARDS; max_row_len <= DSA_DCP_MAX_SHARD_TOKENS
 *             * shards, else DSA_ERR_UNSUPPORTED
 *   stats_out device int32 [rows][3] or NULL: words sent in the first round,
 *             shards that resent, words resent
 *   workspace >= dsa_dcp_topk_workspace_size(rows, k, shards) bytes, 256-B aligned
 * Four launches (candidates, merge, resend candidates, second merge); rows
 * without a resend are written by the first merge.
 */
size_t dsa_dcp_topk_workspace_size(int32_t rows, int32_t k, int32_t shards);
dsa_status_t dsa_dcp_topk(const float* scores, int64_t ld_scores, const int32_t* row_lens, int32_t rows,
                          int32_t max_row_len, int32_t k, int32_t shards, int32_t* idx_out, int32_t* stats_out,
                          void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * Exact sparse MLA decode (stage 3; Day-0 post, sparse-attention section:
 * exact MLA attention restricted to the selected tokens; absorbed form, 96
 * heads).
 * For row r and head h, over the entries i of idx[r] that are >= 0:
 *   c_i       = latent_scale * e4m3(latent row of token idx[r][i])   (576 values)
 *   l_i       = sm_scale * (q[r][h] . c_i)
 *   out[r][h] = sum_i softmax(l)_i * c_i[0:512]        (bf16, round-to-nearest)
 *   lse[r][h] = ln sum_i exp(l_i)                       (fp32; -inf if no entry)
 * Every index must be a visible token of its row; otherwise DSA_ERR_BOUNDS.
 *   q_mla     device bf16 bits [rows][96][576], 16-byte aligned
 *   idx       device int32 [rows][k], k in 1..DSA_MAX_TOPK
 *   out       device bf16 bits [rows][96][512], 8-byte aligned;  lse device fp32 [rows][96]
 *   workspace >= sparse_mla_workspace_size(rows, k) bytes, 256-B aligned
 * Partial results of token chunks are merged through their log-sum-exp
 * (Day-0 post, DCP section: partial outputs combined by LSE).
 */
size_t sparse_mla_workspace_size(int32_t rows, int32_t k);
dsa_status_t sparse_mla_decode(const dsa_paged_cache_t* cache, const dsa_batch_t* batch,
                               const uint16_t* q_mla, const int32_t* idx, int32_t k,
                               float sm_scale, uint16_t* out, float* lse,
                               void* workspace, size_t workspace_bytes,
                               int32_t* dev_status, void* stream);

/*
 * Batch-invariant mode (Day-0 post, section "day 0 的零失配 RL", zero-mismatch
 * RL: with batch-invariant kernels a token's log-prob does not depend on the
 * batch it is computed in).  The indexer and the top-k already give
 * each row the same result whatever the batch; the sparse MLA splits a row's
 * tokens into chunks whose number depends on the number of rows (to fill the
 * SMs), and the merge of the chunks rounds differently for a different split.
 * on != 0 fixes the chunks at 512 tokens for every later call in this process
 * (all threads and devices), so out and lse of a row are bitwise the same in
 * any batch, at the cost of fewer CTAs for small batches.  The workspace
 * sizes reported by sparse_mla_workspace_size and dsa_workspace_size follow
 * the mode at the time of the query: set the mode first, and do not change it
 * while other threads launch.  Returns the previous setting; never fails.
 */
int32_t dsa_batch_invariant(int32_t on);

/*
 * Decode context parallelism, the partial-attention exchange (Day-0 post,
 * decode-context-parallelism section: each GPU attends over its own token
 * shard and the partial outputs are merged through their log-sum-exp),
 * emulated on one GPU with `shards` = W token shards; shard r holds the
 * tokens t with t mod W = r.  For row r and head h, with S_w the entries of
 * idx[r] that are >= 0 and held by shard w:
 *   O_w, LSE_w = the sparse MLA output and LSE over S_w alone (as
 *                sparse_mla_decode defines them), O_w rounded to bf16: what
 *                shard w sends (O_w = 0, LSE_w = -inf for an empty S_w)
 *   lse[r][h]  = ln sum_w exp(LSE_w)
 *   out[r][h]  = sum_w exp(LSE_w - lse[r][h]) * O_w      (bf16, round-to-nearest)
 * This is sparse_mla_decode's result up to the rounding of the O_w to bf16.
 *   cache, batch, q_mla, idx, k, sm_scale, out, lse as for sparse_mla_decode
 *   shards    1 .. DSA_DCP_MAX_SHARDS, else DSA_ERR_UNSUPPORTED
 *   part_out  device bf16 bits [shards][rows][96][512] or NULL: the O_w
 *   part_lse  device fp32 [shards][rows][96] or NULL: the LSE_w
 *   workspace >= dsa_dcp_sparse_mla_workspace_size(rows, k, shards) bytes, 256-B aligned
 * Three launches: grouping of the indices by shard, the MLA kernel over the
 * shards' token groups, and the combine.
 */
size_t dsa_dcp_sparse_mla_workspace_size(int32_t rows, int32_t k, int32_t shards);
dsa_status_t dsa_dcp_sparse_mla(const dsa_paged_cache_t* cache, const dsa_batch_t* batch, const uint16_t* q_mla,
                                const int32_t* idx, int32_t k, int32_t shards, float sm_scale, uint16_t* out,
                                float* lse, uint16_t* part_out, float* part_lse, void* workspace,
                                size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * The fused decode step: page translation, indexer, top-k and sparse MLA on
 * one stream with no host synchronisation (Day-0 post, fused low-latency
 * decode section: a key-balanced scorer and an exact top-k in two kernels,
 * then sparse attention).  Arguments as above; scores_out (fp32
 * [rows][ld_scores]), idx_out (int32 [rows][k]) and phys_out (int32 [rows][k])
 * are optional (NULL: kept in the workspace only).  phys_out receives the
 * physical KV row of each selected token, block_table[b][t / 64] * 64 + t % 64
 * (-1 beside -1 padding): the rows the attention reads (same section: the
 * fused indexer outputs the physical KV rows that attention reads).  When
 * phys_out is given the MLA kernel reads those rows instead of translating the
 * indices again.
 *   workspace >= dsa_workspace_size(batch, k) bytes, 256-B aligned
 */
size_t dsa_workspace_size(const dsa_batch_t* batch, int32_t k);
dsa_status_t dsa_decode_step(const dsa_paged_cache_t* cache, const dsa_batch_t* batch,
                             const uint8_t* q_index, const float* head_w,
                             const uint16_t* q_mla, int32_t k, float sm_scale,
                             uint16_t* out, float* lse,
                             float* scores_out, int64_t ld_scores, int32_t* idx_out, int32_t* phys_out,
                             void* workspace, size_t workspace_bytes,
                             int32_t* dev_status, void* stream);

/*
 * The top-k of the fused step as a call of its own: rows r = b *
 * queries_per_seq + j of the batch with their visible lengths (row j of
 * sequence b sees seq_len_b - (queries_per_seq - 1) + j tokens), the same
 * selection as dsa_topk, and optionally the physical KV rows of the selected
 * tokens through the cache's block table (as phys_out of dsa_decode_step;
 * a table entry outside the pool gives -1 and DSA_ERR_BOUNDS in *dev_status).
 *   scores    device fp32 [rows][ld_scores], ld_scores >= batch->max_seq_len, a multiple of 4
 *   idx_out   device int32 [rows][k];  phys_out device int32 [rows][k] or NULL
 *   workspace >= dsa_topk_workspace_size(rows, batch->max_seq_len, k) bytes, 256-B aligned
 */
dsa_status_t dsa_topk_paged(const dsa_paged_cache_t* cache, const dsa_batch_t* batch, const float* scores,
                            int64_t ld_scores, int32_t k, int32_t* idx_out, int32_t* phys_out, void* workspace,
                            size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * BF16 scores (Day-0 post, decode-context-parallelism section: candidates
 * are picked straight from BF16 scores, and BF16 halves the bytes of the
 * score rows the top-k reads).
 * dsa_index_scores_bf16 is dsa_index_scores with each score rounded to bf16
 * (nearest, ties to even) from the same fp32 value; scores holds bf16 bits
 * [rows][ld_scores].  dsa_topk_bf16 is dsa_topk over bf16 scores (bits),
 * with the same rules: equal scores go to the lower token index, -0 = +0,
 * NaN ranks below every number.  bf16 keeps 8 significant bits, so scores
 * that differ in fp32 can tie in bf16, and a tie at the k-th score goes to
 * the lowest indices: the set can differ from dsa_topk's selection over the
 * fp32 scores wherever a score lies within a bf16 rounding step of the k-th.
 * dsa_decode_step_bf16 is dsa_decode_step with bf16 scores between the
 * indexer and the top-k (scores_out, if not NULL, receives them).
 *   scores    16-byte aligned; ld_scores >= max_row_len (batch->max_seq_len)
 *             and a multiple of 8
 *   dsa_topk_bf16 needs no workspace.  Rows longer than 245,760 tokens take
 *   a cluster of 16 (or 8) CTAs per row; where neither can be scheduled, or
 *   with dsa_topk_force_multipass on, such rows give DSA_ERR_UNSUPPORTED.
 */
dsa_status_t dsa_index_scores_bf16(const dsa_paged_cache_t* cache, const dsa_batch_t* batch,
                                   const uint8_t* q_index, const float* head_w,
                                   uint16_t* scores, int64_t ld_scores,
                                   int32_t* dev_status, void* stream);
dsa_status_t dsa_topk_bf16(const uint16_t* scores, int64_t ld_scores, const int32_t* row_lens, int32_t rows,
                           int32_t max_row_len, int32_t k, int32_t* idx_out, int32_t* dev_status, void* stream);
dsa_status_t dsa_decode_step_bf16(const dsa_paged_cache_t* cache, const dsa_batch_t* batch,
                                  const uint8_t* q_index, const float* head_w,
                                  const uint16_t* q_mla, int32_t k, float sm_scale,
                                  uint16_t* out, float* lse,
                                  uint16_t* scores_out, int64_t ld_scores, int32_t* idx_out, int32_t* phys_out,
                                  void* workspace, size_t workspace_bytes,
                                  int32_t* dev_status, void* stream);

/*
 * New-token cache write: the front end of the fused decode path (Day-0 post,
 * section on the fused low-latency decode path: each step writes the new
 * token's index key and latent into the cache; packed-cache section for the
 * page layout).  For every sequence b and new row j < queries_per_seq, token
 * t = seq_len_b - queries_per_seq + j (the context includes the new tokens)
 * goes to block row block_table[b][t / 64], slot t % 64:
 *   latent (576 values)  codes e4m3(x / latent_scale)
 *   FP8 index key (128)  s = amax / 448 in fp32 (1 if all zero), codes e4m3(x / s),
 *                        s stored as the token's fp32 scale
 *   MXFP4 index key      per 32 elements E = floor(log2 amax) - 2 in [-127, 127]
 *                        (-127 if all zero), codes e2m1(x * 2^-E) packed two per
 *                        byte (element 2i in the low nibble), byte E + 127
 * Rounding: nearest, ties to even; finite values past the largest code saturate.
 *   new_latent     device bf16 bits [batch * queries_per_seq][576]
 *   new_index_key  device bf16 bits [batch * queries_per_seq][128]
 * A table entry outside 0..num_blocks-1 or a length outside the table raises
 * DSA_ERR_BOUNDS in *dev_status and that row is not written.  Rows whose token
 * would precede the sequence start are skipped.
 */
dsa_status_t dsa_cache_append(const dsa_paged_cache_t* cache, const dsa_batch_t* batch,
                              const uint16_t* new_latent, const uint16_t* new_index_key,
                              int32_t* dev_status, void* stream);

/*
 * Indexer query in FP8 (Day-0 post, fused-decode section: the indexer's query
 * is quantised with its scale folded into the head weights).  Per row r and
 * head h: s = amax_d |q[r][h][d]| / 448 in fp32 (1 if all zero),
 * q_index[r][h][d] = e4m3(q / s), head_w_out[r][h] = head_w[r][h] * s.  Since
 * max(0, s * x) = s * max(0, x) for s > 0, the scores of dsa_index_scores on
 * (q_index, head_w_out) are those of the bf16 query up to its FP8 rounding.
 *   q_bf16 device bf16 bits [rows][32][128], 8-byte aligned
 *   head_w / head_w_out device fp32 [rows][32];  q_index device [rows][32][128], 4-byte aligned
 */
dsa_status_t dsa_quantize_index_query(const uint16_t* q_bf16, const float* head_w, int32_t rows,
                                      uint8_t* q_index, float* head_w_out, void* stream);

/*
 * The fused indexer front end (Day-0 post, fused-decode section, second
 * bullet: the query norm, the indexer's query projection, its FP8 or MXFP4
 * quantisation folded into the head weights, and the new token's index key,
 * in one kernel).  For every row r = b * queries_per_seq + j of the batch:
 *   xn[r][i]     = bf16( c_q[r][i] * (1 / sqrt(mean_i c_q[r][i]^2 + eps)) * gamma[i] )
 *                  (RMSNorm in fp32, the product rounded to bf16; the post
 *                  names a "query norm", read as RMSNorm)
 *   q[r][o]      = sum_i w_iq[o][i] * xn[r][i]   for o = h * 128 + d (bf16
 *                  operands, fp32 accumulation)
 *   q_index[r][h][d], head_w_out[r][h]   as dsa_quantize_index_query, from the
 *                  fp32 q: s = amax_d |q| / 448, codes e4m3(q / s), head_w * s;
 *                  for cache->key_format == DSA_KEY_MXFP4_NATIVE the query in
 *                  MXFP4 instead: per head and 32 dims E = floor(log2 amax) - 2
 *                  clamped to [-127, 127] (-127 for an all-zero block), codes
 *                  e2m1(q * 2^-E), scale byte E + 127 (as the MXFP4 keys are
 *                  written), head_w_out = head_w
 *   the row's new token written to the cache exactly as dsa_cache_append does
 *                  (new_latent[r], new_index_key[r])
 * One launch; tcgen05 does the projection.
 *   c_q         device bf16 bits [rows][q_rank], 16-B aligned
 *   q_rank      the compressed query's width D: a multiple of 64, 64 .. 16384,
 *               else DSA_ERR_UNSUPPORTED
 *   gamma       device bf16 bits [q_rank], 16-B aligned;  eps >= 0
 *   w_iq        device bf16 bits [4096][q_rank] (row o = h * 128 + d), 16-B aligned
 *   head_w      device fp32 [rows][32], the head weights before the scale is folded in
 *   new_latent, new_index_key   as for dsa_cache_append
 *   q_index     device [rows][32][128] E4M3 codes (native FP4: [rows][32][64] packed
 *               E2M1, then [rows][32][4] E8M0);  head_w_out device fp32 [rows][32]
 *   q_proj      device fp32 [rows][4096] or NULL: the projected q (for checks)
 * A block-table entry outside the pool raises DSA_ERR_BOUNDS in *dev_status.
 */
dsa_status_t dsa_index_frontend(const dsa_paged_cache_t* cache, const dsa_batch_t* batch, const uint16_t* c_q,
                                int32_t q_rank, const uint16_t* gamma, float eps, const uint16_t* w_iq,
                                const float* head_w, const uint16_t* new_latent, const uint16_t* new_index_key,
                                uint8_t* q_index, float* head_w_out, float* q_proj, int32_t* dev_status,
                                void* stream);

/*
 * A decode step that owns its cache update: dsa_index_frontend (the new
 * tokens into the cache, the indexer query from the compressed query) and
 * then dsa_decode_step over the updated cache, on one stream with no host
 * synchronisation (Day-0 post, fused-decode section: the front end, then the
 * fused indexer and the sparse attention).  The FP8 (or MXFP4) query and the
 * head weights live in the workspace.  Arguments as for the two calls; the step's
 * optional outputs as for dsa_decode_step.
 *   workspace >= dsa_frontend_workspace_size(batch, k) bytes, 256-B aligned
 */
size_t dsa_frontend_workspace_size(const dsa_batch_t* batch, int32_t k);
dsa_status_t dsa_decode_step_frontend(const dsa_paged_cache_t* cache, const dsa_batch_t* batch,
                                      const uint16_t* c_q, int32_t q_rank, const uint16_t* gamma, float eps,
                                      const uint16_t* w_iq, const float* head_w, const uint16_t* new_latent,
                                      const uint16_t* new_index_key, const uint16_t* q_mla, int32_t k,
                                      float sm_scale, uint16_t* out, float* lse, float* scores_out,
                                      int64_t ld_scores, int32_t* idx_out, int32_t* phys_out, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_status, void* stream);

/*
 * Self-test of the bounded in-kernel wait used by every pipelined kernel:
 * launches one CTA that waits on a barrier nothing will ever signal, with a
 * wait limit of `limit_ns` nanoseconds (clamped to 1 ms .. 2 s).  The wait
 * gives up, the kernel writes DSA_ERR_TIMEOUT to *dev_status and returns;
 * the CUDA context stays usable.  No GPU fault or hang is involved.
 */
dsa_status_t dsa_selftest_wait_timeout(int64_t limit_ns, int32_t* dev_status, void* stream);

#ifdef __cplusplus
}  /* extern "C" */
#endif

#endif  /* DSA_H_ */
