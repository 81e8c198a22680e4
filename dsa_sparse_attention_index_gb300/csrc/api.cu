// api.cu — the C ABI of libdsa.so: argument validation, workspace layout and
// the stream-ordered composition of the kernels.  No allocation, no host
// synchronisation on any entry point.
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace dsa {

int num_sms() {
  static std::atomic<int> cache[64];  // zero: not yet asked
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 0 && dev < 64 && cache[dev]) return cache[dev];
  int n = 0;
  if (cudaDeviceGetAttribute(&n, cudaDevAttrMultiProcessorCount, dev) != cudaSuccess || n <= 0) n = 1;
  if (dev >= 0 && dev < 64) cache[dev] = n;
  return n;
}

namespace {
thread_local char g_last_cuda_error[256] = "";
std::atomic<uint64_t> g_launches{0};
}  // namespace

void count_launches(int n) { g_launches.fetch_add((uint64_t)n, std::memory_order_relaxed); }

dsa_status_t cuda_status(cudaError_t e) {
  if (e == cudaSuccess) return DSA_OK;
  snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "%s: %s", cudaGetErrorName(e), cudaGetErrorString(e));
  return DSA_ERR_CUDA;
}

namespace {

using EncodeTiledFn = CUresult (*)(CUtensorMap*, CUtensorMapDataType, cuuint32_t, void*, const cuuint64_t*,
                                   const cuuint64_t*, const cuuint32_t*, const cuuint32_t*, CUtensorMapInterleave,
                                   CUtensorMapSwizzle, CUtensorMapL2promotion, CUtensorMapFloatOOBfill);

EncodeTiledFn encode_fn() {
  static EncodeTiledFn fn = nullptr;
  static std::once_flag once;
  std::call_once(once, [] {
    void* ptr = nullptr;
    cudaDriverEntryPointQueryResult q = cudaDriverEntryPointSymbolNotFound;
    if (cudaGetDriverEntryPointByVersion("cuTensorMapEncodeTiled", &ptr, 12000, cudaEnableDefault, &q) ==
            cudaSuccess &&
        q == cudaDriverEntryPointSuccess)
      fn = reinterpret_cast<EncodeTiledFn>(ptr);
  });
  return fn;
}

inline bool aligned(const void* p, uintptr_t a) { return (reinterpret_cast<uintptr_t>(p) & (a - 1)) == 0; }
inline size_t al256(size_t x) { return (x + 255) & ~size_t(255); }

int latent_record_bytes(int latent_format) { return latent_format == DSA_LATENT_NVFP4 ? 352 : kLatent; }

int index_page_bytes(int key_format) {
  return key_format == DSA_KEY_FP8_E4M3 ? kBlock * (kIdxDim + 4) : kBlock * (kIdxDim / 2 + 4);
}

dsa_status_t check_cache(const dsa_paged_cache_t* c) {
  if (!c || !c->base || !aligned(c->base, 128)) return DSA_ERR_INVALID_ARG;
  if (c->block_size != kBlock) return DSA_ERR_UNSUPPORTED;
  if (c->key_format != DSA_KEY_FP8_E4M3 && c->key_format != DSA_KEY_MXFP4 && c->key_format != DSA_KEY_MXFP4_NATIVE)
    return DSA_ERR_INVALID_ARG;
  if (c->latent_format != DSA_LATENT_FP8_E4M3 && c->latent_format != DSA_LATENT_NVFP4) return DSA_ERR_INVALID_ARG;
  if (c->num_blocks <= 0 || c->row_stride <= 0 || (c->row_stride % 128) || (c->latent_off % 128) ||
      (c->index_off % 128) || c->latent_off < 0 || c->index_off < 0)
    return DSA_ERR_INVALID_ARG;
  if (c->latent_off + kBlock * latent_record_bytes(c->latent_format) > c->row_stride) return DSA_ERR_INVALID_ARG;
  if (c->index_off + index_page_bytes(c->key_format) > c->row_stride) return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}

dsa_status_t check_batch(const dsa_batch_t* b) {
  if (!b || b->batch < 0 || b->max_seq_len < 0 || b->max_blocks_per_seq < 1) return DSA_ERR_INVALID_ARG;
  if (b->queries_per_seq < 1 || b->queries_per_seq > DSA_MAX_QUERIES_PER_SEQ) return DSA_ERR_UNSUPPORTED;
  if (b->batch > 0 && (!b->block_table || !b->seq_lens)) return DSA_ERR_INVALID_ARG;
  if ((int64_t)b->batch * b->queries_per_seq > (1 << 24)) return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

// Row shapes the indexer takes: MXFP4 keys (either query format) one row per sequence; more than 4
// rows per sequence (a prefill chunk) a multiple of 4; at most 4096 sequences.
dsa_status_t check_index_rows(const dsa_paged_cache_t* c, const dsa_batch_t* b) {
  const int nq = b->queries_per_seq;
  if (c->key_format != DSA_KEY_FP8_E4M3 && nq != 1) return DSA_ERR_UNSUPPORTED;
  if (nq > 4 && nq % 4 != 0) return DSA_ERR_UNSUPPORTED;
  if (b->batch > 4096) return DSA_ERR_UNSUPPORTED;
  return DSA_OK;
}

int64_t round_ld(int max_len) { return ((int64_t)std::max(max_len, 1) + 7) & ~int64_t(7); }

}  // namespace

bool encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base, const uint64_t* dims,
                 const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle swizzle) {
  EncodeTiledFn fn = encode_fn();
  if (!fn) return false;
  cuuint64_t d[5], s[4];
  cuuint32_t bx[5], es[5];
  for (int i = 0; i < rank; ++i) {
    d[i] = dims[i];
    bx[i] = box[i];
    es[i] = 1;
  }
  for (int i = 0; i + 1 < rank; ++i) s[i] = strides[i];
  const CUresult r = fn(map, dtype, (cuuint32_t)rank, const_cast<void*>(base), d, s, bx, es,
                        CU_TENSOR_MAP_INTERLEAVE_NONE, swizzle, CU_TENSOR_MAP_L2_PROMOTION_L2_256B,
                        CU_TENSOR_MAP_FLOAT_OOB_FILL_NONE);
  if (r != CUDA_SUCCESS)
    snprintf(g_last_cuda_error, sizeof(g_last_cuda_error), "cuTensorMapEncodeTiled failed with CUresult %d", (int)r);
  return r == CUDA_SUCCESS;
}

}  // namespace dsa

using namespace dsa;

extern "C" {

int32_t dsa_api_version(void) { return DSA_API_VERSION; }

const char* dsa_last_cuda_error(void) { return g_last_cuda_error; }

int32_t dsa_topk_force_multipass(int32_t on) { return dsa::topk_force_multipass(on); }

uint64_t dsa_kernel_launches(void) { return dsa::g_launches.load(std::memory_order_relaxed); }

const char* dsa_status_string(int32_t s) {
  switch (s) {
    case DSA_OK: return "DSA_OK";
    case DSA_ERR_INVALID_ARG: return "DSA_ERR_INVALID_ARG: NULL pointer, bad size or misaligned buffer";
    case DSA_ERR_UNSUPPORTED: return "DSA_ERR_UNSUPPORTED: valid request not handled by this build";
    case DSA_ERR_BOUNDS: return "DSA_ERR_BOUNDS: block-table entry or token index outside the cache";
    case DSA_ERR_TIMEOUT: return "DSA_ERR_TIMEOUT: an in-kernel wait ran out";
    case DSA_ERR_CUDA: return "DSA_ERR_CUDA: CUDA launch or runtime error";
    case DSA_ERR_WORKSPACE: return "DSA_ERR_WORKSPACE: workspace missing or too small";
    default: return "unknown dsa status";
  }
}

dsa_status_t dsa_translate_pages(const dsa_paged_cache_t* cache, const dsa_batch_t* batch, int64_t* latent_pages,
                                 int64_t* index_pages, int32_t* dev_status, void* stream) {
  dsa_status_t s;
  if ((s = check_cache(cache)) != DSA_OK) return s;
  if ((s = check_batch(batch)) != DSA_OK) return s;
  if (!dev_status) return DSA_ERR_INVALID_ARG;
  return launch_translate_pages(*cache, *batch, latent_pages, index_pages, dev_status,
                                static_cast<cudaStream_t>(stream));
}

dsa_status_t dsa_index_scores(const dsa_paged_cache_t* cache, const dsa_batch_t* batch, const uint8_t* q_index,
                              const float* head_w, float* scores, int64_t ld_scores, int32_t* dev_status,
                              void* stream) {
  dsa_status_t s;
  if ((s = check_cache(cache)) != DSA_OK) return s;
  if ((s = check_batch(batch)) != DSA_OK) return s;
  if ((s = check_index_rows(cache, batch)) != DSA_OK) return s;
  if (!dev_status) return DSA_ERR_INVALID_ARG;
  if (batch->batch == 0) return DSA_OK;
  if (!q_index || !head_w || !scores || !aligned(q_index, 16) || !aligned(head_w, 16) || !aligned(scores, 16))
    return DSA_ERR_INVALID_ARG;
  if (ld_scores < batch->max_seq_len || (ld_scores % 4)) return DSA_ERR_INVALID_ARG;
  return launch_index_scores(*cache, *batch, q_index, head_w, scores, false, ld_scores, dev_status,
                             static_cast<cudaStream_t>(stream));
}

dsa_status_t dsa_index_scores_bf16(const dsa_paged_cache_t* cache, const dsa_batch_t* batch, const uint8_t* q_index,
                                   const float* head_w, uint16_t* scores, int64_t ld_scores, int32_t* dev_status,
                                   void* stream) {
  dsa_status_t s;
  if ((s = check_cache(cache)) != DSA_OK) return s;
  if ((s = check_batch(batch)) != DSA_OK) return s;
  if ((s = check_index_rows(cache, batch)) != DSA_OK) return s;
  if (!dev_status) return DSA_ERR_INVALID_ARG;
  if (batch->batch == 0) return DSA_OK;
  if (!q_index || !head_w || !scores || !aligned(q_index, 16) || !aligned(head_w, 16) || !aligned(scores, 16))
    return DSA_ERR_INVALID_ARG;
  if (ld_scores < batch->max_seq_len || (ld_scores % 8)) return DSA_ERR_INVALID_ARG;
  return launch_index_scores(*cache, *batch, q_index, head_w, scores, true, ld_scores, dev_status,
                             static_cast<cudaStream_t>(stream));
}

size_t dsa_topk_workspace_size(int32_t rows, int32_t max_row_len, int32_t k) {
  if (rows < 0 || k < 1 || k > DSA_MAX_TOPK) return 0;
  return topk_workspace_bytes(rows, max_row_len, k);
}

dsa_status_t dsa_topk(const float* scores, int64_t ld_scores, const int32_t* row_lens, int32_t rows,
                      int32_t max_row_len, int32_t k, int32_t* idx_out, void* workspace, size_t workspace_bytes,
                      int32_t* dev_status, void* stream) {
  if (rows < 0 || k < 1 || k > DSA_MAX_TOPK || max_row_len < 0 || !dev_status) return DSA_ERR_INVALID_ARG;
  if (rows == 0) return DSA_OK;
  if (!scores || !row_lens || !idx_out || !aligned(scores, 16) || ld_scores < max_row_len || (ld_scores % 4))
    return DSA_ERR_INVALID_ARG;
  const size_t need = topk_workspace_bytes(rows, max_row_len, k);
  if (need && (!workspace || !aligned(workspace, 256) || workspace_bytes < need)) return DSA_ERR_WORKSPACE;
  return launch_topk(scores, ld_scores, row_lens, nullptr, 1, rows, max_row_len, k, idx_out, workspace, dev_status,
                     static_cast<cudaStream_t>(stream));
}

dsa_status_t dsa_topk_bf16(const uint16_t* scores, int64_t ld_scores, const int32_t* row_lens, int32_t rows,
                           int32_t max_row_len, int32_t k, int32_t* idx_out, int32_t* dev_status, void* stream) {
  if (rows < 0 || k < 1 || k > DSA_MAX_TOPK || max_row_len < 0 || !dev_status) return DSA_ERR_INVALID_ARG;
  if (rows == 0) return DSA_OK;
  if (!scores || !row_lens || !idx_out || !aligned(scores, 16) || ld_scores < max_row_len || (ld_scores % 8))
    return DSA_ERR_INVALID_ARG;
  return launch_topk_bf16(scores, ld_scores, row_lens, nullptr, 1, rows, max_row_len, k, idx_out, dev_status,
                          static_cast<cudaStream_t>(stream));
}

dsa_status_t dsa_topk_noalloc(const float* scores, int64_t ld_scores, const int32_t* row_lens, int32_t rows,
                              int32_t max_row_len, int32_t k, int32_t* idx_out, int32_t* dev_status, void* stream) {
  if (rows < 0 || k < 1 || k > DSA_MAX_TOPK || max_row_len < 0 || !dev_status) return DSA_ERR_INVALID_ARG;
  if (rows > DSA_TOPK_NOALLOC_MAX_ROWS) return DSA_ERR_UNSUPPORTED;
  if (rows == 0) return DSA_OK;
  if (!scores || !row_lens || !idx_out || !aligned(scores, 16) || ld_scores < max_row_len || (ld_scores % 4))
    return DSA_ERR_INVALID_ARG;
  return launch_topk_noalloc(scores, ld_scores, row_lens, rows, max_row_len, k, idx_out, dev_status,
                             static_cast<cudaStream_t>(stream));
}

size_t dsa_dcp_topk_workspace_size(int32_t rows, int32_t k, int32_t shards) {
  if (rows < 0 || k < 1 || k > DSA_MAX_TOPK || shards < 1 || shards > DSA_DCP_MAX_SHARDS) return 0;
  return dcp_workspace_bytes(rows, k, shards);
}

dsa_status_t dsa_dcp_topk(const float* scores, int64_t ld_scores, const int32_t* row_lens, int32_t rows,
                          int32_t max_row_len, int32_t k, int32_t shards, int32_t* idx_out, int32_t* stats_out,
                          void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
  if (rows < 0 || k < 1 || k > DSA_MAX_TOPK || max_row_len < 0 || shards < 1 || !dev_status)
    return DSA_ERR_INVALID_ARG;
  if (shards > DSA_DCP_MAX_SHARDS || (int64_t)max_row_len > (int64_t)DSA_DCP_MAX_SHARD_TOKENS * shards)
    return DSA_ERR_UNSUPPORTED;
  if (rows == 0) return DSA_OK;
  if (!scores || !row_lens || !idx_out || !aligned(scores, 4) || ld_scores < max_row_len) return DSA_ERR_INVALID_ARG;
  const size_t need = dcp_workspace_bytes(rows, k, shards);
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < need) return DSA_ERR_WORKSPACE;
  return launch_dcp_topk(scores, ld_scores, row_lens, rows, max_row_len, k, shards, idx_out, stats_out, workspace,
                         dev_status, static_cast<cudaStream_t>(stream));
}

size_t dsa_dcp_sparse_mla_workspace_size(int32_t rows, int32_t k, int32_t shards) {
  if (rows < 0 || k < 1 || k > DSA_MAX_TOPK || shards < 1 || shards > DSA_DCP_MAX_SHARDS) return 0;
  return dcp_mla_workspace_bytes(rows, k, shards);
}

dsa_status_t dsa_dcp_sparse_mla(const dsa_paged_cache_t* cache, const dsa_batch_t* batch, const uint16_t* q_mla,
                                const int32_t* idx, int32_t k, int32_t shards, float sm_scale, uint16_t* out,
                                float* lse, uint16_t* part_out, float* part_lse, void* workspace,
                                size_t workspace_bytes, int32_t* dev_status, void* stream) {
  dsa_status_t s;
  if ((s = check_cache(cache)) != DSA_OK) return s;
  if ((s = check_batch(batch)) != DSA_OK) return s;
  if (k < 1 || k > DSA_MAX_TOPK || shards < 1 || !dev_status) return DSA_ERR_INVALID_ARG;
  if (shards > DSA_DCP_MAX_SHARDS) return DSA_ERR_UNSUPPORTED;
  const int rows = batch->batch * batch->queries_per_seq;
  if (rows == 0) return DSA_OK;
  if (!q_mla || !idx || !out || !lse || !aligned(q_mla, 16) || !aligned(out, 8) ||
      (part_out && !aligned(part_out, 8)))
    return DSA_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < dcp_mla_workspace_bytes(rows, k, shards))
    return DSA_ERR_WORKSPACE;
  return launch_dcp_sparse_mla(*cache, *batch, q_mla, idx, k, shards, sm_scale, out, lse, part_out, part_lse,
                               workspace, dev_status, static_cast<cudaStream_t>(stream));
}

int32_t dsa_batch_invariant(int32_t on) { return dsa::mla_batch_invariant(on); }

size_t sparse_mla_workspace_size(int32_t rows, int32_t k) {
  if (rows < 0 || k < 1 || k > DSA_MAX_TOPK) return 0;
  return mla_workspace_bytes(rows, k);
}

dsa_status_t sparse_mla_decode(const dsa_paged_cache_t* cache, const dsa_batch_t* batch, const uint16_t* q_mla,
                               const int32_t* idx, int32_t k, float sm_scale, uint16_t* out, float* lse,
                               void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
  dsa_status_t s;
  if ((s = check_cache(cache)) != DSA_OK) return s;
  if ((s = check_batch(batch)) != DSA_OK) return s;
  if (k < 1 || k > DSA_MAX_TOPK || !dev_status) return DSA_ERR_INVALID_ARG;
  const int rows = batch->batch * batch->queries_per_seq;
  if (rows == 0) return DSA_OK;
  if (!q_mla || !idx || !out || !lse || !aligned(q_mla, 16) || !aligned(out, 8)) return DSA_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < mla_workspace_bytes(rows, k))
    return DSA_ERR_WORKSPACE;
  return launch_sparse_mla(*cache, *batch, q_mla, idx, k, sm_scale, out, lse, workspace, dev_status,
                           static_cast<cudaStream_t>(stream));
}

size_t dsa_workspace_size(const dsa_batch_t* batch, int32_t k) {
  if (!batch || batch->batch < 0 || k < 1 || k > DSA_MAX_TOPK) return 0;
  const int rows = batch->batch * std::max(1, batch->queries_per_seq);
  return al256((size_t)rows * round_ld(batch->max_seq_len) * 4) + al256((size_t)rows * k * 4) +
         al256(topk_workspace_bytes(rows, batch->max_seq_len, k)) + al256(mla_workspace_bytes(rows, k));
}

namespace {

dsa_status_t decode_step_impl(const dsa_paged_cache_t* cache, const dsa_batch_t* batch, const uint8_t* q_index,
                              const float* head_w, const uint16_t* q_mla, int32_t k, float sm_scale, uint16_t* out,
                              float* lse, void* scores_out, bool bf16, int64_t ld_scores, int32_t* idx_out,
                              int32_t* phys_out, void* workspace, size_t workspace_bytes, int32_t* dev_status,
                              void* stream) {
  dsa_status_t s;
  if ((s = check_cache(cache)) != DSA_OK) return s;
  if ((s = check_batch(batch)) != DSA_OK) return s;
  if ((s = check_index_rows(cache, batch)) != DSA_OK) return s;
  if (k < 1 || k > DSA_MAX_TOPK || !dev_status) return DSA_ERR_INVALID_ARG;
  const int rows = batch->batch * batch->queries_per_seq;
  if (rows == 0) return DSA_OK;
  if (!q_index || !head_w || !q_mla || !out || !lse) return DSA_ERR_INVALID_ARG;
  if (!aligned(q_index, 16) || !aligned(head_w, 16) || !aligned(q_mla, 16) || !aligned(out, 8))
    return DSA_ERR_INVALID_ARG;
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < dsa_workspace_size(batch, k))
    return DSA_ERR_WORKSPACE;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  uint8_t* w = static_cast<uint8_t*>(workspace);
  void* scores = scores_out;
  int64_t ld = ld_scores;
  const size_t scores_bytes = al256((size_t)rows * round_ld(batch->max_seq_len) * 4);
  if (!scores) {
    scores = w;
    ld = round_ld(batch->max_seq_len);  // a multiple of 8
  } else if (!aligned(scores, 16) || ld < batch->max_seq_len || (ld % (bf16 ? 8 : 4))) {
    return DSA_ERR_INVALID_ARG;
  }
  w += scores_bytes;
  int32_t* idx = idx_out ? idx_out : reinterpret_cast<int32_t*>(w);
  w += al256((size_t)rows * k * 4);
  // the selected tokens' physical KV rows, when the caller asks for them: written
  // by the top-k and read by the MLA (which otherwise translates the indices
  // itself, beside its Q loads, off the critical path)
  int32_t* phys = phys_out;
  void* topk_ws = w;
  w += al256(topk_workspace_bytes(rows, batch->max_seq_len, k));
  void* mla_ws = w;

  if ((s = launch_index_scores(*cache, *batch, q_index, head_w, scores, bf16, ld, dev_status, st)) != DSA_OK)
    return s;
  const int cap = std::min(batch->max_blocks_per_seq * kBlock, batch->max_seq_len);
  TopkPhys po;
  po.phys = phys;
  po.block_table = batch->block_table;
  po.max_blocks = batch->max_blocks_per_seq;
  po.num_blocks = cache->num_blocks;
  if (bf16)
    s = launch_topk_bf16(static_cast<const uint16_t*>(scores), ld, nullptr, batch->seq_lens,
                         batch->queries_per_seq, rows, cap, k, idx, dev_status, st, po);
  else
    s = launch_topk(static_cast<const float*>(scores), ld, nullptr, batch->seq_lens, batch->queries_per_seq, rows,
                    cap, k, idx, topk_ws, dev_status, st, po);
  if (s != DSA_OK) return s;
  return launch_sparse_mla(*cache, *batch, q_mla, idx, k, sm_scale, out, lse, mla_ws, dev_status, st, phys);
}

}  // namespace

dsa_status_t dsa_decode_step(const dsa_paged_cache_t* cache, const dsa_batch_t* batch, const uint8_t* q_index,
                             const float* head_w, const uint16_t* q_mla, int32_t k, float sm_scale, uint16_t* out,
                             float* lse, float* scores_out, int64_t ld_scores, int32_t* idx_out, int32_t* phys_out,
                             void* workspace, size_t workspace_bytes, int32_t* dev_status, void* stream) {
  return decode_step_impl(cache, batch, q_index, head_w, q_mla, k, sm_scale, out, lse, scores_out, false, ld_scores,
                          idx_out, phys_out, workspace, workspace_bytes, dev_status, stream);
}

dsa_status_t dsa_topk_paged(const dsa_paged_cache_t* cache, const dsa_batch_t* batch, const float* scores,
                            int64_t ld_scores, int32_t k, int32_t* idx_out, int32_t* phys_out, void* workspace,
                            size_t workspace_bytes, int32_t* dev_status, void* stream) {
  dsa_status_t s;
  if ((s = check_cache(cache)) != DSA_OK) return s;
  if ((s = check_batch(batch)) != DSA_OK) return s;
  if (k < 1 || k > DSA_MAX_TOPK || !dev_status) return DSA_ERR_INVALID_ARG;
  const int rows = batch->batch * batch->queries_per_seq;
  if (rows == 0) return DSA_OK;
  if (!scores || !idx_out || !aligned(scores, 16) || ld_scores < batch->max_seq_len || (ld_scores % 4))
    return DSA_ERR_INVALID_ARG;
  const size_t need = topk_workspace_bytes(rows, batch->max_seq_len, k);
  if (need && (!workspace || !aligned(workspace, 256) || workspace_bytes < need)) return DSA_ERR_WORKSPACE;
  TopkPhys po;
  po.phys = phys_out;
  po.block_table = batch->block_table;
  po.max_blocks = batch->max_blocks_per_seq;
  po.num_blocks = cache->num_blocks;
  const int cap = std::min(batch->max_blocks_per_seq * kBlock, batch->max_seq_len);
  return launch_topk(scores, ld_scores, nullptr, batch->seq_lens, batch->queries_per_seq, rows, cap, k, idx_out,
                     workspace, dev_status, static_cast<cudaStream_t>(stream), po);
}

dsa_status_t dsa_decode_step_bf16(const dsa_paged_cache_t* cache, const dsa_batch_t* batch, const uint8_t* q_index,
                                  const float* head_w, const uint16_t* q_mla, int32_t k, float sm_scale,
                                  uint16_t* out, float* lse, uint16_t* scores_out, int64_t ld_scores,
                                  int32_t* idx_out, int32_t* phys_out, void* workspace, size_t workspace_bytes,
                                  int32_t* dev_status, void* stream) {
  return decode_step_impl(cache, batch, q_index, head_w, q_mla, k, sm_scale, out, lse, scores_out, true, ld_scores,
                          idx_out, phys_out, workspace, workspace_bytes, dev_status, stream);
}

dsa_status_t dsa_cache_append(const dsa_paged_cache_t* cache, const dsa_batch_t* batch, const uint16_t* new_latent,
                              const uint16_t* new_index_key, int32_t* dev_status, void* stream) {
  dsa_status_t s;
  if ((s = check_cache(cache)) != DSA_OK) return s;
  if ((s = check_batch(batch)) != DSA_OK) return s;
  if (!dev_status) return DSA_ERR_INVALID_ARG;
  if (batch->batch == 0) return DSA_OK;
  if (!new_latent || !new_index_key || !aligned(new_latent, 2) || !aligned(new_index_key, 2))
    return DSA_ERR_INVALID_ARG;
  return launch_cache_append(*cache, *batch, new_latent, new_index_key, dev_status,
                             static_cast<cudaStream_t>(stream));
}

dsa_status_t dsa_quantize_index_query(const uint16_t* q_bf16, const float* head_w, int32_t rows, uint8_t* q_index,
                                      float* head_w_out, void* stream) {
  if (rows < 0) return DSA_ERR_INVALID_ARG;
  if (rows == 0) return DSA_OK;
  if (!q_bf16 || !head_w || !q_index || !head_w_out || !aligned(q_bf16, 8) || !aligned(q_index, 4))
    return DSA_ERR_INVALID_ARG;
  return launch_quantize_query(q_bf16, head_w, rows, q_index, head_w_out, static_cast<cudaStream_t>(stream));
}

namespace {
dsa_status_t check_frontend(const uint16_t* c_q, int32_t q_rank, const uint16_t* gamma, float eps,
                            const uint16_t* w_iq, const float* head_w, const uint16_t* new_latent,
                            const uint16_t* new_index_key) {
  if (q_rank % 64 || q_rank < 64 || q_rank > 16384) return DSA_ERR_UNSUPPORTED;
  if (!c_q || !gamma || !w_iq || !head_w || !new_latent || !new_index_key || !(eps >= 0.f)) return DSA_ERR_INVALID_ARG;
  if (!aligned(c_q, 16) || !aligned(gamma, 16) || !aligned(w_iq, 16) || !aligned(head_w, 4) || !aligned(new_latent, 2) ||
      !aligned(new_index_key, 2))
    return DSA_ERR_INVALID_ARG;
  return DSA_OK;
}
}  // namespace

dsa_status_t dsa_index_frontend(const dsa_paged_cache_t* cache, const dsa_batch_t* batch, const uint16_t* c_q,
                                int32_t q_rank, const uint16_t* gamma, float eps, const uint16_t* w_iq,
                                const float* head_w, const uint16_t* new_latent, const uint16_t* new_index_key,
                                uint8_t* q_index, float* head_w_out, float* q_proj, int32_t* dev_status,
                                void* stream) {
  dsa_status_t s;
  if ((s = check_cache(cache)) != DSA_OK) return s;
  if ((s = check_batch(batch)) != DSA_OK) return s;
  if (!dev_status) return DSA_ERR_INVALID_ARG;
  if (batch->batch == 0) return DSA_OK;
  if ((s = check_frontend(c_q, q_rank, gamma, eps, w_iq, head_w, new_latent, new_index_key)) != DSA_OK) return s;
  if (!q_index || !head_w_out || !aligned(head_w_out, 4) || (q_proj && !aligned(q_proj, 4))) return DSA_ERR_INVALID_ARG;
  return launch_frontend(*cache, *batch, c_q, q_rank, gamma, eps, w_iq, head_w, new_latent, new_index_key, q_index,
                         head_w_out, q_proj, dev_status, static_cast<cudaStream_t>(stream));
}

size_t dsa_frontend_workspace_size(const dsa_batch_t* batch, int32_t k) {
  const size_t step = dsa_workspace_size(batch, k);
  if (!step) return 0;
  const size_t rows = (size_t)batch->batch * std::max(1, batch->queries_per_seq);
  return al256(rows * kIdxHeads * kIdxDim) + al256(rows * kIdxHeads * 4) + step;
}

dsa_status_t dsa_decode_step_frontend(const dsa_paged_cache_t* cache, const dsa_batch_t* batch,
                                      const uint16_t* c_q, int32_t q_rank, const uint16_t* gamma, float eps,
                                      const uint16_t* w_iq, const float* head_w, const uint16_t* new_latent,
                                      const uint16_t* new_index_key, const uint16_t* q_mla, int32_t k,
                                      float sm_scale, uint16_t* out, float* lse, float* scores_out,
                                      int64_t ld_scores, int32_t* idx_out, int32_t* phys_out, void* workspace,
                                      size_t workspace_bytes, int32_t* dev_status, void* stream) {
  dsa_status_t s;
  if ((s = check_cache(cache)) != DSA_OK) return s;
  if ((s = check_batch(batch)) != DSA_OK) return s;
  if ((s = check_index_rows(cache, batch)) != DSA_OK) return s;
  if (k < 1 || k > DSA_MAX_TOPK || !dev_status) return DSA_ERR_INVALID_ARG;
  if (batch->batch == 0) return DSA_OK;
  if ((s = check_frontend(c_q, q_rank, gamma, eps, w_iq, head_w, new_latent, new_index_key)) != DSA_OK) return s;
  if (!workspace || !aligned(workspace, 256) || workspace_bytes < dsa_frontend_workspace_size(batch, k))
    return DSA_ERR_WORKSPACE;
  const size_t rows = (size_t)batch->batch * batch->queries_per_seq;
  uint8_t* w = static_cast<uint8_t*>(workspace);
  uint8_t* q_index = w;
  w += al256(rows * kIdxHeads * kIdxDim);
  float* head_w_out = reinterpret_cast<float*>(w);
  w += al256(rows * kIdxHeads * 4);
  // validate the step's own arguments before the front end writes the cache
  if (!q_mla || !out || !lse || !aligned(q_mla, 16) || !aligned(out, 8)) return DSA_ERR_INVALID_ARG;
  if (scores_out && (!aligned(scores_out, 16) || ld_scores < batch->max_seq_len || (ld_scores % 4)))
    return DSA_ERR_INVALID_ARG;
  cudaStream_t st = static_cast<cudaStream_t>(stream);
  if ((s = launch_frontend(*cache, *batch, c_q, q_rank, gamma, eps, w_iq, head_w, new_latent, new_index_key, q_index,
                           head_w_out, nullptr, dev_status, st)) != DSA_OK)
    return s;
  return dsa_decode_step(cache, batch, q_index, head_w_out, q_mla, k, sm_scale, out, lse, scores_out, ld_scores,
                         idx_out, phys_out, w, workspace_bytes - (size_t)(w - static_cast<uint8_t*>(workspace)),
                         dev_status, stream);
}

dsa_status_t dsa_selftest_wait_timeout(int64_t limit_ns, int32_t* dev_status, void* stream) {
  if (!dev_status) return DSA_ERR_INVALID_ARG;
  return launch_wait_selftest(limit_ns, dev_status, static_cast<cudaStream_t>(stream));
}

}  // extern "C"
