// internal.h — launchers and host helpers shared by the library's .cu files.
#pragma once

#include <cuda.h>
#include <cuda_runtime.h>
#include <stddef.h>
#include <stdint.h>

#include "../../include/dsa.h"

namespace dsa {

// Streaming multiprocessors of the current device (cached per device).
int num_sms();

// Records `e` (if not cudaSuccess) as this thread's last CUDA error and maps
// it to DSA_OK / DSA_ERR_CUDA.
dsa_status_t cuda_status(cudaError_t e);
// cuda_status(cudaGetLastError()): the launch check after a kernel launch.
inline dsa_status_t launch_status() { return cuda_status(cudaGetLastError()); }

// Adds n to the count of kernel launches the library has issued (process-wide,
// read through dsa_kernel_launches).
void count_launches(int n);

// cuTensorMapEncodeTiled through the runtime's driver entry point (no libcuda
// link dependency).  strides: rank-1 byte strides of dims 1..rank-1.
bool encode_tmap(CUtensorMap* map, CUtensorMapDataType dtype, int rank, const void* base, const uint64_t* dims,
                 const uint64_t* strides, const uint32_t* box, CUtensorMapSwizzle swizzle);

dsa_status_t launch_translate_pages(const dsa_paged_cache_t& c, const dsa_batch_t& bt, int64_t* latent_pages,
                                    int64_t* index_pages, int32_t* status, cudaStream_t st);
// FP8 or MXFP4 keys (MXFP4: one query row per sequence, else DSA_ERR_UNSUPPORTED).
// scores: fp32, or bf16 bits when bf16 (ld in elements either way).
dsa_status_t launch_index_scores(const dsa_paged_cache_t& c, const dsa_batch_t& bt, const uint8_t* q_index,
                                 const float* head_w, void* scores, bool bf16, int64_t ld, int32_t* status,
                                 cudaStream_t st);
// The same scores for a prefill chunk (FP8 keys, at least 8 rows per sequence):
// the dense-contraction kernel of prefill.cu.
dsa_status_t launch_prefill_scores(const dsa_paged_cache_t& c, const dsa_batch_t& bt, const uint8_t* q_index,
                                   const float* head_w, void* scores, bool bf16, int64_t ld, int32_t* status,
                                   cudaStream_t st);
size_t topk_workspace_bytes(int rows, int max_row_len, int k);
// Optional physical KV rows beside the top-k's token indices: phys[r][p] =
// block_table[r / nq][t / 64] * 64 + t % 64 for the index t at position p
// (-1 for padding; an entry outside 0..num_blocks-1 is reported as
// DSA_ERR_BOUNDS and gives -1).  phys == nullptr: none.
struct TopkPhys {
  int32_t* phys = nullptr;
  const int32_t* block_table = nullptr;
  int32_t max_blocks = 0, num_blocks = 0;
};
// Process-wide choice of the four-kernel top-k for rows too long for shared memory.
int topk_force_multipass(int on);
dsa_status_t launch_topk(const float* scores, int64_t ld, const int32_t* row_lens, const int32_t* seq_lens, int nq,
                         int rows, int max_row_len, int k, int32_t* out, void* workspace, int32_t* status,
                         cudaStream_t st, const TopkPhys& po = TopkPhys{});
// The same top-k over bf16 scores (bits, widened exactly): the cluster paths
// only (DSA_ERR_UNSUPPORTED where no cluster can be scheduled); no workspace.
dsa_status_t launch_topk_bf16(const uint16_t* scores, int64_t ld, const int32_t* row_lens, const int32_t* seq_lens,
                              int nq, int rows, int max_row_len, int k, int32_t* out, int32_t* status,
                              cudaStream_t st, const TopkPhys& po = TopkPhys{});
// The same top-k with its scratch in a file-scope device array (no allocation).
dsa_status_t launch_topk_noalloc(const float* scores, int64_t ld, const int32_t* row_lens, int rows, int max_row_len,
                                 int k, int32_t* out, int32_t* status, cudaStream_t st);
// Decode-context-parallel top-k merge of `shards` token shards, emulated on one GPU.
size_t dcp_workspace_bytes(int rows, int k, int shards);
dsa_status_t launch_dcp_topk(const float* scores, int64_t ld, const int32_t* row_lens, int rows, int max_row_len,
                             int k, int shards, int32_t* out, int32_t* stats, void* workspace, int32_t* status,
                             cudaStream_t st);
// Decode-context-parallel sparse MLA: per-shard partial attention and the LSE combine.
size_t dcp_mla_workspace_bytes(int rows, int k, int shards);
dsa_status_t launch_dcp_sparse_mla(const dsa_paged_cache_t& c, const dsa_batch_t& bt, const uint16_t* q_mla,
                                   const int32_t* idx, int k, int shards, float sm_scale, uint16_t* out, float* lse,
                                   uint16_t* part_out, float* part_lse, void* workspace, int32_t* status,
                                   cudaStream_t st);
size_t mla_workspace_bytes(int rows, int k);
// Process-wide batch-invariant mode of the MLA chunking; returns the previous setting.
int mla_batch_invariant(int on);
// Tokens of idx one MLA chunk may hold.
int mla_max_chunk();
// The MLA kernel alone over per-row chunk tables: nseg chunks per row,
// boundaries seg[row][0..nseg] in idx[row], each at most mla_max_chunk()
// tokens; partials normalised by their sum of rounded p to opart (fp16 bits)
// [rows][nseg][96][512] and (max, sum of rounded p, sum of p) to ml
// [rows][nseg][96][4].
dsa_status_t launch_sparse_mla_partials(const dsa_paged_cache_t& c, const dsa_batch_t& bt, const uint16_t* q_mla,
                                        const int32_t* idx, int k, const int32_t* seg, int nseg, float sm_scale,
                                        uint16_t* opart, float* ml, int32_t* status, cudaStream_t st);
// phys: the top-k's physical KV rows for idx ([rows][k], -1 padding, already
// bounds-checked and visible) or nullptr: the kernel translates idx itself.
dsa_status_t launch_sparse_mla(const dsa_paged_cache_t& c, const dsa_batch_t& bt, const uint16_t* q_mla,
                               const int32_t* idx, int k, float sm_scale, uint16_t* out, float* lse,
                               void* workspace, int32_t* status, cudaStream_t st, const int32_t* phys = nullptr);
dsa_status_t launch_wait_selftest(int64_t limit_ns, int32_t* status, cudaStream_t st);
dsa_status_t launch_cache_append(const dsa_paged_cache_t& c, const dsa_batch_t& bt, const uint16_t* new_latent,
                                 const uint16_t* new_key, int32_t* status, cudaStream_t st);
// The fused indexer front end: RMSNorm of c_q [rows][dim], the projection by
// w_iq [4096][dim] (bf16), FP8 query codes and folded head weights, optional
// fp32 projected values, and the new tokens into the cache; one launch.
dsa_status_t launch_frontend(const dsa_paged_cache_t& c, const dsa_batch_t& bt, const uint16_t* c_q, int dim,
                             const uint16_t* gamma, float eps, const uint16_t* w_iq, const float* head_w,
                             const uint16_t* new_latent, const uint16_t* new_key, uint8_t* q_index, float* head_w_out,
                             float* q_proj, int32_t* status, cudaStream_t st);
dsa_status_t launch_quantize_query(const uint16_t* q, const float* w, int rows, uint8_t* codes, float* w_out,
                                   cudaStream_t st);

}  // namespace dsa
