// pages.cu — block table -> kernel page addresses, and the bounded-wait self-test.
//
// Page translation follows the vLLM Day-0 post for Kimi K3.1 Pro, section
// "为三类状态服务的 KV 缓存": before every step the block table and cache
// slots are turned into the page addresses the kernels read, so that kernels
// written for small fixed-size pages can read the packed block rows.
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace dsa {

namespace {

__global__ void translate_pages_kernel(const uint8_t* base, int64_t row_stride, int64_t latent_off, int64_t index_off,
                                       int32_t num_blocks, const int32_t* block_table, int32_t max_blocks,
                                       const int32_t* seq_lens, int32_t batch, int32_t cap, int64_t* latent_pages,
                                       int64_t* index_pages, int32_t* status) {
  const int64_t n = (int64_t)batch * max_blocks;
  for (int64_t e = blockIdx.x * (int64_t)blockDim.x + threadIdx.x; e < n; e += (int64_t)gridDim.x * blockDim.x) {
    const int b = (int)(e / max_blocks), j = (int)(e % max_blocks);
    int len = seq_lens[b];
    if (len < 0 || len > cap) {
      if (j == 0) report(status, DSA_ERR_BOUNDS);
      len = len < 0 ? 0 : cap;
    }
    int64_t lat = 0, idx = 0;
    if ((int64_t)j * kBlock < len) {
      const int r = block_table[e];
      if (r >= 0 && r < num_blocks) {
        const int64_t row = reinterpret_cast<int64_t>(base) + (int64_t)r * row_stride;
        lat = row + latent_off;
        idx = row + index_off;
      } else {
        report(status, DSA_ERR_BOUNDS);
      }
    }
    if (latent_pages) latent_pages[e] = lat;
    if (index_pages) index_pages[e] = idx;
  }
}

// Waits on a barrier that nothing signals; the bounded wait must give up,
// report DSA_ERR_TIMEOUT and let the kernel return normally.
__global__ void wait_selftest_kernel(uint64_t limit_ns, int32_t* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x == 0) {
    mbar_init(smem_u32(&bar), 1);
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  if (threadIdx.x == 0) mbar_wait(smem_u32(&bar), 0, &abort_flag, status, limit_ns);
  __syncthreads();
}

}  // namespace

dsa_status_t launch_translate_pages(const dsa_paged_cache_t& c, const dsa_batch_t& bt, int64_t* latent_pages,
                                    int64_t* index_pages, int32_t* status, cudaStream_t st) {
  const int64_t n = (int64_t)bt.batch * bt.max_blocks_per_seq;
  if (n == 0) return DSA_OK;
  const int threads = 256;
  const int grid = (int)std::min<int64_t>((n + threads - 1) / threads, 4 * (int64_t)num_sms());
  const int cap = std::min(bt.max_blocks_per_seq * kBlock, bt.max_seq_len);
  count_launches(1);
  translate_pages_kernel<<<grid, threads, 0, st>>>(static_cast<const uint8_t*>(c.base), c.row_stride, c.latent_off,
                                                   c.index_off, c.num_blocks, bt.block_table,
                                                   bt.max_blocks_per_seq, bt.seq_lens, bt.batch, cap, latent_pages,
                                                   index_pages, status);
  return launch_status();
}

dsa_status_t launch_wait_selftest(int64_t limit_ns, int32_t* status, cudaStream_t st) {
  if (limit_ns < 1000000) limit_ns = 1000000;
  if (limit_ns > 2000000000) limit_ns = 2000000000;
  count_launches(1);
  wait_selftest_kernel<<<1, 32, 0, st>>>((uint64_t)limit_ns, status);
  return launch_status();
}

}  // namespace dsa
