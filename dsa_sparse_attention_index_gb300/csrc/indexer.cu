// indexer.cu — lightning-indexer scores for decode (stage 1 of DSA).
//
// Computes, for every query row r = b*NQ + j and every visible token t,
//     s[r][t] = sum_h w[r][h] * max(0, scale_t * (q[r][h] . k[t]))
// with 32 heads x 128 dims (vLLM Day-0 post for Kimi K3.1 Pro, section
// "K3.1 Pro 中的稀疏注意力": 32 light heads, a 132-byte FP8 key incl. scale;
// AMD section: FP32 accumulation and a weighted reduction across heads).
//
// GB300 design.  Each 132-byte key carries 32*128 multiply-adds, i.e. 62
// FLOP per byte: at HBM speed that is ~0.4 PFLOP/s, several times what the
// CUDA cores can issue, so the dot products run on the 5th-gen tensor cores
// even in decode.  A work unit is one sequence's 256 consecutive tokens (four
// 64-token pages).  The grid is persistent (one CTA per SM) and the units of
// all sequences are split evenly across CTAs ("key-balanced", Day-0 post,
// fused decode section).  Per CTA:
//   warp 0  TMA producer: per unit, four 64 x 128 B code pages (3-D tensor map
//           over the block pool, 128-byte swizzle) and the four pages' fp32
//           scale rows in one tile::gather4 copy, into a 5-6 stage ring; the
//           lanes resolve the block-table rows of the next 32 units while
//           lane 0 issues; the query tile of the current sequence goes into a
//           2-slot ring;
//   warp 1  MMA issuer: tcgen05.mma kind::f8f6f4, two M = 128 key sub-tiles
//           per unit, N = 32*NQ query-heads, K = 128 in four K=32 steps, fp32
//           accumulators in a double-buffered TMEM tile;
//   warps 2-5 epilogue: each thread owns two key rows (one per sub-tile),
//           reads their 32*NQ accumulators with tcgen05.ld, applies scale,
//           ReLU and the head weights, sums the heads in registers (no
//           shuffles) and stores one fp32 score per query row (128-byte
//           coalesced per warp).
// All draft rows of a sequence share one key read (AMD section: keys are
// reused across query rows during speculative verify).
#include <algorithm>

#include "common.cuh"
#include "internal.h"

namespace dsa {

namespace {

constexpr int kUnitKeys = 256;                          // four pages
constexpr int kPagesPerUnit = kUnitKeys / kBlock;       // 4
constexpr int kSubTileBytes = 128 * kIdxDim;            // 16 KB: one M = 128 MMA tile
constexpr int kATileBytes = kUnitKeys * kIdxDim;        // 32 KB of E4M3 codes per unit
constexpr int kPageCodeBytes = kBlock * kIdxDim;        // 8 KB
constexpr int kPageScaleBytes = kBlock * 4;             // 256 B
constexpr int kUnitScaleBytes = kPagesPerUnit * kPageScaleBytes;  // 1 KB (one gather4)
constexpr int kThreads = 192;
constexpr int kMaxBatch = 4096;

struct IdxParams {
  const uint8_t* index_base;  // cache base + index_off
  int64_t row_stride;
  int32_t num_blocks;
  const int32_t* block_table;
  int32_t max_blocks;
  const int32_t* seq_lens;
  int32_t batch;
  int32_t max_seq_len;
  const float* head_w;
  float* scores;
  int64_t ld;
  int32_t* status;
};

template <int NQ>
struct IdxSmem {
  static constexpr int kStages = NQ == 1 ? 6 : 5;  // keeps the CTA within 227 KB of shared memory
  static constexpr int kQSlot = 32 * NQ * kIdxDim;  // bytes
  static constexpr int kOffA = 0;
  static constexpr int kOffQ = kOffA + kStages * kATileBytes;
  static constexpr int kOffScales = kOffQ + 2 * kQSlot;
  static constexpr int kOffBars = kOffScales + kStages * kUnitScaleBytes;
  // barriers: full[S], empty[S], acc_full[2], acc_empty[2], q_full[2], q_empty[2], done
  static constexpr int kNumBars = 2 * kStages + 9;
  static constexpr int kOffMisc = kOffBars + kNumBars * 8;  // tmem slot, abort flag
  static constexpr int kOffPrefix = kOffMisc + 16;
  static size_t bytes(int batch) { return 1024 + kOffPrefix + 4 * (size_t)(batch + 1); }
};

// Sequence of unit u, advancing a cursor (units arrive in increasing order).
__device__ __forceinline__ int seq_of_unit(const int32_t* prefix, int batch, int64_t u, int& cursor) {
  while (cursor + 1 < batch && u >= prefix[cursor + 1]) ++cursor;
  return cursor;
}

__device__ __forceinline__ void tma_gather4(uint32_t dst, const void* map, int c0, int r0, int r1, int r2, int r3,
                                            uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
      ::"r"(dst), "l"(map), "r"(c0), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar)
      : "memory");
}

template <int NQ>
__global__ void __launch_bounds__(kThreads, 1)
    indexer_fp8_kernel(const __grid_constant__ CUtensorMap tmap_keys, const __grid_constant__ CUtensorMap tmap_scales,
                       const __grid_constant__ CUtensorMap tmap_q, const IdxParams p) {
  using L = IdxSmem<NQ>;
  constexpr int kStages = L::kStages;
  constexpr int N = 32 * NQ;
  constexpr uint32_t kTmemCols = (4 * N <= 128) ? 128 : (4 * N <= 256 ? 256 : 512);  // power of two
  constexpr uint32_t kIdesc = make_idesc(kFmtE4M3, kFmtE4M3, 0, 0, 128, N);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + L::kOffBars;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (kStages + s); };
  auto accf_bar = [&](int a) { return bars + 8u * (2 * kStages + a); };
  auto acce_bar = [&](int a) { return bars + 8u * (2 * kStages + 2 + a); };
  auto qf_bar = [&](int q) { return bars + 8u * (2 * kStages + 4 + q); };
  auto qe_bar = [&](int q) { return bars + 8u * (2 * kStages + 6 + q); };
  const uint32_t done_bar = bars + 8u * (2 * kStages + 8);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);
  int32_t* prefix = reinterpret_cast<int32_t*>(smem + L::kOffPrefix);
  const float* scales_smem = reinterpret_cast<const float*>(smem + L::kOffScales);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cap = min(p.max_blocks * kBlock, p.max_seq_len);

  // ---- set-up: barriers, TMEM, per-sequence unit prefix sums
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 4);
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(accf_bar(a), 1);
      mbar_init(acce_bar(a), 4);
      mbar_init(qf_bar(a), 1);
      mbar_init(qe_bar(a), 1);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap_keys);
    prefetch_tmap(&tmap_scales);
    prefetch_tmap(&tmap_q);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  if (warp == 0) {
    int run = 0;
    for (int b0 = 0; b0 < p.batch; b0 += 32) {
      int b = b0 + lane;
      int units = 0;
      if (b < p.batch) {
        int len = p.seq_lens[b];
        if (len < 0 || len > cap) {
          report(p.status, DSA_ERR_BOUNDS);
          len = len < 0 ? 0 : cap;
        }
        units = (len + kUnitKeys - 1) / kUnitKeys;
      }
      int incl = units;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (b < p.batch) prefix[b] = run + incl - units;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) prefix[p.batch] = run;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int64_t total = prefix[p.batch];
  const int64_t u_begin = total * blockIdx.x / gridDim.x;
  const int64_t u_end = total * (blockIdx.x + 1) / gridDim.x;

  auto seq_len_of = [&](int b) {
    int len = p.seq_lens[b];
    return len < 0 ? 0 : (len > cap ? cap : len);
  };
  auto first_seq = [&](int64_t u) {
    int lo = 0, hi = p.batch - 1;  // last b with prefix[b] <= u
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if (prefix[mid] <= u) lo = mid; else hi = mid - 1;
    }
    return lo;
  };

  if (u_begin < u_end) {
    if (warp == 0) {
      // ------------------------------------------------ TMA producer (one warp)
      // The lanes resolve the block-table rows of the next 32 units while lane 0
      // issues the copies of the current 32, so table reads never stall the ring.
      constexpr unsigned kAll = 0xffffffffu;
      auto resolve = [&](int64_t g, int& rb, int& rnp, int (&rr)[kPagesPerUnit]) {
        const int64_t u = g + lane;
        rb = 0;
        rnp = 0;
#pragma unroll
        for (int q = 0; q < kPagesPerUnit; ++q) rr[q] = 0;
        if (u < u_end) {
          rb = first_seq(u);
          const int j = (int)(u - prefix[rb]);
          const int rem = seq_len_of(rb) - kUnitKeys * j;
          rnp = min(kPagesPerUnit, (rem + kBlock - 1) / kBlock);
          const int32_t* bt = p.block_table + (int64_t)rb * p.max_blocks + kPagesPerUnit * j;
#pragma unroll
          for (int q = 0; q < kPagesPerUnit; ++q) rr[q] = q < rnp ? bt[q] : 0;
        }
      };
      int cb, cnp, cr[kPagesPerUnit];
      resolve(u_begin, cb, cnp, cr);
      const uint64_t stream_policy = policy_evict_first();  // keys are read once per step
      int cur_b = -1;
      uint32_t it = 0, qn = 0;
      bool ok = true;
      for (int64_t g = u_begin; ok && g < u_end; g += 32) {
        int nb, nnp, nr[kPagesPerUnit];
        resolve(g + 32, nb, nnp, nr);  // next group's rows, in flight meanwhile
        const int n = (int)((u_end - g) < 32 ? (u_end - g) : 32);
        for (int l = 0; l < n; ++l, ++it) {
          const int b = __shfl_sync(kAll, cb, l);
          const int npages = __shfl_sync(kAll, cnp, l);
          int r[kPagesPerUnit];
#pragma unroll
          for (int q = 0; q < kPagesPerUnit; ++q) r[q] = __shfl_sync(kAll, cr[q], l);
          if (lane == 0) {
            if (b != cur_b) {
              const int slot = qn & 1;
              ok = mbar_wait(qe_bar(slot), ((qn >> 1) & 1) ^ 1, abort_flag, p.status);
              if (ok) {
                mbar_arrive_expect_tx(qf_bar(slot), L::kQSlot);
                tma_load_2d(sbase + L::kOffQ + slot * L::kQSlot, &tmap_q, 0, b * N, qf_bar(slot));
                ++qn;
                cur_b = b;
              }
            }
            const int s = it % kStages;
            ok = ok && mbar_wait(empty_bar(s), ((it / kStages) & 1) ^ 1, abort_flag, p.status);
            if (ok) {
#pragma unroll
              for (int q = 0; q < kPagesPerUnit; ++q) {
                if (q >= npages) r[q] = r[0];  // gather rows must be valid; unused pages repeat page 0
                if (r[q] < 0 || r[q] >= p.num_blocks) {
                  report(p.status, DSA_ERR_BOUNDS);
                  r[q] = 0;  // read a valid row instead; the call's results are void
                }
              }
              mbar_arrive_expect_tx(full_bar(s), npages * kPageCodeBytes + kUnitScaleBytes);
              for (int q = 0; q < npages; ++q)
                tma_load_3d_hint(sbase + L::kOffA + s * kATileBytes + q * kPageCodeBytes, &tmap_keys, 0, 0, r[q],
                                 full_bar(s), stream_policy);
              tma_gather4(sbase + L::kOffScales + s * kUnitScaleBytes, &tmap_scales, 0, r[0], r[1], r[2], r[3],
                          full_bar(s));
            }
          }
          ok = __shfl_sync(kAll, ok, 0);
          if (!ok) break;
        }
        cb = nb;
        cnp = nnp;
#pragma unroll
        for (int q = 0; q < kPagesPerUnit; ++q) cr[q] = nr[q];
      }
      if (lane == 0 && *abort_flag) {  // let copies already in flight land before the CTA exits
        for (uint32_t k = (it > kStages ? it - kStages : 0); k < it; ++k)
          mbar_wait(full_bar(k % kStages), (k / kStages) & 1, abort_flag, nullptr, 10000000ull);
      }
    } else if (warp == 1 && lane == 0) {
      // ------------------------------------------------ MMA issuer
      int cursor = first_seq(u_begin), cur_b = -1;
      uint32_t it = 0, qn = 0;
      for (int64_t u = u_begin; u < u_end; ++u, ++it) {
        const int b = seq_of_unit(prefix, p.batch, u, cursor);
        if (b != cur_b) {
          if (cur_b >= 0) mma_commit(qe_bar((qn - 1) & 1));
          if (!mbar_wait(qf_bar(qn & 1), (qn >> 1) & 1, abort_flag, p.status)) break;
          ++qn;
          cur_b = b;
        }
        const int s = it % kStages, a = it & 1;
        if (!mbar_wait(full_bar(s), (it / kStages) & 1, abort_flag, p.status)) break;
        if (!mbar_wait(acce_bar(a), ((it >> 1) & 1) ^ 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t b_base = sbase + L::kOffQ + ((qn - 1) & 1) * L::kQSlot;
#pragma unroll
        for (int sub = 0; sub < 2; ++sub) {
          const uint32_t a_base = sbase + L::kOffA + s * kATileBytes + sub * kSubTileBytes;
#pragma unroll
          for (int kk = 0; kk < kIdxDim / 32; ++kk) {
            const uint64_t ad = smem_desc(a_base + 32 * kk, 16, 1024, kLayoutSw128);
            const uint64_t bd = smem_desc(b_base + 32 * kk, 16, 1024, kLayoutSw128);
            mma_f8f6f4(tmem + (2 * a + sub) * N, ad, bd, kIdesc, kk > 0 ? 1u : 0u);
          }
        }
        mma_commit(accf_bar(a));
      }
      // all issued MMAs must finish before TMEM is released
      mma_commit(done_bar);
      mbar_wait(done_bar, 0, abort_flag, nullptr, 10000000ull);
    } else if (warp >= 2) {
      // ------------------------------------------------ epilogue
      const int quarter = warp & 3;
      const int row = quarter * 32 + lane;  // TMEM lane = key row of each 128-key sub-tile
      int cursor = first_seq(u_begin), cur_b = -1;
      float w[NQ][kIdxHeads];
      const uint64_t keep_policy = policy_evict_last();  // the top-k reads the scores next
      uint32_t it = 0;
      for (int64_t u = u_begin; u < u_end; ++u, ++it) {
        const int b = seq_of_unit(prefix, p.batch, u, cursor);
        if (b != cur_b) {
#pragma unroll
          for (int q = 0; q < NQ; ++q) {
            const float4* wp = reinterpret_cast<const float4*>(p.head_w + ((int64_t)b * NQ + q) * kIdxHeads);
#pragma unroll
            for (int h4 = 0; h4 < kIdxHeads / 4; ++h4) {
              float4 v = __ldg(wp + h4);
              w[q][4 * h4 + 0] = v.x;
              w[q][4 * h4 + 1] = v.y;
              w[q][4 * h4 + 2] = v.z;
              w[q][4 * h4 + 3] = v.w;
            }
          }
          cur_b = b;
        }
        const int s = it % kStages, a = it & 1;
        bool ok = mbar_wait(accf_bar(a), (it >> 1) & 1, abort_flag, p.status);
        ok = ok && mbar_wait(full_bar(s), (it / kStages) & 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) break;   // warp-uniform: tcgen05.ld below is warp-collective
        tc_fence_after();
        const int j = (int)(u - prefix[b]);
        const int len = seq_len_of(b);
        const int t0 = kUnitKeys * j + row, t1 = t0 + 128;
        const float sc0 = scales_smem[s * (kUnitScaleBytes / 4) + row];
        const float sc1 = scales_smem[s * (kUnitScaleBytes / 4) + 128 + row];
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          uint32_t r0[32], r1[32];
          tmem_ld32(lane_base + (2 * a) * N + 32 * q, r0);
          tmem_ld32(lane_base + (2 * a + 1) * N + 32 * q, r1);
          tmem_ld_wait();
          float s0 = 0.f, s1 = 0.f;
#pragma unroll
          for (int h = 0; h < kIdxHeads; ++h) {
            s0 = fmaf(w[q][h], fmaxf(sc0 * __uint_as_float(r0[h]), 0.f), s0);
            s1 = fmaf(w[q][h], fmaxf(sc1 * __uint_as_float(r1[h]), 0.f), s1);
          }
          const int vis = visible_len(len, NQ, q);
          float* out = p.scores + ((int64_t)b * NQ + q) * p.ld;
          if (t0 < vis) st_global_hint(out + t0, s0, keep_policy);
          if (t1 < vis) st_global_hint(out + t1, s1, keep_policy);
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(acce_bar(a));
          mbar_arrive(empty_bar(s));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <int NQ>
dsa_status_t launch_nq(const IdxParams& p, const CUtensorMap& keys, const CUtensorMap& scales,
                       const CUtensorMap& q, cudaStream_t st) {
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  const size_t smem = IdxSmem<NQ>::bytes(kMaxBatch);
  if (dev < 64 && !attr_set[dev]) {
    if (cuda_status(cudaFuncSetAttribute(indexer_fp8_kernel<NQ>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem)) != DSA_OK)
      return DSA_ERR_CUDA;
    attr_set[dev] = true;
  }
  const int64_t units_bound = (int64_t)p.batch * ((p.max_seq_len + kUnitKeys - 1) / kUnitKeys);
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(units_bound, num_sms()));
  indexer_fp8_kernel<NQ><<<grid, kThreads, IdxSmem<NQ>::bytes(p.batch), st>>>(keys, scales, q, p);
  return launch_status();
}

}  // namespace

dsa_status_t launch_index_scores_fp8(const dsa_paged_cache_t& c, const dsa_batch_t& bt, const uint8_t* q_index,
                                     const float* head_w, float* scores, int64_t ld, int32_t* status,
                                     cudaStream_t st) {
  if (bt.batch > kMaxBatch) return DSA_ERR_UNSUPPORTED;
  const uint8_t* index_base = static_cast<const uint8_t*>(c.base) + c.index_off;
  CUtensorMap keys, scales, qmap;
  // codes: the pool as [num_blocks][64 tokens][128 B], one 64 x 128 box per page
  {
    const uint64_t dims[3] = {(uint64_t)kIdxDim, (uint64_t)kBlock, (uint64_t)c.num_blocks};
    const uint64_t strides[2] = {(uint64_t)kIdxDim, (uint64_t)c.row_stride};
    const uint32_t box[3] = {(uint32_t)kIdxDim, (uint32_t)kBlock, 1};
    if (!encode_tmap(&keys, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, index_base, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return DSA_ERR_CUDA;
  }
  // scales: the pool as [num_blocks][256 B of fp32 scales], one-row boxes for gather4
  {
    const uint64_t dims[2] = {(uint64_t)kPageScaleBytes, (uint64_t)c.num_blocks};
    const uint64_t strides[1] = {(uint64_t)c.row_stride};
    const uint32_t box[2] = {(uint32_t)kPageScaleBytes, 1};
    if (!encode_tmap(&scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, index_base + kPageCodeBytes, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_NONE))
      return DSA_ERR_CUDA;
  }
  const int nq = bt.queries_per_seq;
  {
    const uint64_t rows = (uint64_t)bt.batch * nq * kIdxHeads;
    const uint64_t dims[2] = {(uint64_t)kIdxDim, rows};
    const uint64_t strides[1] = {(uint64_t)kIdxDim};
    const uint32_t box[2] = {(uint32_t)kIdxDim, (uint32_t)(kIdxHeads * nq)};
    if (!encode_tmap(&qmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, q_index, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return DSA_ERR_CUDA;
  }
  IdxParams p{index_base, c.row_stride, c.num_blocks, bt.block_table, bt.max_blocks_per_seq, bt.seq_lens,
              bt.batch, bt.max_seq_len, head_w, scores, ld, status};
  switch (nq) {
    case 1: return launch_nq<1>(p, keys, scales, qmap, st);
    case 2: return launch_nq<2>(p, keys, scales, qmap, st);
    case 3: return launch_nq<3>(p, keys, scales, qmap, st);
    case 4: return launch_nq<4>(p, keys, scales, qmap, st);
    default: return DSA_ERR_UNSUPPORTED;
  }
}

}  // namespace dsa
