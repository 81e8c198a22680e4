// prefill.cu — lightning-indexer scores of a prefill chunk (stage 1 of DSA
// with many query rows per sequence).
//
// The scores are those of indexer.cu,
//     s[r][t] = sum_h w[r][h] * max(0, scale_t * (q[r][h] . k[t])),
// 32 heads x 128 dims, FP8 keys, for the causal rows of a chunk: row j of a
// sequence with context L and nq rows sees L - (nq - 1) + j tokens (vLLM
// Day-0 post for Kimi K3.1 Pro, prefill section: each GPU runs the indexer
// for its own tokens over the whole context with all heads; its cost is
// quadratic in the chunk).  With nq rows per sequence the contraction is
// dense (nq x 32 query-heads against every key), so the rows share each key
// read and the tensor cores see N = 256 per instruction.
//
// GB300 design.  A work item is 512 keys of one sequence (eight 64-token
// pages) and a range of the chunk's 8-row query groups.  The grid is
// persistent, one CTA per SM, items split evenly across CTAs.  Per CTA:
//   warp 0  TMA producer: the item's eight key pages (128-byte swizzle, 64 KB)
//           and their fp32 scale rows (two tile::gather4 copies) into one key
//           buffer; then, per query group, the group's 8 x 32 query-head rows
//           (32 KB, 128-byte swizzle) and 8 x 32 head weights (1 KB) into a
//           4-slot ring;
//   warp 1  MMA issuer: per query group and 128-key sub-tile, four
//           tcgen05.mma kind::f8f6f4 (M = 128 keys, N = 256 query-heads,
//           K = 32) into one of two 256-column TMEM accumulators;
//   warps 2-17 epilogue: warp w reads TMEM lanes 32 (w % 4) .. + 31 (one key
//           each) and the columns of rows 2 ((w - 2) / 4) and the next, 16
//           heads of both rows at a time, frees the accumulator, then: ReLU,
//           head weight and the sum over 32 heads on CUDA cores (pairs of
//           heads in one packed fp32 FMA, the two rows interleaved), the
//           key's scale, one coalesced store per warp and row.  With a
//           non-negative finite scale (every key the cache update writes) the
//           scale is applied once after the sum, since max(0, c x) =
//           c max(0, x) for c >= 0; otherwise inside the ReLU.
// The ReLU and the weighted head sum (48 instructions per key and row at
// best) on CUDA cores, not the MMA, bound this stage: four epilogue warps per
// sub-partition keep the issue slots busy, and the MMA of a group runs
// under the epilogue of the one before.  (Measured alternatives: 4-row groups
// with one row per warp and the weights in registers, and 6-row groups with
// twelve warps, both spent more instructions per score on the per-tile
// handshakes than they saved on weight reads.)
#include <algorithm>
#include <atomic>
#include <cmath>

#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace dsa {

namespace {

constexpr int kPfKeys = 512;                         // keys per work item
constexpr int kPfPages = kPfKeys / kBlock;           // 8
constexpr int kPfSub = kPfKeys / 128;                // M = 128 sub-tiles per item
constexpr int kPfRows = 8;                           // query rows per group: two per epilogue warp of a lane quarter
constexpr int kPfN = kPfRows * kIdxHeads;            // 256 query-heads: the MMA's N
constexpr int kPfQBytes = kPfN * kIdxDim;            // 32 KB per query group
constexpr int kPfWBytes = kPfRows * kIdxHeads * 4;   // 1 KB of head weights per group
constexpr int kPfSlots = 4;                          // query ring
constexpr int kPfAcc = 2;                            // TMEM accumulators (2 x 256 columns)
constexpr int kPfEpiWarps = 16;
constexpr int kPfThreads = (2 + kPfEpiWarps) * 32;   // 576
constexpr int kPfPageBytes = kBlock * kIdxDim;       // 8 KB
constexpr int kPfScaleRowBytes = kBlock * 4;         // 256 B of fp32 scales per page
constexpr int kPfMaxBatch = 4096;
constexpr uint64_t kPfDrainNs = 10000000ull;

constexpr int kPfOffK = 0;
constexpr int kPfOffQ = kPfOffK + kPfPages * kPfPageBytes;      // 65,536
constexpr int kPfOffScale = kPfOffQ + kPfSlots * kPfQBytes;      // 196,608
constexpr int kPfOffW = kPfOffScale + kPfPages * kPfScaleRowBytes;  // 198,656
constexpr int kPfOffBars = kPfOffW + kPfSlots * kPfWBytes;       // 202,752
// key full/empty, query full/empty [slots], accumulator full/empty [kPfAcc], done
constexpr int kPfNumBars = 2 + 2 * kPfSlots + 2 * kPfAcc + 1;
constexpr int kPfOffMisc = (kPfOffBars + kPfNumBars * 8 + 15) / 16 * 16;  // tmem slot, abort flag, gsplit
constexpr int kPfOffPrefix = kPfOffMisc + 16;
static_assert(kPfOffQ % 1024 == 0 && kPfQBytes % 1024 == 0, "swizzle atoms");
static_assert(kPfAcc * kPfN <= 512 && kPfEpiWarps == 2 * kPfRows, "TMEM columns, epilogue rows");
static_assert(kPfOffScale % 16 == 0 && kPfOffW % 16 == 0 && kPfOffBars % 8 == 0, "alignment");

size_t pf_smem_bytes(int batch) { return 1024 + kPfOffPrefix + 4 * (size_t)(batch + 1); }

struct PfParams {
  int32_t num_blocks;
  const int32_t* block_table;
  int32_t max_blocks;
  const int32_t* seq_lens;
  int32_t batch;
  int32_t nq;          // query rows per sequence (>= 8)
  int32_t max_seq_len;
  float* scores;       // [batch * nq][ld], fp32, or bf16 at (uint16_t*)scores
  int64_t ld;
  int32_t score_bf16;
  int32_t* status;
};

__device__ __forceinline__ void pf_gather4(uint32_t dst, const void* map, int r0, int r1, int r2, int r3,
                                           uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile::gather4.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%2, %3, %4, %5, %6}], [%7];"
      ::"r"(dst), "l"(map), "r"(0), "r"(r0), "r"(r1), "r"(r2), "r"(r3), "r"(bar)
      : "memory");
}

// Two fp32 lanes of a 64-bit register: d = a * b + c, each lane rounded once.
__device__ __forceinline__ uint64_t ffma2(uint64_t a, uint64_t b, uint64_t c) {
  uint64_t d;
  asm("fma.rn.f32x2 %0, %1, %2, %3;" : "=l"(d) : "l"(a), "l"(b), "l"(c));
  return d;
}
__device__ __forceinline__ uint64_t pack2(float lo, float hi) {
  return (uint64_t)__float_as_uint(lo) | ((uint64_t)__float_as_uint(hi) << 32);
}
__device__ __forceinline__ float lo_of(uint64_t v) { return __uint_as_float((uint32_t)v); }
__device__ __forceinline__ float hi_of(uint64_t v) { return __uint_as_float((uint32_t)(v >> 32)); }

__global__ void __launch_bounds__(kPfThreads, 1)
    prefill_indexer_kernel(const __grid_constant__ CUtensorMap tmap_keys, const __grid_constant__ CUtensorMap tmap_scales,
                           const __grid_constant__ CUtensorMap tmap_q, const __grid_constant__ CUtensorMap tmap_w,
                           const PfParams p) {
  constexpr uint32_t kIdesc = make_idesc(kFmtE4M3, kFmtE4M3, 0, 0, 128, kPfN);
  constexpr uint32_t kTmemCols = 512;  // kPfAcc accumulators of kPfN columns

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kPfOffBars;
  const uint32_t kfull = bars, kempty = bars + 8u;
  auto qfull = [&](int s) { return bars + 8u * (2 + s); };
  auto qempty = [&](int s) { return bars + 8u * (2 + kPfSlots + s); };
  auto accf = [&](int a) { return bars + 8u * (2 + 2 * kPfSlots + a); };
  auto acce = [&](int a) { return bars + 8u * (2 + 2 * kPfSlots + kPfAcc + a); };
  const uint32_t done_bar = bars + 8u * (2 + 2 * kPfSlots + 2 * kPfAcc);
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kPfOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kPfOffMisc + 4);
  int32_t* gsplit_s = reinterpret_cast<int32_t*>(smem + kPfOffMisc + 8);
  int32_t* prefix = reinterpret_cast<int32_t*>(smem + kPfOffPrefix);  // key items before sequence b
  const float* scale_f = reinterpret_cast<const float*>(smem + kPfOffScale);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cap = min(p.max_blocks * kBlock, p.max_seq_len);
  const int nq = p.nq;
  const int ngroups = (nq + kPfRows - 1) / kPfRows;

  if (threadIdx.x == 0) {
    mbar_init(kfull, 1);
    mbar_init(kempty, 1 + kPfEpiWarps);  // the MMAs' commit and the epilogue (key scales)
    for (int s = 0; s < kPfSlots; ++s) {
      mbar_init(qfull(s), 1);
      mbar_init(qempty(s), 1 + kPfEpiWarps);  // the MMAs' commit and the epilogue (head weights)
    }
    for (int a = 0; a < kPfAcc; ++a) {
      mbar_init(accf(a), 1);
      mbar_init(acce(a), kPfEpiWarps);
    }
    mbar_init(done_bar, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap_keys);
    prefetch_tmap(&tmap_scales);
    prefetch_tmap(&tmap_q);
    prefetch_tmap(&tmap_w);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  auto seq_len_of = [&](int b) {
    const int len = p.seq_lens[b];
    return len < 0 ? 0 : (len > cap ? cap : len);
  };
  if (warp == 0) {
    // key items (512 keys) per sequence, as an exclusive prefix sum
    int run = 0;
    for (int b0 = 0; b0 < p.batch; b0 += 32) {
      const int b = b0 + lane;
      int n = 0;
      if (b < p.batch) {
        const int raw = p.seq_lens[b];
        if (raw < 0 || raw > cap) report(p.status, DSA_ERR_BOUNDS);
        n = (seq_len_of(b) + kPfKeys - 1) / kPfKeys;
      }
      int incl = n;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        const int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (b < p.batch) prefix[b] = run + incl - n;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) {
      prefix[p.batch] = run;
      // split each key item's query groups so that every CTA gets about two items or more
      const int want = (2 * (int)gridDim.x + max(run, 1) - 1) / max(run, 1);
      *gsplit_s = max(1, min(ngroups, want));
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  const int gsplit = *gsplit_s;
  const int gper = (ngroups + gsplit - 1) / gsplit;
  const int64_t total = (int64_t)prefix[p.batch] * gsplit;
  const int64_t i_begin = total * blockIdx.x / gridDim.x;
  const int64_t i_end = total * (blockIdx.x + 1) / gridDim.x;

  // An item: sequence b, key block kb (keys [512 kb, +512)), query groups [g0, g1).
  struct Item {
    int b, kb, g0, g1, len, k0;
  };
  auto item_of = [&](int64_t i) {
    Item it;
    const int ki = (int)(i / gsplit), gs = (int)(i % gsplit);
    int lo = 0, hi = p.batch - 1;  // last b with prefix[b] <= ki
    while (lo < hi) {
      const int mid = (lo + hi + 1) >> 1;
      if (prefix[mid] <= ki) lo = mid; else hi = mid - 1;
    }
    it.b = lo;
    it.kb = ki - prefix[lo];
    it.g0 = gs * gper;
    it.g1 = min(ngroups, it.g0 + gper);
    it.len = seq_len_of(lo);
    it.k0 = it.kb * kPfKeys;
    return it;
  };
  // 128-key sub-tiles of the item that group g sees (0: the group sees none of its keys)
  auto nsub_of = [&](const Item& it, int g) {
    const int vis_hi = visible_len(it.len, nq, min(kPfRows * g + kPfRows - 1, nq - 1));
    return vis_hi > it.k0 ? min(kPfSub, (vis_hi - it.k0 + 127) / 128) : 0;
  };
  auto item_live = [&](const Item& it) {
    for (int g = it.g0; g < it.g1; ++g)
      if (nsub_of(it, g) > 0) return true;
    return false;
  };

  if (i_begin < i_end) {
    if (warp == 0) {
      if (lane == 0) {
        // ------------------------------------------------ TMA producer
        uint32_t kc = 0, qn = 0;
        bool ok = true;
        for (int64_t i = i_begin; ok && i < i_end; ++i) {
          const Item it = item_of(i);
          if (!item_live(it)) continue;
          if (!(ok = mbar_wait(kempty, (kc & 1) ^ 1, abort_flag, p.status))) break;
          const int npages = min(kPfPages, (it.len - it.k0 + kBlock - 1) / kBlock);
          const int32_t* bt = p.block_table + (int64_t)it.b * p.max_blocks + it.kb * kPfPages;
          int rows[kPfPages];
#pragma unroll
          for (int q = 0; q < kPfPages; ++q) {
            int r = q < npages ? bt[q] : -1;
            if (q < npages && (r < 0 || r >= p.num_blocks)) {
              report(p.status, DSA_ERR_BOUNDS);
              r = 0;  // read a valid row instead; the call's results are void
            }
            rows[q] = r;
          }
#pragma unroll
          for (int q = 1; q < kPfPages; ++q)
            if (rows[q] < 0) rows[q] = rows[0];  // gather rows must be valid: unused pages repeat page 0
          mbar_arrive_expect_tx(kfull, npages * kPfPageBytes + kPfPages * kPfScaleRowBytes);
          for (int q = 0; q < npages; ++q)
            tma_load_3d(sbase + kPfOffK + q * kPfPageBytes, &tmap_keys, 0, 0, rows[q], kfull);
          pf_gather4(sbase + kPfOffScale, &tmap_scales, rows[0], rows[1], rows[2], rows[3], kfull);
          pf_gather4(sbase + kPfOffScale + 4 * kPfScaleRowBytes, &tmap_scales, rows[4], rows[5], rows[6], rows[7],
                     kfull);
          ++kc;
          for (int g = it.g0; g < it.g1; ++g) {
            if (nsub_of(it, g) == 0) continue;
            const int s = qn % kPfSlots;
            if (!(ok = mbar_wait(qempty(s), ((qn / kPfSlots) & 1) ^ 1, abort_flag, p.status))) break;
            const int row0 = it.b * nq + kPfRows * g;  // rows past the chunk: the next sequence's or zero fill
            mbar_arrive_expect_tx(qfull(s), kPfQBytes + kPfWBytes);
            tma_load_2d(sbase + kPfOffQ + s * kPfQBytes, &tmap_q, 0, row0 * kIdxHeads, qfull(s));
            tma_load_2d(sbase + kPfOffW + s * kPfWBytes, &tmap_w, 0, row0, qfull(s));
            ++qn;
          }
        }
        if (*abort_flag) {  // let copies already in flight land before the CTA exits
          if (kc > 0) mbar_wait_drain(kfull, (kc - 1) & 1, kPfDrainNs);
          for (uint32_t k = (qn > kPfSlots ? qn - kPfSlots : 0); k < qn; ++k)
            mbar_wait_drain(qfull(k % kPfSlots), (k / kPfSlots) & 1, kPfDrainNs);
        }
      }
    } else if (warp == 1) {
      if (lane == 0) {
        // ------------------------------------------------ MMA issuer
        uint32_t kc = 0, qn = 0, an = 0;
        bool ok = true;
        for (int64_t i = i_begin; ok && i < i_end; ++i) {
          const Item it = item_of(i);
          if (!item_live(it)) continue;
          if (!(ok = mbar_wait(kfull, kc & 1, abort_flag, p.status))) break;
          for (int g = it.g0; ok && g < it.g1; ++g) {
            const int nsub = nsub_of(it, g);
            if (nsub == 0) continue;
            const int s = qn % kPfSlots;
            if (!(ok = mbar_wait(qfull(s), (qn / kPfSlots) & 1, abort_flag, p.status))) break;
            for (int st = 0; st < nsub; ++st) {
              const int a = an % kPfAcc;
              if (!(ok = mbar_wait(acce(a), ((an / kPfAcc) & 1) ^ 1, abort_flag, p.status))) break;
              tc_fence_after();
#pragma unroll
              for (int kk = 0; kk < kIdxDim / 32; ++kk) {
                const uint64_t ad = smem_desc(sbase + kPfOffK + st * 128 * kIdxDim + 32 * kk, 16, 1024, kLayoutSw128);
                const uint64_t bd = smem_desc(sbase + kPfOffQ + s * kPfQBytes + 32 * kk, 16, 1024, kLayoutSw128);
                mma_f8f6f4(tmem + a * kPfN, ad, bd, kIdesc, kk > 0 ? 1u : 0u);
              }
              mma_commit(accf(a));
              ++an;
            }
            mma_commit(qempty(s));  // the slot's query tile is free once these MMAs have read it
            ++qn;
          }
          mma_commit(kempty);
          ++kc;
        }
        // every issued MMA must finish before TMEM is released
        mma_commit(done_bar);
        mbar_wait_drain(done_bar, 0, kPfDrainNs);
      }
    } else {
      // ------------------------------------------------ epilogue
      const int quarter = warp & 3;
      const int r0 = 2 * ((warp - 2) >> 2);        // rows r0, r0 + 1 of each group
      const int key_in_sub = quarter * 32 + lane;  // TMEM lane
      const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16) + r0 * kIdxHeads;
      uint32_t kc = 0, qn = 0, an = 0;
      bool ok = true;
      for (int64_t i = i_begin; ok && i < i_end; ++i) {
        const Item it = item_of(i);
        if (!item_live(it)) continue;
        ok = mbar_wait(kfull, kc & 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
        for (int g = it.g0; ok && g < it.g1; ++g) {
          const int nsub = nsub_of(it, g);
          if (nsub == 0) continue;
          const int s = qn % kPfSlots;
          ok = mbar_wait(qfull(s), (qn / kPfSlots) & 1, abort_flag, p.status);
          if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
          // the two rows' head weights: broadcast shared-memory reads at each use
          const float4* w0 = reinterpret_cast<const float4*>(smem + kPfOffW + s * kPfWBytes) + r0 * (kIdxHeads / 4);
          const float4* w1 = w0 + kIdxHeads / 4;
          const int j0 = kPfRows * g + r0;  // rows j0, j0 + 1 within the sequence's chunk
          const int vis0 = j0 < nq ? visible_len(it.len, nq, j0) : 0;
          const int vis1 = j0 + 1 < nq ? visible_len(it.len, nq, j0 + 1) : 0;
          const int64_t row_off = ((int64_t)it.b * nq + j0) * p.ld;
          for (int st = 0; st < nsub; ++st) {
            const int a = an % kPfAcc;
            ok = mbar_wait(accf(a), (an / kPfAcc) & 1, abort_flag, p.status);
            if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }   // tcgen05.ld below is warp-collective
            tc_fence_after();
            ++an;
            const float sc = scale_f[st * 128 + key_in_sub];
            const bool fast = __all_sync(0xffffffffu, sc >= 0.f && sc < INFINITY);
            // 16 heads of both rows at a time (registers): on the fast path two
            // packed pairs of partial sums per row, the rows interleaved
            uint64_t p0[2] = {0, 0}, p1[2] = {0, 0};
            float s0 = 0.f, s1 = 0.f;
#pragma unroll
            for (int hh = 0; hh < 2; ++hh) {
              uint32_t x0[16], x1[16];
              tmem_ld16(lane_base + a * kPfN + 16 * hh, x0);
              tmem_ld16(lane_base + a * kPfN + kIdxHeads + 16 * hh, x1);
              tmem_ld_wait();
              if (hh == 1) {
                tc_fence_before();
                __syncwarp();
                if (lane == 0) mbar_arrive(acce(a));  // the accumulator is in registers: the next MMAs may start
              }
              if (fast) {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                  const float4 u = w0[4 * hh + q4], v = w1[4 * hh + q4];
                  p0[0] = ffma2(pack2(u.x, u.y), pack2(fmaxf(__uint_as_float(x0[4 * q4]), 0.f),
                                                       fmaxf(__uint_as_float(x0[4 * q4 + 1]), 0.f)), p0[0]);
                  p1[0] = ffma2(pack2(v.x, v.y), pack2(fmaxf(__uint_as_float(x1[4 * q4]), 0.f),
                                                       fmaxf(__uint_as_float(x1[4 * q4 + 1]), 0.f)), p1[0]);
                  p0[1] = ffma2(pack2(u.z, u.w), pack2(fmaxf(__uint_as_float(x0[4 * q4 + 2]), 0.f),
                                                       fmaxf(__uint_as_float(x0[4 * q4 + 3]), 0.f)), p0[1]);
                  p1[1] = ffma2(pack2(v.z, v.w), pack2(fmaxf(__uint_as_float(x1[4 * q4 + 2]), 0.f),
                                                       fmaxf(__uint_as_float(x1[4 * q4 + 3]), 0.f)), p1[1]);
                }
              } else {
#pragma unroll
                for (int q4 = 0; q4 < 4; ++q4) {
                  const float4 u = w0[4 * hh + q4], v = w1[4 * hh + q4];
                  s0 = fmaf(u.x, fmaxf(sc * __uint_as_float(x0[4 * q4 + 0]), 0.f), s0);
                  s0 = fmaf(u.y, fmaxf(sc * __uint_as_float(x0[4 * q4 + 1]), 0.f), s0);
                  s0 = fmaf(u.z, fmaxf(sc * __uint_as_float(x0[4 * q4 + 2]), 0.f), s0);
                  s0 = fmaf(u.w, fmaxf(sc * __uint_as_float(x0[4 * q4 + 3]), 0.f), s0);
                  s1 = fmaf(v.x, fmaxf(sc * __uint_as_float(x1[4 * q4 + 0]), 0.f), s1);
                  s1 = fmaf(v.y, fmaxf(sc * __uint_as_float(x1[4 * q4 + 1]), 0.f), s1);
                  s1 = fmaf(v.z, fmaxf(sc * __uint_as_float(x1[4 * q4 + 2]), 0.f), s1);
                  s1 = fmaf(v.w, fmaxf(sc * __uint_as_float(x1[4 * q4 + 3]), 0.f), s1);
                }
              }
            }
            float sum0 = s0, sum1 = s1;
            if (fast) {
              sum0 = sc * ((lo_of(p0[0]) + hi_of(p0[0])) + (lo_of(p0[1]) + hi_of(p0[1])));
              sum1 = sc * ((lo_of(p1[0]) + hi_of(p1[0])) + (lo_of(p1[1]) + hi_of(p1[1])));
            }
            const int t = it.k0 + st * 128 + key_in_sub;
            if (p.score_bf16) {
              uint16_t* out = reinterpret_cast<uint16_t*>(p.scores) + row_off + t;
              if (t < vis0) out[0] = __bfloat16_as_ushort(__float2bfloat16_rn(sum0));
              if (t < vis1) out[p.ld] = __bfloat16_as_ushort(__float2bfloat16_rn(sum1));
            } else {
              float* out = p.scores + row_off + t;
              if (t < vis0) out[0] = sum0;
              if (t < vis1) out[p.ld] = sum1;
            }
          }
          __syncwarp();
          if (lane == 0) mbar_arrive(qempty(s));  // this warp has read the group's head weights
          ++qn;
        }
        __syncwarp();
        if (lane == 0) mbar_arrive(kempty);  // this warp has read the item's key scales
        ++kc;
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  grid_dep_launch();  // the top-k may be placed now
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

}  // namespace

dsa_status_t launch_prefill_scores(const dsa_paged_cache_t& c, const dsa_batch_t& bt, const uint8_t* q_index,
                                   const float* head_w, void* scores, bool bf16, int64_t ld, int32_t* status,
                                   cudaStream_t st) {
  const int nq = bt.queries_per_seq;
  if (c.key_format != DSA_KEY_FP8_E4M3 || nq < kPfRows) return DSA_ERR_UNSUPPORTED;
  if (bt.batch > kPfMaxBatch) return DSA_ERR_UNSUPPORTED;
  const uint8_t* index_base = static_cast<const uint8_t*>(c.base) + c.index_off;
  CUtensorMap keys, scales, qmap, wmap;
  {  // codes: the pool as [num_blocks][64 tokens][128 bytes], one 64-row box per page
    const uint64_t dims[3] = {(uint64_t)kIdxDim, (uint64_t)kBlock, (uint64_t)c.num_blocks};
    const uint64_t strides[2] = {(uint64_t)kIdxDim, (uint64_t)c.row_stride};
    const uint32_t box[3] = {(uint32_t)kIdxDim, (uint32_t)kBlock, 1};
    if (!encode_tmap(&keys, CU_TENSOR_MAP_DATA_TYPE_UINT8, 3, index_base, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return DSA_ERR_CUDA;
  }
  {  // fp32 scales: the pool as [num_blocks][256 B], one-row boxes for gather4
    const uint64_t dims[2] = {(uint64_t)kPfScaleRowBytes, (uint64_t)c.num_blocks};
    const uint64_t strides[1] = {(uint64_t)c.row_stride};
    const uint32_t box[2] = {(uint32_t)kPfScaleRowBytes, 1};
    if (!encode_tmap(&scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, index_base + kBlock * kIdxDim, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_NONE))
      return DSA_ERR_CUDA;
  }
  const uint64_t rows = (uint64_t)bt.batch * nq;
  {  // query codes: [rows * 32 heads][128 bytes], 8 rows x 32 heads per box
    const uint64_t dims[2] = {(uint64_t)kIdxDim, rows * kIdxHeads};
    const uint64_t strides[1] = {(uint64_t)kIdxDim};
    const uint32_t box[2] = {(uint32_t)kIdxDim, (uint32_t)kPfN};
    if (!encode_tmap(&qmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, q_index, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_128B))
      return DSA_ERR_CUDA;
  }
  {  // head weights: [rows][32] fp32, 8 rows per box
    const uint64_t dims[2] = {(uint64_t)kIdxHeads, rows};
    const uint64_t strides[1] = {(uint64_t)kIdxHeads * 4};
    const uint32_t box[2] = {(uint32_t)kIdxHeads, (uint32_t)kPfRows};
    if (!encode_tmap(&wmap, CU_TENSOR_MAP_DATA_TYPE_FLOAT32, 2, head_w, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_NONE))
      return DSA_ERR_CUDA;
  }
  static std::atomic<bool> attr_set[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    if (cuda_status(cudaFuncSetAttribute(prefill_indexer_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)pf_smem_bytes(kPfMaxBatch))) != DSA_OK)
      return DSA_ERR_CUDA;
    attr_set[dev] = true;
  }
  const int64_t items_bound = (int64_t)bt.batch * ((bt.max_seq_len + kPfKeys - 1) / kPfKeys) *
                              ((nq + kPfRows - 1) / kPfRows);
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(items_bound, num_sms()));
  PfParams p{c.num_blocks, bt.block_table, bt.max_blocks_per_seq, bt.seq_lens, bt.batch, nq, bt.max_seq_len,
             static_cast<float*>(scores), ld, bf16 ? 1 : 0, status};
  count_launches(1);
  prefill_indexer_kernel<<<grid, kPfThreads, pf_smem_bytes(bt.batch), st>>>(keys, scales, qmap, wmap, p);
  return launch_status();
}

}  // namespace dsa
