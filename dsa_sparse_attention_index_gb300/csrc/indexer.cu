// indexer.cu — lightning-indexer scores for decode (stage 1 of DSA).
//
// Computes, for every query row r = b*NQ + j and every visible token t,
//     s[r][t] = sum_h w[r][h] * max(0, scale_t * (q[r][h] . k[t]))
// with 32 heads x 128 dims (vLLM Day-0 post for Kimi K3.1 Pro, section
// "K3.1 Pro 中的稀疏注意力": 32 light heads, a 132-byte FP8 key incl. scale;
// AMD section: FP32 accumulation and a weighted reduction across heads).
// MXFP4 keys (68 bytes: 64 bytes of E2M1 codes, four E8M0 block scales) give
// q[r][h] . k[t] = sum over the four 32-element blocks of 2^(E - 127) times
// the block's dot product, and scale_t = 1.
//
// GB300 design.  Each key carries 32*128 multiply-adds (62 FLOP per FP8 byte,
// 120 per MXFP4 byte): at HBM speed that is several times what the CUDA
// cores can issue, so the dot products run on the 5th-gen tensor cores even
// in decode.  A work unit is one sequence's 256 consecutive tokens (four
// 64-token pages).  The grid is persistent (one CTA per SM) and the units of
// all sequences are split evenly across CTAs ("key-balanced", Day-0 post,
// fused decode section).  Per CTA:
//   warp 0  TMA producer: per unit, four 64-token code pages (3-D tensor map
//           over the block pool, 128-byte swizzle; MXFP4 codes land as
//           8-byte packed chunks 16 bytes apart, the layout the block-scaled
//           MMA reads) into a 5-6 stage code ring, and
//           the four pages' scale rows in one tile::gather4 copy into a
//           deeper scale ring.  The two half-warps issue two units at once;
//           the lanes resolve the block-table rows of the next 32 units; the
//           query tiles go into a 2-slot ring, one sequence ahead;
//   warp 1  MMA issuer: two M = 128 key sub-tiles per unit, N = 32*NQ
//           query-heads, K = 128 in four K=32 steps, fp32 accumulators in a
//           double-buffered TMEM tile.  FP8: tcgen05.mma kind::f8f6f4.
//           MXFP4: kind::mxf8f6f4.block_scale, E2M1 x E4M3 with the keys'
//           E8M0 block scales read from TMEM (queries: scale 2^0), so one
//           accumulator per sub-tile already holds q . k.  Native FP4 (an
//           MXFP4 query too; AMD section: native FP4 matrix instructions):
//           kind::mxf4.block_scale, both operands packed E2M1 (64-byte rows,
//           64-byte swizzle), two K = 64 steps, both sides' E8M0 scales from
//           TMEM; the packed stage is half the FP8 one, so 11 stages hold
//           the keys in flight that HBM needs.  The code stage is released by
//           tcgen05.commit as soon as its MMAs complete;
//   warps 2-5 epilogue: each thread owns two key rows (one per sub-tile),
//           reads their 32*NQ accumulators with tcgen05.ld, applies the FP8
//           scale, ReLU and the head weights, sums the heads in registers
//           and stores one fp32 score per query row (coalesced per warp);
//   warps 6-9 (MXFP4 only) scale staging: per unit, copy the 256 keys' E8M0
//           words from the scale ring into TMEM, laid out as the
//           block-scaled MMA reads them (key row m: lane m % 32, column
//           m / 32, byte = 32-element block); native FP4 also writes the
//           unit's query words (head n: lane n, one column per slot, the
//           slots 32 columns apart as the keys' are).
// All draft rows of a sequence share one key read (AMD section: keys are
// reused across query rows during speculative verify).
#include <algorithm>
#include <atomic>

#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace dsa {

namespace {

constexpr int kUnitKeys = 256;                          // four pages
constexpr int kPagesPerUnit = kUnitKeys / kBlock;       // 4
constexpr int kSubTileBytes = 128 * kIdxDim;            // 16 KB: one M = 128 MMA tile (one byte per element)
constexpr int kATileBytes = kUnitKeys * kIdxDim;        // 32 KB of codes per unit in shared memory
constexpr int kPageCodeBytes = kBlock * kIdxDim;        // 8 KB in shared memory (MXFP4: 4 KB read)
constexpr int kPagePackedBytes = kBlock * kIdxDim / 2;  // 4 KB: a page of packed E2M1 codes (native FP4)
constexpr int kPageScaleBytes = kBlock * 4;             // 256 B
constexpr int kUnitScaleBytes = kPagesPerUnit * kPageScaleBytes;  // 1 KB (one gather4)
constexpr int kMaxBatch = 4096;
constexpr uint64_t kDrainNs = 10000000ull;              // bound on draining in-flight work at exit

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
  int32_t score_bf16;  // scores are bf16 (round to nearest even) at (uint16_t*)scores, else fp32
  const uint32_t* q_scales;  // native FP4: the query's E8M0 words [rows][32] (4 blocks a word), else null
};

constexpr int kSfSlots = 4;  // MXFP4: TMEM scale-factor slots, decoupled from the accumulators

// Shared memory of the indexer.  NAT (native FP4): the code stages hold packed
// E2M1 (16 KB a unit), so nearly twice as many fit and twice the keys are in
// flight for the same bytes.
template <int NQ, bool NAT = false>
struct IdxSmem {
  static constexpr int kATile = NAT ? kUnitKeys * kIdxDim / 2 : kATileBytes;  // bytes of one code stage
  static constexpr int kPageSmem = NAT ? kPagePackedBytes : kPageCodeBytes;   // bytes of one page in a stage
  static constexpr int kStages = NAT ? 11 : (NQ == 1 ? 6 : 5);  // code ring; keeps the CTA within 227 KB
  static constexpr int kScaleStages = kStages + 2;      // scale slots are held until the epilogue ends
  static constexpr int kQSlot = NAT ? 32 * kIdxDim / 2 : 32 * NQ * kIdxDim;  // bytes
  static constexpr int kOffA = 0;
  static constexpr int kOffQ = kOffA + kStages * kATile;
  static constexpr int kOffScales = kOffQ + 2 * kQSlot;
  static constexpr int kOffBars = kOffScales + kScaleStages * kUnitScaleBytes;
  // barriers: code full/empty [S], scale full/empty [SS], acc full/empty [2],
  // q full/empty [2], done, MXFP4 scale-factor slots staged/free [kSfSlots]
  static constexpr int kNumBars = 2 * kStages + 2 * kScaleStages + 9 + 2 * kSfSlots;
  static constexpr int kOffMisc = kOffBars + kNumBars * 8;  // tmem slot, abort flag
  static constexpr int kOffPrefix = kOffMisc + 16;
  static size_t bytes(int batch) { return 1024 + kOffPrefix + 4 * (size_t)(batch + 1); }
};

template <bool MX>
constexpr int idx_threads() { return MX ? 320 : 192; }

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

// KF = 0: FP8 keys (E4M3 codes + fp32 scale).  KF = 1: MXFP4 keys (E2M1 codes
// + E8M0 block scales, applied by the block-scaled MMA) against the E4M3
// query.  KF = 2: the MXFP4 keys against an MXFP4 query, both packed, on the
// native FP4 x FP4 MMA.
template <int NQ, int KF>
__global__ void __launch_bounds__(idx_threads<KF != 0>(), 1)
    indexer_kernel(const __grid_constant__ CUtensorMap tmap_keys, const __grid_constant__ CUtensorMap tmap_scales,
                   const __grid_constant__ CUtensorMap tmap_q, const IdxParams p) {
  constexpr bool MX = KF != 0, NAT = KF == 2;
  using L = IdxSmem<NQ, NAT>;
  static_assert(!MX || NQ == 1, "MXFP4 keys: one query row per sequence");
  constexpr int kStages = L::kStages;
  constexpr int kSS = L::kScaleStages;
  constexpr int N = 32 * NQ;
  // TMEM: accumulators [2 slots][2 sub-tiles][N] at column 0; MXFP4 adds the
  // keys' scale factors (4 columns per sub-tile, at 32-column steps, in
  // kSfSlots slots) and the queries' (2^0; native FP4: the query's words, one
  // column per slot, at 32-column steps like the keys': a scale-factor address
  // off that grid faults)
  constexpr uint32_t kTmemCols = MX ? 512 : ((4 * N <= 128) ? 128 : (4 * N <= 256 ? 256 : 512));
  constexpr uint32_t kSfaCol = 128, kSfbCol = kSfaCol + 64 * kSfSlots;
  static_assert(!MX || kSfbCol + 32 * (kSfSlots - 1) + 1 <= kTmemCols, "TMEM columns");
  constexpr uint32_t kIdesc = NAT  ? make_idesc_mx(kFmtMxf4E2M1, kFmtMxf4E2M1, 128, N)
                              : MX ? make_idesc_mx(kFmtE2M1, kFmtE4M3, 128, N)
                                   : make_idesc(kFmtE4M3, kFmtE4M3, 0, 0, 128, N);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + L::kOffBars;
  auto full_bar = [&](int s) { return bars + 8u * s; };
  auto empty_bar = [&](int s) { return bars + 8u * (kStages + s); };
  auto scf_bar = [&](int s) { return bars + 8u * (2 * kStages + s); };
  auto sce_bar = [&](int s) { return bars + 8u * (2 * kStages + kSS + s); };
  const uint32_t bars2 = bars + 8u * (2 * kStages + 2 * kSS);
  auto accf_bar = [&](int a) { return bars2 + 8u * a; };
  auto acce_bar = [&](int a) { return bars2 + 8u * (2 + a); };
  auto qf_bar = [&](int q) { return bars2 + 8u * (4 + q); };
  auto qe_bar = [&](int q) { return bars2 + 8u * (6 + q); };
  const uint32_t done_bar = bars2 + 8u * 8;
  auto sfr_bar = [&](int f) { return bars2 + 8u * (9 + f); };
  auto sfe_bar = [&](int f) { return bars2 + 8u * (9 + kSfSlots + f); };
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + L::kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + L::kOffMisc + 4);
  int32_t* prefix = reinterpret_cast<int32_t*>(smem + L::kOffPrefix);
  const uint32_t* scale_words = reinterpret_cast<const uint32_t*>(smem + L::kOffScales);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int cap = min(p.max_blocks * kBlock, p.max_seq_len);

  // ---- set-up: barriers, TMEM, per-sequence unit prefix sums
  if (threadIdx.x == 0) {
    for (int s = 0; s < kStages; ++s) {
      mbar_init(full_bar(s), 1);
      mbar_init(empty_bar(s), 1);   // tcgen05.commit of the unit's MMAs
    }
    for (int s = 0; s < kSS; ++s) {
      mbar_init(scf_bar(s), 1);
      mbar_init(sce_bar(s), 4);     // FP8: the epilogue warps; MXFP4: the scale-staging warps
    }
    for (int a = 0; a < 2; ++a) {
      mbar_init(accf_bar(a), 1);
      mbar_init(acce_bar(a), 4);
      mbar_init(qf_bar(a), 1);
      mbar_init(qe_bar(a), 1);
    }
    for (int f = 0; f < kSfSlots; ++f) {
      mbar_init(sfr_bar(f), 4);   // the four scale-staging warps
      mbar_init(sfe_bar(f), 1);   // tcgen05.commit of the MMAs that read the slot
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
  const int nb = p.batch;
  // length of sequence b, clamped to [0, cap]
  auto seq_len_of = [&](int b) {
    const int len = p.seq_lens[b];
    return len < 0 ? 0 : (len > cap ? cap : len);
  };
  if (warp == 0) {
    int run = 0;
    for (int b0 = 0; b0 < nb; b0 += 32) {
      int b = b0 + lane;
      int units = 0;
      if (b < nb) {
        const int raw = p.seq_lens[b];
        if (raw < 0 || raw > cap) report(p.status, DSA_ERR_BOUNDS);
        units = (seq_len_of(b) + kUnitKeys - 1) / kUnitKeys;
      }
      int incl = units;
#pragma unroll
      for (int o = 1; o < 32; o <<= 1) {
        int v = __shfl_up_sync(0xffffffffu, incl, o);
        if (lane >= o) incl += v;
      }
      if (b < nb) prefix[b] = run + incl - units;
      run += __shfl_sync(0xffffffffu, incl, 31);
    }
    if (lane == 0) prefix[nb] = run;
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  const int64_t total = prefix[nb];
  const int64_t u_begin = total * blockIdx.x / gridDim.x;
  const int64_t u_end = total * (blockIdx.x + 1) / gridDim.x;

  auto first_seq = [&](int64_t u) {
    int lo = 0, hi = nb - 1;  // last b with prefix[b] <= u
    while (lo < hi) {
      int mid = (lo + hi + 1) >> 1;
      if (prefix[mid] <= u) lo = mid; else hi = mid - 1;
    }
    return lo;
  };

  if (u_begin < u_end) {
    if (warp == 0) {
      // ------------------------------------------------ TMA producer (one warp)
      // Two units per step: half-warp h (lanes 16h .. 16h+15) issues unit
      // it + h, so the barrier operations and copies of both go out in the
      // same instructions.  The lanes resolve the block-table rows of the next
      // 32 units while the current 32 are issued.
      constexpr unsigned kAll = 0xffffffffu;
      const int half = lane >> 4, hl = lane & 15;
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
      // Query tiles go into the 2-slot ring in the order the MMA meets the
      // sequences.  A load waits (blocking) only for sequences up to `need`,
      // whose earlier units are all issued; one more is loaded ahead when its
      // slot is already free.
      const int q_last = first_seq(u_end - 1);
      int q_seq = first_seq(u_begin);  // next sequence whose query tile is to be loaded
      uint32_t qn = 0;                 // query tiles issued
      auto issue_q = [&](int need) -> bool {
        while (q_seq <= q_last) {
          const int slot = qn & 1;
          const uint32_t par = ((qn >> 1) & 1) ^ 1;
          if (q_seq <= need) {
            if (!mbar_wait(qe_bar(slot), par, abort_flag, p.status)) return false;
          } else if (q_seq > need + 1 || !mbar_try_wait(qe_bar(slot), par)) {
            break;
          }
          mbar_arrive_expect_tx(qf_bar(slot), L::kQSlot);
          tma_load_2d(sbase + L::kOffQ + slot * L::kQSlot, &tmap_q, 0, q_seq * N, qf_bar(slot));
          ++qn;
          do {
            ++q_seq;  // skip sequences without keys: the MMA never meets them
          } while (q_seq <= q_last && prefix[q_seq + 1] == prefix[q_seq]);
        }
        return true;
      };
      int cb, cnp, cr[kPagesPerUnit];
      resolve(u_begin, cb, cnp, cr);
      const uint64_t stream_policy = policy_evict_first();  // keys are read once per step
      uint32_t it = 0;
      bool ok = true;
      for (int64_t g = u_begin; ok && g < u_end; g += 32) {
        int nb, nnp, nr[kPagesPerUnit];
        resolve(g + 32, nb, nnp, nr);  // next group's rows, in flight meanwhile
        const int n = (int)((u_end - g) < 32 ? (u_end - g) : 32);
        for (int l = 0; l < n; l += 2) {
          const int lu = l + half;  // this half-warp's unit within the group
          const bool valid = lu < n;
          const int src = valid ? lu : l;
          const int b = __shfl_sync(kAll, cb, src);
          int npages = __shfl_sync(kAll, cnp, src);
          if (!valid) npages = 0;
          int r[kPagesPerUnit];
#pragma unroll
          for (int q = 0; q < kPagesPerUnit; ++q) r[q] = __shfl_sync(kAll, cr[q], src);
#pragma unroll
          for (int q = 0; q < kPagesPerUnit; ++q) {
            if (q >= npages) r[q] = r[0];  // gather rows must be valid; unused pages repeat page 0
            if (r[q] < 0 || r[q] >= p.num_blocks) {
              if (hl == 0 && valid) report(p.status, DSA_ERR_BOUNDS);
              r[q] = 0;  // read a valid row instead; the call's results are void
            }
          }
          const uint32_t uit = it + half;
          const int s = uit % kStages, s2 = uit % kSS;
          if (lane == 0) ok = issue_q(b);  // lane 0 holds the pair's first unit
          ok = __shfl_sync(kAll, ok, 0);
          bool okh = ok;
          if (ok && hl == 0 && valid) {
            okh = mbar_wait(empty_bar(s), ((uit / kStages) & 1) ^ 1, abort_flag, p.status) &&
                  mbar_wait(sce_bar(s2), ((uit / kSS) & 1) ^ 1, abort_flag, p.status);
            if (okh) {
              // MXFP4 pages are 4 KB in HBM (the unpacking copy of KF = 1 counts its source bytes)
              mbar_arrive_expect_tx(full_bar(s), npages * (MX ? kPagePackedBytes : kPageCodeBytes));
              mbar_arrive_expect_tx(scf_bar(s2), kUnitScaleBytes);
            }
          }
          ok = __all_sync(kAll, okh);
          if (!ok) break;
          // lane hl < npages of each half loads page hl; lane 4 of each half gathers the scale rows
          if (hl < npages) {
            const int rq = hl == 0 ? r[0] : (hl == 1 ? r[1] : (hl == 2 ? r[2] : r[3]));
            tma_load_3d_hint(sbase + L::kOffA + s * L::kATile + hl * L::kPageSmem, &tmap_keys, 0, 0, rq,
                             full_bar(s), stream_policy);
          } else if (hl == kPagesPerUnit && valid) {
            tma_gather4(sbase + L::kOffScales + s2 * kUnitScaleBytes, &tmap_scales, 0, r[0], r[1], r[2], r[3],
                        scf_bar(s2));
          }
          it += (l + 1 < n) ? 2 : 1;
        }
        cb = nb;
        cnp = nnp;
#pragma unroll
        for (int q = 0; q < kPagesPerUnit; ++q) cr[q] = nr[q];
      }
      if (lane == 0 && ok) issue_q(q_last);  // every unit is issued: remaining query tiles may wait
      if (lane == 0 && *abort_flag) {  // let copies already in flight land before the CTA exits
        for (uint32_t k = (it > kStages ? it - kStages : 0); k < it; ++k)
          mbar_wait_drain(full_bar(k % kStages), (k / kStages) & 1, kDrainNs);
        for (uint32_t k = (it > kSS ? it - kSS : 0); k < it; ++k)
          mbar_wait_drain(scf_bar(k % kSS), (k / kSS) & 1, kDrainNs);
        for (uint32_t k = (qn > 2 ? qn - 2 : 0); k < qn; ++k) mbar_wait_drain(qf_bar(k & 1), (k >> 1) & 1, kDrainNs);
      }
    } else if (warp == 1 && lane == 0) {
      // ------------------------------------------------ MMA issuer
      int cursor = first_seq(u_begin), cur_b = -1;
      uint32_t it = 0, qn = 0;
      for (int64_t u = u_begin; u < u_end; ++u, ++it) {
        const int b = seq_of_unit(prefix, nb, u, cursor);
        if (b != cur_b) {
          if (cur_b >= 0) mma_commit(qe_bar((qn - 1) & 1));
          if (!mbar_wait(qf_bar(qn & 1), (qn >> 1) & 1, abort_flag, p.status)) break;
          ++qn;
          cur_b = b;
        }
        const int s = it % kStages, a = it & 1, f = it % kSfSlots;
        if (!mbar_wait(full_bar(s), (it / kStages) & 1, abort_flag, p.status)) break;
        if (MX && !mbar_wait(sfr_bar(f), (it / kSfSlots) & 1, abort_flag, p.status)) break;
        if (!mbar_wait(acce_bar(a), ((it >> 1) & 1) ^ 1, abort_flag, p.status)) break;
        tc_fence_after();
        const uint32_t b_base = sbase + L::kOffQ + ((qn - 1) & 1) * L::kQSlot;
#pragma unroll
        for (int sub = 0; sub < 2; ++sub) {
          if constexpr (NAT) {
            // packed E2M1, 64-byte rows with the 64-byte swizzle (8-row groups 512 B apart);
            // K = 64 per MMA: E8M0 bytes 2 kk and 2 kk + 1 of the scale words
            const uint32_t a_base = sbase + L::kOffA + s * L::kATile + sub * (128 * kIdxDim / 2);
#pragma unroll
            for (int kk = 0; kk < kIdxDim / 64; ++kk)
              mma_mxf4(tmem + (2 * a + sub) * N, smem_desc(a_base + 32 * kk, 16, 512, kLayoutSw64),
                       smem_desc(b_base + 32 * kk, 16, 512, kLayoutSw64), kIdesc | mx_sf_ids(2 * kk, 2 * kk),
                       tmem + kSfaCol + 32 * (2 * f + sub), tmem + kSfbCol + 32 * f, kk > 0 ? 1u : 0u);
            continue;
          }
          const uint32_t a_base = sbase + L::kOffA + s * kATileBytes + sub * kSubTileBytes;
#pragma unroll
          for (int kk = 0; kk < kIdxDim / 32; ++kk) {
            const uint64_t ad = smem_desc(a_base + 32 * kk, 16, 1024, kLayoutSw128);
            const uint64_t bd = smem_desc(b_base + 32 * kk, 16, 1024, kLayoutSw128);
            if constexpr (MX)  // K step kk is E8M0 block kk: scale-factor byte kk
              mma_mxf8f6f4(tmem + (2 * a + sub) * N, ad, bd, kIdesc | mx_sf_ids(kk, kk),
                           tmem + kSfaCol + 32 * (2 * f + sub), tmem + kSfbCol, kk > 0 ? 1u : 0u);
            else
              mma_f8f6f4(tmem + (2 * a + sub) * N, ad, bd, kIdesc, kk > 0 ? 1u : 0u);
          }
        }
        mma_commit(accf_bar(a));
        mma_commit(empty_bar(s));   // the code stage is free once these MMAs have read it
        if (MX) mma_commit(sfe_bar(f));
      }
      // all issued MMAs must finish before TMEM is released
      mma_commit(done_bar);
      mbar_wait_drain(done_bar, 0, kDrainNs);
    } else if (warp >= 2 && warp < 6) {
      // ------------------------------------------------ epilogue
      const int quarter = warp & 3;
      const int row = quarter * 32 + lane;  // TMEM lane = key row of each 128-key sub-tile
      int cursor = first_seq(u_begin), cur_b = -1;
      float w[NQ][kIdxHeads];
      const uint64_t keep_policy = policy_evict_last();  // the top-k reads the scores next
      uint32_t it = 0;
      for (int64_t u = u_begin; u < u_end; ++u, ++it) {
        const int b = seq_of_unit(prefix, nb, u, cursor);
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
        const int s2 = it % kSS, a = it & 1;
        bool ok = mbar_wait(accf_bar(a), (it >> 1) & 1, abort_flag, p.status);
        if (!MX) ok = ok && mbar_wait(scf_bar(s2), (it / kSS) & 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) break;   // warp-uniform: tcgen05.ld below is warp-collective
        tc_fence_after();
        const int j = (int)(u - prefix[b]);
        const int len = seq_len_of(b);
        const int t0 = kUnitKeys * j + row, t1 = t0 + 128;
        const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16);
        // MXFP4: the block scales are inside the accumulators already
        const float sc0 = MX ? 1.f : __uint_as_float(scale_words[s2 * (kUnitScaleBytes / 4) + row]);
        const float sc1 = MX ? 1.f : __uint_as_float(scale_words[s2 * (kUnitScaleBytes / 4) + 128 + row]);
#pragma unroll
        for (int q = 0; q < NQ; ++q) {
          uint32_t r0[32], r1[32];
          tmem_ld32(lane_base + (2 * a) * N + 32 * q, r0);
          tmem_ld32(lane_base + (2 * a + 1) * N + 32 * q, r1);
          tmem_ld_wait();
          float s0 = 0.f, s1 = 0.f;
#pragma unroll
          for (int h = 0; h < kIdxHeads; ++h) {
            if constexpr (MX) {
              s0 = fmaf(w[q][h], fmaxf(__uint_as_float(r0[h]), 0.f), s0);
              s1 = fmaf(w[q][h], fmaxf(__uint_as_float(r1[h]), 0.f), s1);
            } else {
              s0 = fmaf(w[q][h], fmaxf(sc0 * __uint_as_float(r0[h]), 0.f), s0);
              s1 = fmaf(w[q][h], fmaxf(sc1 * __uint_as_float(r1[h]), 0.f), s1);
            }
          }
          const int vis = visible_len(len, NQ, q);
          const int64_t ro = ((int64_t)b * NQ + q) * p.ld;
          if (p.score_bf16) {
            uint16_t* out = reinterpret_cast<uint16_t*>(p.scores) + ro;
            if (t0 < vis) st_global_hint(out + t0, __bfloat16_as_ushort(__float2bfloat16_rn(s0)), keep_policy);
            if (t1 < vis) st_global_hint(out + t1, __bfloat16_as_ushort(__float2bfloat16_rn(s1)), keep_policy);
          } else {
            float* out = p.scores + ro;
            if (t0 < vis) st_global_hint(out + t0, s0, keep_policy);
            if (t1 < vis) st_global_hint(out + t1, s1, keep_policy);
          }
        }
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(acce_bar(a));
          if (!MX) mbar_arrive(sce_bar(s2));
        }
      }
    } else if (MX && warp >= 6) {
      // ------------------------------------------------ MXFP4 scale staging
      // Key row m of a sub-tile takes its E8M0 word from TMEM lane m % 32,
      // column m / 32; every warp writes the same words into its own lane
      // quarter.  The queries' scale words (2^0 in every byte) are written once.
      const uint32_t lane_base = tmem + ((uint32_t)((warp & 3) * 32) << 16);
      if (!NAT) tmem_st4(lane_base + kSfbCol, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu, 0x7F7F7F7Fu);
      int cursor = first_seq(u_begin);
      uint32_t it = 0;
      for (int64_t u = u_begin; u < u_end; ++u, ++it) {
        const int s2 = it % kSS, f = it % kSfSlots;
        // native FP4: head `lane` of the unit's query row (the query's words come from global memory)
        const uint32_t qw = NAT ? __ldg(p.q_scales + (int64_t)seq_of_unit(prefix, nb, u, cursor) * 32 + lane) : 0u;
        bool ok = mbar_wait(scf_bar(s2), (it / kSS) & 1, abort_flag, p.status);
        // slot f's scale factors were last read by the MMAs of unit it - kSfSlots
        ok = ok && mbar_wait(sfe_bar(f), ((it / kSfSlots) & 1) ^ 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) break;   // tcgen05.st is warp-collective
        tc_fence_after();
        const uint32_t* wsrc = scale_words + s2 * (kUnitScaleBytes / 4);
#pragma unroll
        for (int sub = 0; sub < 2; ++sub) {
          const uint32_t* ws = wsrc + 128 * sub + lane;
          tmem_st4(lane_base + kSfaCol + 32 * (2 * f + sub), ws[0], ws[32], ws[64], ws[96]);
        }
        if (NAT) tmem_st1(lane_base + kSfbCol + 32 * f, qw);
        tmem_st_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          mbar_arrive(sfr_bar(f));
          mbar_arrive(sce_bar(s2));
        }
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  // The top-k is launched once every CTA of this grid gets here, i.e. with the
  // scan all but done: its clusters then find the SMs free and are all placed
  // in one wave.  (Triggered at the start, they were placed while the SMs
  // emptied one by one, and the last clusters waited for the first to finish.)
  grid_dep_launch();
  if (warp == 1) tmem_dealloc(tmem, kTmemCols);
}

template <int NQ, int KF>
dsa_status_t launch_nq(const IdxParams& p, const CUtensorMap& keys, const CUtensorMap& scales,
                       const CUtensorMap& q, cudaStream_t st) {
  using L = IdxSmem<NQ, KF == 2>;
  static std::atomic<bool> attr_set[64];
  int dev = 0;
  cudaGetDevice(&dev);
  const size_t smem = L::bytes(kMaxBatch);
  if (dev < 64 && !attr_set[dev]) {
    if (cuda_status(cudaFuncSetAttribute(indexer_kernel<NQ, KF>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem)) != DSA_OK)
      return DSA_ERR_CUDA;
    attr_set[dev] = true;
  }
  const int64_t units_bound = (int64_t)p.batch * ((p.max_seq_len + kUnitKeys - 1) / kUnitKeys);
  const int grid = (int)std::max<int64_t>(1, std::min<int64_t>(units_bound, num_sms()));
  count_launches(1);
  indexer_kernel<NQ, KF><<<grid, idx_threads<KF != 0>(), L::bytes(p.batch), st>>>(keys, scales, q, p);
  return launch_status();
}

}  // namespace

dsa_status_t launch_index_scores(const dsa_paged_cache_t& c, const dsa_batch_t& bt, const uint8_t* q_index,
                                 const float* head_w, void* scores, bool bf16, int64_t ld, int32_t* status,
                                 cudaStream_t st) {
  const bool nat = c.key_format == DSA_KEY_MXFP4_NATIVE;
  const bool mx = c.key_format == DSA_KEY_MXFP4 || nat;
  const int nq = bt.queries_per_seq;
  if (mx && nq != 1) return DSA_ERR_UNSUPPORTED;
  // more than 4 rows per sequence (a prefill chunk): a multiple of 4 rows, scored by
  // the dense-contraction kernel of prefill.cu
  if (nq > 4 && nq % 4 != 0) return DSA_ERR_UNSUPPORTED;
  if (nq > 4) return launch_prefill_scores(c, bt, q_index, head_w, scores, bf16, ld, status, st);
  if (bt.batch > kMaxBatch) return DSA_ERR_UNSUPPORTED;
  const uint8_t* index_base = static_cast<const uint8_t*>(c.base) + c.index_off;
  const int code_bytes = mx ? kIdxDim / 2 : kIdxDim;  // per token in the cache
  const uint64_t rows = (uint64_t)bt.batch * nq;
  CUtensorMap keys, scales, qmap;
  // codes: the pool as [num_blocks][64 tokens][128 elements], one 64-row box per page.  FP8:
  // 128-byte rows, 128-byte swizzle.  MXFP4 against the E4M3 query: the copy unpacks the codes
  // into 8-byte chunks with 8-byte gaps (16 elements per 16 bytes), 128-byte swizzle.  Native
  // FP4: the packed 64-byte rows as they are, 64-byte swizzle.
  {
    const uint64_t dims[3] = {(uint64_t)(nat ? code_bytes : kIdxDim), (uint64_t)kBlock, (uint64_t)c.num_blocks};
    const uint64_t strides[2] = {(uint64_t)code_bytes, (uint64_t)c.row_stride};
    const uint32_t box[3] = {(uint32_t)(nat ? code_bytes : kIdxDim), (uint32_t)kBlock, 1};
    const CUtensorMapDataType type =
        (mx && !nat) ? CU_TENSOR_MAP_DATA_TYPE_16U4_ALIGN16B : CU_TENSOR_MAP_DATA_TYPE_UINT8;
    if (!encode_tmap(&keys, type, 3, index_base, dims, strides, box,
                     nat ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B))
      return DSA_ERR_CUDA;
  }
  // per-token scales (fp32, or four E8M0 bytes): the pool as [num_blocks][256 B], one-row boxes for gather4
  {
    const uint64_t dims[2] = {(uint64_t)kPageScaleBytes, (uint64_t)c.num_blocks};
    const uint64_t strides[1] = {(uint64_t)c.row_stride};
    const uint32_t box[2] = {(uint32_t)kPageScaleBytes, 1};
    if (!encode_tmap(&scales, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, index_base + kBlock * code_bytes, dims, strides, box,
                     CU_TENSOR_MAP_SWIZZLE_NONE))
      return DSA_ERR_CUDA;
  }
  // the query: E4M3 [rows * 32][128] (128-byte swizzle), or native FP4 packed [rows * 32][64]
  // (64-byte swizzle) with its E8M0 words after the codes
  {
    const uint64_t qrow = nat ? kIdxDim / 2 : kIdxDim;
    const uint64_t dims[2] = {qrow, rows * kIdxHeads};
    const uint64_t strides[1] = {qrow};
    const uint32_t box[2] = {(uint32_t)qrow, (uint32_t)(kIdxHeads * nq)};
    if (!encode_tmap(&qmap, CU_TENSOR_MAP_DATA_TYPE_UINT8, 2, q_index, dims, strides, box,
                     nat ? CU_TENSOR_MAP_SWIZZLE_64B : CU_TENSOR_MAP_SWIZZLE_128B))
      return DSA_ERR_CUDA;
  }
  const uint32_t* q_scales = nat ? reinterpret_cast<const uint32_t*>(q_index + rows * kIdxHeads * (kIdxDim / 2))
                                 : nullptr;
  IdxParams p{index_base, c.row_stride, c.num_blocks, bt.block_table, bt.max_blocks_per_seq, bt.seq_lens,
              bt.batch, bt.max_seq_len, head_w, static_cast<float*>(scores), ld, status, bf16 ? 1 : 0, q_scales};
  if (nat) return launch_nq<1, 2>(p, keys, scales, qmap, st);
  if (mx) return launch_nq<1, 1>(p, keys, scales, qmap, st);
  switch (nq) {
    case 1: return launch_nq<1, 0>(p, keys, scales, qmap, st);
    case 2: return launch_nq<2, 0>(p, keys, scales, qmap, st);
    case 3: return launch_nq<3, 0>(p, keys, scales, qmap, st);
    case 4: return launch_nq<4, 0>(p, keys, scales, qmap, st);
    default: return DSA_ERR_UNSUPPORTED;
  }
}

}  // namespace dsa
