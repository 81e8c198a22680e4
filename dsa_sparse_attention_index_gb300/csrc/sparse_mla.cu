// sparse_mla.cu — exact sparse MLA decode over the selected tokens (stage 3).
//
// For every query row and each of the 96 heads: logits over the selected
// tokens' 576-wide latents (absorbed MLA, keys = all 576 columns, values =
// the first 512), an exact softmax, and the weighted sum of values, plus the
// log-sum-exp (vLLM Day-0 post for Kimi K3.1 Pro, sparse-attention section:
// the MLA attention is exact, restricted to the 2,048 selected tokens; the
// prefill section gives the 96 heads).  The selected rows are read straight
// from the packed paged cache through the block table.
//
// GB300 design (one CTA per (query row, token chunk), 12 warps):
//   * Q [96 x 576] bf16 is the A operand of S = Q K^T with the heads on the
//     MMA's M = 128 rows (rows 96..127 are ignored): dims 0..447 loaded once
//     by TMA into shared memory (84 KB, 128-byte swizzle, K-major), dims
//     448..575 written by the softmax warps into TMEM (A from TMEM).  That
//     leaves room for two latent tile buffers of 48 tokens.
//   * warps 4..9 gather 48 latent rows per tile (16-byte loads, three tiles
//     in flight in registers), widen E4M3 -> bf16 exactly and store the tile
//     once, 128-byte swizzled.  That single tile is the B operand of QK^T
//     (K-major, N = 48 tokens) and the A operand of P V (MN-major, M = 128
//     value dims), so V needs no second copy.
//   * two warps issue tcgen05.mma (kind::f16, fp32 accumulation): warp 10
//     S = Q K^T into a 48-column TMEM tile, warp 11 O^T = V^T P^T into
//     4 x 96 TMEM columns (dims on lanes, heads on columns).  The per-MMA
//     cost barely grows with N up to 64, so 48-token tiles issue a third
//     fewer QK^T instructions per token than 32-token ones; TMEM (384 + 48 +
//     64 of 512 columns) then holds one S tile, which the softmax reads out
//     at once so the next QK^T can start.
//   * warps 0..3 (one thread per head) run the online softmax on the S row
//     in registers (exp2 with the scale folded in), write P as bf16 (128-byte
//     swizzled rows, the K-major B operand of PV), and rescale O^T only when
//     a head's running maximum grows by more than 2^8 (exact either way: the
//     final normalisation uses the same reference maximum).
//   * Partial (unnormalised O, max, sums) per chunk go to the workspace and
//     are merged through their log-sum-exp (Day-0 post, DCP section: partial
//     outputs are combined by LSE), inside the row's cluster or by a combine
//     kernel.
#include <algorithm>
#include <atomic>
#include <cmath>

#include <cooperative_groups.h>

#include "common.cuh"
#include "internal.h"

namespace dsa {

namespace {

constexpr int kTileTok = 48;
constexpr int kDBlocks = kLatent / 64;                 // 9 blocks of 64 dims (128 B of bf16)
constexpr int kQTmemBlocks = 2;                        // Q dims 448..575 in TMEM
constexpr int kQSmemBlocks = kDBlocks - kQTmemBlocks;  // Q dims 0..447 in shared memory
constexpr int kQBlockBytes = kHeads * 128;             // 12,288
constexpr int kQBytes = kQSmemBlocks * kQBlockBytes;   // 86,016
constexpr int kTileBufs = 2;
constexpr int kTileDBlockBytes = kTileTok * 128;       // 6,144
constexpr int kTileBytes = kDBlocks * kTileDBlockBytes;  // 55,296
constexpr int kPRowBytes = 128;                        // a head's P row: 48 bf16 in a 128-byte swizzle row
constexpr int kPBytes = kHeads * kPRowBytes;           // 12,288
constexpr int kMaxChunk = 22 * kTileTok;               // 1,056 tokens per CTA
constexpr int kMaskWords = kMaxChunk / 32 + 1;         // token validity bits (+1: tile masks read two words)
constexpr int kInvariantChunk = 512;                   // tokens per CTA in the batch-invariant mode
constexpr int kNvRecord = kValue / 2 + kValue / 16 + (kLatent - kValue);  // 352 B: NVFP4 latent record
constexpr int kNvUnits = kValue / 16;                  // 16-dim units of E2M1 codes (the rest are E4M3)
constexpr int kMaxSplit = 16;                          // chunks per row
constexpr int kMaxFusedSplit = 8;                      // chunks combined inside the kernel (a portable cluster)
// 12 warps: softmax 0-3, loaders 4-9, QK issuer 10, PV issuer 11.  Three warps
// share a sub-partition's register file: room for 168 registers a thread.
constexpr int kThreads = 12 * 32;
constexpr int kLoaderThreads = 192;
constexpr int kMmaWarp = 10;
constexpr int kPvWarp = 11;
constexpr int kChunksPerThread = kTileTok * (kLatent / 16) / kLoaderThreads;  // 9 of the 1,728 16-B units
static_assert(kChunksPerThread * kLoaderThreads == kTileTok * (kLatent / 16), "loader split");
constexpr int kOCols = 4 * kHeads;                     // 384 TMEM columns of O^T
constexpr int kSCol = kOCols;                          // the S tile: columns 384..431
constexpr int kQ8Col = kSCol + 64;                     // Q dims 448..575: 64 columns at 448
constexpr int kTmemCols = 512;
static_assert(kSCol + kTileTok <= kQ8Col && kQ8Col + 32 * kQTmemBlocks <= kTmemCols, "TMEM columns");
constexpr float kRescaleThreshold = 8.0f;              // log2 units

constexpr int kOffQ = 0;
constexpr int kOffTile = kOffQ + kQBytes;                    // 86,016
constexpr int kOffP = kOffTile + kTileBufs * kTileBytes;     // 196,608
constexpr int kOffAlpha = kOffP + 2 * kPBytes;               // 221,184
constexpr int kOffBars = kOffAlpha + 128 * 4;                // 221,696
static_assert(kOffTile % 1024 == 0 && kOffP % 1024 == 0 && kTileDBlockBytes % 1024 == 0, "swizzle atoms");
// q, q8, tiles full/empty, s full/empty, p full, PV done per P buffer, PV drain
constexpr int kNumBars = 2 + 2 * kTileBufs + 2 + 2 + 2 + 1;
constexpr int kOffMisc = kOffBars + kNumBars * 8;
constexpr int kOffTok = kOffMisc + 16;                       // int32 per token: block row * 64 + slot, or -1
constexpr int kOffMask = kOffTok + 4 * kMaxChunk;            // one validity bit per token
constexpr size_t kSmemBytes = 1024 + kOffMask + (size_t)kMaskWords * 4;
static_assert(kSmemBytes <= 232448, "shared memory");

struct MlaParams {
  const uint8_t* latent_base;  // cache base + latent_off
  int64_t row_stride;
  int32_t num_blocks;
  const int32_t* block_table;
  int32_t max_blocks;
  const int32_t* seq_lens;
  int32_t nq;
  int32_t cap;
  const int32_t* idx;
  int32_t k;
  int32_t chunk;    // tokens per CTA
  int32_t nsplit;
  float logit_scale_log2;  // sm_scale * latent_scale * log2(e)
  const uint16_t* q_mla;   // bf16 [rows][96][576]
  uint16_t* opart;  // fp16 [rows][nsplit][96][512]: the chunk's output normalised by its own sum of bf16(p)
  float* ml;        // [rows][nsplit][96][4]: max (log2), sum of bf16(p), sum of p
  int32_t* status;
  // combining in the kernel: a row's nsplit CTAs form a cluster (fuse = 1)
  int32_t fuse;
  float latent_scale;
  uint16_t* out;    // bf16 [rows][96][512]
  float* lse;       // [rows][96]
  // chunk boundaries per row, [rows][nsplit + 1] offsets into idx[row] (chunk
  // `split` is [seg[split], seg[split + 1]), at most `chunk` long), or null:
  // chunk `split` is [split * chunk, (split + 1) * chunk)
  const int32_t* seg;
  // the top-k's physical KV rows beside idx ([rows][k], block row * 64 + slot,
  // -1 padding; visible and bounds-checked by the top-k), or null: the kernel
  // translates idx through the block table itself
  const int32_t* phys;
};

__device__ __forceinline__ float ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

__device__ __forceinline__ bool bar_or_softmax(bool v) {
  uint32_t r;
  asm volatile(
      "{\n .reg .pred p, q;\n setp.ne.u32 q, %1, 0;\n bar.red.or.pred p, 1, 128, q;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(r)
      : "r"((uint32_t)v)
      : "memory");
  return r != 0;
}

// Four fp16 values (bits, low half first) as floats.
__device__ __forceinline__ float4 half4_to_float4(uint2 v) {
  const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&v.x));
  const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&v.y));
  return make_float4(a.x, a.y, b.x, b.y);
}

// The in-cluster merge of a row's NS chunks for this CTA's share [v0, v1) of
// the row's output float4s: every chunk's partial is read from the workspace
// (L2; U x NS 8-byte loads in flight per thread), weighted and summed in
// chunk order with the combine kernel's arithmetic, and written as bf16.  A
// zero weight skips its chunk.  (Reading the peers' partials from their shared
// memory instead was measured slower.)
template <int NS>
__device__ __forceinline__ void merge_share(const uint16_t* opart_row, const float* wgt, int v0, int v1,
                                            uint16_t* out_row) {
  constexpr int U = NS >= 8 ? 2 : NS >= 4 ? 4 : NS >= 2 ? 8 : 16;
  for (int vb = v0 + (int)threadIdx.x; vb < v1; vb += U * kThreads) {
    float4 x[U][NS];
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = vb + u * kThreads;
      if (v < v1) {
        const int hh = v / (kValue / 4), d = (v % (kValue / 4)) * 4;
#pragma unroll
        for (int s = 0; s < NS; ++s)
          if (wgt[hh * kMaxFusedSplit + s] != 0.f)
            x[u][s] = half4_to_float4(*reinterpret_cast<const uint2*>(opart_row + ((int64_t)s * kHeads + hh) * kValue + d));
      }
    }
#pragma unroll
    for (int u = 0; u < U; ++u) {
      const int v = vb + u * kThreads;
      if (v < v1) {
        const int hh = v / (kValue / 4), d = (v % (kValue / 4)) * 4;
        float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
        for (int s = 0; s < NS; ++s) {
          const float w = wgt[hh * kMaxFusedSplit + s];
          if (w != 0.f) {
            a.x = fmaf(w, x[u][s].x, a.x);
            a.y = fmaf(w, x[u][s].y, a.y);
            a.z = fmaf(w, x[u][s].z, a.z);
            a.w = fmaf(w, x[u][s].w, a.w);
          }
        }
        const __nv_bfloat162 lo = __floats2bfloat162_rn(a.x, a.y);
        const __nv_bfloat162 hi = __floats2bfloat162_rn(a.z, a.w);
        uint2 pk;
        pk.x = *reinterpret_cast<const uint32_t*>(&lo);
        pk.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(out_row + hh * kValue + d) = pk;
      }
    }
  }
}

// kNV: NVFP4 latent records (352 B: E2M1 dims 0..511 with an E4M3 scale per
// 16 dims, E4M3 dims 512..575), else E4M3 records (576 B).  Both are widened
// to the same bf16 tile, exactly.
template <bool kNV>
__global__ void __launch_bounds__(kThreads, 1)
    sparse_mla_kernel(const __grid_constant__ CUtensorMap tmap_q, const MlaParams p) {
  constexpr int kRec = kNV ? kNvRecord : kLatent;  // bytes per token record
  // S = Q K^T: A = Q (K-major), B = latent tile (K-major); M = 128, N = 48.
  constexpr uint32_t kIdescQK = make_idesc(kFmtBF16, kFmtBF16, 0, 0, 128, kTileTok);
  // O^T = V^T P^T: A = latent tile (MN-major, M = dims), B = P (K-major); M = 128, N = 96.
  constexpr uint32_t kIdescPV = make_idesc(kFmtBF16, kFmtBF16, 1, 0, 128, kHeads);

  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kOffBars;
  const uint32_t q_full = bars;
  const uint32_t q8_full = bars + 8u;  // Q dims 448..575 written to TMEM by the softmax warps
  auto tile_full = [&](int b) { return bars + 8u * (2 + b); };
  auto tile_empty = [&](int b) { return bars + 8u * (2 + kTileBufs + b); };
  const uint32_t s_full = bars + 8u * (2 + 2 * kTileBufs);
  const uint32_t s_empty = bars + 8u * (3 + 2 * kTileBufs);
  auto p_full = [&](int b) { return bars + 8u * (4 + 2 * kTileBufs + b); };
  auto pv_done = [&](int b) { return bars + 8u * (6 + 2 * kTileBufs + b); };  // PV of the tiles using P buffer b
  const uint32_t pv_drain = bars + 8u * (8 + 2 * kTileBufs);
  // the MMA issuer's teardown barrier reuses q_full's slot after Q has landed
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kOffMisc + 4);
  int32_t* tok_phys = reinterpret_cast<int32_t*>(smem + kOffTok);
  uint32_t* tile_mask = reinterpret_cast<uint32_t*>(smem + kOffMask);
  float* alpha_s = reinterpret_cast<float*>(smem + kOffAlpha);

  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row = blockIdx.y, split = blockIdx.x;
  const int b_seq = row / p.nq;
  const int vis = [&] {
    int len = p.seq_lens[b_seq];
    len = len < 0 ? 0 : (len > p.cap ? p.cap : len);
    return visible_len(len, p.nq, row % p.nq);
  }();
  int c0 = split * p.chunk;
  int count = max(0, min(p.chunk, p.k - c0));

  if (threadIdx.x == 0) {
    mbar_init(q_full, 1);
    mbar_init(q8_full, 4);
    for (int b = 0; b < kTileBufs; ++b) {
      mbar_init(tile_full(b), kLoaderThreads / 32);
      mbar_init(tile_empty(b), 1);
    }
    mbar_init(s_full, 1);
    mbar_init(s_empty, 4);
    for (int b = 0; b < 2; ++b) {
      mbar_init(p_full(b), 4);
      mbar_init(pv_done(b), 1);
    }
    mbar_init(pv_drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap_q);
  }
  if (warp == kMmaWarp) {
    tmem_alloc(smem_u32(tmem_slot), kTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;
  // Q is an input of the step, not an output of the previous kernel, so its
  // loads go out before the wait below when the chunk's size is known without
  // the previous kernel's output (no chunk table): dims 0..447 by TMA into
  // shared memory (the MMA issuer waits for them), dims 448..575 of head h by
  // thread h into TMEM, all sixteen 16-byte loads in flight before the first
  // store.  With a chunk table they go out after the wait, and only for a
  // chunk that is not empty.
  auto issue_q = [&]() {
    if (threadIdx.x == kMmaWarp * 32) {
      mbar_arrive_expect_tx(q_full, kQBytes);
      for (int kb = 0; kb < kQSmemBlocks; ++kb)
        tma_load_2d(sbase + kOffQ + kb * kQBlockBytes, &tmap_q, kb * 64, row * kHeads, q_full);
    }
    if (warp < 4) {
      const int h = threadIdx.x;
      const bool live = h < kHeads;
      const uint4* src = reinterpret_cast<const uint4*>(p.q_mla + ((int64_t)row * kHeads + (live ? h : 0)) * kLatent +
                                                        64 * kQSmemBlocks);
      uint4 v[8 * kQTmemBlocks];
#pragma unroll
      for (int c = 0; c < 8 * kQTmemBlocks; ++c) v[c] = live ? __ldg(src + c) : make_uint4(0, 0, 0, 0);
#pragma unroll
      for (int c = 0; c < 4 * kQTmemBlocks; ++c)
        asm volatile("tcgen05.st.sync.aligned.32x32b.x8.b32 [%0], {%1, %2, %3, %4, %5, %6, %7, %8};"
                     ::"r"(tmem + ((uint32_t)(warp * 32) << 16) + kQ8Col + 8 * c), "r"(v[2 * c].x), "r"(v[2 * c].y),
                     "r"(v[2 * c].z), "r"(v[2 * c].w), "r"(v[2 * c + 1].x), "r"(v[2 * c + 1].y),
                     "r"(v[2 * c + 1].z), "r"(v[2 * c + 1].w)
                     : "memory");
      tmem_st_wait();
      tc_fence_before();
      __syncwarp();
      if (lane == 0) mbar_arrive(q8_full);
    }
  };
  const bool q_early = p.seg == nullptr && count > 0;
  if (q_early) issue_q();
  grid_dep_wait();    // the indices come from the previous kernel
  grid_dep_launch();
  if (p.seg) {
    const int32_t* sg = p.seg + (int64_t)row * (p.nsplit + 1) + split;
    c0 = min(max(sg[0], 0), p.k);
    count = max(0, min(min(sg[1] - c0, p.chunk), p.k - c0));
  }
  const int ntiles = (count + kTileTok - 1) / kTileTok;
  if (!q_early && ntiles > 0) issue_q();
  // physical slots of the chunk's latent rows, block row * 64 + slot (-1: a -1
  // index or padding), and one validity bit per token in 32-token words, by
  // warps 4..11 (warps 0..3 load Q into TMEM meanwhile): every index of a
  // thread is loaded before its block-table entries.  Whole warps run each
  // pass (the bound is a multiple of 32, within kMaxChunk).
  if (warp >= 4) {
    constexpr int kTr = kThreads - 128;
    constexpr int kPer = (kMaxChunk + kTr - 1) / kTr;  // 5
    const int bound = (ntiles * kTileTok + 31) / 32 * 32;
    const int i0 = threadIdx.x - 128;
    int t[kPer], r[kPer];
    if (p.phys) {
      // the top-k's physical rows: visible and bounds-checked already
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int i = i0 + j * kTr;
        const int ph = i < count ? p.phys[(int64_t)row * p.k + c0 + i] : -1;
        t[j] = ph < 0 ? -1 : ph % kBlock;
        r[j] = ph < 0 ? -1 : ph / kBlock;
      }
    } else {
#pragma unroll
      for (int j = 0; j < kPer; ++j) {
        const int i = i0 + j * kTr;
        t[j] = i < count ? p.idx[(int64_t)row * p.k + c0 + i] : -1;
      }
#pragma unroll
      for (int j = 0; j < kPer; ++j)
        r[j] = (t[j] >= 0 && t[j] < vis) ? p.block_table[(int64_t)b_seq * p.max_blocks + t[j] / kBlock] : -1;
    }
#pragma unroll
    for (int j = 0; j < kPer; ++j) {
      const int i = i0 + j * kTr;
      if (i - lane >= bound) break;  // warp-uniform
      int32_t phys = -1;
      if (t[j] >= 0) {
        if (r[j] >= 0 && r[j] < p.num_blocks)
          phys = r[j] * kBlock + t[j] % kBlock;
        else
          report(p.status, DSA_ERR_BOUNDS);
      }
      tok_phys[i] = phys;
      const uint32_t bits = __ballot_sync(0xffffffffu, phys >= 0);  // a warp pass covers 32 consecutive tokens
      if (lane == 0) tile_mask[i >> 5] = bits;
    }
  }
  if (threadIdx.x == 0) tile_mask[(ntiles * kTileTok + 31) / 32] = 0u;  // the word after the last one read
  __syncthreads();

  // this chunk's (running max in log2 units, sum of the rounded p, sum of p)
  // per head, kept by the softmax thread of the head; an empty chunk
  // contributes nothing
  float4 ml_mine = make_float4(-INFINITY, 0.f, 0.f, 0.f);
  if (ntiles > 0) {
    if (warp == kMmaWarp) {
      if (lane == 0) {
        // ------------------------------------------------ QK issuer
        bool ok = mbar_wait(q_full, 0, abort_flag, p.status);
        ok = ok && mbar_wait(q8_full, 0, abort_flag, p.status);
        // Shared-memory descriptors: the start address is the low 14 bits (in
        // 16-byte units) of the low word, so an offset inside shared memory is
        // added to the low word alone; the high word (stride, layout) is fixed.
        const uint64_t q_desc = smem_desc(sbase + kOffQ, 16, 1024, kLayoutSw128);
        const uint32_t q_lo = (uint32_t)q_desc, sw128_hi = (uint32_t)(q_desc >> 32);
        const uint32_t t_lo0 = (uint32_t)smem_desc(sbase + kOffTile, 16, 1024, kLayoutSw128);
        auto issue_qk = [&](int i) {
          const uint32_t d = tmem + kSCol;
          const uint32_t t_lo = t_lo0 + (uint32_t)((i % kTileBufs) * kTileBytes / 16);
#pragma unroll
          for (int kb = 0; kb < kQSmemBlocks; ++kb) {
#pragma unroll
            for (int kk = 0; kk < 4; ++kk)
              mma_bf16(d, desc64(q_lo + (kb * kQBlockBytes + 32 * kk) / 16, sw128_hi),
                       desc64(t_lo + (kb * kTileDBlockBytes + 32 * kk) / 16, sw128_hi), kIdescQK,
                       (kb | kk) ? 1u : 0u);
          }
#pragma unroll
          for (int kk = 0; kk < 4 * kQTmemBlocks; ++kk)  // dims 448..575: A from TMEM, 8 columns per K = 16 step
            mma_bf16_tmem_a(d, tmem + kQ8Col + 8 * kk,
                            desc64(t_lo + ((kQSmemBlocks + kk / 4) * kTileDBlockBytes + 32 * (kk % 4)) / 16, sw128_hi),
                            kIdescQK, 1u);
          mma_commit(s_full);
        };
        for (int i = 0; ok && i < ntiles; ++i) {
          // tile i landed; the S tile read out by the softmax of tile i - 1
          ok = mbar_wait(tile_full(i % kTileBufs), (i / kTileBufs) & 1, abort_flag, p.status) &&
               mbar_wait(s_empty, (i & 1) ^ 1, abort_flag, p.status);
          if (!ok) break;
          tc_fence_after();
          issue_qk(i);
        }
        // wait for every issued MMA before TMEM is released (q_full is free by now)
        mma_commit(q_full);
        mbar_wait_drain(q_full, 1, 10000000ull);
      }
    } else if (warp == kPvWarp) {
      if (lane == 0) {
        // ------------------------------------------------ PV issuer
        // descriptors as in the QK issuer: offsets go to the low word
        const uint64_t a_desc = smem_desc(sbase + kOffTile, kTileDBlockBytes, 1024, kLayoutSw128);
        const uint32_t a_lo0 = (uint32_t)a_desc, a_hi = (uint32_t)(a_desc >> 32);
        const uint64_t p_desc = smem_desc(sbase + kOffP, 16, 1024, kLayoutSw128);
        const uint32_t p_lo0 = (uint32_t)p_desc, p_hi = (uint32_t)(p_desc >> 32);
        for (int i = 0; i < ntiles; ++i) {
          const int b = i & 1;
          if (!mbar_wait(p_full(b), (i >> 1) & 1, abort_flag, p.status)) break;
          tc_fence_after();
          const uint32_t a_lo = a_lo0 + (uint32_t)((i % kTileBufs) * kTileBytes / 16);
          const uint32_t b_lo = p_lo0 + (uint32_t)(b * kPBytes / 16);
#pragma unroll
          for (int mb = 0; mb < 4; ++mb) {
#pragma unroll
            for (int ks = 0; ks < kTileTok / 16; ++ks) {
              // A: dims [128 mb, +128) = two 64-dim atoms (LBO apart), tokens [16 ks, +16) = two 8-row groups
              mma_bf16(tmem + mb * kHeads, desc64(a_lo + (2 * mb * kTileDBlockBytes + 2 * ks * 1024) / 16, a_hi),
                       desc64(b_lo + 32 * ks / 16, p_hi), kIdescPV, (i > 0 || ks > 0) ? 1u : 0u);
            }
          }
          // QK of tile i completed before its P existed, so the tile is free after these
          mma_commit(tile_empty(i % kTileBufs));
          mma_commit(pv_done(b));
        }
        mma_commit(pv_drain);
        mbar_wait_drain(pv_drain, 0, 10000000ull);
      }
    } else if (warp >= 4) {
      // ------------------------------------------------ gather + E4M3 -> bf16
      constexpr int kThreadsPerTok = kLoaderThreads / kTileTok;  // 4
      const int lt = threadIdx.x - 128;                 // 0..191
      const int tok = lt / kThreadsPerTok;               // token row of the tile, 0..47
      const int g = lt % kThreadsPerTok;                 // units g, g+4, ..., g+32 of the 36
      // three tiles in flight per thread (a register ring), so the gather of
      // tile i+3 overlaps the rest; each tile is widened to bf16 in registers
      // before its buffer is free, so only the shared-memory stores wait
      uint4 buf0[kChunksPerThread], buf1[kChunksPerThread], buf2[kChunksPerThread];
      // A unit is 16 dims (32 bytes of bf16 in the tile): for E4M3 records the
      // 16 code bytes; for NVFP4 units below kNvUnits the 8 code bytes (.x, .y)
      // and the scale byte (.z), above them the 16 E4M3 tail bytes.
      auto load = [&](int i, uint4 (&buf)[kChunksPerThread]) {
        if (i >= ntiles) return;
        const int32_t phys = tok_phys[i * kTileTok + tok];
        const uint8_t* rec = p.latent_base + (int64_t)(phys >> 6) * p.row_stride + (phys & (kBlock - 1)) * kRec;
#pragma unroll
        for (int c = 0; c < kChunksPerThread; ++c) {
          const int u = g + kThreadsPerTok * c;
          buf[c] = make_uint4(0, 0, 0, 0);
          if (phys < 0) continue;
          if (!kNV) {
            buf[c] = __ldg(reinterpret_cast<const uint4*>(rec) + u);
          } else if (u < kNvUnits) {
            const uint2 w = __ldg(reinterpret_cast<const uint2*>(rec) + u);
            buf[c] = make_uint4(w.x, w.y, (uint32_t)__ldg(rec + kValue / 2 + u), 0u);
          } else {
            buf[c] = __ldg(reinterpret_cast<const uint4*>(rec + kValue / 2 + kValue / 16) + (u - kNvUnits));
          }
        }
      };
      // widen each unit after the buffer is free (the register ring already
      // holds three raw tiles), then store it 128-byte swizzled
      auto store = [&](int i, const uint4 (&buf)[kChunksPerThread]) -> bool {
        if (i >= ntiles) return true;
        const int b = i % kTileBufs;
        const bool ok = mbar_wait(tile_empty(b), ((i / kTileBufs) & 1) ^ 1, abort_flag, p.status);
        if (!__all_sync(0xffffffffu, ok)) return false;
        uint8_t* tile = smem + kOffTile + b * kTileBytes;
#pragma unroll
        for (int c = 0; c < kChunksPerThread; ++c) {
          const int ch = g + kThreadsPerTok * c;  // 16-dim unit of the 576-dim row: dims [16 ch, +16)
          uint32_t o[8];
          if (kNV && ch < kNvUnits) {
            nvfp4x16_to_bf16x16(buf[c].x, buf[c].y, buf[c].z, o);
          } else {
            const uint32_t w[4] = {buf[c].x, buf[c].y, buf[c].z, buf[c].w};
#pragma unroll
            for (int q = 0; q < 4; ++q) e4m3x4_to_bf16x4(w[q], o[2 * q], o[2 * q + 1]);
          }
          uint8_t* blk = tile + (ch >> 2) * kTileDBlockBytes;
          const uint32_t inner = (uint32_t)((ch & 3) * 32);
          *reinterpret_cast<uint4*>(blk + swz128(tok * 128 + inner)) = make_uint4(o[0], o[1], o[2], o[3]);
          *reinterpret_cast<uint4*>(blk + swz128(tok * 128 + inner + 16)) = make_uint4(o[4], o[5], o[6], o[7]);
        }
        fence_proxy_async_smem();
        __syncwarp();
        if (lane == 0) mbar_arrive(tile_full(b));
        return true;
      };
      load(0, buf0);
      load(1, buf1);
      load(2, buf2);
      for (int i = 0; i < ntiles; i += 3) {
        if (!store(i, buf0)) break;
        load(i + 3, buf0);
        if (!store(i + 1, buf1)) break;
        load(i + 4, buf1);
        if (!store(i + 2, buf2)) break;
        load(i + 5, buf2);
      }
    } else {
      // ------------------------------------------------ softmax (thread = head)
      const int h = threadIdx.x;  // TMEM lane
      const bool live = h < kHeads;
      float m_used = -INFINITY, l_round = 0.f, l_exact = 0.f;
      bool ok = true;
      for (int i = 0; i < ntiles; ++i) {
        const int b = i & 1;
        ok = mbar_wait(s_full, i & 1, abort_flag, p.status);
        if (bar_or_softmax(!ok)) { ok = false; break; }   // uniform over the 128 softmax threads
        tc_fence_after();
        uint32_t r[kTileTok];
        {
          const uint32_t ta = tmem + ((uint32_t)(warp * 32) << 16) + kSCol;
          tmem_ld32(ta, *reinterpret_cast<uint32_t(*)[32]>(r));
          tmem_ld16(ta + 32, r + 32);
        }
        tmem_ld_wait();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(s_empty);  // the QK issuer may overwrite the S tile
        float x[kTileTok];
        // validity bits of tokens [48 i, 48 i + 48) from the 32-token words
        const int t0 = i * kTileTok;
        const uint64_t vmask =
            ((((uint64_t)tile_mask[(t0 >> 5) + 1]) << 32) | (uint64_t)tile_mask[t0 >> 5]) >> (t0 & 31);
        float m0 = -INFINITY, m1 = -INFINITY;
#pragma unroll
        for (int j = 0; j < kTileTok; ++j) {
          x[j] = ((vmask >> j) & 1ull) ? __uint_as_float(r[j]) * p.logit_scale_log2 : -INFINITY;
          if (j & 1) m1 = fmaxf(m1, x[j]); else m0 = fmaxf(m0, x[j]);
        }
        const float m_tile = fmaxf(m0, m1);
        const bool grow = live && m_tile > m_used + kRescaleThreshold;
        if (bar_or_softmax(grow)) {
          const float m_new = grow ? m_tile : m_used;
          const float alpha = (m_used == -INFINITY) ? 0.f : ex2(m_used - m_new);
          if (live) alpha_s[h] = alpha;
          l_round *= alpha;
          l_exact *= alpha;
          m_used = m_new;
          if (i > 0) {
            // O^T holds tiles 0..i-1: wait for the last PV, then scale column h by alpha[h]
            ok = mbar_wait(pv_done((i - 1) & 1), ((i - 1) >> 1) & 1, abort_flag, p.status);
            if (bar_or_softmax(!ok)) { ok = false; break; }   // also publishes alpha_s
            tc_fence_after();
#pragma unroll 1
            for (int c = 0; c < 12; ++c) {  // 4 M-blocks x 3 groups of 32 heads
              uint32_t o[32];
              const uint32_t ta = tmem + ((uint32_t)(warp * 32) << 16) + (c / 3) * kHeads + (c % 3) * 32;
              tmem_ld32(ta, o);
              tmem_ld_wait();
#pragma unroll
              for (int j = 0; j < 32; ++j)
                o[j] = __float_as_uint(__uint_as_float(o[j]) * alpha_s[(c % 3) * 32 + j]);
              tmem_st32(ta, o);
            }
            tmem_st_wait();
          }
        }
        // probabilities -> bf16 P row h (96 of 128 bytes, 128-byte swizzle)
        uint32_t pk[kTileTok / 2];
        float srnd = 0.f, sex = 0.f;
        if (m_used != -INFINITY) {
#pragma unroll
          for (int j = 0; j < kTileTok; j += 2) {
            const float p0 = ex2(x[j] - m_used), p1 = ex2(x[j + 1] - m_used);  // 2^-inf = 0 when masked
            const __nv_bfloat162 bb = __floats2bfloat162_rn(p0, p1);
            const float2 back = __bfloat1622float2(bb);
            srnd += back.x + back.y;
            sex += p0 + p1;
            pk[j >> 1] = *reinterpret_cast<const uint32_t*>(&bb);
          }
        } else {
#pragma unroll
          for (int j = 0; j < kTileTok / 2; ++j) pk[j] = 0;
        }
        l_round += srnd;
        l_exact += sex;
        // P buffer b was last read by the PV of tile i - 2
        ok = mbar_wait(pv_done(b), ((i >> 1) & 1) ^ 1, abort_flag, p.status);
        if (bar_or_softmax(!ok)) { ok = false; break; }
        if (live) {
          uint8_t* prow = smem + kOffP + b * kPBytes;
#pragma unroll
          for (int c = 0; c < kTileTok / 8; ++c)
            *reinterpret_cast<uint4*>(prow + swz128(h * kPRowBytes + c * 16)) =
                make_uint4(pk[4 * c], pk[4 * c + 1], pk[4 * c + 2], pk[4 * c + 3]);
        }
        fence_proxy_async_smem();
        tc_fence_before();
        __syncwarp();
        if (lane == 0) mbar_arrive(p_full(b));
      }
      // ---- this chunk's running max and sums per head
      ok = !bar_or_softmax(!ok);
      if (ok && live) ml_mine = make_float4(m_used, l_round, l_exact, 0.f);
      // the epilogue normalises the chunk's output by its own sum (alpha_s is
      // free now: the softmax threads are its only users)
      alpha_s[h] = (live && l_round > 0.f) ? 1.f / l_round : 0.f;
    }
  }
  // ---- epilogue: the chunk's O^T, normalised by the chunk's sum of the rounded
  //      probabilities, to the workspace as fp16 (values below 448 x the latent
  //      scale: 11 significant bits, far inside the bf16 output's 8), by all twelve
  //      warps.  Every MMA has completed: both issuers waited for theirs before
  //      this barrier.  Warp w reads TMEM lanes 32 (w % 4) .. + 31 (dims of each
  //      128-dim block) and the 32-head column groups w / 4 of the four blocks,
  //      two groups in flight.
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const int64_t part = (int64_t)row * p.nsplit + split;
  if (threadIdx.x < kHeads) reinterpret_cast<float4*>(p.ml)[part * kHeads + threadIdx.x] = ml_mine;
  if (ntiles > 0 && *abort_flag == 0) {
    uint16_t* op = p.opart + part * kHeads * kValue;
    const int quarter = warp & 3, hg = warp >> 2;
    const uint32_t lane_base = tmem + ((uint32_t)(quarter * 32) << 16) + hg * 32;
    const int dim_in_block = quarter * 32 + lane;
#pragma unroll 1
    for (int mb = 0; mb < 4; mb += 2) {
      uint32_t o0[32], o1[32];
      tmem_ld32(lane_base + mb * kHeads, o0);
      tmem_ld32(lane_base + (mb + 1) * kHeads, o1);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        const float il = alpha_s[hg * 32 + j];
        op[(int64_t)(hg * 32 + j) * kValue + mb * 128 + dim_in_block] =
            __half_as_ushort(__float2half_rn(__uint_as_float(o0[j]) * il));
        op[(int64_t)(hg * 32 + j) * kValue + (mb + 1) * 128 + dim_in_block] =
            __half_as_ushort(__float2half_rn(__uint_as_float(o1[j]) * il));
      }
    }
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == kMmaWarp) tmem_dealloc(tmem, kTmemCols);
  if (p.fuse) {
    // ---- the row's chunks are the cluster: once every chunk's partials are
    //      written (the cluster barrier orders them), each CTA merges a share of
    //      the row's outputs through the chunks' log-sum-exp, as the combine
    //      kernel does.  A zero weight (an empty chunk, or one whose maximum
    //      lies far below) skips its partial, which an empty chunk never wrote.
    cooperative_groups::this_cluster().sync();
    float* wgt = reinterpret_cast<float*>(smem + kOffTile);  // [96][kMaxFusedSplit]; the tiles are free
    if (threadIdx.x < kHeads) {
      const int h = threadIdx.x;
      const float4* mlr = reinterpret_cast<const float4*>(p.ml) + (int64_t)row * p.nsplit * kHeads;
      float4 mv[kMaxFusedSplit];
#pragma unroll
      for (int s = 0; s < kMaxFusedSplit; ++s)
        if (s < p.nsplit) mv[s] = mlr[s * kHeads + h];
      float M = -INFINITY;
#pragma unroll
      for (int s = 0; s < kMaxFusedSplit; ++s)
        if (s < p.nsplit) M = fmaxf(M, mv[s].x);
      float den = 0.f, ex = 0.f;
#pragma unroll
      for (int s = 0; s < kMaxFusedSplit; ++s) {
        if (s >= p.nsplit) break;
        const float4 v = mv[s];
        const float w = (M == -INFINITY || v.x == -INFINITY) ? 0.f : ex2(v.x - M);
        den += w * v.y;
        ex += w * v.z;
        wgt[h * kMaxFusedSplit + s] = w * v.y;  // the partial is normalised by v.y
      }
      const float inv = den > 0.f ? p.latent_scale / den : 0.f;
      for (int s = 0; s < p.nsplit; ++s) wgt[h * kMaxFusedSplit + s] *= inv;
      if (split == 0)
        p.lse[(int64_t)row * kHeads + h] =
            (M == -INFINITY || ex <= 0.f) ? -INFINITY : (M + log2f(ex)) * 0.69314718055994531f;
    }
    __syncthreads();
    constexpr int kVec = kHeads * kValue / 4;  // float4s of the row's output
    const int v0 = (int)((int64_t)kVec * split / p.nsplit), v1 = (int)((int64_t)kVec * (split + 1) / p.nsplit);
    uint16_t* out_row = p.out + (int64_t)row * kHeads * kValue;
    const uint16_t* opart_row = p.opart + (int64_t)row * p.nsplit * kHeads * kValue;
    switch (p.nsplit) {
      case 1: merge_share<1>(opart_row, wgt, v0, v1, out_row); break;
      case 2: merge_share<2>(opart_row, wgt, v0, v1, out_row); break;
      case 3: merge_share<3>(opart_row, wgt, v0, v1, out_row); break;
      case 4: merge_share<4>(opart_row, wgt, v0, v1, out_row); break;
      case 5: merge_share<5>(opart_row, wgt, v0, v1, out_row); break;
      case 6: merge_share<6>(opart_row, wgt, v0, v1, out_row); break;
      case 7: merge_share<7>(opart_row, wgt, v0, v1, out_row); break;
      default: merge_share<8>(opart_row, wgt, v0, v1, out_row); break;
    }
  }
}

// Merge the chunks of one row through their log-sum-exp and write bf16 O and
// fp32 LSE (natural log), with the in-cluster merge's arithmetic.  CTA (group,
// row) covers 2 heads, one output float4 per thread; a head's (max, sums) of
// every chunk are loaded before any is used, and so is every chunk's partial of
// a float4 (the loads in flight, not one after another).
constexpr int kCombineHeads = 2;
__global__ void __launch_bounds__(256) mla_combine_kernel(const uint16_t* __restrict__ opart,
                                                           const float* __restrict__ ml, int nsplit,
                                                           float latent_scale, uint16_t* out, float* lse) {
  const int row = blockIdx.y, h0 = blockIdx.x * kCombineHeads;
  __shared__ float wgt[kCombineHeads][kMaxSplit];
  grid_dep_wait();  // the partials come from the previous kernel
  const float4* mlr = reinterpret_cast<const float4*>(ml) + (int64_t)row * nsplit * kHeads;
  if (threadIdx.x < kCombineHeads) {
    const int h = h0 + threadIdx.x;
    float4 mv[kMaxSplit];
#pragma unroll
    for (int s = 0; s < kMaxSplit; ++s)
      if (s < nsplit) mv[s] = mlr[s * kHeads + h];
    float M = -INFINITY;
#pragma unroll
    for (int s = 0; s < kMaxSplit; ++s)
      if (s < nsplit) M = fmaxf(M, mv[s].x);
    float den = 0.f, ex = 0.f;
    float w[kMaxSplit];
#pragma unroll
    for (int s = 0; s < kMaxSplit; ++s) {
      w[s] = 0.f;
      if (s >= nsplit) continue;
      const float4 v = mv[s];
      w[s] = (M == -INFINITY || v.x == -INFINITY) ? 0.f : ex2(v.x - M);
      den += w[s] * v.y;
      ex += w[s] * v.z;
      w[s] *= v.y;  // the partial is normalised by v.y
    }
    const float inv = den > 0.f ? latent_scale / den : 0.f;
#pragma unroll
    for (int s = 0; s < kMaxSplit; ++s) wgt[threadIdx.x][s] = w[s] * inv;
    lse[(int64_t)row * kHeads + h] =
        (M == -INFINITY || ex <= 0.f) ? -INFINITY : (M + log2f(ex)) * 0.69314718055994531f;
  }
  __syncthreads();
  constexpr int kVec = kCombineHeads * kValue / 4;  // 256 float4s per CTA
  for (int v = threadIdx.x; v < kVec; v += blockDim.x) {
    const int hl = v / (kValue / 4), d = (v % (kValue / 4)) * 4;
    const uint16_t* src = opart + ((int64_t)row * nsplit * kHeads + h0 + hl) * kValue + d;
    float4 x[kMaxSplit];
#pragma unroll
    for (int s = 0; s < kMaxSplit; ++s)
      if (s < nsplit && wgt[hl][s] != 0.f) x[s] = half4_to_float4(*reinterpret_cast<const uint2*>(src + (int64_t)s * kHeads * kValue));
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int s = 0; s < kMaxSplit; ++s)
      if (s < nsplit && wgt[hl][s] != 0.f) {
        const float w = wgt[hl][s];
        a.x = fmaf(w, x[s].x, a.x); a.y = fmaf(w, x[s].y, a.y);
        a.z = fmaf(w, x[s].z, a.z); a.w = fmaf(w, x[s].w, a.w);
      }
    const __nv_bfloat162 lo = __floats2bfloat162_rn(a.x, a.y);
    const __nv_bfloat162 hi = __floats2bfloat162_rn(a.z, a.w);
    uint2 pk;
    pk.x = *reinterpret_cast<const uint32_t*>(&lo);
    pk.y = *reinterpret_cast<const uint32_t*>(&hi);
    *reinterpret_cast<uint2*>(out + ((int64_t)row * kHeads + h0 + hl) * kValue + d) = pk;
  }
}

}  // namespace

// Whether clusters of `nsplit` CTAs of the MLA kernel can be resident on this
// device (asked once per device and size).
template <bool kNV>
bool fused_cluster_ok(int nsplit) {
  static std::atomic<int> known[64][kMaxFusedSplit + 1];  // 0 unknown, 1 yes, 2 no
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64 || nsplit < 1 || nsplit > kMaxFusedSplit) return false;
  if (known[dev][nsplit] == 0) {
    bool ok = cudaFuncSetAttribute(sparse_mla_kernel<kNV>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                   (int)kSmemBytes) == cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3((unsigned)nsplit);
    cfg.blockDim = dim3(kThreads);
    cfg.dynamicSmemBytes = kSmemBytes;
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = (unsigned)nsplit;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    ok = ok && cudaOccupancyMaxActiveClusters(&n, sparse_mla_kernel<kNV>, &cfg) == cudaSuccess && n > 0;
    cudaGetLastError();  // a refused query leaves no error behind
    known[dev][nsplit] = ok ? 1 : 2;
  }
  return known[dev][nsplit] == 1;
}

namespace {
std::atomic<int> g_batch_invariant{0};
}  // namespace

int mla_batch_invariant(int on) { return g_batch_invariant.exchange(on ? 1 : 0); }

// Token chunks per row: enough CTAs for one wave over the SMs (one CTA per SM
// fits), at most 16; the workspace is sized for up to 256 SMs.  In the
// batch-invariant mode the chunks are kInvariantChunk tokens whatever the
// number of rows, so a row's arithmetic does not depend on its batch.
static int mla_nsplit_max(int rows, int k, bool inv) {
  const int n = std::max((k + kMaxChunk - 1) / kMaxChunk, std::min(16, 256 / std::max(1, rows)));
  return inv ? std::max(n, (k + kInvariantChunk - 1) / kInvariantChunk) : n;
}
static int mla_nsplit(int rows, int k, bool inv) {
  if (inv) return (k + kInvariantChunk - 1) / kInvariantChunk;
  return std::max((k + kMaxChunk - 1) / kMaxChunk,
                  std::min(mla_nsplit_max(rows, k, false), num_sms() / std::max(1, rows)));
}
static bool batch_invariant() { return g_batch_invariant.load(std::memory_order_relaxed) != 0; }

size_t mla_workspace_bytes(int rows, int k) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t parts = (size_t)rows * mla_nsplit_max(rows, k, batch_invariant());
  return al(parts * kHeads * kValue * 2) + al(parts * kHeads * 16);
}

namespace {

// The Q tensor map and the kernel's parameters for `rows` query rows and
// `nsplit` chunks of `chunk` tokens; false if the tensor map cannot be made or
// the shared-memory size cannot be set.
bool mla_setup(const dsa_paged_cache_t& c, const dsa_batch_t& bt, const uint16_t* q_mla, const int32_t* idx, int k,
               int chunk, int nsplit, float sm_scale, uint16_t* opart, float* ml, uint16_t* out, float* lse,
               int32_t* status, CUtensorMap* qmap, MlaParams* p) {
  const int rows = bt.batch * bt.queries_per_seq;
  const uint64_t dims[2] = {(uint64_t)kLatent, (uint64_t)rows * kHeads};
  const uint64_t strides[1] = {(uint64_t)kLatent * 2};
  const uint32_t box[2] = {64, (uint32_t)kHeads};
  if (!encode_tmap(qmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, q_mla, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
    return false;
  *p = MlaParams{static_cast<const uint8_t*>(c.base) + c.latent_off,
                 c.row_stride,
                 c.num_blocks,
                 bt.block_table,
                 bt.max_blocks_per_seq,
                 bt.seq_lens,
                 bt.queries_per_seq,
                 std::min(bt.max_blocks_per_seq * kBlock, bt.max_seq_len),
                 idx,
                 k,
                 chunk,
                 nsplit,
                 sm_scale * c.latent_scale * 1.4426950408889634f,
                 q_mla,
                 opart,
                 ml,
                 status,
                 0,
                 c.latent_scale,
                 out,
                 lse,
                 nullptr,
                 nullptr};
  static std::atomic<bool> attr_set[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    if (cuda_status(cudaFuncSetAttribute(sparse_mla_kernel<false>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes)) != DSA_OK ||
        cuda_status(cudaFuncSetAttribute(sparse_mla_kernel<true>, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kSmemBytes)) != DSA_OK)
      return false;
    attr_set[dev] = true;
  }
  return true;
}

using MlaKernel = void (*)(const CUtensorMap, const MlaParams);
MlaKernel mla_kernel_for(const dsa_paged_cache_t& c) {
  return c.latent_format == DSA_LATENT_NVFP4 ? sparse_mla_kernel<true> : sparse_mla_kernel<false>;
}

}  // namespace

int mla_max_chunk() { return kMaxChunk; }

dsa_status_t launch_sparse_mla_partials(const dsa_paged_cache_t& c, const dsa_batch_t& bt, const uint16_t* q_mla,
                                        const int32_t* idx, int k, const int32_t* seg, int nseg, float sm_scale,
                                        uint16_t* opart, float* ml, int32_t* status, cudaStream_t st) {
  const int rows = bt.batch * bt.queries_per_seq;
  if (rows == 0) return DSA_OK;
  if (nseg < 1 || nseg > kMaxSplit) return DSA_ERR_UNSUPPORTED;
  CUtensorMap qmap;
  MlaParams p;
  if (!mla_setup(c, bt, q_mla, idx, k, kMaxChunk, nseg, sm_scale, opart, ml, nullptr, nullptr, status, &qmap, &p))
    return DSA_ERR_CUDA;
  p.seg = seg;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)nseg, (unsigned)rows);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  count_launches(1);
  if (cuda_status(cudaLaunchKernelEx(&cfg, mla_kernel_for(c), qmap, p)) != DSA_OK) return DSA_ERR_CUDA;
  return launch_status();
}

dsa_status_t launch_sparse_mla(const dsa_paged_cache_t& c, const dsa_batch_t& bt, const uint16_t* q_mla,
                               const int32_t* idx, int k, float sm_scale, uint16_t* out, float* lse,
                               void* workspace, int32_t* status, cudaStream_t st, const int32_t* phys) {
  const int rows = bt.batch * bt.queries_per_seq;
  if (rows == 0) return DSA_OK;
  const bool inv = batch_invariant();  // read once: the split and the workspace layout agree
  const int nsplit0 = mla_nsplit(rows, k, inv);
  const int tiles = (k + kTileTok - 1) / kTileTok;
  const int chunk = ((tiles + nsplit0 - 1) / nsplit0) * kTileTok;
  const int nsplit = (k + chunk - 1) / chunk;
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  uint16_t* opart = static_cast<uint16_t*>(workspace);
  float* ml = reinterpret_cast<float*>(static_cast<uint8_t*>(workspace) +
                                       al((size_t)rows * mla_nsplit_max(rows, k, inv) * kHeads * kValue * 2));
  CUtensorMap qmap;
  MlaParams p;
  if (!mla_setup(c, bt, q_mla, idx, k, chunk, nsplit, sm_scale, opart, ml, out, lse, status, &qmap, &p))
    return DSA_ERR_CUDA;
  p.phys = phys;
  // Up to kMaxFusedSplit chunks per row: the row's CTAs form a cluster and
  // merge the chunks themselves; more chunks take the combine kernel.
  const bool nv = c.latent_format == DSA_LATENT_NVFP4;
  p.fuse = nsplit <= kMaxFusedSplit && (nv ? fused_cluster_ok<true>(nsplit) : fused_cluster_ok<false>(nsplit)) ? 1 : 0;
  // the launches may overlap the previous kernel's tail; each waits for its inputs
  cudaLaunchAttribute attrs[2];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  attrs[1].id = cudaLaunchAttributeClusterDimension;
  attrs[1].val.clusterDim.x = (unsigned)nsplit;
  attrs[1].val.clusterDim.y = 1;
  attrs[1].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)nsplit, (unsigned)rows);
  cfg.blockDim = dim3(kThreads);
  cfg.dynamicSmemBytes = kSmemBytes;
  cfg.stream = st;
  cfg.attrs = attrs;
  cfg.numAttrs = p.fuse ? 2 : 1;
  count_launches(1);
  if (cuda_status(cudaLaunchKernelEx(&cfg, mla_kernel_for(c), qmap, p)) != DSA_OK) return DSA_ERR_CUDA;
  if (p.fuse) return launch_status();
  cudaLaunchConfig_t cfg2 = cfg;
  cfg2.numAttrs = 1;
  cfg2.gridDim = dim3(kHeads / kCombineHeads, (unsigned)rows);
  cfg2.blockDim = dim3(256);
  cfg2.dynamicSmemBytes = 0;
  count_launches(1);
  if (cuda_status(cudaLaunchKernelEx(&cfg2, mla_combine_kernel, (const uint16_t*)opart, (const float*)ml, nsplit,
                                     c.latent_scale, out, lse)) != DSA_OK)
    return DSA_ERR_CUDA;
  return launch_status();
}

}  // namespace dsa
