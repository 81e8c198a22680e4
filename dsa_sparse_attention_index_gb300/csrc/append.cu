// append.cu — the front end of the fused decode path: the step's new tokens
// into the paged cache, the indexer's query in FP8, and the fused indexer
// front end that does both after the query norm and projection.
//
// vLLM Day-0 post for Kimi K3.1 Pro, section "低延迟解码：融合的 DSA 解码路径"
// (each decode step writes the new token's index key and latent into the
// cache, and the indexer query is FP8 with its scale folded into the head
// weights), and section "为三类状态服务的 KV 缓存" (the packed pages).
//
// Encodings: round to nearest, ties to even, finite values beyond the largest
// magnitude saturate (CUDA's FP8/FP4 conversions).  Scales in fp32:
//   latent    code = e4m3(x / latent_scale)
//   NVFP4     per 16 dims of 0..511: scale code c = e4m3(amax / (6 latent_scale)),
//   latent    codes e2m1(x / (latent_scale * e4m3(c))) (0 where that scale is 0),
//             element 2i in the low nibble of byte i; dims 512..575 as above
//             (the record layout and this rule are readings of the packed-cache
//             section's 352 B NVFP4 latent)
//   FP8 key   s = amax / 448 (1 for an all-zero key), code = e4m3(x / s), s stored
//   MXFP4 key per 32 elements E = floor(log2 amax) - 2 clamped to [-127, 127]
//             (-127 for an all-zero block), code = e2m1(x * 2^-E), byte E + 127
//   query     per (row, head) s = amax / 448, code = e4m3(q / s), w' = w * s
//             (ReLU is positively homogeneous, so the score is unchanged);
//             for native FP4 keys (DSA_KEY_MXFP4_NATIVE) the query per head
//             and 32 dims as an MXFP4 key, w' = w (the E8M0 scales stay with
//             the codes and the block-scaled MMA applies them).
//
// The fused front end (same post, same section, second bullet: the query norm,
// the indexer's query projection, its FP8 or MXFP4 quantisation folded into
// the head weights, and the new token's index key, in one kernel): per row the RMSNorm
// of the compressed query c (xn = bf16(c * (1 / sqrt(mean(c^2) + eps)) *
// gamma), fp32), the projection q = W xn (4,096 outputs, bf16 operands, fp32
// accumulation on tcgen05), the query quantisation above from the fp32 q, and
// the cache write above, in one launch.
#include <algorithm>
#include <atomic>

#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "common.cuh"
#include "internal.h"

namespace dsa {

namespace {

constexpr int kAppendThreads = 128;  // one thread per index-key element

__device__ __forceinline__ float bf16_bits_to_float(uint16_t b) { return __uint_as_float((uint32_t)b << 16); }

__device__ __forceinline__ uint8_t e4m3(float x) {
  return (uint8_t)__nv_cvt_float_to_fp8(x, __NV_SATFINITE, __NV_E4M3);
}

__device__ __forceinline__ float warp_max(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v = fmaxf(v, __shfl_xor_sync(0xffffffffu, v, o));
  return v;
}

struct AppendArgs {
  uint8_t* latent_base;
  uint8_t* index_base;
  int64_t row_stride;
  int32_t num_blocks, key_format, latent_format;
  float latent_scale;
  const int32_t* block_table;
  int32_t max_blocks;
  const int32_t* seq_lens;
  int32_t nq, cap;
  const uint16_t* new_latent;
  const uint16_t* new_key;
  int32_t* status;
};

// Named barrier 1 over the 128 threads that write one token (threads 0..127).
__device__ __forceinline__ void bar_append() { asm volatile("bar.sync 1, 128;" ::: "memory"); }

// New token row nr = b * nq + j (token L_b - nq + j) by threads tid = 0..127;
// `sync` is a barrier over those threads (uniform: every early return below
// depends on nr alone).
template <typename Sync>
__device__ __forceinline__ void append_row(const AppendArgs& a, int nr, int tid, float* warp_amax, Sync sync) {
  uint8_t* latent_base = a.latent_base;
  uint8_t* index_base = a.index_base;
  const int64_t row_stride = a.row_stride;
  const int32_t num_blocks = a.num_blocks, key_format = a.key_format, latent_format = a.latent_format;
  const float latent_scale = a.latent_scale;
  const int32_t* block_table = a.block_table;
  const int32_t max_blocks = a.max_blocks, nq = a.nq, cap = a.cap;
  const uint16_t* new_latent = a.new_latent;
  const uint16_t* new_key = a.new_key;
  int32_t* status = a.status;
  const int b = nr / nq, j = nr % nq, lane = tid & 31, wid = tid >> 5;
  const int L = a.seq_lens[b];
  if (L < 0 || L > cap) {
    if (tid == 0) report(status, DSA_ERR_BOUNDS);
    return;
  }
  const int t = L - nq + j;
  if (t < 0) return;  // a context shorter than its new rows: nothing to write for this one
  const int r = block_table[(int64_t)b * max_blocks + t / kBlock];
  if (r < 0 || r >= num_blocks) {
    if (tid == 0) report(status, DSA_ERR_BOUNDS);
    return;
  }
  const int slot = t % kBlock;
  const uint16_t* lat = new_latent + (int64_t)nr * kLatent;
  if (latent_format == DSA_LATENT_FP8_E4M3) {
    // latent: 576 codes
    uint8_t* lat_dst = latent_base + (int64_t)r * row_stride + (int64_t)slot * kLatent;
    for (int d = tid; d < kLatent; d += kAppendThreads) lat_dst[d] = e4m3(bf16_bits_to_float(lat[d]) / latent_scale);
  } else {
    // NVFP4 record: thread tid owns dims 4 tid .. 4 tid + 3, four threads a 16-dim block
    constexpr int kRec = kValue / 2 + kValue / 16 + (kLatent - kValue);
    uint8_t* rec = latent_base + (int64_t)r * row_stride + (int64_t)slot * kRec;
    float v[4];
#pragma unroll
    for (int q = 0; q < 4; ++q) v[q] = bf16_bits_to_float(lat[4 * tid + q]);
    float amax = fmaxf(fmaxf(fabsf(v[0]), fabsf(v[1])), fmaxf(fabsf(v[2]), fabsf(v[3])));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 1));
    amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, 2));
    const uint8_t sc = e4m3(amax / (6.0f * latent_scale));
    const __half_raw hr = __nv_cvt_fp8_to_halfraw((__nv_fp8_storage_t)sc, __NV_E4M3);
    const float sdec = __half2float(*reinterpret_cast<const __half*>(&hr));
    const float step = latent_scale * sdec;
    uint32_t code[4];
#pragma unroll
    for (int q = 0; q < 4; ++q)
      code[q] = sdec > 0.f ? (uint32_t)__nv_cvt_float_to_fp4(v[q] / step, __NV_E2M1, cudaRoundNearest) & 0xFu : 0u;
    const uint16_t two = (uint16_t)((code[0] | (code[1] << 4)) | ((code[2] | (code[3] << 4)) << 8));
    *reinterpret_cast<uint16_t*>(rec + 2 * tid) = two;
    if ((tid & 3) == 0) rec[kValue / 2 + tid / 4] = sc;
    if (tid < kLatent - kValue)
      rec[kValue / 2 + kValue / 16 + tid] = e4m3(bf16_bits_to_float(lat[kValue + tid]) / latent_scale);
  }
  // index key: thread tid owns element tid
  const float x = bf16_bits_to_float(new_key[(int64_t)nr * kIdxDim + tid]);
  uint8_t* page = index_base + (int64_t)r * row_stride;
  if (key_format == DSA_KEY_FP8_E4M3) {
    const float wm = warp_max(fabsf(x));
    if (lane == 0) warp_amax[wid] = wm;
    sync();
    const float amax = fmaxf(fmaxf(warp_amax[0], warp_amax[1]), fmaxf(warp_amax[2], warp_amax[3]));
    const float s = amax > 0.f ? amax / 448.0f : 1.0f;
    page[(int64_t)slot * kIdxDim + tid] = e4m3(x / s);
    if (tid == 0) *reinterpret_cast<float*>(page + kBlock * kIdxDim + 4 * slot) = s;
  } else {
    // warp wid = 32-element block wid
    const float amax = warp_max(fabsf(x));
    const uint32_t ebits = (__float_as_uint(amax) >> 23) & 0xFFu;  // floor(log2 amax) + 127 for normal amax
    const int e = (amax > 0.f && ebits > 0) ? max(-127, min(127, (int)ebits - 127 - 2)) : -127;
    const uint32_t code = (uint32_t)__nv_cvt_float_to_fp4(ldexpf(x, -e), __NV_E2M1, cudaRoundNearest) & 0xFu;
    const uint32_t hi = __shfl_down_sync(0xffffffffu, code, 1);  // element 2i in the low nibble of byte i
    if ((lane & 1) == 0) page[(int64_t)slot * (kIdxDim / 2) + 16 * wid + lane / 2] = (uint8_t)(code | (hi << 4));
    if (lane == 0) page[kBlock * (kIdxDim / 2) + 4 * slot + wid] = (uint8_t)(e + 127);
  }
}

// One CTA per new token row.
__global__ void __launch_bounds__(kAppendThreads) cache_append_kernel(const AppendArgs a) {
  __shared__ float warp_amax[kAppendThreads / 32];
  append_row(a, blockIdx.x, threadIdx.x, warp_amax, [] { __syncthreads(); });
}

// One warp per (row, head): 128 elements, four per lane.
__global__ void __launch_bounds__(128)
    quantize_query_kernel(const uint16_t* q, const float* w, int64_t pairs, uint8_t* codes, float* w_out) {
  const int64_t rh = (int64_t)blockIdx.x * 4 + (threadIdx.x >> 5);
  const int lane = threadIdx.x & 31;
  if (rh >= pairs) return;
  const uint2 v = reinterpret_cast<const uint2*>(q + rh * kIdxDim)[lane];
  const float x[4] = {bf16_bits_to_float((uint16_t)(v.x & 0xFFFFu)), bf16_bits_to_float((uint16_t)(v.x >> 16)),
                      bf16_bits_to_float((uint16_t)(v.y & 0xFFFFu)), bf16_bits_to_float((uint16_t)(v.y >> 16))};
  const float amax = warp_max(fmaxf(fmaxf(fabsf(x[0]), fabsf(x[1])), fmaxf(fabsf(x[2]), fabsf(x[3]))));
  const float s = amax > 0.f ? amax / 448.0f : 1.0f;
  const uint32_t c = (uint32_t)e4m3(x[0] / s) | ((uint32_t)e4m3(x[1] / s) << 8) | ((uint32_t)e4m3(x[2] / s) << 16) |
                     ((uint32_t)e4m3(x[3] / s) << 24);
  reinterpret_cast<uint32_t*>(codes + rh * kIdxDim)[lane] = c;
  if (lane == 0) w_out[rh] = w[rh] * s;
}


// ---------------------------------------------------------------- fused indexer front end
// Grid (32 * 4 + 64, ceil(rows / 64)), clusters of 4 CTAs along x.  Cluster h
// (CTAs 4h .. 4h + 3) computes the 128 projected values of head h for rows
// 64 g .. 64 g + 63 as one tcgen05 GEMM D[128 dims x N rows] = W_h[128 x D]
// xn^T[D x N] (M = 128, N = the rows rounded up to 16), split over K: CTA rank
// s takes the 64-element K stages [nk s / 4, nk (s + 1) / 4), so 128 CTAs (two
// per SM) stream the weights.  In each CTA warp 0 streams its W_h stages and
// the rows' compressed-query tiles by TMA (128-byte swizzle; rows past the
// batch read as zeros), warp 1 issues the MMAs, and warps 2..5 first sum the
// squares of their K range per row (the four ranks' sums are exchanged through
// distributed shared memory and added in rank order), then turn each stage's
// query tile into xn in place (scale, gamma, bf16; stage j by warp 2 + j % 4),
// and finally write their fp32 accumulators to shared memory.  After a cluster
// barrier rank s adds the four ranks' accumulators (in rank order) for rows
// 16 s .. 16 s + 15, takes each row's amax over the head's 128 dims and writes
// the FP8 codes and the folded head weight (native FP4 keys: per 32 dims, one
// warp's, the MXFP4 codes and E8M0 scale; the head weight as given).
// CTA (128 + j, g): the new token of
// row 64 g + j into the cache (threads 0..127).
constexpr int kFeRows = 64;
constexpr int kFeSplit = 4;                               // K ranks per head (the cluster)
constexpr int kFeStages = 4;
constexpr int kFeK = 64;                                  // K elements per stage: one 128-byte swizzle row
constexpr int kFeWBytes = 128 * kFeK * 2;                 // 16 KB
constexpr int kFeXBytes = kFeRows * kFeK * 2;             // 8 KB
constexpr int kFeThreads = 192;
constexpr int kFeMaxDim = 16384;
constexpr int kFeOffW = 0;
constexpr int kFeOffX = kFeOffW + kFeStages * kFeWBytes;  // 65,536
constexpr int kFeOffBars = kFeOffX + kFeStages * kFeXBytes;  // 98,304
constexpr int kFeNumBars = 4 * kFeStages + 1;             // W full, xn full, stage empty, query tile landed; done
constexpr int kFeOffSs = (kFeOffBars + kFeNumBars * 8 + 127) / 128 * 128;  // partial sums of squares [64]
constexpr int kFeOffNorm = kFeOffSs + kFeRows * 4;                        // RMS factors [64]
constexpr int kFeOffAmax = kFeOffNorm + kFeRows * 4;                      // [4 warps][16 rows]; the writers' amax
constexpr int kFeOffGamma = kFeOffAmax + 4 * kFeRows * 4;                 // gamma of this rank's K range, bf16
constexpr int kFeOffMisc = kFeOffGamma + (kFeMaxDim / kFeSplit) * 2;
constexpr size_t kFeSmem = 1024 + kFeOffMisc + 32;
constexpr int kFePartBytes = kFeRows * 128 * 4;           // this rank's fp32 accumulators [64 rows][128 dims]
static_assert(kFePartBytes <= kFeOffBars, "the accumulators reuse the stage buffers");
static_assert(kFeOffSs % 16 == 0 && kFeOffNorm % 16 == 0 && kFeOffAmax % 16 == 0 && kFeOffGamma % 16 == 0,
              "16-byte vector accesses");
static_assert(2 * kFeSmem <= 233472, "two CTAs per SM");
constexpr int kFeTmemCols = 64;

struct FeParams {
  const uint16_t* c_q;     // bf16 [rows][dim]
  const uint16_t* gamma;   // bf16 [dim]
  int32_t dim;
  float eps;
  const float* head_w;     // fp32 [rows][32]
  int32_t rows;
  uint8_t* q_index;        // E4M3 [rows][32][128]; native FP4: E2M1 [rows][32][64] then E8M0 [rows][32][4]
  float* head_w_out;       // fp32 [rows][32]
  int32_t native;          // the cache's keys are scored against an MXFP4 query (DSA_KEY_MXFP4_NATIVE)
  float* q_proj;           // fp32 [rows][4096] or null
  AppendArgs app;
};

// Named barrier 2 over warps 2..5.
__device__ __forceinline__ void bar_fe() { asm volatile("bar.sync 2, 128;" ::: "memory"); }
// The cluster barrier in two halves (every thread of the cluster arrives, then
// waits), so that warps with other work can arrive early and wait late.
__device__ __forceinline__ void cluster_arrive() { asm volatile("barrier.cluster.arrive.release.aligned;" ::: "memory"); }
__device__ __forceinline__ void cluster_wait() { asm volatile("barrier.cluster.wait.acquire.aligned;" ::: "memory"); }
__device__ __forceinline__ float ld_cluster_f32(uint32_t addr) {
  float v;
  asm volatile("ld.shared::cluster.f32 %0, [%1];" : "=f"(v) : "r"(addr) : "memory");
  return v;
}
__device__ __forceinline__ uint32_t cluster_addr(uint32_t saddr, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(saddr), "r"(rank));
  return r;
}

__global__ void __launch_bounds__(kFeThreads, 2)
    frontend_kernel(const __grid_constant__ CUtensorMap tmap_w, const __grid_constant__ CUtensorMap tmap_c,
                    const FeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = blockIdx.y * kFeRows;
  const int nrow = min(kFeRows, p.rows - row0);
  if (blockIdx.x >= kIdxHeads * kFeSplit) {
    // ---- the new token of one row into the cache (no cluster barrier here)
    const int r = blockIdx.x - kIdxHeads * kFeSplit;
    float* warp_amax = reinterpret_cast<float*>(smem + kFeOffAmax);
    if (r < nrow && threadIdx.x < kAppendThreads)
      append_row(p.app, row0 + r, threadIdx.x, warp_amax, [] { bar_append(); });
    return;
  }
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kFeOffBars;
  auto full_w = [&](int s) { return bars + 8u * s; };
  auto full_x = [&](int s) { return bars + 8u * (kFeStages + s); };
  auto empty = [&](int s) { return bars + 8u * (2 * kFeStages + s); };
  auto raw_x = [&](int s) { return bars + 8u * (3 * kFeStages + s); };  // the stage's query tile landed
  const uint32_t done = bars + 8u * (4 * kFeStages);
  float* ss_s = reinterpret_cast<float*>(smem + kFeOffSs);
  float* norm = reinterpret_cast<float*>(smem + kFeOffNorm);
  float* amax_s = reinterpret_cast<float*>(smem + kFeOffAmax);
  uint16_t* gamma_s = reinterpret_cast<uint16_t*>(smem + kFeOffGamma);
  float* part = reinterpret_cast<float*>(smem + kFeOffW);    // [64 rows][128 dims], after the MMAs
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kFeOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kFeOffMisc + 4);
  const int h = blockIdx.x / kFeSplit, rank = blockIdx.x % kFeSplit;  // clusters are 4 consecutive CTAs along x
  const int n_mma = max(16, (nrow + 15) & ~15);
  const int nk = p.dim / kFeK;
  const int kc0 = nk * rank / kFeSplit, nkm = nk * (rank + 1) / kFeSplit - kc0;  // this rank's K stages
  if (threadIdx.x == 0) {
    for (int s = 0; s < kFeStages; ++s) {
      mbar_init(full_w(s), 1);
      mbar_init(full_x(s), 1);
      mbar_init(empty(s), 1);
      mbar_init(raw_x(s), 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap_w);
    prefetch_tmap(&tmap_c);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kFeTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp < 2) {
    cluster_arrive();  // phase 1 (the sums of squares): nothing to give
    if (warp == 0 && lane == 0) {
      // ------------------------------------------------ this rank's W_h and query stages by TMA
      int issued = 0;
      for (int j = 0; j < nkm; ++j) {
        const int s = j % kFeStages, kc = kc0 + j;
        if (!mbar_wait(empty(s), ((j / kFeStages) & 1) ^ 1, abort_flag, p.app.status)) break;
        mbar_arrive_expect_tx(full_w(s), kFeWBytes);
        tma_load_2d(sbase + kFeOffW + s * kFeWBytes, &tmap_w, kc * kFeK, h * 128, full_w(s));
        mbar_arrive_expect_tx(raw_x(s), kFeXBytes);
        tma_load_2d(sbase + kFeOffX + s * kFeXBytes, &tmap_c, kc * kFeK, row0, raw_x(s));
        ++issued;
      }
      // the copies still in flight land before the buffers are reused (all of
      // them have landed already unless another role gave up)
      for (int j = max(0, issued - kFeStages); j < issued; ++j) {
        mbar_wait_drain(full_w(j % kFeStages), (j / kFeStages) & 1, 100000000ull);
        mbar_wait_drain(raw_x(j % kFeStages), (j / kFeStages) & 1, 100000000ull);
      }
    } else if (warp == 1 && lane == 0) {
      // ------------------------------------------------ MMA issuer
      const uint32_t idesc = make_idesc(kFmtBF16, kFmtBF16, 0, 0, 128, (uint32_t)n_mma);
      for (int j = 0; j < nkm; ++j) {
        const int s = j % kFeStages;
        if (!(mbar_wait(full_w(s), (j / kFeStages) & 1, abort_flag, p.app.status) &&
              mbar_wait(full_x(s), (j / kFeStages) & 1, abort_flag, p.app.status)))
          break;
        tc_fence_after();
        const uint32_t a0 = sbase + kFeOffW + s * kFeWBytes, b0 = sbase + kFeOffX + s * kFeXBytes;
#pragma unroll
        for (int kk = 0; kk < kFeK / 16; ++kk)
          mma_bf16(tmem, smem_desc(a0 + 32 * kk, 16, 1024, kLayoutSw128), smem_desc(b0 + 32 * kk, 16, 1024, kLayoutSw128),
                   idesc, (j | kk) ? 1u : 0u);
        mma_commit(empty(s));
      }
      mma_commit(done);  // also after an abort: every issued MMA completes before TMEM is released
    }
    __syncwarp();
    cluster_wait();    // phase 1
    cluster_arrive();  // phase 2 (the accumulators): nothing to give
    cluster_wait();
    cluster_arrive();  // phase 3 (the peers have read the accumulators)
    cluster_wait();
  } else {
    // ------------------------------------------------ warps 2..5
    const int t = threadIdx.x - 64, eq = warp - 2;
    const float hw_t = t < nrow ? p.head_w[(int64_t)(row0 + t) * kIdxHeads + h] : 0.f;
    // gamma of this rank's K range into shared memory
    for (int i = t; i < nkm * (kFeK / 8); i += 128)
      reinterpret_cast<uint4*>(gamma_s)[i] = reinterpret_cast<const uint4*>(p.gamma + kc0 * kFeK)[i];
    // this rank's part of sum(c^2) per row: a warp takes four rows at a time,
    // every lane's 16-byte loads of all four (up to 6 of each) in flight first
    auto sq_acc = [](const uint4& v, float& ss) {
      const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const float lo = __uint_as_float(w4[q] << 16), hi = __uint_as_float(w4[q] & 0xFFFF0000u);
        ss = fmaf(lo, lo, ss);
        ss = fmaf(hi, hi, ss);
      }
    };
    const int nv = nkm * (kFeK / 8);  // 16-byte chunks of a row in this rank's range
    for (int rb = eq; rb < kFeRows; rb += 16) {
      float ss[4] = {0.f, 0.f, 0.f, 0.f};
      for (int j0 = lane; j0 < nv; j0 += 6 * 32) {
        uint4 v[4][6];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int r = rb + 4 * q;
          const uint4* c = reinterpret_cast<const uint4*>(p.c_q + (int64_t)(row0 + min(r, nrow - 1)) * p.dim + kc0 * kFeK);
#pragma unroll
          for (int j = 0; j < 6; ++j) {
            const int jj = j0 + 32 * j;
            v[q][j] = (r < nrow && jj < nv) ? c[jj] : make_uint4(0u, 0u, 0u, 0u);
          }
        }
#pragma unroll
        for (int q = 0; q < 4; ++q)
#pragma unroll
          for (int j = 0; j < 6; ++j) sq_acc(v[q][j], ss[q]);
      }
#pragma unroll
      for (int q = 0; q < 4; ++q) {
#pragma unroll
        for (int o = 16; o > 0; o >>= 1) ss[q] += __shfl_xor_sync(0xffffffffu, ss[q], o);
        if (lane == 0) ss_s[rb + 4 * q] = ss[q];
      }
    }
    cluster_arrive();  // phase 1: this rank's sums of squares are written
    cluster_wait();
    // the RMS factors from the four ranks' sums, added in rank order (0 for the
    // zero rows past the batch)
    if (t < kFeRows) {
      float tot = 0.f;
#pragma unroll
      for (int q = 0; q < kFeSplit; ++q) tot += ld_cluster_f32(cluster_addr(smem_u32(ss_s + t), (uint32_t)q));
      norm[t] = t < nrow ? 1.0f / sqrtf(tot / (float)p.dim + p.eps) : 0.f;
    }
    bar_fe();
    // xn stages: each landed query tile (rows x 64 elements, 128-byte swizzle)
    // is scaled in place by one warp (stage j by warp 2 + j % 4, so that the
    // proxy fences of four stages overlap).  Lane l takes the 16-byte chunks at
    // physical column pc = l % 8 of rows l / 8 + 4 i, whose logical column is
    // pc ^ (row % 8).
    const int pc = lane & 7;
    bool ok = true;
    for (int j = eq; j < nkm; j += 4) {
      const int s = j % kFeStages;
      ok = mbar_wait(raw_x(s), (j / kFeStages) & 1, abort_flag, p.app.status);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      uint8_t* xs = smem + kFeOffX + s * kFeXBytes;
      const uint4* gk = reinterpret_cast<const uint4*>(gamma_s + j * kFeK);
#pragma unroll 4
      for (int r = lane >> 3; r < n_mma; r += 4) {
        uint4* cell = reinterpret_cast<uint4*>(xs + r * 128 + pc * 16);
        const uint4 cv = *cell;
        const uint4 gv = gk[pc ^ (r & 7)];
        const float nr = norm[r];
        const uint32_t c4[4] = {cv.x, cv.y, cv.z, cv.w}, g4[4] = {gv.x, gv.y, gv.z, gv.w};
        uint32_t o4[4];
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float lo = __uint_as_float(c4[q] << 16) * nr * __uint_as_float(g4[q] << 16);
          const float hi = __uint_as_float(c4[q] & 0xFFFF0000u) * nr * __uint_as_float(g4[q] & 0xFFFF0000u);
          const __nv_bfloat162 b2 = __floats2bfloat162_rn(lo, hi);
          o4[q] = *reinterpret_cast<const uint32_t*>(&b2);
        }
        *cell = make_uint4(o4[0], o4[1], o4[2], o4[3]);
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(full_x(s));
    }
    ok = !__any_sync(0xffffffffu, !ok);
    // ---- this rank's accumulators into shared memory (zeros for a rank with no
    //      K stage): TMEM lane = dim 32 (warp % 4) + lane, column = row
    const bool fin = mbar_wait(done, 0, abort_flag, p.app.status) && ok;
    tc_fence_after();
    const int quarter = warp & 3, d = quarter * 32 + lane;
    {
      uint32_t r0[32], r1[32];
      const uint32_t ta = tmem + ((uint32_t)(quarter * 32) << 16);
      tmem_ld32(ta, r0);
      tmem_ld32(ta + 32, r1);
      tmem_ld_wait();
      const bool have = fin && nkm > 0;
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        part[j * 128 + d] = have ? __uint_as_float(r0[j]) : 0.f;
        part[(32 + j) * 128 + d] = have ? __uint_as_float(r1[j]) : 0.f;
      }
    }
    cluster_arrive();  // phase 2: this rank's accumulators are written
    cluster_wait();
    // ---- rows 16 rank .. + 15: the four ranks' accumulators added in rank
    //      order, each row's amax over the head's 128 dims, the FP8 codes and
    //      the folded head weight
    const uint32_t part_u = smem_u32(part);
    float v[16];
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int r = 16 * rank + i;
      float a = 0.f;
#pragma unroll
      for (int q = 0; q < kFeSplit; ++q) a += ld_cluster_f32(cluster_addr(part_u + (uint32_t)(r * 128 + d) * 4u, (uint32_t)q));
      v[i] = a;
    }
    cluster_arrive();  // phase 3: the peers' accumulators are read
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int r = 16 * rank + i;
      if (r >= nrow) break;
      if (p.q_proj) p.q_proj[(int64_t)(row0 + r) * (kIdxHeads * kIdxDim) + h * kIdxDim + d] = v[i];
      const uint32_t m = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v[i])));  // |v| bits order as |v|
      if (lane == 0) amax_s[eq * 16 + i] = __uint_as_float(m);
    }
    bar_fe();
    const bool good = !*abort_flag;
#pragma unroll
    for (int i = 0; i < 16; ++i) {
      const int r = 16 * rank + i;
      if (r >= nrow || !good) break;
      const int64_t rh = (int64_t)(row0 + r) * kIdxHeads + h;
      if (p.native) {
        // MXFP4: this warp's 32 dims are one block; E = floor(log2 amax) - 2
        // clamped to [-127, 127] (-127 for an all-zero block), codes
        // e2m1(q 2^-E), as the MXFP4 keys are written; the head weight as given
        const float am = amax_s[eq * 16 + i];
        const uint32_t ebits = (__float_as_uint(am) >> 23) & 0xFFu;  // floor(log2 amax) + 127 for normal amax
        const int e = (am > 0.f && ebits > 0) ? max(-127, min(127, (int)ebits - 127 - 2)) : -127;
        const uint32_t code = (uint32_t)__nv_cvt_float_to_fp4(ldexpf(v[i], -e), __NV_E2M1, cudaRoundNearest) & 0xFu;
        const uint32_t hi = __shfl_down_sync(0xffffffffu, code, 1);  // element 2i in the low nibble of byte i
        if ((lane & 1) == 0) p.q_index[rh * (kIdxDim / 2) + d / 2] = (uint8_t)(code | (hi << 4));
        if (lane == 0) p.q_index[(int64_t)p.rows * kIdxHeads * (kIdxDim / 2) + rh * 4 + quarter] = (uint8_t)(e + 127);
        if (t == r) p.head_w_out[rh] = hw_t;
      } else {
        const float amax = fmaxf(fmaxf(amax_s[i], amax_s[16 + i]), fmaxf(amax_s[32 + i], amax_s[48 + i]));
        const float sc = amax > 0.f ? amax / 448.0f : 1.0f;
        p.q_index[rh * kIdxDim + d] = e4m3(v[i] / sc);
        if (t == r) p.head_w_out[rh] = hw_t * sc;
      }
    }
    cluster_wait();    // phase 3: no peer reads this rank's accumulators any more
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  if (warp == 1) tmem_dealloc(tmem, kFeTmemCols);
}

}  // namespace

dsa_status_t launch_cache_append(const dsa_paged_cache_t& c, const dsa_batch_t& bt, const uint16_t* new_latent,
                                 const uint16_t* new_key, int32_t* status, cudaStream_t st) {
  const int rows = bt.batch * bt.queries_per_seq;
  if (rows == 0) return DSA_OK;
  uint8_t* base = static_cast<uint8_t*>(c.base);
  const int cap = std::min(bt.max_blocks_per_seq * kBlock, bt.max_seq_len);
  const AppendArgs a{base + c.latent_off, base + c.index_off, c.row_stride, c.num_blocks, c.key_format,
                     c.latent_format, c.latent_scale, bt.block_table, bt.max_blocks_per_seq, bt.seq_lens,
                     bt.queries_per_seq, cap, new_latent, new_key, status};
  count_launches(1);
  cache_append_kernel<<<rows, kAppendThreads, 0, st>>>(a);
  return launch_status();
}

dsa_status_t launch_quantize_query(const uint16_t* q, const float* w, int rows, uint8_t* codes, float* w_out,
                                   cudaStream_t st) {
  const int64_t pairs = (int64_t)rows * kIdxHeads;
  if (pairs == 0) return DSA_OK;
  count_launches(1);
  quantize_query_kernel<<<(unsigned)((pairs + 3) / 4), 128, 0, st>>>(q, w, pairs, codes, w_out);
  return launch_status();
}

dsa_status_t launch_frontend(const dsa_paged_cache_t& c, const dsa_batch_t& bt, const uint16_t* c_q, int dim,
                             const uint16_t* gamma, float eps, const uint16_t* w_iq, const float* head_w,
                             const uint16_t* new_latent, const uint16_t* new_key, uint8_t* q_index, float* head_w_out,
                             float* q_proj, int32_t* status, cudaStream_t st) {
  const int rows = bt.batch * bt.queries_per_seq;
  if (rows == 0) return DSA_OK;
  CUtensorMap wmap;
  const uint64_t dims[2] = {(uint64_t)dim, (uint64_t)(kIdxHeads * kIdxDim)};
  const uint64_t strides[1] = {(uint64_t)dim * 2};
  const uint32_t box[2] = {(uint32_t)kFeK, 128u};
  if (!encode_tmap(&wmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, w_iq, dims, strides, box, CU_TENSOR_MAP_SWIZZLE_128B))
    return DSA_ERR_CUDA;
  // the compressed queries, 64 rows x 64 elements a box; rows past the batch read as zeros
  CUtensorMap cmap;
  const uint64_t cdims[2] = {(uint64_t)dim, (uint64_t)rows};
  const uint32_t cbox[2] = {(uint32_t)kFeK, (uint32_t)kFeRows};
  if (!encode_tmap(&cmap, CU_TENSOR_MAP_DATA_TYPE_BFLOAT16, 2, c_q, cdims, strides, cbox, CU_TENSOR_MAP_SWIZZLE_128B))
    return DSA_ERR_CUDA;
  static std::atomic<bool> attr_set[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    if (cuda_status(cudaFuncSetAttribute(frontend_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kFeSmem)) != DSA_OK)
      return DSA_ERR_CUDA;
    attr_set[dev] = true;
  }
  uint8_t* base = static_cast<uint8_t*>(c.base);
  FeParams p;
  p.c_q = c_q;
  p.gamma = gamma;
  p.dim = dim;
  p.eps = eps;
  p.head_w = head_w;
  p.rows = rows;
  p.q_index = q_index;
  p.head_w_out = head_w_out;
  p.native = c.key_format == DSA_KEY_MXFP4_NATIVE ? 1 : 0;
  p.q_proj = q_proj;
  p.app = AppendArgs{base + c.latent_off, base + c.index_off, c.row_stride, c.num_blocks, c.key_format,
                     c.latent_format, c.latent_scale, bt.block_table, bt.max_blocks_per_seq, bt.seq_lens,
                     bt.queries_per_seq, std::min(bt.max_blocks_per_seq * kBlock, bt.max_seq_len), new_latent,
                     new_key, status};
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = kFeSplit;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kIdxHeads * kFeSplit + kFeRows, (unsigned)((rows + kFeRows - 1) / kFeRows));
  cfg.blockDim = dim3(kFeThreads);
  cfg.dynamicSmemBytes = kFeSmem;
  cfg.stream = st;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  count_launches(1);
  if (cuda_status(cudaLaunchKernelEx(&cfg, frontend_kernel, wmap, cmap, p)) != DSA_OK) return DSA_ERR_CUDA;
  return launch_status();
}

}  // namespace dsa
