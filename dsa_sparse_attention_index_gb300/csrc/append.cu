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
//             (ReLU is positively homogeneous, so the score is unchanged).
//
// The fused front end (same post, same section, second bullet: the query norm,
// the indexer's query projection, its FP8 quantisation folded into the head
// weights, and the new token's index key, in one kernel): per row the RMSNorm
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
// Grid (33, ceil(rows / 64)).  CTA (h < 32, g): the 128 projected values of
// head h for rows 64 g .. 64 g + 63, as one tcgen05 GEMM D[128 dims x N rows]
// = W_h[128 x D] xn^T[D x N] (M = 128, N = the rows rounded up to 16, K in
// 64-element stages): warp 0 streams W_h by TMA (128-byte swizzle), warps 2..5
// normalise the rows and write each stage's xn tile (the same swizzle), warp 1
// issues the MMAs; then warps 2..5 (one TMEM lane quarter each: 32 dims) read
// the fp32 accumulators, take each row's amax over the head's 128 dims and
// write the FP8 codes and the folded head weight.  CTA (32, g): the new
// tokens of rows 64 g .. 64 g + 63 into the cache (threads 0..127).
constexpr int kFeRows = 64;
constexpr int kFeStages = 4;
constexpr int kFeK = 64;                                  // K elements per stage: one 128-byte swizzle row
constexpr int kFeWBytes = 128 * kFeK * 2;                 // 16 KB
constexpr int kFeXBytes = kFeRows * kFeK * 2;             // 8 KB
constexpr int kFeThreads = 192;
constexpr int kFeOffW = 0;
constexpr int kFeOffX = kFeOffW + kFeStages * kFeWBytes;  // 65,536
constexpr int kFeOffBars = kFeOffX + kFeStages * kFeXBytes;  // 98,304
constexpr int kFeNumBars = 3 * kFeStages + 1;             // W full, xn full, stage empty; done
constexpr int kFeOffNorm = kFeOffBars + kFeNumBars * 8;
constexpr int kFeOffAmax = kFeOffNorm + kFeRows * 4;
constexpr int kFeOffMisc = kFeOffAmax + 4 * kFeRows * 4;
constexpr size_t kFeSmem = 1024 + kFeOffMisc + 32;
constexpr int kFeTmemCols = 64;

struct FeParams {
  const uint16_t* c_q;     // bf16 [rows][dim]
  const uint16_t* gamma;   // bf16 [dim]
  int32_t dim;
  float eps;
  const float* head_w;     // fp32 [rows][32]
  int32_t rows;
  uint8_t* q_index;        // E4M3 [rows][32][128]
  float* head_w_out;       // fp32 [rows][32]
  float* q_proj;           // fp32 [rows][4096] or null
  AppendArgs app;
};

// Named barrier 2 over warps 2..5.
__device__ __forceinline__ void bar_fe() { asm volatile("bar.sync 2, 128;" ::: "memory"); }

__global__ void __launch_bounds__(kFeThreads, 1)
    frontend_kernel(const __grid_constant__ CUtensorMap tmap_w, const FeParams p) {
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  const int warp = threadIdx.x >> 5, lane = threadIdx.x & 31;
  const int row0 = blockIdx.y * kFeRows;
  const int nrow = min(kFeRows, p.rows - row0);
  if (blockIdx.x == kIdxHeads) {
    // ---- the new tokens of this CTA's rows into the cache
    float* warp_amax = reinterpret_cast<float*>(smem + kFeOffAmax);
    if (threadIdx.x < kAppendThreads)
      for (int r = 0; r < nrow; ++r) {
        append_row(p.app, row0 + r, threadIdx.x, warp_amax, [] { bar_append(); });
        bar_append();  // warp_amax is rewritten by the next row
      }
    return;
  }
  const uint32_t sbase = smem_u32(smem);
  const uint32_t bars = sbase + kFeOffBars;
  auto full_w = [&](int s) { return bars + 8u * s; };
  auto full_x = [&](int s) { return bars + 8u * (kFeStages + s); };
  auto empty = [&](int s) { return bars + 8u * (2 * kFeStages + s); };
  const uint32_t done = bars + 8u * (3 * kFeStages);
  float* norm = reinterpret_cast<float*>(smem + kFeOffNorm);
  float* amax_s = reinterpret_cast<float*>(smem + kFeOffAmax);  // [4 warps][64 rows]
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(smem + kFeOffMisc);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(smem + kFeOffMisc + 4);
  const int h = blockIdx.x;
  const int n_mma = max(16, (nrow + 15) & ~15);
  const int nk = p.dim / kFeK;
  if (threadIdx.x == 0) {
    for (int s = 0; s < kFeStages; ++s) {
      mbar_init(full_w(s), 1);
      mbar_init(full_x(s), 4);
      mbar_init(empty(s), 1);
    }
    mbar_init(done, 1);
    *abort_flag = 0;
    fence_mbar_init();
    prefetch_tmap(&tmap_w);
  }
  if (warp == 1) {
    tmem_alloc(smem_u32(tmem_slot), kFeTmemCols);
    tmem_relinquish();
  }
  tc_fence_before();
  __syncthreads();
  tc_fence_after();
  const uint32_t tmem = *tmem_slot;

  if (warp == 0) {
    if (lane == 0) {
      // ------------------------------------------------ W_h stages by TMA
      int issued = 0;
      for (int kc = 0; kc < nk; ++kc) {
        const int s = kc % kFeStages;
        if (!mbar_wait(empty(s), ((kc / kFeStages) & 1) ^ 1, abort_flag, p.app.status)) break;
        mbar_arrive_expect_tx(full_w(s), kFeWBytes);
        tma_load_2d(sbase + kFeOffW + s * kFeWBytes, &tmap_w, kc * kFeK, h * 128, full_w(s));
        ++issued;
      }
      // the copies still in flight land before the CTA exits (all of them have
      // landed already unless another role gave up)
      for (int kc = max(0, issued - kFeStages); kc < issued; ++kc)
        mbar_wait_drain(full_w(kc % kFeStages), (kc / kFeStages) & 1, 100000000ull);
    }
  } else if (warp == 1) {
    if (lane == 0) {
      // ------------------------------------------------ MMA issuer
      const uint32_t idesc = make_idesc(kFmtBF16, kFmtBF16, 0, 0, 128, (uint32_t)n_mma);
      bool ok = true;
      for (int kc = 0; kc < nk && ok; ++kc) {
        const int s = kc % kFeStages;
        ok = mbar_wait(full_w(s), (kc / kFeStages) & 1, abort_flag, p.app.status) &&
             mbar_wait(full_x(s), (kc / kFeStages) & 1, abort_flag, p.app.status);
        if (!ok) break;
        tc_fence_after();
        const uint32_t a0 = sbase + kFeOffW + s * kFeWBytes, b0 = sbase + kFeOffX + s * kFeXBytes;
#pragma unroll
        for (int kk = 0; kk < kFeK / 16; ++kk)
          mma_bf16(tmem, smem_desc(a0 + 32 * kk, 16, 1024, kLayoutSw128), smem_desc(b0 + 32 * kk, 16, 1024, kLayoutSw128),
                   idesc, (kc | kk) ? 1u : 0u);
        mma_commit(empty(s));
      }
      mma_commit(done);  // also after an abort: every issued MMA completes before TMEM is released
    }
  } else {
    // ------------------------------------------------ norm, xn stages, epilogue
    const int t = threadIdx.x - 64, eq = warp - 2;
    // 1 / sqrt(mean(c^2) + eps) per row, one warp per row
    for (int r = eq; r < nrow; r += 4) {
      const uint16_t* c = p.c_q + (int64_t)(row0 + r) * p.dim;
      float ss = 0.f;
      for (int i = 8 * lane; i < p.dim; i += 256) {
        const uint4 v = *reinterpret_cast<const uint4*>(c + i);
        const uint32_t w4[4] = {v.x, v.y, v.z, v.w};
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const float lo = __uint_as_float(w4[q] << 16), hi = __uint_as_float(w4[q] & 0xFFFF0000u);
          ss = fmaf(lo, lo, ss);
          ss = fmaf(hi, hi, ss);
        }
      }
#pragma unroll
      for (int o = 16; o > 0; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) norm[r] = 1.0f / sqrtf(ss / (float)p.dim + p.eps);
    }
    bar_fe();
    // xn stages: row r, 16-byte chunk cc (8 elements) of the stage's 64
    bool ok = true;
    for (int kc = 0; kc < nk; ++kc) {
      const int s = kc % kFeStages;
      ok = mbar_wait(empty(s), ((kc / kFeStages) & 1) ^ 1, abort_flag, p.app.status);
      if (!__all_sync(0xffffffffu, ok)) { ok = false; break; }
      uint8_t* xs = smem + kFeOffX + s * kFeXBytes;
      for (int idx = t; idx < n_mma * 8; idx += 128) {
        const int r = idx >> 3, cc = idx & 7;
        uint4 o = make_uint4(0u, 0u, 0u, 0u);
        if (r < nrow) {
          const int e0 = kc * kFeK + 8 * cc;
          const uint4 cv = *reinterpret_cast<const uint4*>(p.c_q + (int64_t)(row0 + r) * p.dim + e0);
          const uint4 gv = *reinterpret_cast<const uint4*>(p.gamma + e0);
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
          o = make_uint4(o4[0], o4[1], o4[2], o4[3]);
        }
        *reinterpret_cast<uint4*>(xs + swz128((uint32_t)(r * 128 + cc * 16))) = o;
      }
      fence_proxy_async_smem();
      __syncwarp();
      if (lane == 0) mbar_arrive(full_x(s));
    }
    // ---- epilogue: TMEM lane = dim 32 (warp % 4) + lane of the head, column = row
    const bool fin = mbar_wait(done, 0, abort_flag, p.app.status) && ok;
    tc_fence_after();
    const int quarter = warp & 3, d = quarter * 32 + lane;
    float v[kFeRows];
    {
      uint32_t r0[32], r1[32];
      const uint32_t ta = tmem + ((uint32_t)(quarter * 32) << 16);
      tmem_ld32(ta, r0);
      tmem_ld32(ta + 32, r1);
      tmem_ld_wait();
#pragma unroll
      for (int j = 0; j < 32; ++j) {
        v[j] = __uint_as_float(r0[j]);
        v[32 + j] = __uint_as_float(r1[j]);
      }
    }
    if (fin) {
#pragma unroll
      for (int r = 0; r < kFeRows; ++r) {
        if (r >= nrow) break;
        if (p.q_proj) p.q_proj[(int64_t)(row0 + r) * (kIdxHeads * kIdxDim) + h * kIdxDim + d] = v[r];
        const uint32_t m = __reduce_max_sync(0xffffffffu, __float_as_uint(fabsf(v[r])));  // |v| bits order as |v|
        if (lane == 0) amax_s[quarter * kFeRows + r] = __uint_as_float(m);
      }
    }
    bar_fe();
    if (fin) {
#pragma unroll
      for (int r = 0; r < kFeRows; ++r) {
        if (r >= nrow) break;
        const float amax = fmaxf(fmaxf(amax_s[r], amax_s[kFeRows + r]), fmaxf(amax_s[2 * kFeRows + r], amax_s[3 * kFeRows + r]));
        const float sc = amax > 0.f ? amax / 448.0f : 1.0f;
        p.q_index[(int64_t)(row0 + r) * (kIdxHeads * kIdxDim) + h * kIdxDim + d] = e4m3(v[r] / sc);
        if (t == r) p.head_w_out[(int64_t)(row0 + r) * kIdxHeads + h] = p.head_w[(int64_t)(row0 + r) * kIdxHeads + h] * sc;
      }
    }
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
  p.q_proj = q_proj;
  p.app = AppendArgs{base + c.latent_off, base + c.index_off, c.row_stride, c.num_blocks, c.key_format,
                     c.latent_format, c.latent_scale, bt.block_table, bt.max_blocks_per_seq, bt.seq_lens,
                     bt.queries_per_seq, std::min(bt.max_blocks_per_seq * kBlock, bt.max_seq_len), new_latent,
                     new_key, status};
  count_launches(1);
  frontend_kernel<<<dim3(kIdxHeads + 1, (unsigned)((rows + kFeRows - 1) / kFeRows)), kFeThreads, kFeSmem, st>>>(
      wmap, p);
  return launch_status();
}

}  // namespace dsa
