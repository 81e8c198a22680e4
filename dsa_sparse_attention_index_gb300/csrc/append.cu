// append.cu — the step's new tokens into the paged cache, and the indexer's
// query in FP8 (the front end of the fused decode path).
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

// One CTA per new token row nr = b * nq + j (token L_b - nq + j).
__global__ void __launch_bounds__(kAppendThreads)
    cache_append_kernel(uint8_t* latent_base, uint8_t* index_base, int64_t row_stride, int32_t num_blocks,
                        int32_t key_format, int32_t latent_format, float latent_scale,
                        const int32_t* block_table, int32_t max_blocks,
                        const int32_t* seq_lens, int32_t nq, int32_t cap, const uint16_t* new_latent,
                        const uint16_t* new_key, int32_t* status) {
  __shared__ float warp_amax[kAppendThreads / 32];
  const int nr = blockIdx.x, b = nr / nq, j = nr % nq, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int L = seq_lens[b];
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
    __syncthreads();
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

}  // namespace

dsa_status_t launch_cache_append(const dsa_paged_cache_t& c, const dsa_batch_t& bt, const uint16_t* new_latent,
                                 const uint16_t* new_key, int32_t* status, cudaStream_t st) {
  const int rows = bt.batch * bt.queries_per_seq;
  if (rows == 0) return DSA_OK;
  uint8_t* base = static_cast<uint8_t*>(c.base);
  const int cap = std::min(bt.max_blocks_per_seq * kBlock, bt.max_seq_len);
  count_launches(1);
  cache_append_kernel<<<rows, kAppendThreads, 0, st>>>(base + c.latent_off, base + c.index_off, c.row_stride,
                                                       c.num_blocks, c.key_format, c.latent_format,
                                                       c.latent_scale, bt.block_table,
                                                       bt.max_blocks_per_seq, bt.seq_lens, bt.queries_per_seq, cap,
                                                       new_latent, new_key, status);
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

}  // namespace dsa
