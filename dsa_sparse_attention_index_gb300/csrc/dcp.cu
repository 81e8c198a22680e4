// dcp.cu — decode context parallelism emulated on one GPU: the exact top-k
// merge across W token shards.
//
// vLLM Day-0 post for Kimi K3.1 Pro, decode-context-parallelism section.
// Shard r of W holds the tokens t with t mod W = r (local position t div W).
// Each shard sends only its best ceil(1.5 k / W) candidates, picked on bf16
// scores, each packed with its score into one 32-bit word (about ten times
// fewer bytes than a full local top-k of (fp32 score, token id) pairs); every
// shard then radix-selects the same global top-k from the gathered words.
// The merge stays exact: a shard all of whose words were taken, and which
// has not sent its full local top-k, may hold more of the top-k, so it
// resends its full local top-k for that row and the selection runs again.
//
// Here the W shards are CTAs of one grid and the exchange is global memory:
//   1. dcp_candidates_kernel, one CTA per (row, shard): the shard's keys in
//      shared memory, a two-digit radix selection of its best `c`, and the
//      words in local order;
//   2. dcp_merge_kernel, one CTA per row: the global top-k of the gathered
//      words, by (bf16 key desc, global index asc), a six-digit radix
//      selection over 48-bit composites in shared memory; shards that must
//      resend are flagged and the row is left for the second round;
//   3. the candidate kernel again for the flagged (row, shard) pairs, now with
//      their full local top-k, and
//   4. the merge kernel again for the flagged rows.
// Readings (as the oracle's): the word is the 16-bit order key of the
// bf16-rounded score above the 16-bit local position, so a shard holds at
// most 65,536 tokens of a row; keys order as the fp32 top-k does (NaN below
// every number, -0 = +0) and equal keys go to the lower global index.  The
// result is the top-k of the bf16-rounded scores, in ascending token order.
#include <algorithm>

#include <cuda_bf16.h>

#include "common.cuh"
#include "internal.h"

namespace dsa {

namespace {

constexpr int kDcpThreads = 512;
constexpr int kDcpWarps = kDcpThreads / 32;

// 16-bit order key of the bf16-rounded score: higher score -> larger key,
// NaN -> 0 (below every number), -0 folded into +0.
__device__ __forceinline__ uint32_t bf16_order_key(float x) {
  const uint32_t u = __float_as_uint(x);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0u;
  uint32_t b = (uint32_t)__bfloat16_as_ushort(__float2bfloat16_rn(x));
  if (b == 0x8000u) b = 0u;
  return (b & 0x8000u) ? (~b & 0xFFFFu) : (b | 0x8000u);
}

// Block-wide exclusive prefix sum of one value per thread; `total` gets the sum.
__device__ __forceinline__ uint32_t dcp_block_scan(uint32_t v, uint32_t* sh, uint32_t& total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t u = __shfl_up_sync(0xffffffffu, x, d);
    if (lane >= d) x += u;
  }
  if (lane == 31) sh[wid] = x;
  __syncthreads();
  if (wid == 0) {
    uint32_t w = lane < kDcpWarps ? sh[lane] : 0u;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t u = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += u;
    }
    sh[lane] = w;
  }
  __syncthreads();
  total = sh[kDcpWarps - 1];
  const uint32_t r = (wid ? sh[wid - 1] : 0u) + x - v;
  __syncthreads();
  return r;
}

// The bin of `hist` (nb bins, ascending values) holding the need-th largest
// element, counting from the top; `need` becomes the count still needed
// inside that bin and `pop` its population.
__device__ void dcp_pick(const uint32_t* hist, int nb, uint32_t* sh, uint32_t& need, int& bin, uint32_t& pop) {
  const int per = (nb + kDcpThreads - 1) / kDcpThreads;  // bins per thread, from the top
  uint32_t c = 0;
  for (int i = 0; i < per; ++i) {
    const int b = nb - 1 - ((int)threadIdx.x * per + i);
    if (b >= 0) c += hist[b];
  }
  uint32_t total;
  const uint32_t excl = dcp_block_scan(c, sh, total);
  __shared__ int s_bin;
  __shared__ uint32_t s_need, s_pop;
  if (excl < need && excl + c >= need) {
    uint32_t run = excl;
    for (int i = 0; i < per; ++i) {
      const int b = nb - 1 - ((int)threadIdx.x * per + i);
      if (b < 0) break;
      if (run + hist[b] >= need) {
        s_bin = b;
        s_need = need - run;
        s_pop = hist[b];
        break;
      }
      run += hist[b];
    }
  }
  __syncthreads();
  bin = s_bin;
  need = s_need;
  pop = s_pop;
  __syncthreads();
}

// A row's length, clamped to [0, cap]; an out-of-range length is reported.
__device__ __forceinline__ int dcp_row_len(const int32_t* row_lens, int r, int cap, int32_t* status) {
  const int len = row_lens[r];
  if (len < 0 || len > cap) {
    if (status && threadIdx.x == 0) report(status, DSA_ERR_BOUNDS);
    return len < 0 ? 0 : cap;
  }
  return len;
}

struct DcpWs {
  uint32_t* cand;   // [rows][W][cap] words: key << 16 | local position, in local order
  int32_t* nsent;   // [rows][W] words a shard has sent
  int32_t* flag;    // [rows][W] the shard resends its full local top-k
  int32_t* rowflag; // [rows] the row needs the second round
  int cap;          // max(ceil(1.5 k / W), k)
};

// ---- 1 / 3: one shard's best `c` of a row (second round: flagged shards, c = min(k, n)).
__global__ void __launch_bounds__(kDcpThreads, 1)
    dcp_candidates_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* row_lens, int cap, int k,
                          int W, int c1, bool resend, int n_cap, DcpWs ws, int32_t* status) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint16_t* key = reinterpret_cast<uint16_t*>(smem_raw);                 // [n_cap], n_cap a multiple of 8
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem_raw + 2 * n_cap);  // [2048]
  uint32_t* sh = hist + 2048;                                          // [32]
  const int s = blockIdx.x, r = blockIdx.y, tid = threadIdx.x;
  const int64_t rs = (int64_t)r * W + s;
  grid_dep_wait();
  if (resend && ws.flag[rs] == 0) return;
  if (!resend && tid == 0) ws.flag[rs] = 0;
  const int len = dcp_row_len(row_lens, r, cap, resend ? nullptr : status);
  const int n = len > s ? (len - s + W - 1) / W : 0;  // this shard's tokens of the row
  const int cnt = resend ? min(k, n) : min(c1, n);
  const float* row = scores + (int64_t)r * ld;
  for (int l = tid; l < n; l += kDcpThreads) key[l] = (uint16_t)bf16_order_key(row[(int64_t)l * W + s]);
  // the threshold key T and how many keys equal to T are taken (lowest local positions)
  uint32_t thr = 0, take_eq = 0;
  bool all = cnt >= n;
  if (!all) {
    for (int i = tid; i < 2048; i += kDcpThreads) hist[i] = 0u;
    __syncthreads();
    for (int l = tid; l < n; l += kDcpThreads) atomicAdd(&hist[key[l] >> 5], 1u);
    __syncthreads();
    uint32_t need = (uint32_t)cnt, pop;
    int hi;
    dcp_pick(hist, 2048, sh, need, hi, pop);
    for (int i = tid; i < 32; i += kDcpThreads) hist[i] = 0u;
    __syncthreads();
    for (int l = tid; l < n; l += kDcpThreads)
      if ((key[l] >> 5) == (uint32_t)hi) atomicAdd(&hist[key[l] & 31], 1u);
    __syncthreads();
    int lo;
    dcp_pick(hist, 32, sh, need, lo, pop);
    thr = ((uint32_t)hi << 5) | (uint32_t)lo;
    take_eq = need;
  }
  // the words in local order: thread t owns positions [t m, t m + m)
  const int m = (n + kDcpThreads - 1) / kDcpThreads;
  const int l0 = min(n, tid * m), l1 = min(n, l0 + m);
  uint32_t c_gt = 0, c_eq = 0;
  if (!all)
    for (int l = l0; l < l1; ++l) {
      c_gt += key[l] > thr;
      c_eq += key[l] == thr;
    }
  uint32_t tot;
  const uint32_t eq_before = dcp_block_scan(c_eq, sh, tot);
  const uint32_t eq_mine = all ? 0u : (eq_before >= take_eq ? 0u : min(c_eq, take_eq - eq_before));
  uint32_t pos = dcp_block_scan(all ? (uint32_t)(l1 - l0) : c_gt + eq_mine, sh, tot);
  uint32_t* out = ws.cand + rs * ws.cap;
  uint32_t eq_left = eq_mine;
  for (int l = l0; l < l1; ++l) {
    bool take = all || key[l] > thr;
    if (!take && key[l] == thr && eq_left) {
      take = true;
      --eq_left;
    }
    if (take) out[pos++] = ((uint32_t)key[l] << 16) | (uint32_t)l;
  }
  if (tid == 0) ws.nsent[rs] = cnt;
  grid_dep_launch();
}

// ---- 2 / 4: the global top-k of a row from its shards' words (second round:
//      the flagged rows, with the resent full local top-ks).
__global__ void __launch_bounds__(kDcpThreads, 1)
    dcp_merge_kernel(const int32_t* row_lens, int cap, int k, int W, bool final_round, int len_cap, int m_cap,
                     DcpWs ws, int32_t* out, int32_t* stats, int32_t* status) {
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint64_t* comp = reinterpret_cast<uint64_t*>(smem_raw);                      // [m_cap] composites
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(smem_raw + 8 * (size_t)m_cap);  // [len_cap / 32]
  uint32_t* hist = bitmap + len_cap / 32;                                       // [256]
  uint32_t* sh = hist + 256;                                                    // [32]
  __shared__ int s_base[16 + 1];
  __shared__ uint32_t s_taken[16];
  __shared__ int s_again;
  const int r = blockIdx.x, tid = threadIdx.x;
  grid_dep_wait();
  if (final_round && ws.rowflag[r] == 0) return;
  const int len = dcp_row_len(row_lens, r, cap, nullptr);
  // the gathered words, as composites (key << 32) | ~global: larger = earlier in the order
  if (tid == 0) {
    int b = 0;
    for (int s = 0; s < W; ++s) {
      s_base[s] = b;
      b += ws.nsent[(int64_t)r * W + s];
    }
    s_base[W] = b;
    s_again = 0;
  }
  if (tid < 16) s_taken[tid] = 0u;
  __syncthreads();
  const int m = s_base[W];
  if (m > m_cap) {  // cannot happen for the sizes the host allows
    if (tid == 0) report(status, DSA_ERR_BOUNDS);
    return;
  }
  for (int s = 0; s < W; ++s) {
    const uint32_t* src = ws.cand + ((int64_t)r * W + s) * ws.cap;
    const int ns = s_base[s + 1] - s_base[s];
    for (int i = tid; i < ns; i += kDcpThreads) {
      const uint32_t w = src[i];
      const uint32_t global = (w & 0xFFFFu) * (uint32_t)W + (uint32_t)s;
      comp[s_base[s] + i] = ((uint64_t)(w >> 16) << 32) | (uint64_t)(~global);
    }
  }
  __syncthreads();
  const int sel = min(k, m);
  // the sel-th largest composite (all distinct): six 8-bit digits, bits 47..0
  uint64_t prefix = 0;
  uint32_t need = (uint32_t)sel, pop = 0;
  int shift = 48;
  if (sel < m) {
    while (shift > 0) {
      shift -= 8;
      for (int i = tid; i < 256; i += kDcpThreads) hist[i] = 0u;
      __syncthreads();
      for (int i = tid; i < m; i += kDcpThreads) {
        const uint64_t v = comp[i];
        if ((v >> (shift + 8)) == (prefix >> (shift + 8))) atomicAdd(&hist[(v >> shift) & 0xFFu], 1u);
      }
      __syncthreads();
      int bin;
      dcp_pick(hist, 256, sh, need, bin, pop);
      prefix |= (uint64_t)bin << shift;
      if (need == pop) break;  // the whole bin is taken: prefix bounds the selection
    }
  }
  // taken: composites >= prefix (the bin at `shift` taken whole), or all when sel == m
  const uint64_t thr = sel < m ? prefix : 0ull;
  for (int i = tid; i < len_cap / 32; i += kDcpThreads) bitmap[i] = 0u;
  __syncthreads();
  for (int i = tid; i < m; i += kDcpThreads) {
    const uint64_t v = comp[i];
    if (v >= thr) {
      const uint32_t global = ~(uint32_t)v;
      atomicAdd(&s_taken[global % (uint32_t)W], 1u);
      if (global < (uint32_t)len_cap) atomicOr(&bitmap[global >> 5], 1u << (global & 31));
    }
  }
  __syncthreads();
  if (!final_round && tid < W) {
    // a shard whose words were all taken and which has not sent its full
    // local top-k may hold more of the top-k: it resends
    const int n = len > tid ? (len - tid + W - 1) / W : 0;
    const int sent = s_base[tid + 1] - s_base[tid];
    const bool again = (int)s_taken[tid] == sent && sent < min(k, n);
    ws.flag[(int64_t)r * W + tid] = again ? 1 : 0;
    if (again) atomicAdd(&s_again, 1);
  }
  __syncthreads();
  if (!final_round) {
    if (tid == 0) {
      ws.rowflag[r] = s_again ? 1 : 0;
      if (stats) {
        stats[3 * r] = m;
        stats[3 * r + 1] = s_again;
        stats[3 * r + 2] = 0;
      }
    }
    if (s_again) return;  // the second round writes this row
  } else if (tid == 0 && stats) {
    int resent = 0;
    for (int s = 0; s < W; ++s)
      if (ws.flag[(int64_t)r * W + s]) resent += ws.nsent[(int64_t)r * W + s];
    stats[3 * r + 2] = resent;
  }
  // the chosen indices in ascending order, from the bitmap
  const int words = (len + 31) / 32;
  const int per = (words + kDcpThreads - 1) / kDcpThreads;
  const int w0 = min(words, tid * per), w1 = min(words, w0 + per);
  uint32_t c = 0;
  for (int w = w0; w < w1; ++w) c += __popc(bitmap[w]);
  uint32_t tot;
  uint32_t p = dcp_block_scan(c, sh, tot);
  int32_t* o = out + (int64_t)r * k;
  for (int w = w0; w < w1; ++w) {
    uint32_t bits = bitmap[w];
    while (bits) {
      const int b = __ffs(bits) - 1;
      bits &= bits - 1;
      if (p < (uint32_t)k) o[p] = w * 32 + b;
      ++p;
    }
  }
  for (int i = (int)tot + tid; i < k; i += kDcpThreads) o[i] = -1;
  if (tid == 0 && tot != (uint32_t)sel) report(status, DSA_ERR_BOUNDS);  // consistency check
  grid_dep_launch();
}


// ---------------------------------------------------------------- LSE combine
// The second half of the DCP exchange (same section): every shard attends
// only over the selected tokens it holds, and the shards' partial outputs are
// merged through their log-sum-exp.  Emulated here with the shard's token
// groups as chunks of the MLA kernel:
//   1. dcp_group_kernel, one CTA per (shard, row): the row's selected indices grouped
//      by shard (t mod W), in their original order inside a shard, each
//      shard's group cut into P pieces of the MLA kernel's chunk (1,024
//      tokens; P = 2 covers a shard that holds all 2,048);
//   2. the MLA kernel over those pieces (unnormalised partials, max and sums);
//   3. dcp_combine_kernel: per shard, the output it would send (its pieces
//      merged: bf16 O_r and fp32 LSE_r, the exchanged format), then the LSE
//      combine of the W shards from those rounded values.

// Selected indices of a row grouped by shard, one CTA per (shard r, row):
// seg[row][r * P + j] is where piece j of shard r starts in gidx[row],
// seg[row][W * P] the number of entries >= 0; the rest of gidx[row] is -1.
// Pieces are `piece` tokens long from the group's start, so a group of at
// most `piece` tokens leaves its later pieces empty (their CTAs of the MLA
// kernel return at once).  One block scan of packed counts places the group:
// the low 16 bits count shard r's entries, the high 16 bits those of shards
// below r (each at most 2,048, so no carry crosses).
__global__ void __launch_bounds__(kDcpThreads) dcp_group_kernel(const int32_t* __restrict__ idx, int k, int W,
                                                                int P, int piece, int32_t* __restrict__ gidx,
                                                                int32_t* __restrict__ seg) {
  __shared__ uint32_t sh[32];
  constexpr int kPer = (kMaxTopk + kDcpThreads - 1) / kDcpThreads;
  const int r = blockIdx.x, row = blockIdx.y;
  const int per = (k + kDcpThreads - 1) / kDcpThreads;
  const int i0 = (int)threadIdx.x * per;
  int32_t t[kPer];
  uint32_t c = 0;
#pragma unroll
  for (int j = 0; j < kPer; ++j) {
    t[j] = (j < per && i0 + j < k) ? idx[(int64_t)row * k + i0 + j] : -1;
    if (t[j] >= 0) {
      const int s = t[j] % W;
      c += s == r ? 1u : (s < r ? 0x10000u : 0u);
    }
  }
  uint32_t tot;
  const uint32_t e = dcp_block_scan(c, sh, tot);
  const uint32_t base = tot >> 16, n = tot & 0xFFFFu;
  int32_t* g = gidx + (int64_t)row * k;
  int32_t* sg = seg + (int64_t)row * (W * P + 1);
  uint32_t pos = base + (e & 0xFFFFu);
#pragma unroll
  for (int j = 0; j < kPer; ++j)
    if (t[j] >= 0 && t[j] % W == r) g[pos++] = t[j];
  if (threadIdx.x == 0)
    for (int j = 0; j < P; ++j) sg[r * P + j] = (int32_t)(base + min(n, (uint32_t)(j * piece)));
  if (r == W - 1) {  // the last group ends where the entries end: pad the rest
    for (int i = (int)(base + n) + (int)threadIdx.x; i < k; i += kDcpThreads) g[i] = -1;
    if (threadIdx.x == 0) sg[W * P] = (int32_t)(base + n);
  }
}

__device__ __forceinline__ float dcp_ex2(float x) {
  float y;
  asm("ex2.approx.ftz.f32 %0, %1;" : "=f"(y) : "f"(x));
  return y;
}

constexpr int kDcpCombineHeads = 8;
constexpr int kDcpMaxPieces = 16;

// Per (row, 8 heads): each shard's output from its pieces, as the MLA's own
// chunk merge forms it (max, weights 2^(m - M), output normalised by the sum of
// the rounded probabilities, LSE from the exact sum), rounded to bf16; then
// out = sum_r 2^(LSE_r - LSE) * O_r with LSE = log2 sum_r 2^LSE_r (log2 units
// inside, natural log stored).  part_out / part_lse (nullable) receive the
// shards' outputs, [W][rows][96][512] bf16 and [W][rows][96] fp32.
template <int P>
__global__ void __launch_bounds__(256) dcp_combine_kernel(const uint16_t* __restrict__ opart,
                                                           const float* __restrict__ ml, int W, int rows,
                                                           float latent_scale, uint16_t* __restrict__ out,
                                                           float* __restrict__ lse, uint16_t* __restrict__ part_out,
                                                           float* __restrict__ part_lse) {
  const int row = blockIdx.y, h0 = blockIdx.x * kDcpCombineHeads;
  const int nseg = W * P;
  __shared__ float wgt[kDcpCombineHeads][kDcpMaxPieces];      // a piece's weight inside its shard
  __shared__ float swt[kDcpCombineHeads][DSA_DCP_MAX_SHARDS];  // a shard's weight in the output
  grid_dep_wait();  // the partials come from the previous kernel
  const float4* mlr = reinterpret_cast<const float4*>(ml) + (int64_t)row * nseg * kHeads;
  constexpr float kLn2 = 0.69314718055994531f;
  if (threadIdx.x < kDcpCombineHeads) {
    const int hl = threadIdx.x, h = h0 + hl;
    float lse2[DSA_DCP_MAX_SHARDS];
    float G = -INFINITY;
#pragma unroll
    for (int r = 0; r < DSA_DCP_MAX_SHARDS; ++r) {
      lse2[r] = -INFINITY;
      if (r >= W) continue;
      float M = -INFINITY;
      for (int j = 0; j < P; ++j) M = fmaxf(M, mlr[(r * P + j) * kHeads + h].x);
      float den = 0.f, ex = 0.f;
      for (int j = 0; j < P; ++j) {
        const float4 v = mlr[(r * P + j) * kHeads + h];
        const float w = (M == -INFINITY || v.x == -INFINITY) ? 0.f : dcp_ex2(v.x - M);
        den += w * v.y;
        ex += w * v.z;
        wgt[hl][r * P + j] = w * v.y;  // the piece's partial is normalised by v.y
      }
      const float inv = den > 0.f ? latent_scale / den : 0.f;
      for (int j = 0; j < P; ++j) wgt[hl][r * P + j] *= inv;
      lse2[r] = (M == -INFINITY || ex <= 0.f) ? -INFINITY : M + log2f(ex);
      G = fmaxf(G, lse2[r]);
      if (part_lse) part_lse[((int64_t)r * rows + row) * kHeads + h] = lse2[r] * kLn2;
    }
    float U = 0.f;
#pragma unroll
    for (int r = 0; r < DSA_DCP_MAX_SHARDS; ++r) {
      const float u = (lse2[r] == -INFINITY) ? 0.f : dcp_ex2(lse2[r] - G);  // 0 past the W shards
      swt[hl][r] = u;
      U += u;
    }
    const float invU = U > 0.f ? 1.f / U : 0.f;
#pragma unroll
    for (int r = 0; r < DSA_DCP_MAX_SHARDS; ++r) swt[hl][r] *= invU;
    lse[(int64_t)row * kHeads + h] = (G == -INFINITY) ? -INFINITY : (G + log2f(U)) * kLn2;
  }
  __syncthreads();
  constexpr int kVec = kDcpCombineHeads * kValue / 4;  // 1024 float4s per CTA
  for (int v = threadIdx.x; v < kVec; v += blockDim.x) {
    const int hl = v / (kValue / 4), d = (v % (kValue / 4)) * 4;
    const uint16_t* src = opart + ((int64_t)row * nseg * kHeads + h0 + hl) * kValue + d;
    // an empty piece wrote no partial: only pieces with weight are read
    float4 x[DSA_DCP_MAX_SHARDS * P];
#pragma unroll
    for (int s = 0; s < DSA_DCP_MAX_SHARDS * P; ++s)
      if (s < nseg && wgt[hl][s] != 0.f) {
        const uint2 hv = *reinterpret_cast<const uint2*>(src + (int64_t)s * kHeads * kValue);
        const float2 a = __half22float2(*reinterpret_cast<const __half2*>(&hv.x));
        const float2 b = __half22float2(*reinterpret_cast<const __half2*>(&hv.y));
        x[s] = make_float4(a.x, a.y, b.x, b.y);
      }
    float4 a = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
    for (int r = 0; r < DSA_DCP_MAX_SHARDS; ++r) {
      if (r >= W) break;
      float4 o = make_float4(0.f, 0.f, 0.f, 0.f);
#pragma unroll
      for (int j = 0; j < P; ++j) {
        const int s = r * P + j;
        const float w = wgt[hl][s];
        if (w != 0.f) {
          o.x = fmaf(w, x[s].x, o.x); o.y = fmaf(w, x[s].y, o.y);
          o.z = fmaf(w, x[s].z, o.z); o.w = fmaf(w, x[s].w, o.w);
        }
      }
      const __nv_bfloat162 lo = __floats2bfloat162_rn(o.x, o.y);
      const __nv_bfloat162 hi = __floats2bfloat162_rn(o.z, o.w);
      if (part_out) {
        uint2 pk;
        pk.x = *reinterpret_cast<const uint32_t*>(&lo);
        pk.y = *reinterpret_cast<const uint32_t*>(&hi);
        *reinterpret_cast<uint2*>(part_out + (((int64_t)r * rows + row) * kHeads + h0 + hl) * kValue + d) = pk;
      }
      const float2 l2 = __bfloat1622float2(lo), h2 = __bfloat1622float2(hi);
      const float u = swt[hl][r];
      a.x = fmaf(u, l2.x, a.x); a.y = fmaf(u, l2.y, a.y);
      a.z = fmaf(u, h2.x, a.z); a.w = fmaf(u, h2.y, a.w);
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

size_t dcp_workspace_bytes(int rows, int k, int shards) {
  if (rows <= 0 || shards < 1) return 0;
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  const int c1 = (3 * k + 2 * shards - 1) / (2 * shards);
  const size_t cap = (size_t)std::max(c1, k);
  return al((size_t)rows * shards * cap * 4) + 3 * al((size_t)rows * shards * 4);
}

dsa_status_t launch_dcp_topk(const float* scores, int64_t ld, const int32_t* row_lens, int rows, int max_row_len,
                             int k, int shards, int32_t* out, int32_t* stats, void* workspace, int32_t* status,
                             cudaStream_t st) {
  if (rows == 0) return DSA_OK;
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  const int W = shards;
  const int c1 = (3 * k + 2 * W - 1) / (2 * W);
  DcpWs ws;
  ws.cap = std::max(c1, k);
  uint8_t* w = static_cast<uint8_t*>(workspace);
  ws.cand = reinterpret_cast<uint32_t*>(w);
  w += al((size_t)rows * W * ws.cap * 4);
  ws.nsent = reinterpret_cast<int32_t*>(w);
  w += al((size_t)rows * W * 4);
  ws.flag = reinterpret_cast<int32_t*>(w);
  w += al((size_t)rows * W * 4);
  ws.rowflag = reinterpret_cast<int32_t*>(w);
  // shared memory: a shard's keys (2 B each); the merge's composites and the row's bitmap
  const int n_cap = (((max_row_len + W - 1) / W) + 7) & ~7;
  const size_t smem1 = 2 * (size_t)n_cap + 4 * (2048 + 32);
  // words a row can gather: after resends, at most 2W/3 shards send k, the rest c1
  const int m_cap = std::min(W * ws.cap, (2 * W / 3) * k + W * c1 + k);
  const int len_cap = ((max_row_len + 31) / 32) * 32;
  const size_t smem2 = 8 * (size_t)m_cap + (size_t)len_cap / 8 + 4 * (256 + 32);
  // room is raised per device as larger launches come (each kernel also has a
  // few hundred bytes of static shared memory within the 227 KB)
  constexpr size_t kMaxDyn = 226 * 1024;
  if (smem1 > kMaxDyn || smem2 > kMaxDyn) return DSA_ERR_UNSUPPORTED;
  static size_t set1[64] = {}, set2[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 0 || dev >= 64) return DSA_ERR_UNSUPPORTED;
  if (smem1 > set1[dev]) {
    if (cuda_status(cudaFuncSetAttribute(dcp_candidates_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem1)) != DSA_OK)
      return DSA_ERR_CUDA;
    set1[dev] = smem1;
  }
  if (smem2 > set2[dev]) {
    if (cuda_status(cudaFuncSetAttribute(dcp_merge_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem2)) != DSA_OK)
      return DSA_ERR_CUDA;
    set2[dev] = smem2;
  }
  const dim3 g1((unsigned)W, (unsigned)rows);
  count_launches(4);
  dcp_candidates_kernel<<<g1, kDcpThreads, smem1, st>>>(scores, ld, row_lens, max_row_len, k, W, c1, false, n_cap,
                                                         ws, status);
  dcp_merge_kernel<<<rows, kDcpThreads, smem2, st>>>(row_lens, max_row_len, k, W, false, len_cap, m_cap, ws, out,
                                                     stats, status);
  dcp_candidates_kernel<<<g1, kDcpThreads, smem1, st>>>(scores, ld, row_lens, max_row_len, k, W, c1, true, n_cap,
                                                         ws, status);
  dcp_merge_kernel<<<rows, kDcpThreads, smem2, st>>>(row_lens, max_row_len, k, W, true, len_cap, m_cap, ws, out,
                                                     stats, status);
  return launch_status();
}

// Pieces per shard: a shard may hold all k selected tokens, and a piece is at
// most one MLA chunk.
static int dcp_pieces(int k) { return (k + mla_max_chunk() - 1) / mla_max_chunk(); }

size_t dcp_mla_workspace_bytes(int rows, int k, int shards) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t nseg = (size_t)shards * dcp_pieces(k);
  return al((size_t)rows * k * 4) + al((size_t)rows * (nseg + 1) * 4) + al((size_t)rows * nseg * kHeads * kValue * 2) +
         al((size_t)rows * nseg * kHeads * 16);
}

dsa_status_t launch_dcp_sparse_mla(const dsa_paged_cache_t& c, const dsa_batch_t& bt, const uint16_t* q_mla,
                                   const int32_t* idx, int k, int shards, float sm_scale, uint16_t* out, float* lse,
                                   uint16_t* part_out, float* part_lse, void* workspace, int32_t* status,
                                   cudaStream_t st) {
  const int rows = bt.batch * bt.queries_per_seq;
  if (rows == 0) return DSA_OK;
  const int W = shards, P = dcp_pieces(k), nseg = W * P;
  if (P > 2) return DSA_ERR_UNSUPPORTED;  // k <= 2,048 and chunks of 1,024 tokens
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  uint8_t* w = static_cast<uint8_t*>(workspace);
  int32_t* gidx = reinterpret_cast<int32_t*>(w);
  w += al((size_t)rows * k * 4);
  int32_t* seg = reinterpret_cast<int32_t*>(w);
  w += al((size_t)rows * (nseg + 1) * 4);
  uint16_t* opart = reinterpret_cast<uint16_t*>(w);
  w += al((size_t)rows * nseg * kHeads * kValue * 2);
  float* ml = reinterpret_cast<float*>(w);
  count_launches(1);
  dcp_group_kernel<<<dim3((unsigned)W, (unsigned)rows), kDcpThreads, 0, st>>>(idx, k, W, P, mla_max_chunk(), gidx,
                                                                             seg);
  dsa_status_t s = launch_status();
  if (s != DSA_OK) return s;
  s = launch_sparse_mla_partials(c, bt, q_mla, gidx, k, seg, nseg, sm_scale, opart, ml, status, st);
  if (s != DSA_OK) return s;
  cudaLaunchAttribute attrs[1];
  attrs[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attrs[0].val.programmaticStreamSerializationAllowed = 1;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3(kHeads / kDcpCombineHeads, (unsigned)rows);
  cfg.blockDim = dim3(256);
  cfg.stream = st;
  cfg.attrs = attrs;
  cfg.numAttrs = 1;
  count_launches(1);
  const cudaError_t e =
      P == 1 ? cudaLaunchKernelEx(&cfg, dcp_combine_kernel<1>, (const uint16_t*)opart, (const float*)ml, W, rows,
                                  c.latent_scale, out, lse, part_out, part_lse)
             : cudaLaunchKernelEx(&cfg, dcp_combine_kernel<2>, (const uint16_t*)opart, (const float*)ml, W, rows,
                                  c.latent_scale, out, lse, part_out, part_lse);
  if (cuda_status(e) != DSA_OK) return DSA_ERR_CUDA;
  return launch_status();
}

}  // namespace dsa
