// topk.cu — exact per-row top-k selection (stage 2 of DSA).
//
// Keeps the k (= 2,048 in the model) highest-scoring visible tokens of each
// query row (vLLM Day-0 post for Kimi K3.1 Pro, sparse-attention section:
// "then keep the top 2,048 tokens"; fused-decode section: an exact top-k
// selection kernel).  Equal scores go to the lower token index, so the
// selected set is unique; it is written in ascending token order with -1
// padding when a row has fewer than k tokens.
//
// Scores are compared as order-preserving 32-bit keys (integer radix).
//   1. hist:    multi-CTA per row: 4096-bin histogram of the key's top 12
//               bits, merged into a per-row global histogram.
//   2. threshold: one CTA per row finds the bin T holding the k-th largest
//               key and the count above it.
//   3. collect: multi-CTA per row: every CTA scans its segment: keys above T
//               are selected outright (fewer than k of them); keys in T become
//               candidates (key, index), reserved with one atomic per CTA.
//   4. final:   one CTA per row: radix-selects the remaining (k - selected)
//               candidates by (key desc, index asc) on 52 packed bits, then
//               writes the chosen indices in ascending order through a
//               shared-memory bitmap of the index range.  If the candidate
//               buffer overflowed (heavily tied scores) it re-derives the
//               candidates from the scores directly.
// The multi-CTA split keeps all SMs busy for the few-long-rows case (4 rows
// of 1M tokens) as well as for many shorter rows.
#include <algorithm>
#include <mutex>

#include "common.cuh"
#include "internal.h"

namespace dsa {

namespace {

constexpr int kBins = 4096;           // 12-bit first digit
constexpr int kSeg = 8192;            // tokens per CTA in hist/collect
constexpr int kThreads = 256;
constexpr int kCandCap = 8192;        // candidates kept per row
constexpr int kFinalThreads = 512;
constexpr int kWindowBits = 1 << 20;  // bitmap window of the final sort (128 KB)
constexpr int kVecPerThread = kSeg / 4 / kThreads;  // float4 loads per thread and segment

struct TopkWs {
  uint32_t* hist;    // [rows][kBins]
  uint32_t* counts;  // [rows][4]: selected, candidates
  int32_t* sel;      // [rows][k]
  uint64_t* cand;    // [rows][kCandCap]
};

__device__ __forceinline__ int row_len(const int32_t* row_lens, const int32_t* seq_lens, int nq, int r, int cap,
                                       int32_t* status) {
  int len = row_lens ? row_lens[r] : visible_len(seq_lens[r / nq], nq, r % nq);
  if (len < 0 || len > cap) {
    report(status, DSA_ERR_BOUNDS);
    len = len < 0 ? 0 : cap;
  }
  return len;
}

__global__ void __launch_bounds__(kThreads) topk_hist_kernel(const float* __restrict__ scores, int64_t ld,
                                                              const int32_t* row_lens, const int32_t* seq_lens,
                                                              int nq, int cap, int k, TopkWs ws, int32_t* status) {
  __shared__ uint32_t h[kBins];
  const int r = blockIdx.y;
  const int len = row_len(row_lens, seq_lens, nq, r, cap, status);
  const int64_t t0 = (int64_t)blockIdx.x * kSeg;
  if (len <= k || t0 >= len) return;
  for (int i = threadIdx.x; i < kBins; i += kThreads) h[i] = 0;
  __syncthreads();
  const int n = (int)std::min<int64_t>(kSeg, len - t0);
  const float* row = scores + (int64_t)r * ld + t0;
  const int n4 = n >> 2;
  const float4* row4 = reinterpret_cast<const float4*>(row);
  float4 v[kVecPerThread];  // every load of this thread in flight before the first use
#pragma unroll
  for (int c = 0; c < kVecPerThread; ++c) {
    const int i = threadIdx.x + c * kThreads;
    v[c] = i < n4 ? row4[i] : make_float4(0.f, 0.f, 0.f, 0.f);
  }
#pragma unroll
  for (int c = 0; c < kVecPerThread; ++c) {
    if (threadIdx.x + c * kThreads < n4) {
      atomicAdd(&h[score_key(v[c].x) >> 20], 1u);
      atomicAdd(&h[score_key(v[c].y) >> 20], 1u);
      atomicAdd(&h[score_key(v[c].z) >> 20], 1u);
      atomicAdd(&h[score_key(v[c].w) >> 20], 1u);
    }
  }
  for (int i = 4 * n4 + threadIdx.x; i < n; i += kThreads) atomicAdd(&h[score_key(row[i]) >> 20], 1u);
  __syncthreads();
  uint32_t* g = ws.hist + (int64_t)r * kBins;
  for (int i = threadIdx.x; i < kBins; i += kThreads)
    if (h[i]) atomicAdd(&g[i], h[i]);
}

// Per row: the threshold bin T of the first digit (the bin holding the k-th
// largest key) and the count strictly above it, from the row's histogram;
// T = -1 for rows with at most k tokens.  Written to counts[r][2..3].
__global__ void __launch_bounds__(kThreads) topk_threshold_kernel(const int32_t* row_lens, const int32_t* seq_lens,
                                                                   int nq, int cap, int k, TopkWs ws) {
  __shared__ uint32_t wsum[kThreads / 32];
  const int r = blockIdx.x, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const int len = row_len(row_lens, seq_lens, nq, r, cap, nullptr);
  uint32_t* cnt = ws.counts + 4 * (int64_t)r;
  if (len <= k) {
    if (tid == 0) cnt[2] = 0xFFFFFFFFu;
    return;
  }
  constexpr int per = kBins / kThreads;  // 16 consecutive bins per thread
  uint32_t h[per];
  const uint4* src = reinterpret_cast<const uint4*>(ws.hist + (int64_t)r * kBins + tid * per);
#pragma unroll
  for (int c = 0; c < per / 4; ++c) {
    const uint4 v = src[c];
    h[4 * c] = v.x; h[4 * c + 1] = v.y; h[4 * c + 2] = v.z; h[4 * c + 3] = v.w;
  }
  uint32_t sum = 0;
#pragma unroll
  for (int i = 0; i < per; ++i) sum += h[i];
  uint32_t incl = sum;  // inclusive prefix over threads (ascending bins)
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t u = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += u;
  }
  if (lane == 31) wsum[wid] = incl;
  __syncthreads();
  uint32_t before = 0, total = 0;
  for (int w = 0; w < kThreads / 32; ++w) {
    if (w < wid) before += wsum[w];
    total += wsum[w];
  }
  incl += before;
  const uint32_t above_mine = total - incl;  // keys in bins above this thread's range
  if (above_mine < (uint32_t)k && above_mine + sum >= (uint32_t)k) {
    uint32_t run = above_mine;
    for (int i = per - 1; i >= 0; --i) {
      if (run + h[i] >= (uint32_t)k) {
        cnt[2] = (uint32_t)(tid * per + i);
        cnt[3] = run;
        break;
      }
      run += h[i];
    }
  }
}

// Block-wide exclusive scan of one value per thread (kThreads threads).
__device__ __forceinline__ uint32_t cta_excl_scan(uint32_t v, uint32_t* sh, uint32_t& total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t u = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += u;
  }
  if (lane == 31) sh[wid] = incl;
  __syncthreads();
  uint32_t before = 0;
  total = 0;
#pragma unroll
  for (int w = 0; w < kThreads / 32; ++w) {
    const uint32_t x = sh[w];
    before += w < wid ? x : 0u;
    total += x;
  }
  return before + incl - v;
}

// Each thread owns 32 consecutive tokens of the CTA's segment: it loads them
// (8 x 16 B), keys them in registers, and the CTA places its selected and
// candidate tokens with two block scans and one global reservation per list.
__global__ void __launch_bounds__(kThreads) topk_collect_kernel(const float* __restrict__ scores, int64_t ld,
                                                                 const int32_t* row_lens, const int32_t* seq_lens,
                                                                 int nq, int cap, int k, TopkWs ws,
                                                                 int32_t* status) {
  constexpr int kPer = kSeg / kThreads;  // 32 tokens per thread
  __shared__ uint32_t sh_s[kThreads / 32], sh_c[kThreads / 32];
  __shared__ uint32_t s_base[2];
  const int r = blockIdx.y;
  const int len = row_len(row_lens, seq_lens, nq, r, cap, nullptr);
  const int64_t t0 = (int64_t)blockIdx.x * kSeg;
  if (len <= k || t0 >= len) return;
  const int T = (int)ws.counts[4 * (int64_t)r + 2];
  const int n = (int)std::min<int64_t>(kSeg, len - t0);
  const int i0 = threadIdx.x * kPer;  // first token of this thread, relative to t0
  const float* row = scores + (int64_t)r * ld + t0;
  uint32_t key[kPer];
  if (i0 + kPer <= n) {
    const float4* src = reinterpret_cast<const float4*>(row + i0);
#pragma unroll
    for (int c = 0; c < kPer / 4; ++c) {
      const float4 v = src[c];
      key[4 * c] = score_key(v.x);
      key[4 * c + 1] = score_key(v.y);
      key[4 * c + 2] = score_key(v.z);
      key[4 * c + 3] = score_key(v.w);
    }
  } else {
#pragma unroll
    for (int c = 0; c < kPer; ++c) key[c] = (i0 + c < n) ? score_key(row[i0 + c]) : 0u;
  }
  uint32_t ns = 0, nc = 0;
#pragma unroll
  for (int c = 0; c < kPer; ++c) {
    const bool valid = i0 + c < n;
    const int bin = (int)(key[c] >> 20);
    ns += (valid && bin > T);
    nc += (valid && bin == T);
  }
  uint32_t tot_s, tot_c;
  const uint32_t off_s = cta_excl_scan(ns, sh_s, tot_s);
  const uint32_t off_c = cta_excl_scan(nc, sh_c, tot_c);
  uint32_t* cnt = ws.counts + 4 * (int64_t)r;
  if (threadIdx.x == 0) {  // one global reservation per list per CTA
    s_base[0] = tot_s ? atomicAdd(&cnt[0], tot_s) : 0u;
    s_base[1] = tot_c ? atomicAdd(&cnt[1], tot_c) : 0u;
  }
  __syncthreads();
  if (ns | nc) {
    uint32_t ps = s_base[0] + off_s, pc = s_base[1] + off_c;
    int32_t* sel = ws.sel + (int64_t)r * k;
    uint64_t* cand = ws.cand + (int64_t)r * kCandCap;
#pragma unroll
    for (int c = 0; c < kPer; ++c) {
      const bool valid = i0 + c < n;
      const int bin = (int)(key[c] >> 20);
      const uint32_t t = (uint32_t)(t0 + i0 + c);
      if (valid && bin > T) {
        if (ps < (uint32_t)k) sel[ps] = (int32_t)t;
        ++ps;
      } else if (valid && bin == T) {
        if (pc < (uint32_t)kCandCap) cand[pc] = ((uint64_t)key[c] << 32) | (uint64_t)(0xFFFFFFFFu - t);
        ++pc;
      }
    }
  }
}

// Block-wide exclusive scan of one value per thread (kFinalThreads threads).
__device__ __forceinline__ uint32_t block_excl_scan(uint32_t v, uint32_t* sh, uint32_t& total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t incl = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t u = __shfl_up_sync(0xffffffffu, incl, d);
    if (lane >= d) incl += u;
  }
  if (lane == 31) sh[wid] = incl;
  __syncthreads();
  if (wid == 0) {
    uint32_t w = lane < kFinalThreads / 32 ? sh[lane] : 0;
#pragma unroll
    for (int d = 1; d < 32; d <<= 1) {
      const uint32_t u = __shfl_up_sync(0xffffffffu, w, d);
      if (lane >= d) w += u;
    }
    sh[lane] = w;  // inclusive warp totals
  }
  __syncthreads();
  total = sh[kFinalThreads / 32 - 1];
  const uint32_t r = (wid ? sh[wid - 1] : 0) + incl - v;
  __syncthreads();
  return r;
}

// Finds, in the digit histogram `hist` (nbins bins, larger digit = larger
// value), the digit holding the need-th largest value; updates `need` to the
// rank inside that bin and returns the digit and the bin's population.
__device__ void pick_digit(const uint32_t* hist, int nbins, uint32_t* sh, uint32_t& need, int& digit,
                           uint32_t& pop) {
  const int per = (nbins + kFinalThreads - 1) / kFinalThreads;  // bins per thread, descending order
  uint32_t c = 0;
  for (int i = 0; i < per; ++i) {
    const int bin = nbins - 1 - (threadIdx.x * per + i);
    if (bin >= 0) c += hist[bin];
  }
  uint32_t total;
  const uint32_t excl = block_excl_scan(c, sh, total);
  __shared__ int s_digit;
  __shared__ uint32_t s_need, s_pop;
  if (excl < need && excl + c >= need) {
    uint32_t run = excl;
    for (int i = 0; i < per; ++i) {
      const int bin = nbins - 1 - (threadIdx.x * per + i);
      if (bin < 0) break;
      if (run + hist[bin] >= need) {
        s_digit = bin;
        s_need = need - run;
        s_pop = hist[bin];
        break;
      }
      run += hist[bin];
    }
  }
  __syncthreads();
  digit = s_digit;
  need = s_need;
  pop = s_pop;
  __syncthreads();
}

__global__ void __launch_bounds__(kFinalThreads) topk_final_kernel(const float* __restrict__ scores, int64_t ld,
                                                                    const int32_t* row_lens,
                                                                    const int32_t* seq_lens, int nq, int cap, int k,
                                                                    TopkWs ws, int32_t* out, int32_t* status) {
  extern __shared__ uint8_t smem_raw[];
  // bitmap[kWindowBits/32] u32 | cand[kCandCap] u64 | chosen[kMaxTopk] i32 | hist[kBins] u32 | scan[32] u32
  uint32_t* bitmap = reinterpret_cast<uint32_t*>(smem_raw);
  uint64_t* cand = reinterpret_cast<uint64_t*>(smem_raw + kWindowBits / 8);
  int32_t* chosen = reinterpret_cast<int32_t*>(smem_raw + kWindowBits / 8 + 8 * kCandCap);
  uint32_t* hist = reinterpret_cast<uint32_t*>(smem_raw + kWindowBits / 8 + 8 * kCandCap + 4 * kMaxTopk);
  uint32_t* scan = hist + kBins;
  __shared__ uint32_t s_count;

  const int r = blockIdx.x, tid = threadIdx.x;
  const int len = row_len(row_lens, seq_lens, nq, r, cap, nullptr);
  int32_t* o = out + (int64_t)r * k;
  if (len <= k) {
    for (int i = tid; i < k; i += kFinalThreads) o[i] = i < len ? i : -1;
    return;
  }
  const uint32_t* cnt = ws.counts + 4 * (int64_t)r;
  const uint32_t n_sel = cnt[0], n_cand = cnt[1];
  const int T = (int)cnt[2];
  if (n_sel >= (uint32_t)k || n_cand == 0) {  // impossible with a consistent histogram
    report(status, DSA_ERR_BOUNDS);
    for (int i = tid; i < k; i += kFinalThreads) o[i] = -1;
    return;
  }
  // rows up to one bitmap window set their bits directly; longer rows collect a list first
  const bool direct = len <= kWindowBits;
  const int words0 = direct ? (len + 31) >> 5 : 0;
  for (int i = tid; i < words0; i += kFinalThreads) bitmap[i] = 0;
  const bool overflow = n_cand > (uint32_t)kCandCap;
  const uint64_t* gcand = ws.cand + (int64_t)r * kCandCap;
  if (!overflow) {
    for (uint32_t i0 = 0; i0 < n_cand; i0 += 4 * kFinalThreads) {  // four loads in flight per thread
      uint64_t v[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t i = i0 + c * kFinalThreads + tid;
        v[c] = i < n_cand ? gcand[i] : 0;
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const uint32_t i = i0 + c * kFinalThreads + tid;
        if (i < n_cand) cand[i] = v[c];
      }
    }
  }
  __syncthreads();
  {
    const int32_t* gs = ws.sel + (int64_t)r * k;
    for (int i0 = 0; i0 < (int)n_sel; i0 += 4 * kFinalThreads) {
      int32_t v[4];
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int i = i0 + c * kFinalThreads + tid;
        v[c] = i < (int)n_sel ? gs[i] : 0;
      }
#pragma unroll
      for (int c = 0; c < 4; ++c) {
        const int i = i0 + c * kFinalThreads + tid;
        if (i < (int)n_sel) {
          if (direct) atomicOr(&bitmap[v[c] >> 5], 1u << (v[c] & 31));
          else chosen[i] = v[c];
        }
      }
    }
  }
  uint32_t need = (uint32_t)k - n_sel;
  const float* row = scores + (int64_t)r * ld;

  // ---- the `need` largest packed values v = (key << 32) | ~index among the
  //      candidates: 12-bit digits of bits 51..0 (bits 63..52 equal T), stopping
  //      as soon as the digit's bin is taken whole.
  auto packed = [&](int t) -> uint64_t {
    return ((uint64_t)score_key(row[t]) << 32) | (uint64_t)(0xFFFFFFFFu - (uint32_t)t);
  };
  uint64_t prefix = 0;
  int shift = 52;
  while (shift > 0) {
    const int bits = shift >= 12 ? 12 : shift;
    const int nshift = shift - bits;
    for (int i = tid; i < (1 << bits); i += kFinalThreads) hist[i] = 0;
    __syncthreads();
    const uint32_t dmask = (1u << bits) - 1;
    if (!overflow) {
      for (uint32_t i = tid; i < n_cand; i += kFinalThreads) {
        const uint64_t v = cand[i] & ((1ull << 52) - 1);
        if ((v >> shift) == prefix) atomicAdd(&hist[(uint32_t)(v >> nshift) & dmask], 1u);
      }
    } else {
      for (int t = tid; t < len; t += kFinalThreads) {
        const uint64_t full = packed(t);
        if ((int)(full >> 52) != T) continue;
        const uint64_t v = full & ((1ull << 52) - 1);
        if ((v >> shift) == prefix) atomicAdd(&hist[(uint32_t)(v >> nshift) & dmask], 1u);
      }
    }
    __syncthreads();
    int digit;
    uint32_t pop;
    pick_digit(hist, 1 << bits, scan, need, digit, pop);
    prefix = (prefix << bits) | (uint64_t)digit;
    shift = nshift;
    if (need == pop) break;  // the whole bin is taken: select by prefix
  }
  // candidates whose bits 51..shift are >= prefix complete the selection
  if (tid == 0) s_count = n_sel;
  __syncthreads();
  auto take = [&](int32_t t) {
    if (direct) {
      atomicOr(&bitmap[t >> 5], 1u << (t & 31));
    } else {
      const uint32_t pos = atomicAdd(&s_count, 1u);
      if (pos < (uint32_t)k) chosen[pos] = t;
    }
  };
  if (!overflow) {
    for (uint32_t i = tid; i < n_cand; i += kFinalThreads) {
      const uint64_t v = cand[i] & ((1ull << 52) - 1);
      if ((v >> shift) >= prefix) take((int32_t)(0xFFFFFFFFu - (uint32_t)cand[i]));
    }
  } else {
    for (int t = tid; t < len; t += kFinalThreads) {
      const uint64_t full = packed(t);
      if ((int)(full >> 52) != T) continue;
      if (((full & ((1ull << 52) - 1)) >> shift) >= prefix) take(t);
    }
  }
  __syncthreads();
  const int nchosen = direct ? k : (int)std::min<uint32_t>(s_count, (uint32_t)k);
  if (!direct && s_count != (uint32_t)k) report(status, DSA_ERR_BOUNDS);  // internal consistency check

  // ---- ascending order through the bitmap of the index range, one window at a time
  uint32_t written = 0;
  for (int64_t w0 = 0; w0 < len; w0 += kWindowBits) {
    const int span = (int)std::min<int64_t>(kWindowBits, len - w0);
    const int words = (span + 31) >> 5;
    const int per = (words + kFinalThreads - 1) / kFinalThreads;
    if (!direct) {
      for (int i = tid; i < words; i += kFinalThreads) bitmap[i] = 0;
      __syncthreads();
      for (int i = tid; i < nchosen; i += kFinalThreads) {
        const int64_t t = chosen[i];
        if (t >= w0 && t < w0 + span) atomicOr(&bitmap[(t - w0) >> 5], 1u << ((t - w0) & 31));
      }
      __syncthreads();
    }
    uint32_t c = 0;
    for (int i = 0; i < per; ++i) {
      const int wi = tid * per + i;
      if (wi < words) c += __popc(bitmap[wi]);
    }
    uint32_t total;
    uint32_t pos = written + block_excl_scan(c, scan, total);
    for (int i = 0; i < per; ++i) {
      const int wi = tid * per + i;
      if (wi >= words) break;
      uint32_t bits = bitmap[wi];
      while (bits) {
        const int b = __ffs(bits) - 1;
        bits &= bits - 1;
        if (pos < (uint32_t)k) o[pos] = (int32_t)(w0 + (int64_t)wi * 32 + b);
        ++pos;
      }
    }
    written += total;
    __syncthreads();
  }
  if (direct && written != (uint32_t)k) report(status, DSA_ERR_BOUNDS);  // internal consistency check
  for (int i = (int)written + tid; i < k; i += kFinalThreads) o[i] = -1;
}

size_t ws_bytes(int rows, int k) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  return al((size_t)rows * kBins * 4) + al((size_t)rows * 16) + al((size_t)rows * k * 4) +
         al((size_t)rows * kCandCap * 8);
}

}  // namespace

size_t topk_workspace_bytes(int rows, int max_row_len, int k) {
  (void)max_row_len;
  return ws_bytes(rows, k);
}

size_t topk_final_smem_bytes() { return (size_t)kWindowBits / 8 + 8 * kCandCap + 4 * kMaxTopk + 4 * kBins + 128; }

dsa_status_t launch_topk(const float* scores, int64_t ld, const int32_t* row_lens, const int32_t* seq_lens, int nq,
                         int rows, int max_row_len, int k, int32_t* out, void* workspace, int32_t* status,
                         cudaStream_t st) {
  if (rows == 0) return DSA_OK;
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  uint8_t* w = static_cast<uint8_t*>(workspace);
  TopkWs ws;
  ws.hist = reinterpret_cast<uint32_t*>(w);
  w += al((size_t)rows * kBins * 4);
  ws.counts = reinterpret_cast<uint32_t*>(w);
  w += al((size_t)rows * 16);
  ws.sel = reinterpret_cast<int32_t*>(w);
  w += al((size_t)rows * k * 4);
  ws.cand = reinterpret_cast<uint64_t*>(w);
  const int cap = max_row_len;
  const int nseg = std::max(1, (max_row_len + kSeg - 1) / kSeg);
  if (max_row_len > k) {
    dim3 grid(nseg, rows);
    // histograms and counters start at zero
    const size_t zero_bytes = al((size_t)rows * kBins * 4) + al((size_t)rows * 16);
    if (cuda_status(cudaMemsetAsync(workspace, 0, zero_bytes, st)) != DSA_OK) return DSA_ERR_CUDA;
    topk_hist_kernel<<<grid, kThreads, 0, st>>>(scores, ld, row_lens, seq_lens, nq, cap, k, ws, status);
    topk_threshold_kernel<<<rows, kThreads, 0, st>>>(row_lens, seq_lens, nq, cap, k, ws);
    topk_collect_kernel<<<grid, kThreads, 0, st>>>(scores, ld, row_lens, seq_lens, nq, cap, k, ws, status);
  }
  static bool attr_set[64] = {};
  int dev = 0;
  cudaGetDevice(&dev);
  const size_t smem = topk_final_smem_bytes();
  if (dev < 64 && !attr_set[dev]) {
    if (cuda_status(cudaFuncSetAttribute(topk_final_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem)) != DSA_OK)
      return DSA_ERR_CUDA;
    attr_set[dev] = true;
  }
  topk_final_kernel<<<rows, kFinalThreads, smem, st>>>(scores, ld, row_lens, seq_lens, nq, cap, k, ws, out, status);
  return launch_status();
}

// ---------------------------------------------------------------- top-k with built-in scratch
// The scratch the top-k needs (histograms, counters, selected and candidate
// lists) for up to kNoAllocMaxRows rows of any length with k <= 2048, kept in
// a device array that exists for as long as the library is loaded, so the
// entry point below never allocates.  Every call reuses it: launch_topk zeroes
// the histograms and counters at the start of each call, the lists are written
// before they are read, and calls whose work overlaps on the GPU would race.
namespace {
constexpr int kNoAllocMaxRows = DSA_TOPK_NOALLOC_MAX_ROWS;
constexpr size_t al256c(size_t x) { return (x + 255) & ~size_t(255); }
constexpr size_t kNoAllocBytes = al256c((size_t)kNoAllocMaxRows * kBins * 4) + al256c((size_t)kNoAllocMaxRows * 16) +
                                 al256c((size_t)kNoAllocMaxRows * kMaxTopk * 4) +
                                 al256c((size_t)kNoAllocMaxRows * kCandCap * 8);  // 5.5 MiB
static __device__ __align__(256) uint8_t g_topk_scratch[kNoAllocBytes];
std::mutex g_scratch_mu;
void* g_scratch_addr[64] = {};  // the array's device address, per device, resolved on first use
}  // namespace

dsa_status_t launch_topk_noalloc(const float* scores, int64_t ld, const int32_t* row_lens, int rows, int max_row_len,
                                 int k, int32_t* out, int32_t* status, cudaStream_t st) {
  if (rows > kNoAllocMaxRows || ws_bytes(rows, k) > kNoAllocBytes) return DSA_ERR_UNSUPPORTED;
  int dev = 0;
  if (cuda_status(cudaGetDevice(&dev)) != DSA_OK) return DSA_ERR_CUDA;
  if (dev < 0 || dev >= 64) return DSA_ERR_UNSUPPORTED;
  void* scratch = nullptr;
  {
    std::lock_guard<std::mutex> lock(g_scratch_mu);
    if (g_scratch_addr[dev] == nullptr) {
      // the host-side name of the array is not a device address: ask the runtime, with this device current
      void* addr = nullptr;
      if (cuda_status(cudaGetSymbolAddress(&addr, g_topk_scratch)) != DSA_OK) return DSA_ERR_CUDA;
      g_scratch_addr[dev] = addr;
    }
    scratch = g_scratch_addr[dev];
  }
  return launch_topk(scores, ld, row_lens, nullptr, 1, rows, max_row_len, k, out, scratch, status, st);
}

}  // namespace dsa
