// topk.cu — exact per-row top-k selection (stage 2 of DSA).
//
// Keeps the k (= 2,048 in the model) highest-scoring visible tokens of each
// query row (vLLM Day-0 post for Kimi K3.1 Pro, sparse-attention section:
// the indexer's scores choose 2,048 tokens per query; fused-decode section:
// the selection is exact).  Equal scores go to the lower token index, so the
// selected set is unique; it is written in ascending token order with -1
// padding when a row has fewer than k tokens.  Scores are compared as
// order-preserving 32-bit keys (integer radix).
//
// Rows up to 8 x 30,720 tokens: one kernel, a thread-block cluster per row
// (topk_cluster_kernel).  Each CTA of the cluster keeps its slice of the row
// as keys in shared memory (bulk copies from L2).  The first digit (11 bits)
// is picked from the CTAs' histograms, merged through distributed shared
// memory.  One more pass over the keys then marks, per lane run, the keys
// above that digit's bin (taken whatever follows) and moves the keys in the
// bin to the front of the run; the second and third digits (11 and 10 bits)
// and the output use only those candidates.  Ties on the k-th key go to the
// lowest indices in CTA-rank and token order; each lane writes its run's
// chosen indices in ascending order at a place from warp and cluster scans.
// No workspace is used.
//
// Many rows of at most 163,840 tokens (more than one wave of clusters, such
// as a prefill chunk's rows) take topk_row_kernel instead: one CTA per row at
// a time, two per SM, persistent over the rows.  A sample of the row sets a
// bar with about 1.3 k keys above it; one pass streams the row, comparing
// scores against the bar as floats, and keeps every key above it as a
// candidate in shared memory; the selection then runs over the candidates
// and the output goes through bitmaps of the row.  If the sample misleads
// (fewer than k keys pass, or more than fit), exact digit passes over the
// row take over.
//
// Longer rows (the 1M-token rows) with fp32 scores and a workspace take two
// levels of the same kernel: pass 1 selects the top-k of every segment of at
// most 163,840 tokens (one cluster per segment, as many segments as fill the
// SMs, so few long rows still use them all) and writes it, with the scores,
// into the row's compact candidate list in token order; pass 2 selects the
// row's top-k among those candidates.  The result is exact: a token of the
// row's top-k is also in its own segment's top-k, and the compact rows keep
// token order, so ties still go to the lower index.
// Without a workspace (bf16 scores, the no-allocation entry point) they take
// the kernel's streaming form: a cluster of 16 CTAs per row (8 where the
// device cannot schedule 16) that reads its slice again from L2 in every pass
// and keeps only the histograms in shared memory.  Where the four-kernel form
// is forced, or no cluster can be scheduled, four kernels over a workspace do
// the selection:
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
#include <algorithm>
#include <atomic>
#include <type_traits>
#include <mutex>

#include <cooperative_groups.h>

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

// The physical KV row of token t of row r's sequence (block row * 64 + slot),
// -1 for padding; an entry outside the pool is reported and gives -1.
__device__ __forceinline__ int32_t phys_row(const TopkPhys& po, int nq, int r, int t, int32_t* status) {
  if (t < 0) return -1;
  const int32_t b = po.block_table[(int64_t)(r / nq) * po.max_blocks + t / kBlock];
  if (b < 0 || b >= po.num_blocks) {
    report(status, DSA_ERR_BOUNDS);
    return -1;
  }
  return b * kBlock + t % kBlock;
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
                                                                    TopkWs ws, int32_t* out, int32_t* status,
                                                                    const TopkPhys po) {
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
  auto emit = [&](int64_t pos_, int t_) {  // index t_ at output position pos_, and its physical row
    o[pos_] = t_;
    if (po.phys) po.phys[(int64_t)r * k + pos_] = phys_row(po, nq, r, t_, status);
  };
  if (len <= k) {
    for (int i = tid; i < k; i += kFinalThreads) emit(i, i < len ? i : -1);
    return;
  }
  const uint32_t* cnt = ws.counts + 4 * (int64_t)r;
  const uint32_t n_sel = cnt[0], n_cand = cnt[1];
  const int T = (int)cnt[2];
  if (n_sel >= (uint32_t)k || n_cand == 0) {  // impossible with a consistent histogram
    report(status, DSA_ERR_BOUNDS);
    for (int i = tid; i < k; i += kFinalThreads) emit(i, -1);
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
        if (pos < (uint32_t)k) emit(pos, (int32_t)(w0 + (int64_t)wi * 32 + b));
        ++pos;
      }
    }
    written += total;
    __syncthreads();
  }
  if (direct && written != (uint32_t)k) report(status, DSA_ERR_BOUNDS);  // internal consistency check
  for (int i = (int)written + tid; i < k; i += kFinalThreads) emit(i, -1);
}

// ---------------------------------------------------------------- row-resident path
namespace cg = cooperative_groups;

constexpr int kResKeys = 30720;     // most keys a CTA holds in shared memory (120 KB): a lane's
                                    // run of a 16-warp CTA is then at most 15 groups of 4 (60 bits)
static_assert((kResKeys / 4 + 15) / 16 <= 15 * 32, "lane runs must fit a 64-bit mask");
constexpr int kResPairKeys = 20480; // keys per CTA that still let two CTAs share an SM
constexpr int kResThreads = kFinalThreads;
constexpr int kResWarps = kResThreads / 32;
constexpr int kResMaxCluster = 8;   // portable cluster size: rows up to 245,760 tokens
// digits of the 32-bit key: bits 31..21, 20..10, 9..0
constexpr int kD1 = 11, kD2 = 11, kD3 = 10;
constexpr int kB1 = 1 << kD1, kB2 = 1 << kD2, kB3 = 1 << kD3;
// shared memory (32-bit words): keys[slice] | h1[kB1] | h2[kB2] | h3[kB3] |
// stage[kB1] | coarse[3][64] | scan[32] | misc[32] | 4 mbarriers
constexpr int kCoarse = 64;      // super-bins of 32 bins per digit level
constexpr int kLoadChunks = 4;   // bulk copies of a resident slice, each with its own mbarrier
constexpr size_t kResFixed = 4 * ((size_t)kB1 + kB2 + kB3 + kB1 + 3 * kCoarse + 32 + 32 + 2 * kLoadChunks);
constexpr int kOverflow = 25;    // misc slot: a warp took more indices than it can stage
constexpr int kPick = 26;        // misc slots 26..28: the merge's digit, need and pop
constexpr int kStageCap = kB1 / kResWarps;  // indices a warp stages (128)
size_t res_smem(int slice) { return 4 * (size_t)slice + kResFixed; }

// Warp-wide exclusive prefix sum of one value 0..7 per lane, from three
// ballots of its bits; `total` gets the sum.
__device__ __forceinline__ uint32_t warp_excl_scan_small(uint32_t v, uint32_t lanes_below, uint32_t& total) {
  const uint32_t b0 = __ballot_sync(0xffffffffu, v & 1u), b1 = __ballot_sync(0xffffffffu, v & 2u),
                 b2 = __ballot_sync(0xffffffffu, v & 4u);
  total = __popc(b0) + 2u * __popc(b1) + 4u * __popc(b2);
  return __popc(b0 & lanes_below) + 2u * __popc(b1 & lanes_below) + 4u * __popc(b2 & lanes_below);
}

// A key range [klo, khi] of score_key order as scores, so that the streaming
// passes compare scores without converting them: a score's key lies in the
// range iff lo <= s <= hi, and above it iff s > hi.  The compares are IEEE (the
// library is built without flush-to-zero), so -0 == +0 as in score_key.  NaN
// scores (key 0) fail every compare; a range that starts at key 0 holds
// exactly the NaN scores (no score has a key in 1..0x7FFFFE), flagged by
// `nan`, and then every other score is above it.  Ranges chosen by a digit
// pass always hold a key that occurs, so khi never falls in 1..0x7FFFFE.
struct ScoreRange {
  float lo, hi;
  bool nan;
};

__device__ __forceinline__ float key_score(uint32_t key) {  // the score of a key that occurs
  return __uint_as_float((key & 0x80000000u) ? (key & 0x7FFFFFFFu) : ~key);
}

__device__ __forceinline__ ScoreRange score_range(uint32_t klo, uint32_t khi) {
  ScoreRange r;
  r.nan = klo == 0u;
  r.lo = klo <= 0x007FFFFFu ? __uint_as_float(0xFF800000u) : key_score(klo);  // key of -inf: 0x007FFFFF
  r.hi = khi >= 0xFF800000u   ? __uint_as_float(0x7F800000u)                  // key of +inf: 0xFF800000
         : khi == 0x7FFFFFFFu ? __uint_as_float(0x80000001u)  // just below the zeros' key: -denorm_min
                              : key_score(khi);
  return r;
}

// A threshold range in both forms: keys [klo, klo + span] and their scores.
struct KeyRange {
  uint32_t klo, span;
  ScoreRange s;
};

__device__ __forceinline__ KeyRange key_range(uint32_t prefix, int shift) {
  KeyRange r;
  r.klo = prefix << shift;
  r.span = (1u << shift) - 1u;
  r.s = score_range(r.klo, r.klo + r.span);
  return r;
}

// Bit j: element j of a group (keys, or scores when streaming) lies in the
// range / above it.
__device__ __forceinline__ uint32_t bits_in(const uint4& v, const KeyRange& r) {
  return (uint32_t)(v.x - r.klo <= r.span) | ((uint32_t)(v.y - r.klo <= r.span) << 1) |
         ((uint32_t)(v.z - r.klo <= r.span) << 2) | ((uint32_t)(v.w - r.klo <= r.span) << 3);
}
__device__ __forceinline__ uint32_t bits_above(const uint4& v, const KeyRange& r) {
  const uint32_t hi = r.klo + r.span;
  return (uint32_t)(v.x > hi) | ((uint32_t)(v.y > hi) << 1) | ((uint32_t)(v.z > hi) << 2) | ((uint32_t)(v.w > hi) << 3);
}
__device__ __forceinline__ uint32_t bits_in(const float4& v, const KeyRange& r) {
  const ScoreRange& s = r.s;
  if (s.nan)
    return (uint32_t)(v.x != v.x) | ((uint32_t)(v.y != v.y) << 1) | ((uint32_t)(v.z != v.z) << 2) |
           ((uint32_t)(v.w != v.w) << 3);
  return (uint32_t)(v.x >= s.lo && v.x <= s.hi) | ((uint32_t)(v.y >= s.lo && v.y <= s.hi) << 1) |
         ((uint32_t)(v.z >= s.lo && v.z <= s.hi) << 2) | ((uint32_t)(v.w >= s.lo && v.w <= s.hi) << 3);
}
__device__ __forceinline__ uint32_t bits_above(const float4& v, const KeyRange& r) {
  const ScoreRange& s = r.s;
  if (s.nan)
    return (uint32_t)(v.x == v.x) | ((uint32_t)(v.y == v.y) << 1) | ((uint32_t)(v.z == v.z) << 2) |
           ((uint32_t)(v.w == v.w) << 3);
  return (uint32_t)(v.x > s.hi) | ((uint32_t)(v.y > s.hi) << 1) | ((uint32_t)(v.z > s.hi) << 2) |
         ((uint32_t)(v.w > s.hi) << 3);
}
__device__ __forceinline__ uint32_t elem_key(const uint4& v, int j) {
  return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w;
}
__device__ __forceinline__ uint32_t elem_key(const float4& v, int j) {
  return score_key(j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w);
}


// Warp-wide exclusive prefix sum of one value per lane; `total` gets the sum.
__device__ __forceinline__ uint32_t warp_excl_scan(uint32_t v, uint32_t& total) {
  const int lane = threadIdx.x & 31;
  uint32_t x = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t u = __shfl_up_sync(0xffffffffu, x, d);
    if (lane >= d) x += u;
  }
  total = __shfl_sync(0xffffffffu, x, 31);
  return x - v;
}

// kStream = false: each CTA keeps its slice of the row as keys in shared
// memory.  kStream = true (rows too long for that): every pass reads the
// slice's scores again from global memory (L2), and shared memory holds only
// the histograms.  Resident: two CTAs of 512 threads per SM (at most 64
// registers); streaming: one.
// In: the score element, float or uint16_t (bf16 bits, widened exactly to
// fp32 as they are read; the selection is then the fp32 one).
// The two-level form for long rows.  Pass 1 (nseg > 0): launch row v is
// segment p = v % nseg of score row r = v / nseg, tokens [p seg, (p+1) seg),
// and its top-k goes straight into row r's compact candidate list at
// positions p k + i (every segment before p is full, so holds k of them):
// the token index to cand_idx, its score to cand_score.  Pass 2 (pass2 set):
// launch row r is that compact row, floor(len / seg) k + min(k, len % seg)
// candidates for a score row of len tokens, and an output position i is
// written as cand_idx[r][i], the candidate's token index.  The compact rows
// are in token order.  All zero: the plain top-k of each score row.
struct TopkSeg {
  int32_t seg_tokens = 0;
  int32_t nseg = 0;
  bool pass2 = false;
  float* cand_score = nullptr;
  int32_t* cand_idx = nullptr;
  int64_t ldc = 0;
  int32_t longest = 0;  // the longest launch row (0: cap)
};

template <int C, bool kStream, typename In>
__global__ void __launch_bounds__(kResThreads, kStream ? 1 : 2)
    topk_cluster_kernel(const In* __restrict__ scores, int64_t ld, const int32_t* row_lens,
                        const int32_t* seq_lens, int nq, int cap, int k, int32_t* out, int32_t* status,
                        int slice_cap, const TopkPhys po, const TopkSeg sg) {
  constexpr bool kF32 = std::is_same<In, float>::value;
  using G = typename std::conditional<kStream, float4, uint4>::type;  // a group of 4 elements
  cg::cluster_group cluster = cg::this_cluster();
  const int c = (int)cluster.block_rank();
  const int rv = blockIdx.x / C, tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;  // the launch's row
  const int r = sg.nseg ? rv / sg.nseg : rv;       // the score row
  const int seg_p = sg.nseg ? rv % sg.nseg : 0;    // the segment of it (pass 1)
  auto csync = [&]() {  // a one-CTA cluster needs only the block barrier
    if (C == 1) __syncthreads();
    else cluster.sync();
  };
  extern __shared__ __align__(16) uint8_t smem_raw[];
  uint4* keys4 = reinterpret_cast<uint4*>(smem_raw);  // the slice's keys (resident form)
  uint32_t* h1 = reinterpret_cast<uint32_t*>(smem_raw) + (kStream ? 0 : slice_cap);  // slice_cap: a multiple of 4
  uint32_t* h2 = h1 + kB1;
  uint32_t* h3 = h2 + kB2;
  uint32_t* stage = h3 + kB3;  // the warps' taken indices, kStageCap each
  uint32_t* coarse = stage + kB1;  // per digit level: sums of 32 consecutive bins
  uint32_t* scan = coarse + 3 * kCoarse;
  uint32_t* misc = scan + 32;
  const uint32_t load_bars = smem_u32(misc + 32);  // kLoadChunks mbarriers, 8 bytes each

  // the scores (and in the two-level form's second pass the row lengths and
  // index map) come from the previous kernel, which may also still read `out`
  grid_dep_wait();
  grid_dep_launch();
  int len = row_len(row_lens, seq_lens, nq, r, cap, (c == 0 && seg_p == 0 && !sg.pass2) ? status : nullptr);
  if (sg.nseg) len = max(0, min(sg.seg_tokens, len - seg_p * sg.seg_tokens));
  if (sg.pass2) len = (len / sg.seg_tokens) * k + min(k, len % sg.seg_tokens);
  int32_t* o = sg.nseg ? nullptr : out + (int64_t)rv * k;  // pass 1 writes the candidate rows instead
  auto emit = [&](int64_t pos_, int t_) {  // index t_ at output position pos_, and its physical row
    if (sg.nseg) {  // pass 1: into the compact candidate row
      if (t_ >= 0) {
        const int64_t tok = (int64_t)seg_p * sg.seg_tokens + t_;
        const int64_t at = (int64_t)r * sg.ldc + (int64_t)seg_p * k + pos_;
        sg.cand_idx[at] = (int32_t)tok;
        const In x = scores[(int64_t)r * ld + tok];
        if constexpr (kF32) sg.cand_score[at] = x;
        else sg.cand_score[at] = __uint_as_float((uint32_t)x << 16);
      }
      return;
    }
    if (sg.pass2 && t_ >= 0) t_ = sg.cand_idx[(int64_t)r * sg.ldc + t_];
    o[pos_] = t_;
    if (po.phys) po.phys[(int64_t)rv * k + pos_] = phys_row(po, nq, r, t_, status);
  };
  if (len <= k) {  // the same branch for every CTA of the cluster
    if (c == 0)
      for (int i = tid; i < k; i += kResThreads) emit(i, i < len ? i : -1);
    return;
  }
  // this CTA's slice of the row: S tokens from `start` (S a multiple of 4)
  const int S = (((len + C - 1) / C) + 3) & ~3;
  const int start = c * S;
  const int n = max(0, min(S, len - start));
  const int n4 = (n + 3) >> 2;  // groups of 4; the last one is padded with NaN / key 0 (never counted)
  const In* row = scores + (int64_t)r * ld + (int64_t)seg_p * sg.seg_tokens + start;
  const int full4 = n >> 2;
  auto widen = [](In x) -> float {
    if constexpr (kF32) return x;
    else return __uint_as_float((uint32_t)x << 16);
  };
  auto score_group = [&](int i) -> float4 {  // scores 4i..4i+3 from global memory
    if (i < full4) {
      if constexpr (kF32) {
        return reinterpret_cast<const float4*>(row)[i];
      } else {
        const uint2 w = reinterpret_cast<const uint2*>(row)[i];
        return make_float4(__uint_as_float(w.x << 16), __uint_as_float(w.x & 0xFFFF0000u),
                           __uint_as_float(w.y << 16), __uint_as_float(w.y & 0xFFFF0000u));
      }
    }
    const int b = 4 * i;  // the slice's ragged last group
    const float nan = __uint_as_float(0x7FC00000u);
    return make_float4(widen(row[b]), b + 1 < n ? widen(row[b + 1]) : nan, b + 2 < n ? widen(row[b + 2]) : nan,
                       b + 3 < n ? widen(row[b + 3]) : nan);
  };
  auto load_group = [&](int i) -> G {
    if constexpr (kStream) return score_group(i);
    else return keys4[i];
  };
  // the valid elements of group i (padding past the slice's end excluded)
  auto valid_bits = [&](int i) -> uint32_t { return 4 * i + 4 > n ? (1u << (n - 4 * i)) - 1u : 0xFu; };
  // the first digit's histogram entries of group i's keys
  auto count_first = [&](int i, const uint4& kk) {
    const bool pad = 4 * i + 3 >= n;  // padding keys are not counted
    atomicAdd(&h1[kk.x >> (32 - kD1)], 1u);
    if (!pad || 4 * i + 1 < n) atomicAdd(&h1[kk.y >> (32 - kD1)], 1u);
    if (!pad || 4 * i + 2 < n) atomicAdd(&h1[kk.z >> (32 - kD1)], 1u);
    if (!pad) atomicAdd(&h1[kk.w >> (32 - kD1)], 1u);
  };
  auto to_keys = [](const float4& v) {
    return make_uint4(score_key(v.x), score_key(v.y), score_key(v.z), score_key(v.w));
  };

  // ---- 1. histogram of the first digit (bits 31..21); resident: the slice
  //         into shared memory as keys
  for (int i = tid; i < (kB1 + kB2 + kB3) / 4; i += kResThreads) reinterpret_cast<uint4*>(h1)[i] = make_uint4(0, 0, 0, 0);
  if (tid == 0) {
    misc[kOverflow] = 0u;
    if (!kStream) {
      for (int q = 0; q < kLoadChunks; ++q) mbar_init(load_bars + 8 * q, 1);
      fence_mbar_init();
    }
  }
  __syncthreads();
  if constexpr (!kStream && !kF32) {
    // bf16 scores: 8-byte loads widened to keys (half the bytes of fp32)
    for (int i = tid; i < n4; i += kResThreads) {
      const uint4 kk = to_keys(score_group(i));
      keys4[i] = kk;
      count_first(i, kk);
    }
  } else if constexpr (!kStream) {
    // the slice's whole groups by bulk copies in kLoadChunks pieces, converted to
    // keys in place as each lands; the ragged last group by plain loads
    const float4* row4 = reinterpret_cast<const float4*>(row);
    const int per = (full4 + kLoadChunks - 1) / kLoadChunks;
    if (tid == 0) {
#pragma unroll
      for (int q = 0; q < kLoadChunks; ++q) {
        const int a = min(full4, q * per), b = min(full4, a + per);
        mbar_arrive_expect_tx(load_bars + 8 * q, (uint32_t)(b - a) * 16u);
        if (b > a) bulk_load(smem_u32(keys4 + a), row4 + a, (uint32_t)(b - a) * 16u, load_bars + 8 * q);
      }
    }
    if (full4 < n4 && tid == kResThreads - 1) {
      const uint4 kk = to_keys(score_group(full4));
      keys4[full4] = kk;
      count_first(full4, kk);
    }
#pragma unroll 1
    for (int q = 0; q < kLoadChunks; ++q) {
      const int a = min(full4, q * per), b = min(full4, a + per);
      if (!mbar_wait_drain(load_bars + 8 * q, 0, 1000000000ull)) report(status, DSA_ERR_TIMEOUT);
      for (int i = a + tid; i < b; i += kResThreads) {
        const uint4 raw = keys4[i];
        const uint4 kk = to_keys(make_float4(__uint_as_float(raw.x), __uint_as_float(raw.y),
                                             __uint_as_float(raw.z), __uint_as_float(raw.w)));
        keys4[i] = kk;
        count_first(i, kk);
      }
    }
  } else {
    for (int i0 = 0; i0 < n4; i0 += 8 * kResThreads) {
      float4 v[8];  // eight 16-byte loads in flight per thread
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * kResThreads + tid;
        if (i < n4) v[u] = score_group(i);
      }
#pragma unroll
      for (int u = 0; u < 8; ++u) {
        const int i = i0 + u * kResThreads + tid;
        if (i < n4) count_first(i, to_keys(v[u]));
      }
    }
  }
  // The cluster-wide choice of a digit from the CTAs' histograms `local`
  // (nbins = 32 * nc bins each, nc <= 64) with one cluster barrier: each CTA
  // sums its histogram in nc super-bins of 32 bins (`cs`), then warp 0 adds up
  // every CTA's super-bins (distributed shared memory), finds the one holding
  // the need-th largest key counting from the top, adds up the 32 bins of that
  // super-bin over the CTAs and picks the bin.  The peers' arrays are only read
  // after the barrier and never written again in this launch.
  auto merge_pick = [&](const uint32_t* local, int nc, uint32_t* cs, uint32_t& need, int& digit, uint32_t& pop) {
    __syncthreads();  // this CTA's histogram is complete
    for (int sb = wid; sb < nc; sb += kResWarps) {
      const uint32_t v = __reduce_add_sync(0xffffffffu, local[sb * 32 + lane]);
      if (lane == 0) cs[sb] = v;
    }
    csync();  // every CTA's histogram and super-bins are complete
    if (wid == 0) {
      // lane l: super-bins l (lo) and 32 + l (hi)
      uint32_t lo = 0, hi = 0;
#pragma unroll
      for (int q = 0; q < C; ++q) {
        const uint32_t* pc = C == 1 ? cs : cluster.map_shared_rank(cs, q);
        lo += pc[lane];
        if (nc > 32) hi += pc[32 + lane];
      }
      // inclusive sums from the top: super-bins above and including each
      uint32_t shi = hi, slo = lo;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const uint32_t a = __shfl_down_sync(0xffffffffu, shi, d), b = __shfl_down_sync(0xffffffffu, slo, d);
        if (lane + d < 32) {
          shi += a;
          slo += b;
        }
      }
      const uint32_t tot_hi = __shfl_sync(0xffffffffu, shi, 0);
      slo += tot_hi;
      // the super-bin where the running count from the top first reaches need
      const bool in_hi = shi - hi < need && need <= shi;
      const bool in_lo = slo - lo < need && need <= slo;
      const uint32_t m_hi = __ballot_sync(0xffffffffu, in_hi), m_lo = __ballot_sync(0xffffffffu, in_lo);
      // exactly one lane qualifies (the clamp only keeps indices in range if the
      // counts were inconsistent)
      const int sb = max(0, m_hi ? 32 + __ffs(m_hi) - 1 : __ffs(m_lo) - 1);
      const uint32_t above = __shfl_sync(0xffffffffu, m_hi ? shi - hi : slo - lo, (sb & 31));
      // the 32 bins of super-bin sb over the cluster
      uint32_t f = 0;
#pragma unroll
      for (int q = 0; q < C; ++q) f += (C == 1 ? local : cluster.map_shared_rank(local, q))[sb * 32 + lane];
      uint32_t sf = f;
#pragma unroll
      for (int d = 1; d < 32; d <<= 1) {
        const uint32_t a = __shfl_down_sync(0xffffffffu, sf, d);
        if (lane + d < 32) sf += a;
      }
      const uint32_t want = need - above;
      const uint32_t mb = __ballot_sync(0xffffffffu, sf - f < want && want <= sf);
      const int l = max(0, __ffs(mb) - 1);
      if (lane == l) {
        misc[kPick] = (uint32_t)(sb * 32 + l);
        misc[kPick + 1] = want - (sf - f);
        misc[kPick + 2] = f;
      }
    }
    __syncthreads();
    digit = (int)misc[kPick];
    need = misc[kPick + 1];
    pop = misc[kPick + 2];
  };
  uint32_t need = (uint32_t)k, pop;
  int digit;
  merge_pick(h1, kB1 / 32, coarse, need, digit, pop);
  // Keys whose bits above `shift` exceed `prefix` are taken; keys equal to it on
  // those bits form the threshold group, taken whole unless `tie` (only on the
  // full 32 bits), where the first `quota` of them in token order are taken.
  uint32_t prefix = (uint32_t)digit;
  int shift = 32 - kD1;
  bool tie = false;
  uint32_t quota = 0;
  auto tie_quota = [&]() {  // equal keys: `need` of them, lowest indices first (lower CTA ranks hold lower indices)
    tie = true;
    uint32_t before = 0;
#pragma unroll
    for (int q = 0; q < C; ++q)
      if (q < c) before += cluster.map_shared_rank(h3, q)[digit];
    const uint32_t mine = h3[digit];
    quota = need > before ? min(need - before, mine) : 0u;
  };
  // Warp w owns the contiguous run of groups [g0, g1) of the slice.
  const int wg = (n4 + kResWarps - 1) / kResWarps;
  const int g0 = min(n4, wid * wg), g1 = min(n4, g0 + wg);
  const uint32_t lanes_below = (1u << lane) - 1u;
  // The warp's place in the row's output from its counts: `n_sel` taken or in
  // the threshold group, `n_eq` of those in the group when it is tied.  Returns
  // the first output position and the warp's share of the group quota.
  auto place = [&](uint32_t n_sel, uint32_t n_eq, bool stage_overflow, uint32_t& eq_take, bool& overflow) {
    if (lane == 0) {
      scan[wid] = tie ? n_eq : 0u;                 // threshold-group keys that need a quota
      misc[1 + wid] = tie ? n_sel - n_eq : n_sel;  // taken outright
      if (stage_overflow) misc[kOverflow] = 1u;
    }
    __syncthreads();
    uint32_t eq_before = 0, sel_before = 0, sel_total = 0;
    eq_take = 0;
    for (int w = 0; w < kResWarps; ++w) {
      const uint32_t e = scan[w], gtw = misc[1 + w];
      const uint32_t take_e = eq_before >= quota ? 0u : min(e, quota - eq_before);
      if (w < wid) sel_before += gtw + take_e;
      if (w == wid) eq_take = take_e;
      sel_total += gtw + take_e;
      eq_before += e;
    }
    overflow = misc[kOverflow] != 0u;
    // each CTA's total into slot c of every higher-ranked CTA (distributed
    // shared memory), so that after the barrier the offsets are read locally
    // and no CTA's shared memory is read by a peer any more
    if (tid > c && tid < C) cluster.map_shared_rank(scan + 16, tid)[c] = sel_total;
    csync();
    uint32_t offset = 0;
#pragma unroll
    for (int q = 0; q < C; ++q) offset += q < c ? scan[16 + q] : 0u;
    if (c == C - 1 && tid == 0 && offset + sel_total != (uint32_t)k) report(status, DSA_ERR_BOUNDS);  // consistency check
    return offset + sel_before;
  };

  if constexpr (!kStream) {
    // Lane l owns the contiguous groups [q0, q1) of its warp's run: an odd
    // number, at most 15 (slices of at most kResKeys keys), so a warp's
    // 16-byte loads fall in distinct banks and the run fits a 64-bit mask.
    const int wl = ((g1 - g0 + 31) / 32) | 1;
    const int q0 = min(g1, g0 + lane * wl), q1 = min(g1, q0 + wl);
    uint32_t* run = reinterpret_cast<uint32_t*>(keys4) + 4 * q0;  // the run's keys, then its candidates
    // ---- 2. one pass over the run: keys above the first digit's bin are taken
    //         whatever follows (bit set in `above`); keys in the bin are the
    //         candidates (bit set in `cand`), moved to the front of the run in
    //         token order and counted for the second digit
    const bool count2 = need != pop;
    uint64_t above = 0, cand = 0;
    int nc = 0;
    for (int i = q0; i < q1; ++i) {
      const uint4 kk = keys4[i];
      const uint32_t valid = valid_bits(i);
      const uint32_t a[4] = {kk.x, kk.y, kk.z, kk.w};
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const uint32_t bin = a[j] >> (32 - kD1);
        const int b = 4 * (i - q0) + j;
        if (((valid >> j) & 1u) && bin >= prefix) {
          if (bin > prefix) {
            above |= 1ull << b;
          } else {
            cand |= 1ull << b;
            run[nc++] = a[j];  // never past the key just read
            if (count2) atomicAdd(&h2[(a[j] >> kD3) & (kB2 - 1)], 1u);
          }
        }
      }
    }
    if (count2) {
      merge_pick(h2, kB2 / 32, coarse + kCoarse, need, digit, pop);
      prefix = (prefix << kD2) | (uint32_t)digit;
      shift = kD3;
      if (need != pop) {
        // ---- 3. last digit (bits 9..0), over the candidates only
        for (int t = 0; t < nc; ++t) {
          const uint32_t key = run[t];
          if ((key >> kD3) == prefix) atomicAdd(&h3[key & (kB3 - 1)], 1u);
        }
        merge_pick(h3, kB3 / 32, coarse + 2 * kCoarse, need, digit, pop);
        prefix = (prefix << kD3) | (uint32_t)digit;
        shift = 0;
        if (need != pop) tie_quota();
      }
    }
    // ---- 4. emit in ascending token order
    const KeyRange fin = key_range(prefix, shift);  // the threshold group
    const uint32_t fin_hi = fin.klo + fin.span;
    uint32_t c_gt = (uint32_t)__popcll(above), c_eq = 0;
    for (int t = 0; t < nc; ++t) {
      const uint32_t key = run[t];
      c_gt += key > fin_hi;
      c_eq += key - fin.klo <= fin.span;
    }
    const uint32_t n_eq = __reduce_add_sync(0xffffffffu, c_eq);
    const uint32_t n_sel = __reduce_add_sync(0xffffffffu, c_gt) + n_eq;
    uint32_t eq_take;
    bool overflow;
    const uint32_t pos = place(n_sel, n_eq, false, eq_take, overflow);
    // this lane's place in the warp: the lanes below took their keys above the
    // group and, up to the warp's quota, their keys in it
    uint32_t eq_tot, taken_tot;
    const uint32_t eq_before_lane = warp_excl_scan(c_eq, eq_tot);
    const uint32_t eq_mine = !tie ? c_eq : (eq_before_lane >= eq_take ? 0u : min(c_eq, eq_take - eq_before_lane));
    uint32_t p = pos + warp_excl_scan(c_gt + eq_mine, taken_tot);
    uint32_t eq_left = eq_mine;
    int t = 0;
    for (uint64_t m = above | cand; m; m &= m - 1) {
      const int b = __ffsll((long long)m) - 1;
      bool take = (above >> b) & 1ull;
      if (!take) {  // the t-th candidate
        const uint32_t key = run[t++];
        if (key > fin_hi) {
          take = true;
        } else if (key - fin.klo <= fin.span && eq_left) {
          take = true;
          --eq_left;
        }
      }
      if (take) {
        if (p < (uint32_t)k) emit(p, start + 4 * q0 + b);
        ++p;
      }
    }
    return;
  }

  // ---------------------------------------------------------------- streaming
  // U groups loaded ahead per thread
  constexpr int U = 8;
  auto for_my_groups = [&](auto&& body) {  // body(i, group) for groups i = tid + j * kResThreads
    for (int i0 = tid; i0 < n4; i0 += U * kResThreads) {
      G v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = i0 + u * kResThreads;
        if (i < n4) v[u] = load_group(i);
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (i0 + u * kResThreads < n4) body(i0 + u * kResThreads, v[u]);
    }
  };
  if (need != pop) {
    // ---- 2. second digit (bits 20..10) within the threshold group
    const KeyRange rg = key_range(prefix, shift);
    for_my_groups([&](int i, const G& v) {
      const uint32_t m = bits_in(v, rg) & valid_bits(i);
      if (m) {
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if ((m >> j) & 1u) atomicAdd(&h2[(elem_key(v, j) >> kD3) & (kB2 - 1)], 1u);
      }
    });
    merge_pick(h2, kB2 / 32, coarse + kCoarse, need, digit, pop);
    prefix = (prefix << kD2) | (uint32_t)digit;
    shift = kD3;
    if (need != pop) {
      // ---- 3. last digit (bits 9..0)
      const KeyRange rg3 = key_range(prefix, shift);
      for_my_groups([&](int i, const G& v) {
        const uint32_t m = bits_in(v, rg3) & valid_bits(i);
        if (m) {
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if ((m >> j) & 1u) atomicAdd(&h3[elem_key(v, j) & (kB3 - 1)], 1u);
        }
      });
      merge_pick(h3, kB3 / 32, coarse + 2 * kCoarse, need, digit, pop);
      prefix = (prefix << kD3) | (uint32_t)digit;
      shift = 0;
      if (need != pop) tie_quota();
    }
  }
  const KeyRange fin = key_range(prefix, shift);  // the threshold group

  // ---- 4. emit in ascending token order, 128 scores per warp step (a 16-byte
  //         group per lane)
  auto for_warp_groups = [&](auto&& body) {  // body(i, group) for i = g0 + 32 s + lane while g0 + 32 s < g1
    for (int b0 = g0; b0 < g1; b0 += 32 * U) {
      G v[U];
#pragma unroll
      for (int u = 0; u < U; ++u) {
        const int i = b0 + 32 * u + lane;
        if (i < g1) v[u] = load_group(i);
      }
#pragma unroll
      for (int u = 0; u < U; ++u)
        if (b0 + 32 * u < g1) body(b0 + 32 * u + lane, v[u]);  // the same for the whole warp
    }
  };
  auto classify = [&](int i, const G& v, uint32_t& gt, uint32_t& eq) {  // bit j: element 4i+j above / in the group
    gt = eq = 0;
    if (i < g1) {
      const uint32_t valid = valid_bits(i);
      gt = bits_above(v, fin) & valid;
      eq = bits_in(v, fin) & valid;
    }
  };
  // 4a. one pass: the warp counts what it takes and stages the slice-local
  //     indices in token order (bit 31: a key of the threshold group)
  uint32_t* my_stage = stage + wid * kStageCap;
  uint32_t n_sel = 0, n_eq = 0;
  for_warp_groups([&](int i, const G& v) {
    uint32_t gt, eq;
    classify(i, v, gt, eq);
    const uint32_t sel = gt | eq;
    if (__any_sync(0xffffffffu, sel != 0)) {  // most steps select nothing
      uint32_t tot;
      uint32_t p = n_sel + warp_excl_scan_small(__popc(sel), lanes_below, tot);
#pragma unroll
      for (int j = 0; j < 4; ++j)
        if ((sel >> j) & 1u) {
          if (p < (uint32_t)kStageCap) my_stage[p] = (uint32_t)(4 * i + j) | (((eq >> j) & 1u) << 31);
          ++p;
        }
      n_sel += tot;
      if (tie) n_eq += __reduce_add_sync(0xffffffffu, __popc(eq));
    }
  });
  uint32_t eq_take;
  bool overflow;
  uint32_t pos = place(n_sel, n_eq, n_sel > (uint32_t)kStageCap, eq_take, overflow);
  if (!overflow) {
    // 4b. the staged indices out, 32 at a time; threshold-group keys past the
    //     warp's quota are dropped
    uint32_t eq_seen = 0;
    for (uint32_t t0 = 0; t0 < n_sel; t0 += 32) {
      const uint32_t t = t0 + lane;
      const uint32_t e = t < n_sel ? my_stage[t] : 0u;
      bool take = t < n_sel;
      if (tie) {
        const bool is_eq = take && (e >> 31);
        const uint32_t eq_mask = __ballot_sync(0xffffffffu, is_eq);
        if (is_eq) take = eq_seen + __popc(eq_mask & lanes_below) < eq_take;
        eq_seen += __popc(eq_mask);
      }
      const uint32_t take_mask = __ballot_sync(0xffffffffu, take);
      const uint32_t p = pos + __popc(take_mask & lanes_below);
      if (take && p < (uint32_t)k) emit(p, start + (int)(e & 0x7FFFFFFFu));
      pos += __popc(take_mask);
    }
    return;
  }
  // 4b'. a warp took more than it can stage (many keys of one warp's run at the
  //      top, or a large tie): classify the run again and write as it goes
  uint32_t eq_seen = 0;
  {
    for_warp_groups([&](int i, const G& v) {
      uint32_t gt, eq;
      classify(i, v, gt, eq);
      uint32_t take = gt;
      if (!tie) {
        take |= eq;
      } else if (__any_sync(0xffffffffu, eq != 0)) {
        // the group's keys in token order until the warp's quota
        uint32_t eq_tot;
        const uint32_t eq_pre = warp_excl_scan_small(__popc(eq), lanes_below, eq_tot);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if ((eq >> j) & 1u) {
            if (eq_seen + eq_pre + __popc(eq & ((1u << j) - 1u)) < eq_take) take |= 1u << j;
          }
        eq_seen += eq_tot;
      }
      if (__any_sync(0xffffffffu, take != 0)) {
        uint32_t t_tot;
        uint32_t p = pos + warp_excl_scan_small(__popc(take), lanes_below, t_tot);
#pragma unroll
        for (int j = 0; j < 4; ++j)
          if ((take >> j) & 1u) {
            if (p < (uint32_t)k) emit(p, start + 4 * i + j);
            ++p;
          }
        pos += t_tot;
      }
    });
  }
}

template <int C, bool kStream, typename In>
dsa_status_t launch_cluster(const In* scores, int64_t ld, const int32_t* row_lens, const int32_t* seq_lens,
                            int nq, int rows, int cap, int k, int32_t* out, int32_t* status, cudaStream_t st,
                            const TopkPhys& po, const TopkSeg& sg = TopkSeg{}) {
  static std::atomic<bool> attr_set[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    if (cuda_status(cudaFuncSetAttribute(topk_cluster_kernel<C, kStream, In>,
                                         cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)res_smem(kStream ? 0 : kResKeys))) != DSA_OK)
      return DSA_ERR_CUDA;
    if (C > kResMaxCluster &&
        cuda_status(cudaFuncSetAttribute(topk_cluster_kernel<C, kStream, In>,
                                         cudaFuncAttributeNonPortableClusterSizeAllowed, 1)) != DSA_OK)
      return DSA_ERR_CUDA;
    attr_set[dev] = true;
  }
  // each CTA's slice of the longest row (segment), rounded up to 4 keys
  const int longest = sg.longest ? sg.longest : cap;
  const int slice = (((longest + C - 1) / C) + 3) & ~3;
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)(rows * (sg.nseg ? sg.nseg : 1) * C));
  cfg.blockDim = dim3(kResThreads);
  cfg.dynamicSmemBytes = res_smem(kStream ? 0 : slice);
  cfg.stream = st;
  cudaLaunchAttribute attr[2];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = C;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  attr[1].id = cudaLaunchAttributeProgrammaticStreamSerialization;  // overlaps the indexer's tail
  attr[1].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 2;
  count_launches(1);
  if (cuda_status(cudaLaunchKernelEx(&cfg, topk_cluster_kernel<C, kStream, In>, scores, ld, row_lens, seq_lens, nq, cap,
                                     k, out, status, slice, po, sg)) != DSA_OK)
    return DSA_ERR_CUDA;
  return launch_status();
}

// Whether clusters of C streaming CTAs can be resident at all on this device
// (asked once per device; a cluster of 16 needs the non-portable size).
template <int C, typename In>
bool stream_cluster_ok() {
  static std::atomic<int> known[64];  // 0 unknown, 1 yes, 2 no
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev >= 64) return false;
  if (known[dev] == 0) {
    bool ok = cudaFuncSetAttribute(topk_cluster_kernel<C, true, In>, cudaFuncAttributeNonPortableClusterSizeAllowed,
                                   C > kResMaxCluster ? 1 : 0) == cudaSuccess;
    cudaLaunchConfig_t cfg = {};
    cfg.gridDim = dim3(C);
    cfg.blockDim = dim3(kResThreads);
    cfg.dynamicSmemBytes = res_smem(0);
    cudaLaunchAttribute attr[1];
    attr[0].id = cudaLaunchAttributeClusterDimension;
    attr[0].val.clusterDim.x = C;
    attr[0].val.clusterDim.y = 1;
    attr[0].val.clusterDim.z = 1;
    cfg.attrs = attr;
    cfg.numAttrs = 1;
    int n = 0;
    ok = ok && cudaOccupancyMaxActiveClusters(&n, topk_cluster_kernel<C, true, In>, &cfg) == cudaSuccess && n > 0;
    cudaGetLastError();  // a refused query leaves no error behind
    known[dev] = ok ? 1 : 2;
  }
  return known[dev] == 1;
}

size_t ws_bytes(int rows, int k) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  return al((size_t)rows * kBins * 4) + al((size_t)rows * 16) + al((size_t)rows * k * 4) +
         al((size_t)rows * kCandCap * 8);
}

// ------------------------------------------------------------ many rows
// Many rows of at most kRowMaxLen tokens (a prefill chunk's rows): one CTA
// per row at a time, persistent over the rows, each row streamed from global
// memory rather than held on chip, so that a row per SM is in flight instead
// of a row per cluster.
//   1. One pass over the row: histogram of the keys' top 12 bits, and the bin
//      holding the k-th key (the threshold group).
//   2. While the group holds more than half the candidate buffer, one more
//      pass refines it by the next 10 bits.
//   3. One pass marks the keys above the group in bitmap A and moves the
//      group's keys with their indices into shared memory, each warp into a
//      region of its own (no shared counter); a group of one key value (all
//      32 bits fixed) goes straight into bitmap B.  If a warp's region
//      overflows, the group is refined once more and the pass repeated.
//   4. The remaining digits over the candidates in shared memory give the
//      exact k-th key; candidates above it go into A, those equal to it into B.
//   5. B keeps its `need` lowest indices (ties to the lower index), and the
//      indices of A | B are written in ascending order.
constexpr int kRowThreads = 512;              // two CTAs per SM: one streams while the other selects
constexpr int kRowWarps = kRowThreads / 32;
constexpr int kRowMaxLen = 163840;           // bitmaps of 5,120 words each
constexpr int kRowWords = kRowMaxLen / 32;
constexpr int kRowB1 = 4096;                 // first digit: key bits 31..20
constexpr int kRowD = 10;                    // later digits: bits 19..10, then 9..0
constexpr int kRowCand = 6144;               // group keys held in shared memory, ...
constexpr int kRowWarpCand = kRowCand / kRowWarps;  // ... in one region per warp
constexpr int kRowGroupMax = kRowCand / 2;   // larger groups are narrowed first
constexpr int kRowU = 4;                     // 16-byte loads in flight per thread
constexpr int kRowAhead = 4;                 // L2 prefetch distance in loop steps (32 KB each)
constexpr size_t kRowSmem = (size_t)(kRowB1 + 2 * kRowWords + 2 * kRowCand + 96) * 4;
static_assert(kRowWarps <= 32, "the block scan holds the warp totals in one warp's lanes");
// a row of at most kRowCand tokens puts at most kRowWarpCand of them in each warp's stripe
static_assert(kRowCand % (4 * kRowThreads) == 0, "whole passes of the stream loop");

// Exclusive prefix sum of v over the CTA's threads in thread order; `total`
// is the sum over all of them.  ws: kRowWarps words.  Two barriers.
__device__ __forceinline__ uint32_t row_block_scan(uint32_t v, uint32_t* ws, uint32_t& total) {
  const int lane = threadIdx.x & 31, wid = threadIdx.x >> 5;
  uint32_t x = v;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, x, d);
    if (lane >= d) x += y;
  }
  __syncthreads();  // ws is free
  if (lane == 31) ws[wid] = x;
  __syncthreads();
  const uint32_t w = lane < kRowWarps ? ws[lane] : 0u;
  uint32_t wsum = w;
#pragma unroll
  for (int d = 1; d < 32; d <<= 1) {
    const uint32_t y = __shfl_up_sync(0xffffffffu, wsum, d);
    if (lane >= d) wsum += y;
  }
  total = __shfl_sync(0xffffffffu, wsum, 31);
  return __shfl_sync(0xffffffffu, wsum - w, wid) + x - v;
}

// The bin of histogram h (nb bins, nb a multiple of the thread count) that
// holds the need-th largest key counting from the top, need within it, and
// its count.  Thread t sums the bins [nb - (t+1) per, nb - t per), so the
// scan in thread order counts the keys above each thread's bins.  res: 3
// words, read after the closing barrier.  Opens with a barrier, so the
// histogram's last increments are complete.
struct RowPick {
  uint32_t bin, need, pop;
};
__device__ __forceinline__ RowPick row_pick(const uint32_t* h, int nb, uint32_t need, uint32_t* ws, uint32_t* res) {
  const int per = nb / kRowThreads;
  const int hi = nb - (int)threadIdx.x * per;
  __syncthreads();  // the histogram is complete
  if (threadIdx.x == 0) {  // only kept if the counts were inconsistent
    res[0] = 0u;
    res[1] = 1u;
    res[2] = 0u;
  }
  uint32_t sum = 0;
  for (int j = 1; j <= per; ++j) sum += h[hi - j];
  uint32_t tot;
  const uint32_t above = row_block_scan(sum, ws, tot);
  if (above < need && need <= above + sum) {
    uint32_t a = above;
    for (int j = 1; j <= per; ++j) {
      const uint32_t c = h[hi - j];
      if (need <= a + c) {
        res[0] = (uint32_t)(hi - j);
        res[1] = need - a;
        res[2] = c;
        break;
      }
      a += c;
    }
  }
  __syncthreads();
  return RowPick{res[0], res[1], res[2]};
}

__global__ void __launch_bounds__(kRowThreads, 2)
    topk_row_kernel(const float* __restrict__ scores, int64_t ld, const int32_t* row_lens, const int32_t* seq_lens,
                    int nq, int rows, int cap, int k, int32_t* out, int32_t* status, const TopkPhys po) {
  extern __shared__ __align__(16) uint32_t rsm[];
  uint32_t* hist = rsm;               // kRowB1 bins (1,024 in the later digits)
  uint32_t* bmA = hist + kRowB1;      // tokens above the k-th key
  uint32_t* bmB = bmA + kRowWords;    // tokens equal to it
  uint32_t* ckey = bmB + kRowWords;   // the group's keys ...
  uint32_t* cidx = ckey + kRowCand;   // ... and their token indices
  uint32_t* ws = cidx + kRowCand;     // 32 words: scan scratch
  uint32_t* res = ws + 32;            // 0..2: a pick
  uint32_t* wcnt = res + 32;          // kRowWarps words: candidates per warp region
  const int tid = threadIdx.x, lane = tid & 31, wid = tid >> 5;
  const uint32_t lanes_below = (1u << lane) - 1u;
  grid_dep_wait();  // the scores come from the previous kernel, which may also still read `out`
  grid_dep_launch();
  for (int r = blockIdx.x; r < rows; r += gridDim.x) {
    const int len = row_len(row_lens, seq_lens, nq, r, cap, status);
    int32_t* o = out + (int64_t)r * k;
    auto emit = [&](int pos, int t) {
      o[pos] = t;
      if (po.phys) po.phys[(int64_t)r * k + pos] = phys_row(po, nq, r, t, status);
    };
    if (len <= k) {  // every token, then padding; no shared memory used
      for (int i = tid; i < k; i += kRowThreads) emit(i, i < len ? i : -1);
      continue;
    }
    const float* row = scores + (int64_t)r * ld;
    const int nw = (len + 31) >> 5;
    const int full4 = len >> 2;
    // body(t0, keys, valid) for every group of 4 tokens t0..t0+3 (valid: a bit
    // per token of the row); every thread of a warp calls it equally often,
    // so warp votes inside are allowed
    const int n4 = (len + 3) >> 2;
    // group i of the row (16-byte aligned; the ragged last one padded with NaN)
    auto load_group = [&](int i) -> float4 {
      if (i < full4) return reinterpret_cast<const float4*>(row)[i];
      const float nan = __uint_as_float(0x7FC00000u);
      if (i >= n4) return make_float4(nan, nan, nan, nan);
      return make_float4(row[4 * i], 4 * i + 1 < len ? row[4 * i + 1] : nan, 4 * i + 2 < len ? row[4 * i + 2] : nan,
                         nan);
    };
    auto group_valid = [&](int i) -> uint32_t {
      return i < full4 ? 0xFu : (i < n4 ? (1u << (len - 4 * i)) - 1u : 0u);
    };
    auto group_keys = [](const float4& v) {
      return make_uint4(score_key(v.x), score_key(v.y), score_key(v.z), score_key(v.w));
    };
    // four groups in flight per thread, held in named registers (no array)
    static_assert(kRowU == 4, "stream() holds four groups");
    // L2 prefetch of step `it` of a pass (its 4 x kRowThreads groups), kRowAhead
    // steps before the loads: the loads then mostly wait on L2, not HBM
    auto prefetch = [&](int it) {
      const int g0 = it * 4 * kRowThreads;
      if (tid == 0 && g0 < full4) prefetch_l2(row + 4 * (int64_t)g0, (uint32_t)min(4 * kRowThreads, full4 - g0) * 16u);
    };
    bool primed = false;  // the row's first pass finds its first prefetches issued
    auto stream = [&](auto&& body) {
      if (!primed)
        for (int d = 0; d < kRowAhead; ++d) prefetch(d);
      primed = false;
      for (int base = 0; base < n4; base += 4 * kRowThreads) {  // the same trip count in every thread
        prefetch(base / (4 * kRowThreads) + kRowAhead);
        const int i0 = base + tid, i1 = i0 + kRowThreads, i2 = i0 + 2 * kRowThreads, i3 = i0 + 3 * kRowThreads;
        const float4 v0 = load_group(i0), v1 = load_group(i1), v2 = load_group(i2), v3 = load_group(i3);
        body(4 * i0, group_keys(v0), group_valid(i0));
        body(4 * i1, group_keys(v1), group_valid(i1));
        body(4 * i2, group_keys(v2), group_valid(i2));
        body(4 * i3, group_keys(v3), group_valid(i3));
      }
    };

    for (int i = tid; i < kRowB1; i += kRowThreads) hist[i] = 0u;
    for (int i = tid; i < nw; i += kRowThreads) {
      bmA[i] = 0u;
      bmB[i] = 0u;
    }
    for (int d = 0; d < kRowAhead; ++d) prefetch(d);  // the row's first pass, while the sample is read
    primed = true;
    __syncthreads();
    uint32_t* const wkey = ckey + wid * kRowWarpCand;  // this warp's candidate region
    uint32_t* const widx = cidx + wid * kRowWarpCand;
    // Stores the keys of the 4-token group at t0 flagged in `grp` in the
    // warp's region from slot wc on (every lane of the warp calls it with the
    // same wc, which then counts all of the warp's flagged keys).
    auto store_cands = [&](int t0, const uint4& kk, uint32_t grp, uint32_t& wc) {
      uint32_t tot;
      uint32_t slot = wc + warp_excl_scan_small((uint32_t)__popc(grp), lanes_below, tot);
      wc += tot;
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        if ((grp >> j) & 1u) {
          if (slot < (uint32_t)kRowWarpCand) {
            wkey[slot] = j == 0 ? kk.x : j == 1 ? kk.y : j == 2 ? kk.z : kk.w;
            widx[slot] = (uint32_t)(t0 + j);
          }
          ++slot;
        }
      }
    };
    RowPick p;
    uint32_t prefix = 0, need = 0, pop = 0;  // the threshold group: keys whose bits above `shift` equal `prefix`
    int shift = 20;

    // ---- 0. one pass, where a sample predicts the bar: the first 128 tokens
    //         of every 2,048 estimate a first-digit bin L with about 1.3 k keys
    //         above its lower edge; one pass then keeps every key of bin L or above as a
    //         candidate (the sample's lines are still in L2).  If they number
    //         at least k and fit their regions, the row's top-k is among them.
    bool fast = false;
    {
      const int64_t n_s = (int64_t)(len / 2048) * 128 + min(128, len % 2048);  // sampled tokens
      const int64_t need_s = (13 * (int64_t)k * n_s + 10 * (int64_t)len - 1) / (10 * (int64_t)len) + 32;
      uint32_t bar = kRowB1;  // no candidates pass: go to the general steps
      if (need_s <= n_s) {
        const int nchunk = (len + 2047) / 2048;
        // warp w reads chunks w, w + kRowWarps, ...: their first 32 groups (128 tokens)
        auto sample = [&](int c) { return load_group(c < nchunk ? c * 512 + lane : n4); };
        auto count = [&](int c, const float4& v) {
          const uint32_t valid = c < nchunk ? group_valid(c * 512 + lane) : 0u;
          const uint4 kk = group_keys(v);
          if (valid & 1u) atomicAdd(&hist[kk.x >> 20], 1u);
          if (valid & 2u) atomicAdd(&hist[kk.y >> 20], 1u);
          if (valid & 4u) atomicAdd(&hist[kk.z >> 20], 1u);
          if (valid & 8u) atomicAdd(&hist[kk.w >> 20], 1u);
        };
        for (int c0 = wid; c0 < nchunk; c0 += 4 * kRowWarps) {
          const int c1 = c0 + kRowWarps, c2 = c0 + 2 * kRowWarps, c3 = c0 + 3 * kRowWarps;
          const float4 v0 = sample(c0), v1 = sample(c1), v2 = sample(c2), v3 = sample(c3);
          count(c0, v0);
          count(c1, v1);
          count(c2, v2);
          count(c3, v3);
        }
        bar = row_pick(hist, kRowB1, (uint32_t)need_s, ws, res).bin;
      } else if (len <= kRowCand) {
        bar = 0;  // every key: a warp's stripe of such a row holds at most kRowWarpCand tokens
      }
      if (bar < (uint32_t)kRowB1) {
        for (int i = tid; i < kRowB1; i += kRowThreads) hist[i] = 0u;
        __syncthreads();
        // keys of bin `bar` or above, compared as scores (score_range: NaN
        // scores are below every bin but bin 0, where every score passes)
        const KeyRange kr = key_range(bar, 20);
        auto pass = [&](const float4& v, uint32_t valid) -> uint32_t {
          return (kr.s.nan ? 0xFu : ((uint32_t)(v.x >= kr.s.lo) | ((uint32_t)(v.y >= kr.s.lo) << 1) |
                                     ((uint32_t)(v.z >= kr.s.lo) << 2) | ((uint32_t)(v.w >= kr.s.lo) << 3))) &
                 valid;
        };
        auto elem = [](const float4& v, int j) { return j == 0 ? v.x : j == 1 ? v.y : j == 2 ? v.z : v.w; };
        uint32_t wc = 0;  // this warp's candidates so far (the same in every lane)
        if (tid == 0 && !primed)
          for (int d = 0; d < kRowAhead; ++d) prefetch(d);
        primed = false;
        for (int base = 0; base < n4; base += 4 * kRowThreads) {  // the same trip count in every thread
          prefetch(base / (4 * kRowThreads) + kRowAhead);
          const int i0 = base + tid;
          const float4 v0 = load_group(i0), v1 = load_group(i0 + kRowThreads), v2 = load_group(i0 + 2 * kRowThreads),
                       v3 = load_group(i0 + 3 * kRowThreads);
          // bit 4u + j: element j of group i0 + u * kRowThreads passes
          const uint32_t m = pass(v0, group_valid(i0)) | (pass(v1, group_valid(i0 + kRowThreads)) << 4) |
                             (pass(v2, group_valid(i0 + 2 * kRowThreads)) << 8) |
                             (pass(v3, group_valid(i0 + 3 * kRowThreads)) << 12);
          // the warp's exclusive prefix of the lanes' counts (0..16: five bit planes)
          const uint32_t c = (uint32_t)__popc(m);
          uint32_t before = 0, tot = 0;
#pragma unroll
          for (int bit = 0; bit < 5; ++bit) {
            const uint32_t plane = __ballot_sync(0xffffffffu, (c >> bit) & 1u);
            before += (uint32_t)__popc(plane & lanes_below) << bit;
            tot += (uint32_t)__popc(plane) << bit;
          }
          uint32_t slot = wc + before;
          wc += tot;
          for (uint32_t mm = m; mm; mm &= mm - 1) {
            const int b = __ffs(mm) - 1, u = b >> 2, j = b & 3;
            const float e0 = elem(v0, j), e1 = elem(v1, j), e2 = elem(v2, j), e3 = elem(v3, j);
            const uint32_t key = score_key(u == 0 ? e0 : u == 1 ? e1 : u == 2 ? e2 : e3);
            atomicAdd(&hist[key >> 20], 1u);
            if (slot < (uint32_t)kRowWarpCand) {
              wkey[slot] = key;
              widx[slot] = (uint32_t)(4 * (i0 + u * kRowThreads) + j);
            }
            ++slot;
          }
        }
        if (lane == 0) wcnt[wid] = wc;
        __syncthreads();
        bool over = false;
        uint32_t total = 0;
        for (int w = 0; w < kRowWarps; ++w) {
          over |= wcnt[w] > (uint32_t)kRowWarpCand;
          total += wcnt[w];
        }
        if (!over && total >= (uint32_t)k) {
          fast = true;
          p = row_pick(hist, kRowB1, (uint32_t)k, ws, res);
          prefix = p.bin;
          need = p.need;
          pop = p.pop;
        }
      }
    }

    // ---- 1. first digit (where the one pass did not settle it)
    if (!fast) {
      for (int i = tid; i < kRowB1; i += kRowThreads) hist[i] = 0u;
      __syncthreads();
      stream([&](int, const uint4& kk, uint32_t valid) {
        if (valid & 1u) atomicAdd(&hist[kk.x >> 20], 1u);
        if (valid & 2u) atomicAdd(&hist[kk.y >> 20], 1u);
        if (valid & 4u) atomicAdd(&hist[kk.z >> 20], 1u);
        if (valid & 8u) atomicAdd(&hist[kk.w >> 20], 1u);
      });
      p = row_pick(hist, kRowB1, (uint32_t)k, ws, res);
      prefix = p.bin;
      need = p.need;
      pop = p.pop;
    }
    bool narrow = false;  // a warp's candidate region overflowed: narrow the group once more
    while (!fast) {
      // ---- 2. narrower groups until the candidates fit comfortably
      while ((pop > (uint32_t)kRowGroupMax || narrow) && shift > 0) {
        narrow = false;
        for (int i = tid; i < (1 << kRowD); i += kRowThreads) hist[i] = 0u;
        __syncthreads();
        const int s2 = shift - kRowD;
        stream([&](int, const uint4& kk, uint32_t valid) {
          const uint32_t a[4] = {kk.x, kk.y, kk.z, kk.w};
#pragma unroll
          for (int j = 0; j < 4; ++j)
            if (((valid >> j) & 1u) && (a[j] >> shift) == prefix)
              atomicAdd(&hist[(a[j] >> s2) & ((1u << kRowD) - 1u)], 1u);
        });
        p = row_pick(hist, 1 << kRowD, need, ws, res);
        prefix = (prefix << kRowD) | p.bin;
        need = p.need;
        pop = p.pop;
        shift = s2;
      }
      // ---- 3. keys above the group into A (a group's 4 tokens share a bitmap
      //         word); the group into the warp's candidate region (or B)
      uint32_t wc = 0;  // this warp's candidates so far (the same in every lane)
      stream([&](int t0, const uint4& kk, uint32_t valid) {
        const uint32_t a[4] = {kk.x, kk.y, kk.z, kk.w};
        uint32_t above = 0, grp = 0;
#pragma unroll
        for (int j = 0; j < 4; ++j) {
          const uint32_t top = a[j] >> shift;
          if (top > prefix) above |= 1u << j;
          if (top == prefix) grp |= 1u << j;
        }
        above &= valid;
        grp &= valid;
        if (above) atomicOr(&bmA[t0 >> 5], above << (t0 & 31));
        if (shift == 0) {
          if (grp) atomicOr(&bmB[t0 >> 5], grp << (t0 & 31));
        } else {
          store_cands(t0, kk, grp, wc);
        }
      });
      if (lane == 0) wcnt[wid] = wc;
      __syncthreads();
      if (shift == 0) break;
      bool over = false;
      for (int w = 0; w < kRowWarps; ++w) over |= wcnt[w] > (uint32_t)kRowWarpCand;
      if (!over) break;
      narrow = true;  // A keeps its bits: keys above this group are above any narrower one
      __syncthreads();  // every thread has read the counts
    }
    // ---- 4. the last digits over the candidates: the exact k-th key (in
    //         the one-pass case the candidates hold every key above the group
    //         too, and they go into A with the others above it)
    auto for_cands = [&](auto&& body) {  // body(key, token) for every stored candidate
      for (int c = tid; c < kRowCand; c += kRowThreads)
        if ((uint32_t)(c % kRowWarpCand) < wcnt[c / kRowWarpCand]) body(ckey[c], cidx[c]);
    };
    if (shift > 0) {
      while (shift > 0) {
        for (int i = tid; i < (1 << kRowD); i += kRowThreads) hist[i] = 0u;
        __syncthreads();
        const int s2 = shift - kRowD;
        for_cands([&](uint32_t key, uint32_t) {
          if ((key >> shift) == prefix) atomicAdd(&hist[(key >> s2) & ((1u << kRowD) - 1u)], 1u);
        });
        p = row_pick(hist, 1 << kRowD, need, ws, res);
        prefix = (prefix << kRowD) | p.bin;
        need = p.need;
        pop = p.pop;
        shift = s2;
      }
      for_cands([&](uint32_t key, uint32_t t) {
        if (key > prefix) atomicOr(&bmA[t >> 5], 1u << (t & 31));
        else if (key == prefix) atomicOr(&bmB[t >> 5], 1u << (t & 31));
      });
      __syncthreads();
    }
    // ---- 5. the lowest `need` of the tied indices, then the output in order;
    //         thread t owns the bitmap words [w0, w1)
    const int per = (nw + kRowThreads - 1) / kRowThreads;
    const int w0 = min(nw, tid * per), w1 = min(nw, w0 + per);
    uint32_t tot;
    if (need < pop) {
      uint32_t cnt = 0;
      for (int w = w0; w < w1; ++w) cnt += __popc(bmB[w]);
      uint32_t run = row_block_scan(cnt, ws, tot);
      for (int w = w0; w < w1; ++w) {
        uint32_t x = bmB[w], keep = 0;
        while (x && run < need) {
          const uint32_t b = x & (0u - x);
          keep |= b;
          x ^= b;
          ++run;
        }
        bmB[w] = keep;
      }
      __syncthreads();
    }
    uint32_t cnt = 0;
    for (int w = w0; w < w1; ++w) cnt += __popc(bmA[w] | bmB[w]);
    uint32_t pos = row_block_scan(cnt, ws, tot);
    for (int w = w0; w < w1; ++w) {
      for (uint32_t x = bmA[w] | bmB[w]; x; x &= x - 1) {
        if (pos < (uint32_t)k) emit((int)pos, w * 32 + __ffs(x) - 1);
        ++pos;
      }
    }
    if (tid == 0 && tot != (uint32_t)k) report(status, DSA_ERR_BOUNDS);  // consistency check
    __syncthreads();  // shared memory is reused by the next row
  }
}

// Whether the per-row CTA form serves these rows: more rows than one wave of
// row-resident clusters holds (two CTAs of 20,480 keys per SM), and rows
// short enough for its bitmaps.
bool use_row_form(int rows, int max_row_len, int k) {
  if (max_row_len <= k || max_row_len > kRowMaxLen) return false;
  const int64_t ctas = (int64_t)rows * ((max_row_len + kResPairKeys - 1) / kResPairKeys);
  return ctas > 2 * (int64_t)num_sms();
}

dsa_status_t launch_topk_rows(const float* scores, int64_t ld, const int32_t* row_lens, const int32_t* seq_lens,
                              int nq, int rows, int cap, int k, int32_t* out, int32_t* status, cudaStream_t st,
                              const TopkPhys& po) {
  static std::atomic<bool> attr_set[64];
  int dev = 0;
  cudaGetDevice(&dev);
  if (dev < 64 && !attr_set[dev]) {
    if (cuda_status(cudaFuncSetAttribute(topk_row_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)kRowSmem)) != DSA_OK)
      return DSA_ERR_CUDA;
    attr_set[dev] = true;
  }
  cudaLaunchConfig_t cfg = {};
  cfg.gridDim = dim3((unsigned)std::min(rows, 2 * num_sms()));  // two CTAs per SM, persistent over the rows
  cfg.blockDim = dim3(kRowThreads);
  cfg.dynamicSmemBytes = kRowSmem;
  cfg.stream = st;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeProgrammaticStreamSerialization;
  attr[0].val.programmaticStreamSerializationAllowed = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  count_launches(1);
  if (cuda_status(cudaLaunchKernelEx(&cfg, topk_row_kernel, scores, ld, row_lens, seq_lens, nq, rows, cap, k, out,
                                     status, po)) != DSA_OK)
    return DSA_ERR_CUDA;
  return launch_status();
}

// The two-level form for rows longer than a cluster holds: segments of at
// most kSegMax tokens (8 CTAs of 20,480 keys, two CTAs per SM), more of them
// where that fills the SMs better (down to kSegMin tokens), each reduced to
// its top-k; then one more top-k over the rows' candidates.  Few long rows
// then spread over all SMs.  The workspace holds the candidates of up to
// kSlotsMax / 8 segments per row (or the fewest that cover the row).
constexpr int kSegMax = 8 * 20480;
constexpr int kSegMin = 8 * 4096;
constexpr int kSlotsMax = 2 * 192;  // CTA slots the segment count aims at, on devices up to 192 SMs
int two_level_max_nseg(int rows, int max_row_len) {
  const int need = (max_row_len + kSegMax - 1) / kSegMax;
  const int fill = std::min(kSlotsMax / (8 * std::max(rows, 1)), (max_row_len + kSegMin - 1) / kSegMin);
  return std::max(need, fill);
}
int64_t two_level_ldc(int nseg, int k) { return ((int64_t)nseg * k + 3) & ~int64_t(3); }
size_t two_level_bytes(int rows, int max_row_len, int k) {
  auto al = [](size_t x) { return (x + 255) & ~size_t(255); };
  const size_t plane = al((size_t)rows * two_level_ldc(two_level_max_nseg(rows, max_row_len), k) * 4);
  return 2 * plane;  // candidate scores, then their token indices
}

}  // namespace

size_t topk_workspace_bytes(int rows, int max_row_len, int k) {
  // rows that fit a cluster's shared memory (or need no selection) use none;
  // longer rows: the two-level form, or the four-kernel form where clusters
  // cannot be scheduled or it is forced
  if (max_row_len <= k || (max_row_len + kResKeys - 1) / kResKeys <= kResMaxCluster) return 0;
  return std::max(ws_bytes(rows, k), two_level_bytes(rows, max_row_len, k));
}

namespace {
std::atomic<int> g_force_multipass{0};
}  // namespace

int topk_force_multipass(int on) { return g_force_multipass.exchange(on ? 1 : 0); }

size_t topk_final_smem_bytes() { return (size_t)kWindowBits / 8 + 8 * kCandCap + 4 * kMaxTopk + 4 * kBins + 128; }

namespace {

// Cluster size of the row-resident form for `rows` rows of at most `len`
// keys: enough CTAs to hold a row, small enough slices for two CTAs per SM
// where a cluster of 8 allows it, and for few rows enough CTAs to spread them
// over the SMs (at least 8,192 keys per CTA).
int resident_cluster(int rows, int len) {
  const int c_min = (len + kResKeys - 1) / kResKeys;
  // two CTAs per SM pay off only while the grid stays within one wave
  int c_pair = std::min(kResMaxCluster, (len + kResPairKeys - 1) / kResPairKeys);
  if ((int64_t)rows * c_pair > 2 * (int64_t)num_sms()) c_pair = 1;
  const int c_fill = std::min(num_sms() / std::max(rows, 1), len / 8192);
  return std::min(kResMaxCluster, std::max(std::max(c_min, c_pair), std::max(c_fill, 1)));
}

template <bool kStream, typename In>
dsa_status_t launch_cluster_sized(int cluster, const In* scores, int64_t ld, const int32_t* row_lens,
                                  const int32_t* seq_lens, int nq, int rows, int cap, int k, int32_t* out,
                                  int32_t* status, cudaStream_t st, const TopkPhys& po, const TopkSeg& sg) {
#define DSA_RES(C) launch_cluster<C, kStream, In>(scores, ld, row_lens, seq_lens, nq, rows, cap, k, out, status, st, po, sg)
  switch (cluster) {
    case 1: return DSA_RES(1);
    case 2: return DSA_RES(2);
    case 3: return DSA_RES(3);
    case 4: return DSA_RES(4);
    case 5: return DSA_RES(5);
    case 6: return DSA_RES(6);
    case 7: return DSA_RES(7);
    default: return DSA_RES(8);
  }
#undef DSA_RES
}

// Rows longer than a cluster holds (fp32 scores, a workspace): pass 1 reduces
// every segment to its top-k, written into each row's compact candidate list
// (token order, with the scores), and pass 2 selects the row's top-k among
// them, writing token indices (and physical rows).  The result is the top-k
// of the whole row: every token of it is among its own segment's top-k.  Two
// launches, chained by programmatic dependent launch.  Both passes use
// clusters of up to 8 CTAs, as many as two CTAs per SM allow.
dsa_status_t launch_topk_two_level(const float* scores, int64_t ld, const int32_t* row_lens, const int32_t* seq_lens,
                                   int nq, int rows, int max_row_len, int k, int32_t* out, void* workspace,
                                   int32_t* status, cudaStream_t st, const TopkPhys& po) {
  const int slots = 2 * num_sms();
  const int need = (max_row_len + kSegMax - 1) / kSegMax;
  const int nseg = std::min(two_level_max_nseg(rows, max_row_len),
                            std::max(need, std::min(slots / (8 * rows), (max_row_len + kSegMin - 1) / kSegMin)));
  const int seg = (((max_row_len + nseg - 1) / nseg) + 3) & ~3;  // bulk copies start on 16 bytes
  const int64_t ldc = two_level_ldc(nseg, k);
  const size_t plane = ((size_t)rows * ldc * 4 + 255) & ~size_t(255);
  TopkSeg s1;
  s1.seg_tokens = seg;
  s1.nseg = nseg;
  s1.cand_score = static_cast<float*>(workspace);
  s1.cand_idx = reinterpret_cast<int32_t*>(static_cast<uint8_t*>(workspace) + plane);
  s1.ldc = ldc;
  s1.longest = std::min(max_row_len, seg);
  auto cluster_for = [&](int vrows, int len) {
    const int c_min = (len + kResKeys - 1) / kResKeys;
    if ((int64_t)vrows * kResMaxCluster <= slots) return kResMaxCluster;
    return std::max(c_min, resident_cluster(vrows, len));
  };
  dsa_status_t res = launch_cluster_sized<false, float>(cluster_for(rows * nseg, s1.longest), scores, ld, row_lens,
                                                        seq_lens, nq, rows, max_row_len, k, nullptr, status, st,
                                                        TopkPhys{}, s1);
  if (res != DSA_OK) return res;
  TopkSeg s2 = s1;
  s2.nseg = 0;
  s2.pass2 = true;
  s2.longest = (max_row_len / seg) * k + std::min(k, max_row_len % seg);
  return launch_cluster_sized<false, float>(cluster_for(rows, s2.longest), s1.cand_score, ldc, row_lens, seq_lens, nq,
                                            rows, max_row_len, k, out, status, st, po, s2);
}

// The cluster paths: true with *res set when one of them took the rows.
template <typename In>
bool launch_topk_cluster(const In* scores, int64_t ld, const int32_t* row_lens, const int32_t* seq_lens, int nq,
                         int rows, int max_row_len, int k, int32_t* out, int32_t* status, cudaStream_t st,
                         dsa_status_t* res, const TopkPhys& po) {
  // row-resident path: one cluster per row (resident_cluster), no workspace
  const int c_min = (max_row_len + kResKeys - 1) / kResKeys;
  if (max_row_len > k && c_min <= kResMaxCluster) {
    *res = launch_cluster_sized<false, In>(resident_cluster(rows, max_row_len), scores, ld, row_lens, seq_lens, nq,
                                           rows, max_row_len, k, out, status, st, po, TopkSeg{});
    return true;
  }
  if (max_row_len > k && !g_force_multipass.load(std::memory_order_relaxed)) {
    // rows too long to hold on chip: the streaming cluster kernel, 16 CTAs per
    // row where the device schedules such clusters, else 8
    if (stream_cluster_ok<16, In>()) {
      *res = launch_cluster<16, true, In>(scores, ld, row_lens, seq_lens, nq, rows, max_row_len, k, out, status, st, po);
      return true;
    }
    if (stream_cluster_ok<8, In>()) {
      *res = launch_cluster<8, true, In>(scores, ld, row_lens, seq_lens, nq, rows, max_row_len, k, out, status, st, po);
      return true;
    }
  }
  return false;
}

}  // namespace

dsa_status_t launch_topk_bf16(const uint16_t* scores, int64_t ld, const int32_t* row_lens, const int32_t* seq_lens,
                              int nq, int rows, int max_row_len, int k, int32_t* out, int32_t* status,
                              cudaStream_t st, const TopkPhys& po) {
  if (rows == 0) return DSA_OK;
  dsa_status_t res = DSA_OK;
  if (max_row_len <= k)  // nothing to select: the kernel writes 0..len-1 and the padding, reading no score
    return launch_cluster<1, false, uint16_t>(scores, ld, row_lens, seq_lens, nq, rows, max_row_len, k, out, status,
                                              st, po);
  if (launch_topk_cluster(scores, ld, row_lens, seq_lens, nq, rows, max_row_len, k, out, status, st, &res, po))
    return res;
  // long rows with the four-kernel path forced, or no cluster schedulable: that path reads fp32 scores only
  return DSA_ERR_UNSUPPORTED;
}

namespace {

// two_level: rows longer than a cluster holds may take the two-level form
// (the workspace then holds at least two_level(...).bytes); otherwise the
// streaming cluster, or the four-kernel form where it is forced or no cluster
// can be scheduled.
dsa_status_t launch_topk_impl(const float* scores, int64_t ld, const int32_t* row_lens, const int32_t* seq_lens,
                              int nq, int rows, int max_row_len, int k, int32_t* out, void* workspace,
                              int32_t* status, cudaStream_t st, const TopkPhys& po, bool two_level_ok) {
  if (rows == 0) return DSA_OK;
  dsa_status_t res = DSA_OK;
  const bool forced = g_force_multipass.load(std::memory_order_relaxed);
  if (two_level_ok && max_row_len > kResMaxCluster * kResKeys && workspace && !forced)
    return launch_topk_two_level(scores, ld, row_lens, seq_lens, nq, rows, max_row_len, k, out, workspace, status, st,
                                 po);
  // many rows: one CTA per row at a time (the forced four-kernel form keeps
  // the rows longer than a cluster holds)
  if (use_row_form(rows, max_row_len, k) && !(forced && max_row_len > kResMaxCluster * kResKeys))
    return launch_topk_rows(scores, ld, row_lens, seq_lens, nq, rows, max_row_len, k, out, status, st, po);
  if (launch_topk_cluster(scores, ld, row_lens, seq_lens, nq, rows, max_row_len, k, out, status, st, &res, po))
    return res;
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
    count_launches(3);
    topk_hist_kernel<<<grid, kThreads, 0, st>>>(scores, ld, row_lens, seq_lens, nq, cap, k, ws, status);
    topk_threshold_kernel<<<rows, kThreads, 0, st>>>(row_lens, seq_lens, nq, cap, k, ws);
    topk_collect_kernel<<<grid, kThreads, 0, st>>>(scores, ld, row_lens, seq_lens, nq, cap, k, ws, status);
  }
  static std::atomic<bool> attr_set[64];
  int dev = 0;
  cudaGetDevice(&dev);
  const size_t smem = topk_final_smem_bytes();
  if (dev < 64 && !attr_set[dev]) {
    if (cuda_status(cudaFuncSetAttribute(topk_final_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                         (int)smem)) != DSA_OK)
      return DSA_ERR_CUDA;
    attr_set[dev] = true;
  }
  count_launches(1);
  topk_final_kernel<<<rows, kFinalThreads, smem, st>>>(scores, ld, row_lens, seq_lens, nq, cap, k, ws, out, status, po);
  return launch_status();
}

}  // namespace

dsa_status_t launch_topk(const float* scores, int64_t ld, const int32_t* row_lens, const int32_t* seq_lens, int nq,
                         int rows, int max_row_len, int k, int32_t* out, void* workspace, int32_t* status,
                         cudaStream_t st, const TopkPhys& po) {
  return launch_topk_impl(scores, ld, row_lens, seq_lens, nq, rows, max_row_len, k, out, workspace, status, st, po,
                          true);
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
  // the streaming cluster for long rows (the scratch is sized for the four-kernel form)
  return launch_topk_impl(scores, ld, row_lens, nullptr, 1, rows, max_row_len, k, out, scratch, status, st, TopkPhys{},
                          false);
}

}  // namespace dsa
