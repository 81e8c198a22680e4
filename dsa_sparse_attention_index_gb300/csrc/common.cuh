// common.cuh — device building blocks shared by the sm_103a kernels:
// mbarriers with bounded waits, TMA / bulk copies, tcgen05 (TMEM, MMA,
// loads/stores), shared-memory matrix descriptors and status reporting.
#pragma once

#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_fp16.h>
#include <cuda_fp8.h>
#include <cuda_runtime.h>
#include <stdint.h>

#include "../../include/dsa.h"

namespace dsa {

constexpr int kBlock = DSA_BLOCK_SIZE;
constexpr int kIdxHeads = DSA_INDEX_HEADS;
constexpr int kIdxDim = DSA_INDEX_DIM;
constexpr int kHeads = DSA_MLA_HEADS;
constexpr int kLatent = DSA_LATENT_DIM;
constexpr int kValue = DSA_VALUE_DIM;
constexpr int kMaxTopk = DSA_MAX_TOPK;

// Longest a pipelined wait may take before the kernel gives up (ns).  Real
// waits last microseconds; this only bounds a wait that can never finish.
constexpr uint64_t kWaitLimitNs = 2000000000ull;

// ---------------------------------------------------------------- status
__device__ __forceinline__ void report(int32_t* status, int32_t code) {
  if (status != nullptr) atomicCAS(status, 0, code);
}

__device__ __forceinline__ uint64_t globaltimer() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint32_t bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(bar), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint32_t bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(bar) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint32_t bar, uint32_t bytes) {
  asm volatile("mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;" ::"r"(bar), "r"(bytes) : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n .reg .pred p;\n mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n selp.u32 %0, 1, 0, p;\n}\n"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait for the phase of parity `parity` to complete.  Gives up when `abort`
// (a CTA-wide shared flag) is raised by another role, or after `limit_ns`;
// in the latter case it raises the flag and reports DSA_ERR_TIMEOUT.
// Returns true when the phase completed.
__device__ __forceinline__ bool mbar_wait(uint32_t bar, uint32_t parity, volatile int* abort, int32_t* status,
                                          uint64_t limit_ns = kWaitLimitNs) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0) {
      if (*abort) return false;
      if (globaltimer() - t0 > limit_ns) {
        *abort = 1;
        report(status, DSA_ERR_TIMEOUT);
        return false;
      }
    }
  }
}

// Wait for a phase without looking at the abort flag: used when draining
// copies or MMAs already in flight before a CTA exits or frees TMEM, which
// must happen even after another role gave up.  Bounded by `limit_ns`.
__device__ __forceinline__ bool mbar_wait_drain(uint32_t bar, uint32_t parity, uint64_t limit_ns) {
  if (mbar_try_wait(bar, parity)) return true;
  const uint64_t t0 = globaltimer();
  for (uint32_t it = 1;; ++it) {
    if (mbar_try_wait(bar, parity)) return true;
    if ((it & 31u) == 0 && globaltimer() - t0 > limit_ns) return false;
  }
}

// ---------------------------------------------------------------- programmatic dependent launch
// A kernel launched with programmatic stream serialization may start while the
// previous kernel in the stream is still running; grid_dep_wait() blocks until
// that kernel has completed and its memory is visible (it returns at once for
// an ordinary launch).  grid_dep_launch() lets this grid's dependent launch as
// soon as every CTA of this grid has issued it.
__device__ __forceinline__ void grid_dep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void grid_dep_launch() { asm volatile("griddepcontrol.launch_dependents;" ::: "memory"); }

// ---------------------------------------------------------------- copies
__device__ __forceinline__ void prefetch_tmap(const void* map) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(map) : "memory");
}
__device__ __forceinline__ void tma_load_2d(uint32_t dst, const void* map, int c0, int c1, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3}], [%4];"
      ::"r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(bar)
      : "memory");
}
__device__ __forceinline__ void tma_load_3d(uint32_t dst, const void* map, int c0, int c1, int c2, uint32_t bar) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes [%0], [%1, {%2, %3, %4}], [%5];"
      ::"r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(bar)
      : "memory");
}
// L2 cache policies: streamed-once data (evict first) and data read again
// soon by the next kernel (evict last).
__device__ __forceinline__ uint64_t policy_evict_first() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ uint64_t policy_evict_last() {
  uint64_t p;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(p));
  return p;
}
__device__ __forceinline__ void tma_load_3d_hint(uint32_t dst, const void* map, int c0, int c1, int c2, uint32_t bar,
                                                 uint64_t policy) {
  asm volatile(
      "cp.async.bulk.tensor.3d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%2, %3, %4}], [%5], %6;"
      ::"r"(dst), "l"(map), "r"(c0), "r"(c1), "r"(c2), "r"(bar), "l"(policy)
      : "memory");
}
__device__ __forceinline__ void st_global_hint(float* addr, float v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.f32 [%0], %1, %2;" ::"l"(addr), "f"(v), "l"(policy) : "memory");
}
__device__ __forceinline__ void st_global_hint(uint16_t* addr, uint16_t v, uint64_t policy) {
  asm volatile("st.global.L2::cache_hint.b16 [%0], %1, %2;" ::"l"(addr), "h"(v), "l"(policy) : "memory");
}
// Plain bulk copy; both addresses 16-byte aligned, bytes a multiple of 16.
__device__ __forceinline__ void bulk_load(uint32_t dst, const void* src, uint32_t bytes, uint32_t bar) {
  asm volatile("cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%3];"
               ::"r"(dst), "l"(src), "r"(bytes), "r"(bar)
               : "memory");
}
// Asks L2 to fetch [src, src + bytes) (16-byte aligned, a multiple of 16 bytes)
// without waiting for it.
__device__ __forceinline__ void prefetch_l2(const void* src, uint32_t bytes) {
  asm volatile("cp.async.bulk.prefetch.L2.global [%0], %1;" ::"l"(src), "r"(bytes) : "memory");
}
// Make this thread's generic-proxy shared-memory writes visible to the async
// proxy (tensor core / TMA) before signalling the consumer.
__device__ __forceinline__ void fence_proxy_async_smem() {
  asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
}

// ---------------------------------------------------------------- tcgen05
__device__ __forceinline__ void tmem_alloc(uint32_t dst_smem, uint32_t ncols) {
  asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(dst_smem), "r"(ncols)
               : "memory");
}
__device__ __forceinline__ void tmem_relinquish() {
  asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}
// D[tmem] (+)= A[smem] * B[smem]; 8-bit (E4M3/E5M2/...) operands.
__device__ __forceinline__ void mma_f8f6f4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, p;\n}\n"
      ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[smem] * B[smem]; 16-bit (bf16 or f16, both the same) operands.
__device__ __forceinline__ void mma_bf16(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, p;\n}\n"
      ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= A[tmem] * B[smem]; 16-bit operands.  A (K-major) sits in TMEM:
// lane = row, each 32-bit column two consecutive K elements (low half first).
__device__ __forceinline__ void mma_bf16_tmem_a(uint32_t d, uint32_t a_tmem, uint64_t b, uint32_t idesc,
                                                uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %4, 0;\n"
      " tcgen05.mma.cta_group::1.kind::f16 [%0], [%1], %2, %3, p;\n}\n"
      ::"r"(d), "r"(a_tmem), "l"(b), "r"(idesc), "r"(accumulate)
      : "memory");
}
// D[tmem] (+)= (A * B) with MX block scaling: per 32-element K block, A row m
// is scaled by 2^(E - 127) with E the byte `sf_id` (instruction descriptor
// bits [29,31)) of the TMEM word at lane m % 32, column sfa + m / 32; B
// likewise from `sfb` (descriptor bits [4,6)).  A and B: E2M1 (unpacked byte
// containers), E4M3, ...; fp32 accumulator.
__device__ __forceinline__ void mma_mxf8f6f4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                             uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf8f6f4.block_scale [%0], %1, %2, %3, [%4], [%5], p;\n}\n"
      ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}
// The same with packed E2M1 operands on both sides (kind::mxf4, K = 64 per
// instruction, two E8M0 scales per row: bytes sf_id and sf_id + 1 of the
// scale word, sf_id 0 or 2).
__device__ __forceinline__ void mma_mxf4(uint32_t d, uint64_t a, uint64_t b, uint32_t idesc, uint32_t sfa,
                                         uint32_t sfb, uint32_t accumulate) {
  asm volatile(
      "{\n .reg .pred p;\n setp.ne.b32 p, %6, 0;\n"
      " tcgen05.mma.cta_group::1.kind::mxf4.block_scale.scale_vec::2X [%0], %1, %2, %3, [%4], [%5], p;\n}\n"
      ::"r"(d), "l"(a), "l"(b), "r"(idesc), "r"(sfa), "r"(sfb), "r"(accumulate)
      : "memory");
}
// Arrive once on `bar` when every tcgen05.mma issued so far by this thread completes.
__device__ __forceinline__ void mma_commit(uint32_t bar) {
  asm volatile("tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];" ::"r"(bar) : "memory");
}

#define DSA_R32(r)                                                                                          \
  "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]), "=r"(r[8]), \
      "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15]), "=r"(r[16]),   \
      "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]), "=r"(r[22]), "=r"(r[23]), "=r"(r[24]),  \
      "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]), "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
#define DSA_W32(r)                                                                                        \
  "r"(r[0]), "r"(r[1]), "r"(r[2]), "r"(r[3]), "r"(r[4]), "r"(r[5]), "r"(r[6]), "r"(r[7]), "r"(r[8]),      \
      "r"(r[9]), "r"(r[10]), "r"(r[11]), "r"(r[12]), "r"(r[13]), "r"(r[14]), "r"(r[15]), "r"(r[16]),       \
      "r"(r[17]), "r"(r[18]), "r"(r[19]), "r"(r[20]), "r"(r[21]), "r"(r[22]), "r"(r[23]), "r"(r[24]),      \
      "r"(r[25]), "r"(r[26]), "r"(r[27]), "r"(r[28]), "r"(r[29]), "r"(r[30]), "r"(r[31])

// 32 consecutive 32-bit TMEM columns of this thread's lane (warp-collective;
// a warp may only touch lanes 32*(warp%4) .. +31).
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,"
      "%16,%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31}, [%32];"
      : DSA_R32(r)
      : "r"(taddr));
}
// 16 consecutive 32-bit TMEM columns of this thread's lane (warp-collective).
__device__ __forceinline__ void tmem_ld16(uint32_t taddr, uint32_t* r) {
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x16.b32 {%0,%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15}, [%16];"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]), "=r"(r[15])
      : "r"(taddr));
}
__device__ __forceinline__ void tmem_st32(uint32_t taddr, const uint32_t (&r)[32]) {
  asm volatile(
      "tcgen05.st.sync.aligned.32x32b.x32.b32 [%0], {%1,%2,%3,%4,%5,%6,%7,%8,%9,%10,%11,%12,%13,%14,%15,%16,"
      "%17,%18,%19,%20,%21,%22,%23,%24,%25,%26,%27,%28,%29,%30,%31,%32};" ::"r"(taddr),
      DSA_W32(r)
      : "memory");
}
// One 32-bit TMEM column of this thread's lane (warp-collective).
__device__ __forceinline__ void tmem_st1(uint32_t taddr, uint32_t v) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x1.b32 [%0], {%1};" ::"r"(taddr), "r"(v) : "memory");
}
// Four consecutive 32-bit TMEM columns of this thread's lane (warp-collective).
__device__ __forceinline__ void tmem_st4(uint32_t taddr, uint32_t v0, uint32_t v1, uint32_t v2, uint32_t v3) {
  asm volatile("tcgen05.st.sync.aligned.32x32b.x4.b32 [%0], {%1, %2, %3, %4};" ::"r"(taddr), "r"(v0), "r"(v1),
               "r"(v2), "r"(v3)
               : "memory");
}
__device__ __forceinline__ void tmem_ld_wait() { asm volatile("tcgen05.wait::ld.sync.aligned;" ::: "memory"); }
__device__ __forceinline__ void tmem_st_wait() { asm volatile("tcgen05.wait::st.sync.aligned;" ::: "memory"); }

// ---------------------------------------------------------------- descriptors
// Shared-memory matrix descriptor of tcgen05: start address >> 4 in bits
// [0,14), leading-dimension byte offset >> 4 in [16,30), stride-dimension byte
// offset >> 4 in [32,46), descriptor version 1 in [46,48), base offset 0,
// layout (swizzle) in [61,64).
enum : uint64_t { kLayoutNone = 0, kLayoutSw128 = 2, kLayoutSw64 = 4, kLayoutSw32 = 6 };

__device__ __forceinline__ uint64_t smem_desc(uint32_t addr, uint32_t lbo, uint32_t sbo, uint64_t layout) {
  return static_cast<uint64_t>((addr & 0x3FFFFu) >> 4) | (static_cast<uint64_t>((lbo >> 4) & 0x3FFFu) << 16) |
         (static_cast<uint64_t>((sbo >> 4) & 0x3FFFu) << 32) | (1ull << 46) | (layout << 61);
}

// A descriptor from its two 32-bit words.
__device__ __forceinline__ uint64_t desc64(uint32_t lo, uint32_t hi) { return ((uint64_t)hi << 32) | lo; }

// Instruction descriptor (kind::f16 and kind::f8f6f4): fp32 accumulator,
// operand formats, K-major (0) / MN-major (1) per operand, N >> 3, M >> 4.
enum : uint32_t { kFmtE4M3 = 0, kFmtE2M1 = 5, kFmtBF16 = 1 };
// E2M1 in the operand-format field of kind::mxf4 (the only format of that kind)
constexpr uint32_t kFmtMxf4E2M1 = 1;
// Instruction descriptor of kind::mxf8f6f4.block_scale (fp32 accumulator
// implied): operand formats, K-major operands, N >> 3, E8M0 scale type (bit
// 23), M >> 4; the per-MMA scale-factor byte ids are ORed in with mx_sf_ids.
__host__ __device__ constexpr uint32_t make_idesc_mx(uint32_t a_fmt, uint32_t b_fmt, uint32_t M, uint32_t N) {
  return (a_fmt << 7) | (b_fmt << 10) | ((N >> 3) << 17) | (1u << 23) | ((M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t mx_sf_ids(uint32_t sfa_id, uint32_t sfb_id) {
  return (sfa_id << 29) | (sfb_id << 4);
}
__host__ __device__ constexpr uint32_t make_idesc(uint32_t a_fmt, uint32_t b_fmt, uint32_t a_mn, uint32_t b_mn,
                                                  uint32_t M, uint32_t N) {
  return (1u << 4) | (a_fmt << 7) | (b_fmt << 10) | (a_mn << 15) | (b_mn << 16) | ((N >> 3) << 17) |
         ((M >> 4) << 24);
}

// Byte offset inside a swizzled region: the 16-byte chunk index (bits 4..6)
// is XORed with address bits 7..9 (128B), 7..8 (64B) or 7 (32B).  `off` is
// relative to a base aligned to the pattern (1024 / 512 / 256 bytes).
__device__ __forceinline__ uint32_t swz128(uint32_t off) { return off ^ (((off >> 7) & 7u) << 4); }
__device__ __forceinline__ uint32_t swz64(uint32_t off) { return off ^ (((off >> 7) & 3u) << 4); }

// ---------------------------------------------------------------- numerics
// Order-preserving key of an fp32 score: larger score -> larger key; -0 is
// folded into +0; NaN maps to 0 (below every number).
__device__ __forceinline__ uint32_t score_key(float s) {
  uint32_t u = __float_as_uint(s);
  if ((u & 0x7FFFFFFFu) > 0x7F800000u) return 0u;
  if (u == 0x80000000u) u = 0u;
  return (u & 0x80000000u) ? ~u : (u | 0x80000000u);
}

// Four E4M3 bytes -> four bf16, exactly, on full-rate pipes.  An E4M3 value
// S.EEEE.MMM equals the bf16 with the same sign, exponent field EEEE and
// mantissa MMM0000 times 2^120, for normal and subnormal codes alike (the
// bf16 of a zero exponent field is the subnormal 0.MMM * 2^-126); the
// product is exact.  The NaN codes 0x7F / 0xFF are not special-cased.
// lo = elements 0 and 1, hi = elements 2 and 3 (low half = lower element).
__device__ __forceinline__ void e4m3x4_to_bf16x4(uint32_t w, uint32_t& lo, uint32_t& hi) {
  const uint32_t x0 = __byte_perm(w, 0u, 0x4140);  // [0, b1, 0, b0] as 16-bit lanes
  const uint32_t x1 = __byte_perm(w, 0u, 0x4342);  // [0, b3, 0, b2]
  // magnitude bits 6..0 -> 10..4 and sign bit 7 -> 15 of each 16-bit lane (one LOP3 each)
  const uint32_t f0 = ((x0 << 4) & 0x07F007F0u) | ((x0 << 8) & 0x80008000u);
  const uint32_t f1 = ((x1 << 4) & 0x07F007F0u) | ((x1 << 8) & 0x80008000u);
  const uint32_t k2_120 = 0x7B807B80u;  // bf16 2^120 in both halves
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(lo) : "r"(f0), "r"(k2_120));
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(hi) : "r"(f1), "r"(k2_120));
}

// 16 E2M1 codes (w0, w1: element 2i in the low nibble of byte i) times one
// E4M3 block scale -> 16 bf16 (o[j]: elements 2j, 2j + 1), exactly: an E2M1
// value has 2 significant bits and an E4M3 scale 4, so the product fits
// bf16's 8.  Each nibble's exponent and mantissa bits go to bf16's lowest
// exponent bits and top mantissa bit, so the bf16 reads 2^-126 times the E2M1
// value (E2M1's zero exponent lands on bf16 subnormals the same way); one
// multiply by 2^126 and one by the scale (itself widened as E4M3 is above).
__device__ __forceinline__ void nvfp4x16_to_bf16x16(uint32_t w0, uint32_t w1, uint32_t scale_byte,
                                                    uint32_t (&o)[8]) {
  const uint32_t sx = scale_byte * 0x00010001u;
  const uint32_t sf = ((sx << 4) & 0x07F007F0u) | ((sx << 8) & 0x80008000u);
  uint32_t s2;
  asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(s2) : "r"(sf), "r"(0x7B807B80u));  // 2^120: E4M3's bias
#pragma unroll
  for (int j = 0; j < 8; ++j) {
    const uint32_t byte = ((j < 4 ? w0 : w1) >> (8 * (j & 3))) & 0xFFu;
    const uint32_t y = (byte & 0x0Fu) | ((byte & 0xF0u) << 12);  // the two nibbles in the two 16-bit lanes
    const uint32_t f = ((y << 6) & 0x01C001C0u) | ((y << 12) & 0x80008000u);
    uint32_t v;
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(v) : "r"(f), "r"(0x7E807E80u));  // 2^126
    asm("mul.rn.bf16x2 %0, %1, %2;" : "=r"(o[j]) : "r"(v), "r"(s2));
  }
}

// Two E4M3 bytes (low byte = first element) -> two bf16 (low half = first).
__device__ __forceinline__ uint32_t e4m3x2_to_bf16x2(uint16_t v) {
  __half2_raw h = __nv_cvt_fp8x2_to_halfraw2(static_cast<__nv_fp8x2_storage_t>(v), __NV_E4M3);
  float2 f = __half22float2(*reinterpret_cast<__half2*>(&h));
  __nv_bfloat162 b = __floats2bfloat162_rn(f.x, f.y);
  return *reinterpret_cast<uint32_t*>(&b);
}

__device__ __forceinline__ int visible_len(int L, int nq, int j) {
  int v = L - (nq - 1) + j;
  return v < 0 ? 0 : v;
}

}  // namespace dsa
