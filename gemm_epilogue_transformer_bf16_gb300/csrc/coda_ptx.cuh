// Inline-PTX wrappers for sm_103a: mbarrier (with bounded waits), TMA tile
// loads, tcgen05 (TMEM allocation, UMMA issue/commit, TMEM loads) and the
// shared-memory / instruction descriptors the UMMA reads.
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>

#include "coda_status.h"

namespace coda {

__device__ __forceinline__ uint32_t smem_u32(const void* p) {
  return static_cast<uint32_t>(__cvta_generic_to_shared(p));
}

__device__ __forceinline__ uint64_t globaltimer_ns() {
  uint64_t t;
  asm volatile("mov.u64 %0, %%globaltimer;" : "=l"(t));
  return t;
}

// ---------------------------------------------------------------- mbarrier
__device__ __forceinline__ void mbar_init(uint64_t* bar, uint32_t count) {
  asm volatile("mbarrier.init.shared::cta.b64 [%0], %1;" ::"r"(smem_u32(bar)), "r"(count) : "memory");
}
__device__ __forceinline__ void fence_mbar_init() {
  asm volatile("fence.mbarrier_init.release.cluster;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive(uint64_t* bar) {
  asm volatile("mbarrier.arrive.shared::cta.b64 _, [%0];" ::"r"(smem_u32(bar)) : "memory");
}
__device__ __forceinline__ void mbar_arrive_expect_tx(uint64_t* bar, uint32_t bytes, uint32_t p) {
  asm volatile(
      "{\n\t.reg .pred P;\n\tsetp.ne.b32 P, %2, 0;\n\t"
      "@P mbarrier.arrive.expect_tx.shared::cta.b64 _, [%0], %1;\n\t}" ::"r"(smem_u32(bar)), "r"(bytes), "r"(p)
      : "memory");
}
__device__ __forceinline__ bool mbar_try_wait(uint32_t bar, uint32_t parity) {
  uint32_t ok;
  asm volatile(
      "{\n\t.reg .pred p;\n\t"
      "mbarrier.try_wait.parity.shared::cta.b64 p, [%1], %2;\n\t"
      "selp.u32 %0, 1, 0, p;\n\t}"
      : "=r"(ok)
      : "r"(bar), "r"(parity)
      : "memory");
  return ok != 0;
}

// Wait until the phase with the given parity of `bar` has completed.  The
// wait is bounded: it gives up when `*abort` becomes non-zero (another role
// of the CTA gave up) or after `limit_ns` of wall time, in which case it sets
// `*abort`, records CODA_DEV_TIMEOUT in the status word and returns false.
__device__ __forceinline__ bool mbar_wait_bounded(uint64_t* bar, uint32_t parity, volatile int* abort,
                                                  int* status, uint64_t limit_ns, uint32_t sleep_ns = 0) {
  const uint32_t b = smem_u32(bar);
  if (mbar_try_wait(b, parity)) return true;
  const uint64_t t0 = globaltimer_ns();
  while (true) {
#pragma unroll 1
    for (int i = 0; i < 32; ++i) {
      if (mbar_try_wait(b, parity)) return true;
      if (sleep_ns) __nanosleep(sleep_ns);  // a waiter with slack backs off
    }
    if (*abort) return false;
    if (globaltimer_ns() - t0 > limit_ns) {
      *abort = 1;
      if (status) atomicOr(status, CODA_DEV_TIMEOUT);
      return false;
    }
  }
}

// Same, but ignores the abort flag (used while draining in-flight copies).
__device__ __forceinline__ bool mbar_wait_drain(uint64_t* bar, uint32_t parity, uint64_t limit_ns) {
  const uint32_t b = smem_u32(bar);
  const uint64_t t0 = globaltimer_ns();
  while (!mbar_try_wait(b, parity)) {
    if (globaltimer_ns() - t0 > limit_ns) return false;
  }
  return true;
}

// ---------------------------------------------------------------- TMA
__device__ __forceinline__ void tma_prefetch_desc(const CUtensorMap* m) {
  asm volatile("prefetch.tensormap [%0];" ::"l"(reinterpret_cast<uint64_t>(m)) : "memory");
}

// 2-D tiled bulk tensor copy global -> shared, completion counted in bytes
// on `bar`.  x is the innermost (contiguous) coordinate in elements.
// The copy and MMA helpers below take an issue predicate `p`: the whole warp
// executes them with the same (warp-uniform) operands and only the lane with
// p != 0 issues the instruction (see elect_one), so the operands stay in
// uniform registers and the loop around them runs without divergence.
__device__ __forceinline__ void tma_load_2d(void* dst, const CUtensorMap* m, uint64_t* bar, int x, int y,
                                            uint32_t p) {
  asm volatile(
      "{\n\t.reg .pred P;\n\tsetp.ne.b32 P, %5, 0;\n\t"
      "@P cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes"
      " [%0], [%1, {%3, %4}], [%2];\n\t}" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(p)
      : "memory");
}

// L2 eviction-priority policies for the TMA loads below.
// Untiled bulk copy global -> shared (16-byte aligned, size a multiple of
// 16), completion counted in bytes on `bar`; issued when p != 0.
__device__ __forceinline__ void bulk_load(void* dst, const void* src, uint32_t bytes, uint64_t* bar, uint32_t p) {
  asm volatile(
      "{\n\t.reg .pred P;\n\tsetp.ne.b32 P, %3, 0;\n\t"
      "@P cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes [%0], [%1], %2, [%4];\n\t}" ::"r"(
          smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(p), "r"(smem_u32(bar))
      : "memory");
}

__device__ __forceinline__ uint64_t l2_policy_evict_last() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_last.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}
__device__ __forceinline__ uint64_t l2_policy_evict_first() {
  uint64_t pol;
  asm volatile("createpolicy.fractional.L2::evict_first.b64 %0, 1.0;" : "=l"(pol));
  return pol;
}

// Same as tma_load_2d with an L2 cache-eviction policy.
__device__ __forceinline__ void tma_load_2d_hint(void* dst, const CUtensorMap* m, uint64_t* bar, int x, int y,
                                                 uint64_t policy, uint32_t p) {
  asm volatile(
      "{\n\t.reg .pred P;\n\tsetp.ne.b32 P, %6, 0;\n\t"
      "@P cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.L2::cache_hint"
      " [%0], [%1, {%3, %4}], [%2], %5;\n\t}" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y), "l"(policy), "r"(p)
      : "memory");
}

// 2-D tiled copy for a CTA pair (cta_group::2): the data lands in this CTA's
// shared memory, the byte count is signalled on `bar_cluster`, a
// shared::cluster address that may name the peer CTA's mbarrier.
__device__ __forceinline__ void tma_load_2d_pair(void* dst, const CUtensorMap* m, uint32_t bar_cluster, int x, int y,
                                                 uint32_t p) {
  asm volatile(
      "{\n\t.reg .pred P;\n\tsetp.ne.b32 P, %5, 0;\n\t"
      "@P cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      " [%0], [%1, {%3, %4}], [%2];\n\t}" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(x), "r"(y), "r"(p)
      : "memory");
}

__device__ __forceinline__ void tma_load_2d_pair_hint(void* dst, const CUtensorMap* m, uint32_t bar_cluster, int x,
                                                      int y, uint64_t policy, uint32_t p) {
  asm volatile(
      "{\n\t.reg .pred P;\n\tsetp.ne.b32 P, %6, 0;\n\t"
      "@P cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.cta_group::2"
      ".L2::cache_hint [%0], [%1, {%3, %4}], [%2], %5;\n\t}" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(x), "r"(y), "l"(policy), "r"(p)
      : "memory");
}

// The same copy multicast to every CTA in `cta_mask` (same shared-memory
// offset in each).  With cta_group::2 the byte count of each destination is
// signalled on the mbarrier at `bar_cluster`'s offset in the even CTA of that
// destination's pair.
__device__ __forceinline__ void tma_load_2d_pair_mc(void* dst, const CUtensorMap* m, uint32_t bar_cluster, int x,
                                                    int y, uint16_t cta_mask, uint32_t p) {
  asm volatile(
      "{\n\t.reg .pred P;\n\tsetp.ne.b32 P, %6, 0;\n\t"
      "@P cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
      ".cta_group::2 [%0], [%1, {%3, %4}], [%2], %5;\n\t}" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(bar_cluster), "r"(x), "r"(y), "h"(cta_mask), "r"(p)
      : "memory");
}

// 1 in exactly one active lane of the warp, 0 in the others.
__device__ __forceinline__ uint32_t elect_one() {
  uint32_t e;
  asm volatile(
      "{\n\t.reg .pred P;\n\telect.sync _|P, 0xffffffff;\n\tselp.u32 %0, 1, 0, P;\n\t}"
      : "=r"(e));
  return e;
}

// ---------------------------------------------------------------- programmatic dependent launch
// A kernel launched with programmatic stream serialization may start while
// the previous kernel in its stream is still running; griddep_wait blocks
// until that kernel has completed and its memory operations are visible, so
// it must precede every global-memory access of such a kernel.
// griddep_launch_dependents lets the next such kernel start its own
// prologue early (it still waits for this one to complete).
__device__ __forceinline__ void griddep_wait() { asm volatile("griddepcontrol.wait;" ::: "memory"); }
__device__ __forceinline__ void griddep_launch_dependents() {
  asm volatile("griddepcontrol.launch_dependents;" ::: "memory");
}

// ---------------------------------------------------------------- clusters
__device__ __forceinline__ uint32_t cluster_ctarank() {
  uint32_t r;
  asm volatile("mov.u32 %0, %%cluster_ctarank;" : "=r"(r));
  return r;
}
// shared::cluster address of the variable at `p` (this CTA's layout) in CTA `rank`.
__device__ __forceinline__ uint32_t mapa_shared(const void* p, uint32_t rank) {
  uint32_t r;
  asm volatile("mapa.shared::cluster.u32 %0, %1, %2;" : "=r"(r) : "r"(smem_u32(p)), "r"(rank));
  return r;
}
__device__ __forceinline__ void cluster_sync() {
  asm volatile("barrier.cluster.arrive.release;\n\tbarrier.cluster.wait.acquire;" ::: "memory");
}
__device__ __forceinline__ void mbar_arrive_cluster(uint32_t bar_cluster) {
  asm volatile("mbarrier.arrive.release.cluster.shared::cluster.b64 _, [%0];" ::"r"(bar_cluster) : "memory");
}

// ---------------------------------------------------------------- tcgen05
// PAIR = true: the cta_group::2 forms, executed by both CTAs of a pair.
template <bool PAIR>
__device__ __forceinline__ void tmem_alloc(uint32_t* slot, uint32_t ncols) {
  if constexpr (PAIR)
    asm volatile("tcgen05.alloc.cta_group::2.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
  else
    asm volatile("tcgen05.alloc.cta_group::1.sync.aligned.shared::cta.b32 [%0], %1;" ::"r"(smem_u32(slot)),
                 "r"(ncols)
                 : "memory");
}
template <bool PAIR>
__device__ __forceinline__ void tmem_relinquish() {
  if constexpr (PAIR)
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::2.sync.aligned;" ::: "memory");
  else
    asm volatile("tcgen05.relinquish_alloc_permit.cta_group::1.sync.aligned;" ::: "memory");
}
template <bool PAIR>
__device__ __forceinline__ void tmem_dealloc(uint32_t taddr, uint32_t ncols) {
  if constexpr (PAIR)
    asm volatile("tcgen05.dealloc.cta_group::2.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
  else
    asm volatile("tcgen05.dealloc.cta_group::1.sync.aligned.b32 %0, %1;" ::"r"(taddr), "r"(ncols) : "memory");
}
__device__ __forceinline__ void tc_fence_before() {
  asm volatile("tcgen05.fence::before_thread_sync;" ::: "memory");
}
__device__ __forceinline__ void tc_fence_after() {
  asm volatile("tcgen05.fence::after_thread_sync;" ::: "memory");
}

// D[tmem] (+)= A[smem] * B[smem]^T, bf16 inputs, fp32 accumulator, issued by
// one thread.
__device__ __forceinline__ void umma_bf16(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                          uint32_t accumulate, uint32_t p) {
  asm volatile(
      "{\n\t.reg .pred A, P;\n\t"
      "setp.ne.b32 A, %4, 0;\n\t"
      "setp.ne.b32 P, %5, 0;\n\t"
      "@P tcgen05.mma.cta_group::1.kind::f16 [%0], %1, %2, %3, A;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(p)
      : "memory");
}

// D[tmem] (+)= A * B^T over a CTA pair: M = 256 (128 rows of A in each CTA's
// shared memory at the same offset), B split along N between the two CTAs,
// each CTA's TMEM receiving its own 128 rows.  Issued by one thread of the
// even CTA.
__device__ __forceinline__ void umma_bf16_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                               uint32_t accumulate, uint32_t p) {
  asm volatile(
      "{\n\t.reg .pred A, P;\n\t"
      "setp.ne.b32 A, %4, 0;\n\t"
      "setp.ne.b32 P, %5, 0;\n\t"
      "@P tcgen05.mma.cta_group::2.kind::f16 [%0], %1, %2, %3, A;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(p)
      : "memory");
}

// The same with e4m3 operands (kind::f8f6f4, K = 32 elements per
// instruction = the same 32 bytes as a bf16 K = 16 step).
__device__ __forceinline__ void umma_f8(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                        uint32_t accumulate, uint32_t p) {
  asm volatile(
      "{\n\t.reg .pred A, P;\n\t"
      "setp.ne.b32 A, %4, 0;\n\t"
      "setp.ne.b32 P, %5, 0;\n\t"
      "@P tcgen05.mma.cta_group::1.kind::f8f6f4 [%0], %1, %2, %3, A;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(p)
      : "memory");
}
__device__ __forceinline__ void umma_f8_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                             uint32_t accumulate, uint32_t p) {
  asm volatile(
      "{\n\t.reg .pred A, P;\n\t"
      "setp.ne.b32 A, %4, 0;\n\t"
      "setp.ne.b32 P, %5, 0;\n\t"
      "@P tcgen05.mma.cta_group::2.kind::f8f6f4 [%0], %1, %2, %3, A;\n\t}" ::"r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(accumulate), "r"(p)
      : "memory");
}

// Arrive on `bar` once every tcgen05 operation issued so far by this thread
// has completed.
__device__ __forceinline__ void umma_commit(uint64_t* bar, uint32_t p) {
  asm volatile(
      "{\n\t.reg .pred P;\n\tsetp.ne.b32 P, %1, 0;\n\t"
      "@P tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar)),
      "r"(p)
      : "memory");
}
// CTA-pair form: arrive on the mbarrier at `bar`'s offset in every CTA of
// `cta_mask`.
__device__ __forceinline__ void umma_commit_pair_mc(uint64_t* bar, uint16_t cta_mask, uint32_t p) {
  asm volatile(
      "{\n\t.reg .pred P;\n\tsetp.ne.b32 P, %2, 0;\n\t"
      "@P tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}"
      ::"r"(smem_u32(bar)), "h"(cta_mask), "r"(p)
      : "memory");
}
__device__ __forceinline__ void umma_commit_pair(uint64_t* bar, uint32_t p) {
  asm volatile(
      "{\n\t.reg .pred P;\n\tsetp.ne.b32 P, %1, 0;\n\t"
      "@P tcgen05.commit.cta_group::2.mbarrier::arrive::one.shared::cluster.b64 [%0];\n\t}" ::"r"(smem_u32(bar)),
      "r"(p)
      : "memory");
}

// 32 consecutive fp32 columns of one TMEM lane per thread (warp w reads lanes
// 32*(w%4) .. 32*(w%4)+31).  The wait is fused so the registers are valid on
// return.
__device__ __forceinline__ void tmem_ld32(uint32_t taddr, float (&v)[32]) {
  uint32_t r[32];
  asm volatile(
      "tcgen05.ld.sync.aligned.32x32b.x32.b32 "
      "{%0, %1, %2, %3, %4, %5, %6, %7, %8, %9, %10, %11, %12, %13, %14, %15, "
      "%16, %17, %18, %19, %20, %21, %22, %23, %24, %25, %26, %27, %28, %29, %30, %31}, [%32];\n\t"
      "tcgen05.wait::ld.sync.aligned;"
      : "=r"(r[0]), "=r"(r[1]), "=r"(r[2]), "=r"(r[3]), "=r"(r[4]), "=r"(r[5]), "=r"(r[6]), "=r"(r[7]),
        "=r"(r[8]), "=r"(r[9]), "=r"(r[10]), "=r"(r[11]), "=r"(r[12]), "=r"(r[13]), "=r"(r[14]),
        "=r"(r[15]), "=r"(r[16]), "=r"(r[17]), "=r"(r[18]), "=r"(r[19]), "=r"(r[20]), "=r"(r[21]),
        "=r"(r[22]), "=r"(r[23]), "=r"(r[24]), "=r"(r[25]), "=r"(r[26]), "=r"(r[27]), "=r"(r[28]),
        "=r"(r[29]), "=r"(r[30]), "=r"(r[31])
      : "r"(taddr)
      : "memory");
#pragma unroll
  for (int i = 0; i < 32; ++i) v[i] = __uint_as_float(r[i]);
}

// ---------------------------------------------------------------- descriptors
// Shared-memory matrix descriptor (sm_100 family layout): start address,
// leading-dimension byte offset, stride-dimension byte offset (all >> 4),
// descriptor version 1 at bits 46-47, 128-byte swizzle (layout type 2) at
// bits 61-63.  Tiles start on 1024-byte boundaries so the base offset is 0.
__device__ __forceinline__ uint64_t sdesc_sw128(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  d |= static_cast<uint64_t>(2) << 61;
  return d;
}

// Instruction descriptor of tcgen05.mma kind::f16: fp32 accumulator (bits
// 4-5 = 1), A and B bf16 (bits 7-9 and 10-12 = 1), A/B major-ness (bit 15 /
// 16: 1 = MN-major), N>>3 at bits 17-22, M>>4 at bits 24-28.
// kind::f8f6f4 with e4m3 A and B (type code 0 at bits 7-9 and 10-12), fp32
// accumulator, K-major operands.
__host__ __device__ constexpr uint32_t idesc_e4m3(int M, int N) {
  return (1u << 4) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}
__host__ __device__ constexpr uint32_t idesc_bf16(int M, int N, int a_mn, int b_mn) {
  return (1u << 4) | (1u << 7) | (1u << 10) | (static_cast<uint32_t>(a_mn) << 15) |
         (static_cast<uint32_t>(b_mn) << 16) | (static_cast<uint32_t>(N >> 3) << 17) |
         (static_cast<uint32_t>(M >> 4) << 24);
}

// ---------------------------------------------------------------- misc
__device__ __forceinline__ uint32_t pack_bf16x2(float lo, float hi) {
  __nv_bfloat162 h = __floats2bfloat162_rn(lo, hi);
  return *reinterpret_cast<uint32_t*>(&h);
}
__device__ __forceinline__ float bf16_lo(uint32_t w) { return __uint_as_float(w << 16); }
__device__ __forceinline__ float bf16_hi(uint32_t w) { return __uint_as_float(w & 0xFFFF0000u); }

// Request the bytes [p, p + bytes) into L2 (a hint: nothing is returned and
// nothing waits on it).  One prefetch per 128-byte line, plus the line that
// holds the last byte when p is not line-aligned; every address issued lies
// inside the span.
__device__ __forceinline__ void prefetch_l2_span(const void* p, int bytes) {
  const char* c = static_cast<const char*>(p);
  for (int o = 0; o < bytes; o += 128) asm volatile("prefetch.global.L2 [%0];" ::"l"(c + o));
  if (bytes > 0) asm volatile("prefetch.global.L2 [%0];" ::"l"(c + bytes - 1));
}

// 8 bf16 packed in 16 bytes, widened to fp32.
__device__ __forceinline__ void bf16x8_to_f32(const uint4& q, float* out) {
  out[0] = bf16_lo(q.x); out[1] = bf16_hi(q.x);
  out[2] = bf16_lo(q.y); out[3] = bf16_hi(q.y);
  out[4] = bf16_lo(q.z); out[5] = bf16_hi(q.z);
  out[6] = bf16_lo(q.w); out[7] = bf16_hi(q.w);
}

// Load 8 consecutive bf16 (16 bytes) as fp32.
__device__ __forceinline__ void load_bf16x8(const __nv_bfloat16* p, float* out) {
  uint4 q = *reinterpret_cast<const uint4*>(p);
  out[0] = bf16_lo(q.x); out[1] = bf16_hi(q.x);
  out[2] = bf16_lo(q.y); out[3] = bf16_hi(q.y);
  out[4] = bf16_lo(q.z); out[5] = bf16_hi(q.z);
  out[6] = bf16_lo(q.w); out[7] = bf16_hi(q.w);
}
// Round 8 fp32 to bf16 (RNE) and store 16 bytes.
__device__ __forceinline__ void store_bf16x8(__nv_bfloat16* p, const float* v) {
  uint4 q;
  q.x = pack_bf16x2(v[0], v[1]);
  q.y = pack_bf16x2(v[2], v[3]);
  q.z = pack_bf16x2(v[4], v[5]);
  q.w = pack_bf16x2(v[6], v[7]);
  *reinterpret_cast<uint4*>(p) = q;
}
// Same, as a streaming store (.cs) when `stream` is set: an output tile is
// written once and need not displace the L2-resident operand panel.
__device__ __forceinline__ void store_bf16x8(__nv_bfloat16* p, const float* v, bool stream) {
  const uint32_t x = pack_bf16x2(v[0], v[1]), y = pack_bf16x2(v[2], v[3]);
  const uint32_t z = pack_bf16x2(v[4], v[5]), w = pack_bf16x2(v[6], v[7]);
  if (stream)
    asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(p), "r"(x), "r"(y), "r"(z), "r"(w)
                 : "memory");
  else
    *reinterpret_cast<uint4*>(p) = make_uint4(x, y, z, w);
}

}  // namespace coda
