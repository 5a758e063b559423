// Persistent, warp-specialised bf16 GEMM for sm_103a with a programmable
// epilogue.
//
//   D[m, n] = epilogue( sum_k A(m, k) * B(n, k) )   (fp32 accumulation)
//
// This is the fixed GEMM mainloop plus per-output-tile epilogue of "CODA:
// Rewriting Transformer Blocks as GEMM-Epilogue Programs" (§2.2 and §3.1: the
// epilogue sees one output tile, its accumulator and consistently-indexed
// auxiliary tensors).  The GB300 mapping:
//
//   warp 0        TMA producer: one elected thread streams A/B k-slices
//                 (64 bf16 = 128 bytes wide, 128-byte swizzle) into a
//                 STAGES-deep shared-memory ring, completion counted on
//                 per-stage mbarriers.
//   warp 1        TMEM owner and UMMA issuer: one thread issues
//                 tcgen05.mma (M=128, N=BN, K=16) into one of two TMEM
//                 accumulators, frees smem stages with tcgen05.commit and
//                 signals a finished accumulator to the epilogue.
//   warps 2..5    epilogue: tcgen05.ld of their 32-lane quarter of the
//                 accumulator (thread = output row), the epilogue functor's
//                 math, vectorised 16-byte global stores.  Two accumulators
//                 let the epilogue of tile i overlap the mainloop of tile i+1.
//
// Operands can be K-major (row-major [rows, K], the nn.Linear weight layout)
// or MN-major (row-major [K, rows]); backward GEMMs need both.  A second
// (A, B) descriptor pair continues the contraction (concatenated K), and a
// second B descriptor can fill the upper half of the tile's N (the SwiGLU
// gate/up pair).  Every wait is bounded: on expiry the CTA records
// CODA_DEV_TIMEOUT, drains its in-flight copies and MMAs, frees TMEM and
// returns.
#pragma once
#include <cstdint>
#include <type_traits>
#include <cuda.h>
#include <cuda_bf16.h>

#include "coda_ptx.cuh"

namespace coda {

constexpr int BM = 128;
constexpr int BK = 64;
constexpr int NUM_THREADS = 192;

// PAIR: a cluster of two CTAs on two SMs computes a 256 x BN tile with
// tcgen05.mma.cta_group::2; each CTA stages its own 128 rows of A and half of
// B (BN/2 rows), so a stage is 32 KB and six of them fit.
#ifndef CODA_PAIR_STAGES
#define CODA_PAIR_STAGES 6
#endif
// Epilogue ring: an epilogue that reads bf16 [M, N] tensors tile by tile
// (the residual) has them copied by TMA, 32 rows x 32 columns (2 KB, 64-byte
// swizzle) per copy, into RING_SLOTS slots per epilogue warp, issued before
// the tile's accumulator is ready and RING_SLOTS chunks ahead of the chunk
// being read.  RING = tensors per slot (0: no ring).
constexpr int RING_SLOTS = 3;
constexpr uint32_t RING_CHUNK_BYTES = 32 * 32 * 2;

template <int BN, bool PAIR = false, int RING = 0>
struct GemmCfg {
  static constexpr int B_ROWS = PAIR ? BN / 2 : BN;  // B rows staged by one CTA
  static constexpr uint32_t A_BYTES = BM * BK * 2;
  static constexpr uint32_t B_BYTES = B_ROWS * BK * 2;
  static constexpr uint32_t STAGE_BYTES = A_BYTES + B_BYTES;
  static constexpr uint32_t TMEM_COLS = 2 * BN;
  static constexpr uint32_t BAR_BYTES = 512;
  static constexpr uint32_t EPI_STAGE_BYTES = 4 * 2048;  // 2 KB store-transpose buffer per epilogue warp
  static constexpr uint32_t RING_BYTES = 4u * RING_SLOTS * RING_CHUNK_BYTES * RING;
  static constexpr int STAGES_WANT = PAIR ? CODA_PAIR_STAGES : (BN >= 256 ? 4 : 6);
  static constexpr int STAGES_FIT =
      static_cast<int>((232448u - 1024u - BAR_BYTES - EPI_STAGE_BYTES - RING_BYTES) / STAGE_BYTES);
  static constexpr int STAGES = STAGES_WANT < STAGES_FIT ? STAGES_WANT : STAGES_FIT;
  static constexpr uint32_t SMEM_BYTES = 1024 + STAGES * STAGE_BYTES + RING_BYTES + BAR_BYTES + EPI_STAGE_BYTES;
  static_assert(SMEM_BYTES <= 232448, "shared memory per CTA");
};

// Tensors an epilogue stages through the ring (Epi::RING, 0 if absent).
template <class E, class = void>
struct EpiRing {
  static constexpr int value = 0;
};
template <class E>
struct EpiRing<E, std::void_t<decltype(E::RING)>> {
  static constexpr int value = E::RING;
};

// Everything an epilogue may read or write.  Unused fields are null/zero.
struct EpiArgs {
  void* D;
  int64_t ldd;
  int d_f32;
  int beta;
  const float* row_scale;
  const float* col_scale;
  const __nv_bfloat16* aux0;
  int64_t ld_aux0;
  const __nv_bfloat16* aux1;
  int64_t ld_aux1;
  const float* row_coef;
  const int32_t* gather_rows;   // aux1 row read for output row i (skipped when < 0)
  const __nv_bfloat16* aux2;    // rows subtracted through the CSR below
  int64_t ld_aux2;
  const int32_t* csr_off;       // [M+1] per output row: range of csr_idx
  const int32_t* csr_idx;       // aux2 row indices
  const float* csr_w;           // weight of each aux2 row
  const float* row_scale2;      // SWIGLU: second per-row factor (FP8 token scale)
  const float* col_scale2;      // SWIGLU: per-column factor of the up half (col_scale: gate half); PLAIN: gamma of out1
  const float* row_coef2;       // PLAIN: D -= row_coef2_i * aux3[i, j]
  const __nv_bfloat16* aux3;
  int64_t ld_aux3;
  __nv_bfloat16* out1;
  int64_t ld_out1;
  __nv_bfloat16* out2;
  int64_t ld_out2;
  __nv_bfloat16* out3;
  int64_t ld_out3;
  float* partials;
  int64_t ld_part;
  // cross-entropy
  const int32_t* labels;
  int32_t ignore_index;
  const float* lse;
  const int32_t* n_valid;
  float dloss;
  int onehot;                   // CE_DLOGITS: include -w at the label column
  int st_stream;                // epilogue tile stores as streaming (.cs) stores
  int aux_prefetch;             // request the tile's auxiliary rows into L2 before its accumulator is ready
  int ring;                     // tensors the epilogue reads through the TMA ring (0: plain loads)
  int no_lean;                  // 1: the plain epilogue runs its general chunk loop (for comparisons)
  int mode;                     // SIGMOID: 0 forward, 1 backward on the recomputed logits
  float* target_logit;
  int64_t col_base;             // CE_DLOGITS: vocabulary column of the launch's column 0 (a vocabulary slice)
  int64_t n_total;              // CE_DLOGITS: vocabulary size (0: the launch's N)
  const float* acc_in;          // PLAIN (bf16 D): fp32 tile added to the result (a running sum over slices)
  int64_t ld_acc_in;
  // FP8 operands: the accumulator is acc * acc_rs[i] * acc_cs[j] (the two
  // operands' per-row scales) before any epilogue math; null = 1.  PLAIN and
  // SWIGLU take these scales through their row/column scale fields instead.
  const float* acc_rs;
  const float* acc_cs;
  // QK-RMSNorm + RoPE
  const int32_t* pos;
  const float2* cos_sin;
  int max_pos;
  int n_q;
  int n_kv;
  float eps;
  const float* gamma_q;
  const float* gamma_k;
  __nv_bfloat16* Q;
  __nv_bfloat16* Kh;
  __nv_bfloat16* V;
  int64_t ldq;
  int64_t ldk;
  int64_t ldv;
};

struct GemmArgs {
  int M, N;          // output rows / columns seen by the epilogue
  int num_m, num_n;  // tile grid
  int kb0, kb1;      // k-blocks of descriptor pair 0 and pair 1
  int a_mn, b_mn;    // operand major-ness (1 = MN-major)
  int b_dual;        // B tile = [B0 rows | B1 rows], BN/2 each
  int n_per_unit;    // consecutive N tiles handled as one unit (running state)
  int num_units;
  int group_m;       // raster: M blocks per group
  int nb_base;       // first N tile of this launch (a launch may cover a slice of N)
  uint32_t idesc;
  int* status;
  uint64_t timeout_ns;
  int l2_hints;                // bit 0: A loads evict_last, bit 1: B loads evict_first
  uint32_t producer_sleep_ns;  // back-off of the producer's and the epilogue's
  uint32_t epilogue_sleep_ns;  // barrier waits (0 = spin)
  EpiArgs e;
  // host side only (the kernel ignores them)
  int max_clusters;     // > 0: launch at most this many clusters
  int* query_clusters;  // non-null: report the resident-cluster limit and launch nothing
};

struct TileInfo {
  int mb, nb, unit_chunk;
  int row;          // global output row of this thread
  int M, N;
  uint32_t taddr;   // TMEM address of this warp's lane quarter, column 0
  int* status;
  uint8_t* stage;   // this warp's 2 KB shared-memory store-transpose buffer
  // epilogue ring (used when EpiArgs::ring is set)
  uint8_t* ring;            // this warp's RING_SLOTS slots
  uint64_t* ring_bar;       // one barrier per slot
  uint32_t* ring_cnt;       // [0] chunks issued, [1] chunks consumed (this warp's, in shared memory)
  const CUtensorMap* emap0; // first ring tensor
  const CUtensorMap* emap1; // second ring tensor
  volatile int* abort_flag;
  uint64_t timeout_ns;
};

// Ring chunk g (this warp's running chunk count) = columns [col, col + 32)
// of rows [row0, row0 + 32) of each ring tensor, into slot g % RING_SLOTS.
// Called by the whole warp with uniform arguments; lane 0 issues.  Rows and
// columns outside the tensor arrive as zeros.  The fence orders the warp's
// earlier reads of the slot (generic proxy) before the copy's writes.
__device__ __forceinline__ void ring_issue(const TileInfo& t, int ntens, uint32_t g, int col, int row0) {
  const int sl = static_cast<int>(g % RING_SLOTS);
  uint8_t* dst = t.ring + sl * ntens * RING_CHUNK_BYTES;
  const uint32_t l0 = (threadIdx.x & 31) == 0;
  if (l0) asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
  mbar_arrive_expect_tx(&t.ring_bar[sl], ntens * RING_CHUNK_BYTES, l0);
  tma_load_2d(dst, t.emap0, &t.ring_bar[sl], col, row0, l0);
  if (ntens > 1) tma_load_2d(dst + RING_CHUNK_BYTES, t.emap1, &t.ring_bar[sl], col, row0, l0);
}

// Wait for ring chunk g; warp-uniform result (false: timed out or aborted).
__device__ __forceinline__ bool ring_wait(const TileInfo& t, uint32_t g) {
  const bool ok = mbar_wait_bounded(&t.ring_bar[g % RING_SLOTS], (g / RING_SLOTS) & 1, t.abort_flag, t.status,
                                    t.timeout_ns);
  return __all_sync(0xffffffffu, ok);
}

// 16-byte piece p (columns 8p .. 8p + 7) of this lane's row in tensor `k` of
// slot g % RING_SLOTS (64-byte swizzle: piece p of row r at r * 64 + (p ^ ((r >> 1) & 3)) * 16).
__device__ __forceinline__ uint4 ring_read(const TileInfo& t, int ntens, uint32_t g, int k, int p) {
  const int r = threadIdx.x & 31;
  const uint8_t* slot = t.ring + static_cast<int>(g % RING_SLOTS) * ntens * RING_CHUNK_BYTES + k * RING_CHUNK_BYTES;
  return *reinterpret_cast<const uint4*>(slot + r * 64 + ((p ^ ((r >> 1) & 3)) * 16));
}

// Unit -> (m block, first n block, number of n blocks).
__device__ __forceinline__ void unit_coords(const GemmArgs& a, int u, int& mb, int& nb0, int& nlen, int& chunk) {
  if (a.n_per_unit <= 1) {
    const int per_group = a.group_m * a.num_n;
    const int g = u / per_group;
    const int first_m = g * a.group_m;
    const int gm = min(a.group_m, a.num_m - first_m);
    const int r = u - g * per_group;
    mb = first_m + r % gm;
    nb0 = a.nb_base + r / gm;
    nlen = 1;
    chunk = nb0;
  } else {
    chunk = u / a.num_m;
    mb = u - chunk * a.num_m;
    nb0 = chunk * a.n_per_unit;
    nlen = min(a.n_per_unit, a.num_n - nb0);
  }
}

// CG: CTAs per cluster.  1 = single CTAs (M = 128 tiles); 2 = a CTA pair
// (cta_group::2, M = 256); 4 = two CTA pairs on adjacent 256-row blocks that
// share the B tile: each CTA loads half of its B rows and multicasts them to
// the CTA at the same position in the other pair, so every SM stages 24 KB
// per k-slice instead of 32 KB.
// FP8: e4m3 operands, tcgen05.mma kind::f8f6f4, 128 elements per 128-byte
// k-slice (a compile-time variant, so the bf16 kernels hold only kind::f16).
template <int BN, class Epi, int CG, bool FP8 = false>
__global__ void __launch_bounds__(NUM_THREADS, 1)
    coda_gemm_kernel(const __grid_constant__ CUtensorMap mA0, const __grid_constant__ CUtensorMap mB0,
                     const __grid_constant__ CUtensorMap mA1, const __grid_constant__ CUtensorMap mB1,
                     const __grid_constant__ CUtensorMap mE0, const __grid_constant__ CUtensorMap mE1,
                     const GemmArgs args) {
  constexpr bool PAIR = CG >= 2;
  constexpr bool QUAD = CG == 4;
  static_assert(CG == 1 || CG == 2 || CG == 4, "cluster size");
  constexpr int RING = EpiRing<Epi>::value;
  using Cfg = GemmCfg<BN, PAIR, RING>;
  constexpr int S = Cfg::STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* tiles = smem;
  uint8_t* ring = smem + S * Cfg::STAGE_BYTES;  // 1024-byte aligned
  uint64_t* full = reinterpret_cast<uint64_t*>(ring + Cfg::RING_BYTES);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 2;
  uint64_t* drain = tempty + 2;
  uint64_t* ring_bar = drain + 1;  // RING_SLOTS per epilogue warp
  uint32_t* ring_cnt = reinterpret_cast<uint32_t*>(ring_bar + 4 * RING_SLOTS);  // 2 per epilogue warp
  uint32_t* tmem_slot = ring_cnt + 8;
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  static_assert((2 * 6 + 5 + 4 * RING_SLOTS) * 8 + 10 * 4 <= Cfg::BAR_BYTES, "barrier area");
  uint8_t* epi_stage = ring + Cfg::RING_BYTES + Cfg::BAR_BYTES;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  // In a pair, the even CTA issues the MMAs and owns the "full" and
  // "TMEM empty" barriers; both CTAs load, and both run epilogues.
  const uint32_t rank = PAIR ? cluster_ctarank() : 0u;
  const uint32_t pair_lead = rank & ~1u;
  const bool leader = (rank & 1u) == 0;
  const int cluster_id = static_cast<int>(blockIdx.x) / CG;
  const int num_clusters = static_cast<int>(gridDim.x) / CG;

  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], QUAD ? 2 : 1);  // one commit per pair reading the stage
    }
    for (int b = 0; b < 2; ++b) {
      mbar_init(&tfull[b], 1);
      mbar_init(&tempty[b], PAIR ? 8 : 4);
    }
    mbar_init(drain, 1);
    for (int i = 0; i < 4 * RING_SLOTS; ++i) mbar_init(&ring_bar[i], 1);
    for (int i = 0; i < 8; ++i) ring_cnt[i] = 0;
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mA0);
    tma_prefetch_desc(&mB0);
    if (args.kb1 > 0) {
      tma_prefetch_desc(&mA1);
      tma_prefetch_desc(&mB1);
    }
    if (args.b_dual) tma_prefetch_desc(&mB1);
    if (RING > 0 && args.e.ring > 0) tma_prefetch_desc(&mE0);
    if (RING > 1 && args.e.ring > 1) tma_prefetch_desc(&mE1);
  }
  if (warp == 1) {
    tmem_alloc<PAIR>(tmem_slot, Cfg::TMEM_COLS);
    tmem_relinquish<PAIR>();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // peer barriers initialised before any remote arrive
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int num_kb = args.kb0 + args.kb1;
  bool aborted = false;
  // Everything above touched only shared memory, TMEM and the kernel
  // parameters: with programmatic launch it overlaps the previous kernel's
  // tail.  From here on global memory is read and written.
  griddep_wait();
  griddep_launch_dependents();

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    // The whole warp runs the loop; one elected lane issues the copies.
    const uint32_t el = elect_one();
    {
      // A panels are shared by the raster group's successive waves; B tiles
      // only by the tiles of one wave.
      const bool hint_a = args.l2_hints & 1, hint_b = args.l2_hints & 2;
      const uint64_t pol_a = l2_policy_evict_last();
      const uint64_t pol_b = l2_policy_evict_first();
      uint32_t it = 0;
      for (int u = cluster_id; u < args.num_units && !aborted; u += num_clusters) {
        int mb2, nb0, nlen, chunk;
        unit_coords(args, u, mb2, nb0, nlen, chunk);
        const int mb = mb2 * CG + static_cast<int>(rank);
        for (int j = 0; j < nlen && !aborted; ++j) {
          const int nb = nb0 + j;
          for (int kb = 0; kb < num_kb; ++kb, ++it) {
            const int s = it % S;
            const uint32_t ph = (it / S) & 1;
            if (!mbar_wait_bounded(&empty[s], ph ^ 1, abort_flag, args.status, args.timeout_ns,
                                   args.producer_sleep_ns)) {
              aborted = true;
              break;
            }
            if (leader) mbar_arrive_expect_tx(&full[s], PAIR ? 2 * Cfg::STAGE_BYTES : Cfg::STAGE_BYTES, el);
            const bool second = kb >= args.kb0;
            const CUtensorMap* ma = second ? &mA1 : &mA0;
            const CUtensorMap* mbp = second ? &mB1 : &mB0;
            const int k = (second ? kb - args.kb0 : kb) * (FP8 ? 2 * BK : BK);
            uint8_t* sa = tiles + s * Cfg::STAGE_BYTES;
            uint8_t* sb = sa + Cfg::A_BYTES;
            if constexpr (PAIR) {
              const uint32_t bar = mapa_shared(&full[s], pair_lead);
              if (!args.a_mn) {
                hint_a ? tma_load_2d_pair_hint(sa, ma, bar, k, mb * BM, pol_a, el)
                       : tma_load_2d_pair(sa, ma, bar, k, mb * BM, el);
              } else {
#pragma unroll
                for (int c = 0; c < BM / 64; ++c)
                  hint_a ? tma_load_2d_pair_hint(sa + c * 8192, ma, bar, mb * BM + c * 64, k, pol_a, el)
                         : tma_load_2d_pair(sa + c * 8192, ma, bar, mb * BM + c * 64, k, el);
              }
              if constexpr (QUAD) {
                // this CTA's B rows (as in a pair) split in two 64-row halves:
                // half h is loaded by the CTA of pair h and lands in both pairs
                const int h = static_cast<int>(rank >> 1);
                const uint16_t mask = static_cast<uint16_t>((1u << rank) | (1u << (rank ^ 2u)));
                const int odd = static_cast<int>(rank & 1u);
                if (args.b_dual)
                  tma_load_2d_pair_mc(sb + h * 8192, odd ? &mB1 : &mB0, bar, k, nb * (BN / 2) + h * 64, mask, el);
                else if (!args.b_mn)
                  tma_load_2d_pair_mc(sb + h * 8192, mbp, bar, k, nb * BN + odd * Cfg::B_ROWS + h * 64, mask, el);
                else
                  tma_load_2d_pair_mc(sb + h * 8192, mbp, bar, nb * BN + odd * Cfg::B_ROWS + h * 64, k, mask, el);
              } else if (args.b_dual) {
                // the pair's N = [gate rows | up rows]: rank 0 stages the gate half, rank 1 the up half
                hint_b ? tma_load_2d_pair_hint(sb, rank ? &mB1 : &mB0, bar, k, nb * (BN / 2), pol_b, el)
                       : tma_load_2d_pair(sb, rank ? &mB1 : &mB0, bar, k, nb * (BN / 2), el);
              } else if (!args.b_mn) {
                hint_b ? tma_load_2d_pair_hint(sb, mbp, bar, k, nb * BN + static_cast<int>(rank) * Cfg::B_ROWS, pol_b,
                                               el)
                       : tma_load_2d_pair(sb, mbp, bar, k, nb * BN + static_cast<int>(rank) * Cfg::B_ROWS, el);
              } else {
#pragma unroll
                for (int c = 0; c < Cfg::B_ROWS / 64; ++c)
                  hint_b ? tma_load_2d_pair_hint(sb + c * 8192, mbp, bar,
                                                 nb * BN + static_cast<int>(rank) * Cfg::B_ROWS + c * 64, k, pol_b, el)
                         : tma_load_2d_pair(sb + c * 8192, mbp, bar,
                                            nb * BN + static_cast<int>(rank) * Cfg::B_ROWS + c * 64, k, el);
              }
            } else {
              if (!args.a_mn) {
                hint_a ? tma_load_2d_hint(sa, ma, &full[s], k, mb * BM, pol_a, el)
                       : tma_load_2d(sa, ma, &full[s], k, mb * BM, el);
              } else {
#pragma unroll
                for (int c = 0; c < BM / 64; ++c)
                  hint_a ? tma_load_2d_hint(sa + c * 8192, ma, &full[s], mb * BM + c * 64, k, pol_a, el)
                         : tma_load_2d(sa + c * 8192, ma, &full[s], mb * BM + c * 64, k, el);
              }
              if (args.b_dual) {
                hint_b ? tma_load_2d_hint(sb, &mB0, &full[s], k, nb * (BN / 2), pol_b, el)
                       : tma_load_2d(sb, &mB0, &full[s], k, nb * (BN / 2), el);
                hint_b ? tma_load_2d_hint(sb + (BN / 2) * 128, &mB1, &full[s], k, nb * (BN / 2), pol_b, el)
                       : tma_load_2d(sb + (BN / 2) * 128, &mB1, &full[s], k, nb * (BN / 2), el);
              } else if (!args.b_mn) {
                hint_b ? tma_load_2d_hint(sb, mbp, &full[s], k, nb * BN, pol_b, el)
                       : tma_load_2d(sb, mbp, &full[s], k, nb * BN, el);
              } else {
#pragma unroll
                for (int c = 0; c < BN / 64; ++c)
                  hint_b ? tma_load_2d_hint(sb + c * 8192, mbp, &full[s], nb * BN + c * 64, k, pol_b, el)
                         : tma_load_2d(sb + c * 8192, mbp, &full[s], nb * BN + c * 64, k, el);
              }
            }
          }
        }
      }
      if (aborted) {
        if (leader) {
          // let every copy already issued land before the CTA's smem is reused
          const uint32_t first = it > static_cast<uint32_t>(S) ? it - S : 0;
          for (uint32_t j = first; j < it; ++j) mbar_wait_drain(&full[j % S], (j / S) & 1, 200000000ull);
        } else {
          // the peer's copies complete on the leader's barrier; give them time
          const uint64_t t0 = globaltimer_ns();
          while (globaltimer_ns() - t0 < 2000000ull) {
          }
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ UMMA issuer
    // The whole warp of the pair's even CTA runs the loop; one elected lane
    // issues the MMAs and commits.
    if (leader) {
      const uint32_t el = elect_one();
      uint32_t it = 0, t = 0;
      bool issued = false;
      const uint32_t idesc = args.idesc;
      for (int u = cluster_id; u < args.num_units && !aborted; u += num_clusters) {
        int mb2, nb0, nlen, chunk;
        unit_coords(args, u, mb2, nb0, nlen, chunk);
        for (int j = 0; j < nlen && !aborted; ++j, ++t) {
          const uint32_t buf = t & 1;
          if (!mbar_wait_bounded(&tempty[buf], ((t >> 1) & 1) ^ 1, abort_flag, args.status, args.timeout_ns)) {
            aborted = true;
            break;
          }
          tc_fence_after();
          const uint32_t d_tmem = tmem_base + buf * BN;
          for (int kb = 0; kb < num_kb; ++kb, ++it) {
            const int s = it % S;
            if (!mbar_wait_bounded(&full[s], (it / S) & 1, abort_flag, args.status, args.timeout_ns)) {
              aborted = true;
              break;
            }
            tc_fence_after();
            const uint32_t sa = smem_u32(tiles + s * Cfg::STAGE_BYTES);
            const uint32_t sb = sa + Cfg::A_BYTES;
#pragma unroll
            for (int k16 = 0; k16 < BK / 16; ++k16) {
              // K-major: rows of 128 B, 8-row swizzle atoms 1024 B apart; a
              // 16-element k step is +32 B inside the atom.  MN-major: 64-wide
              // MN chunks 8 KB apart (LBO), 8-row k groups 1 KB apart (SBO);
              // a 16-row k step is +2 KB.
              const uint64_t ad = args.a_mn ? sdesc_sw128(sa + k16 * 2048, 8192, 1024)
                                            : sdesc_sw128(sa + k16 * 32, 16, 1024);
              const uint64_t bd = args.b_mn ? sdesc_sw128(sb + k16 * 2048, 8192, 1024)
                                            : sdesc_sw128(sb + k16 * 32, 16, 1024);
              const uint32_t acc = (kb | k16) != 0;
              if constexpr (PAIR && FP8)
                umma_f8_pair(d_tmem, ad, bd, idesc, acc, el);
              else if constexpr (PAIR)
                umma_bf16_pair(d_tmem, ad, bd, idesc, acc, el);
              else if constexpr (FP8)
                umma_f8(d_tmem, ad, bd, idesc, acc, el);
              else
                umma_bf16(d_tmem, ad, bd, idesc, acc, el);
            }
            issued = true;
            if constexpr (QUAD)
              umma_commit_pair_mc(&empty[s], 0xF, el);  // the stage's B halves live in all four CTAs
            else if constexpr (PAIR)
              umma_commit_pair_mc(&empty[s], 0x3, el);
            else
              umma_commit(&empty[s], el);
          }
          if (aborted) break;
          if constexpr (PAIR)
            umma_commit_pair_mc(&tfull[buf], static_cast<uint16_t>(0x3u << pair_lead), el);
          else
            umma_commit(&tfull[buf], el);
        }
      }
      if (aborted && issued) {
        if constexpr (PAIR)
          umma_commit_pair(drain, el);
        else
          umma_commit(drain, el);
        mbar_wait_drain(drain, 0, 200000000ull);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue
    const int q = warp & 3;  // TMEM lane quarter this warp may access
    uint32_t t = 0;
    for (int u = cluster_id; u < args.num_units && !aborted; u += num_clusters) {
      int mb2, nb0, nlen, chunk;
      unit_coords(args, u, mb2, nb0, nlen, chunk);
      const int mb = mb2 * CG + static_cast<int>(rank);
      TileInfo ti;
      ti.mb = mb;
      ti.unit_chunk = chunk;
      ti.row = mb * BM + q * 32 + lane;
      ti.M = args.M;
      ti.N = args.N;
      ti.status = args.status;
      ti.stage = epi_stage + q * 2048;
      ti.ring = ring + q * RING_SLOTS * RING * RING_CHUNK_BYTES;
      ti.ring_bar = ring_bar + q * RING_SLOTS;
      ti.ring_cnt = ring_cnt + q * 2;
      ti.emap0 = &mE0;
      ti.emap1 = &mE1;
      ti.abort_flag = abort_flag;
      ti.timeout_ns = args.timeout_ns;
      typename Epi::State st;
      Epi::begin(st, args.e, ti);
      for (int j = 0; j < nlen; ++j, ++t) {
        const uint32_t buf = t & 1;
        ti.nb = nb0 + j;
        Epi::prefetch(args.e, ti);  // the tile's auxiliary rows into L2 while its mainloop runs
        if (!mbar_wait_bounded(&tfull[buf], (t >> 1) & 1, abort_flag, args.status, args.timeout_ns,
                               args.epilogue_sleep_ns)) {
          aborted = true;
          break;
        }
        tc_fence_after();
        __syncwarp();
        ti.nb = nb0 + j;
        ti.taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16) + buf * BN;
        Epi::tile(st, args.e, ti);
        tc_fence_before();
        __syncwarp();
        if (lane == 0) {
          if constexpr (PAIR)
            mbar_arrive_cluster(mapa_shared(&tempty[buf], pair_lead));
          else
            mbar_arrive(&tempty[buf]);
        }
      }
      if (aborted) break;
      Epi::end(st, args.e, ti);
    }
    if (RING > 0 && args.e.ring > 0) {
      // ring copies issued but not consumed (an aborted tile) land before
      // the CTA's shared memory is released
      __syncwarp();
      uint64_t* rb = ring_bar + q * RING_SLOTS;
      const uint32_t issued = ring_cnt[q * 2], done = ring_cnt[q * 2 + 1];
      for (uint32_t g = done; g < issued; ++g) mbar_wait_drain(&rb[g % RING_SLOTS], (g / RING_SLOTS) & 1, 200000000ull);
    }
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (PAIR) cluster_sync();  // no CTA leaves while its peer may still signal it
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc<PAIR>(tmem_base, Cfg::TMEM_COLS);
  }
}

}  // namespace coda
