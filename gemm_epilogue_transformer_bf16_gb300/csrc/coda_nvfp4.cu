// NVFP4 operands: 4-bit e2m1 elements with one e4m3 scale per 16 elements
// along K and an fp32 scale per row, and the persistent GEMM that consumes
// them with tcgen05.mma kind::mxf4nvf4 (block-scaled, scale vector 4X).
//
// "CODA: Rewriting Transformer Blocks as GEMM-Epilogue Programs" (§1) and
// the news flash on it name FP4 beside FP8 as the formats that make the
// matrix multiplications fast and the data movement around them dominant;
// the epilogues are the ones of the bf16 and e4m3 kernels.
//
// Quantised operand layout (what coda_quantize_nvfp4_rows writes):
//   codes  [rows, K/2] bytes: element 2j in the low nibble of byte j, 2j+1 in
//          the high nibble (e2m1: bit 3 sign, bits 0-2 magnitude index);
//   scale  [rows] fp32: s = amax(row) / (6 * 448), 1 for a zero row;
//   sf     e4m3 block scales in the order the tensor core reads them: rows in
//          blocks of 128, K in tiles of 256 elements (16 scales per row);
//          the 2 KB of one (row block, k tile) are contiguous, four 512-byte
//          groups of 64 elements, each holding row r's 4 scales at byte
//          (r % 32) * 16 + ((r % 128) / 32) * 4.  Rows are padded to a
//          multiple of 512 (a cluster of four 128-row blocks) and K to a
//          multiple of 256 with zero scales.
//
// GEMM structure: warp 0 TMA producer, warp 1 TMEM owner and MMA issuer,
// warps 2-9 epilogue (two per TMEM lane quarter); M = 128, N = 256, k-slices
// of 256 elements (128 bytes of codes per row, the same 128-byte swizzled
// rows as the bf16 kernel), four stages.  Per stage the producer also copies
// the k-slice's block scales (2 KB for A, 4 KB for B) to shared memory; the
// MMA thread moves them into TMEM with tcgen05.cp (32 lanes x 128 bits,
// replicated to the four lane quarters) before the four MMAs (K = 64 each)
// that read them.  TMEM: the accumulator in columns 0-255 and, per stage,
// 64 columns of scales (A at +0, B at +16).  With a single accumulator the
// epilogue warps pull their columns into registers and free it before their
// math and stores, which then overlap the next tile's mainloop.  Variants:
// clusters of 2 or 4 CTAs sharing the B tile by multicast, and CTA pairs
// (cta_group::2, 256 x 256 tiles) further down.
#include <algorithm>
#include <atomic>
#include <cstdio>
#include <cstdlib>
#include <cstring>
#include <mutex>
#include <type_traits>
#include <utility>

#include <cuda_fp4.h>
#include <cuda_fp8.h>

#include "coda_epilogues.cuh"
#include "coda_internal.h"

namespace coda {

namespace {

constexpr int F4_BN = 256;
constexpr uint32_t F4_A_BYTES = BM * 128;
constexpr uint32_t F4_B_BYTES = F4_BN * 128;
constexpr uint32_t F4_SFA_BYTES = 2048;
constexpr uint32_t F4_SFB_BYTES = 4096;
constexpr uint32_t F4_STAGE_BYTES = F4_A_BYTES + F4_B_BYTES + F4_SFA_BYTES + F4_SFB_BYTES;
constexpr uint32_t F4_BAR_BYTES = 256;
constexpr uint32_t F4_TMEM_COLS = 512;
constexpr uint32_t F4_SF_COL0 = 256;     // first TMEM column of the scale slots
constexpr uint32_t F4_SF_SLOT_COLS = 64;
static_assert(F4_STAGE_BYTES % 1024 == 0, "stages keep 1024-byte alignment");

// Eight epilogue warps, two per TMEM lane quarter, each on half of the
// tile's columns, with 1 KB store buffers; four stages.
constexpr int F4_EW = 8;
constexpr int F4_STAGES = 4;
constexpr int F4_THREADS = 64 + 32 * F4_EW;
constexpr uint32_t F4_EPI_WARP_BYTES = 1024;
constexpr uint32_t F4_EPI_BYTES = F4_EW * F4_EPI_WARP_BYTES;
constexpr uint32_t F4_SMEM = 1024 + F4_STAGES * F4_STAGE_BYTES + F4_BAR_BYTES + F4_EPI_BYTES;
static_assert(F4_SMEM <= 232448, "shared memory per CTA");
static_assert(F4_SF_COL0 + F4_STAGES * F4_SF_SLOT_COLS <= F4_TMEM_COLS, "TMEM columns");

// The same, written to the same offset in every CTA of `mask` in the
// cluster, completion counted on each destination CTA's barrier at `bar`'s
// offset.
__device__ __forceinline__ void bulk_load_mc(void* dst, const void* src, uint32_t bytes, uint64_t* bar,
                                             uint16_t mask, uint32_t p) {
  asm volatile(
      "{\n\t.reg .pred P;\n\tsetp.ne.b32 P, %3, 0;\n\t"
      "@P cp.async.bulk.shared::cluster.global.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1], %2, [%4], %5;\n\t}" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(src)), "r"(bytes), "r"(p), "r"(smem_u32(bar)), "h"(mask)
      : "memory");
}

// Tiled tensor copy multicast to the CTAs of `mask` (same smem offset and
// barrier offset in each).
__device__ __forceinline__ void tma_load_2d_mc(void* dst, const CUtensorMap* m, uint64_t* bar, int x, int y,
                                               uint16_t mask, uint32_t p) {
  asm volatile(
      "{\n\t.reg .pred P;\n\tsetp.ne.b32 P, %5, 0;\n\t"
      "@P cp.async.bulk.tensor.2d.shared::cluster.global.tile.mbarrier::complete_tx::bytes.multicast::cluster"
      " [%0], [%1, {%3, %4}], [%2], %6;\n\t}" ::"r"(smem_u32(dst)),
      "l"(reinterpret_cast<uint64_t>(m)), "r"(smem_u32(bar)), "r"(x), "r"(y), "r"(p), "h"(mask)
      : "memory");
}

// Arrive once on the barrier at `bar`'s offset in every CTA of `mask` when
// the tcgen05 operations issued so far by this thread have completed.
__device__ __forceinline__ void umma_commit_mc(uint64_t* bar, uint16_t mask, uint32_t p) {
  asm volatile(
      "{\n\t.reg .pred P;\n\tsetp.ne.b32 P, %2, 0;\n\t"
      "@P tcgen05.commit.cta_group::1.mbarrier::arrive::one.shared::cluster.multicast::cluster.b64 [%0], %1;\n\t}" ::
          "r"(smem_u32(bar)),
      "h"(mask), "r"(p)
      : "memory");
}

// Shared-memory descriptor without swizzling: 8-row x 16-byte core
// matrices, `sbo` bytes between consecutive 8-row groups.
__device__ __forceinline__ uint64_t sdesc_plain(uint32_t saddr, uint32_t lbo_bytes, uint32_t sbo_bytes) {
  uint64_t d = 0;
  d |= static_cast<uint64_t>((saddr >> 4) & 0x3FFFu);
  d |= static_cast<uint64_t>((lbo_bytes >> 4) & 0x3FFFu) << 16;
  d |= static_cast<uint64_t>((sbo_bytes >> 4) & 0x3FFFu) << 32;
  d |= static_cast<uint64_t>(1) << 46;
  return d;  // layout type 0 (no swizzle) at bits 61-63
}

// 32 rows x 128 bits from shared memory into TMEM lanes 0-31, replicated to
// the four 32-lane quarters (4 columns).
__device__ __forceinline__ void tmem_cp_32x128_x4(uint32_t taddr, uint64_t sdesc, uint32_t p) {
  asm volatile(
      "{\n\t.reg .pred P;\n\tsetp.ne.b32 P, %2, 0;\n\t"
      "@P tcgen05.cp.cta_group::1.32x128b.warpx4 [%0], %1;\n\t}" ::"r"(taddr),
      "l"(sdesc), "r"(p)
      : "memory");
}

// D[tmem] (+)= (A . sfA) * (B . sfB)^T: e2m1 operands, e4m3 scale per 16
// elements (scale vector 4X), K = 64 per instruction, fp32 accumulator.
__device__ __forceinline__ void umma_nvfp4(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                           uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate,
                                           uint32_t p) {
  asm volatile(
      "{\n\t.reg .pred A, P;\n\t"
      "setp.ne.b32 A, %6, 0;\n\t"
      "setp.ne.b32 P, %7, 0;\n\t"
      "@P tcgen05.mma.cta_group::1.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], A;\n\t}" ::
          "r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate), "r"(p)
      : "memory");
}

// Instruction descriptor of the block-scaled kinds: B scale-factor id 0
// (bits 4-5), A and B e2m1 (type 1 at bits 7-9 and 10-12), K-major, N>>3 at
// bits 17-22, scale type e4m3 (bit 23 = 0), M>>4 at bits 24-28, A
// scale-factor id 0 (bits 29-30), K = 64 (bit 31 = 0).
constexpr uint32_t idesc_nvfp4(int M, int N) {
  return (1u << 7) | (1u << 10) | (static_cast<uint32_t>(N >> 3) << 17) | (static_cast<uint32_t>(M >> 4) << 24);
}

// e4m3 code -> value (1 sign, 4 exponent bits with bias 7, 3 mantissa bits;
// exponent 0 subnormal); scale codes are never NaN (<= 448 by construction).
__device__ __forceinline__ float e4m3_value(uint32_t b) {
  const uint32_t e = (b >> 3) & 15u, m = b & 7u;
  const float v = e ? __uint_as_float(((e + 120u) << 23) | (m << 20)) : static_cast<float>(m) * 0.001953125f;
  return (b & 0x80u) ? -v : v;
}

// x[0..15] *= gamma[16j ..] (one fp32 product each).
__device__ __forceinline__ void apply_gamma(const float* gamma, int64_t j, float* x) {
  const float4* gp = reinterpret_cast<const float4*>(gamma + j * 16);
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const float4 g = gp[i];
    x[4 * i] = __fmul_rn(x[4 * i], g.x);
    x[4 * i + 1] = __fmul_rn(x[4 * i + 1], g.y);
    x[4 * i + 2] = __fmul_rn(x[4 * i + 2], g.z);
    x[4 * i + 3] = __fmul_rn(x[4 * i + 3], g.w);
  }
}

// Block j (16 elements) of a bf16 row as fp32.
__device__ __forceinline__ void load_block16(const __nv_bfloat16* row, int64_t j, float* x) {
  const uint4* p = reinterpret_cast<const uint4*>(row + j * 16);
  const uint4 w[2] = {p[0], p[1]};
  const uint32_t* u = reinterpret_cast<const uint32_t*>(w);
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    x[2 * i] = bf16_lo(u[i]);
    x[2 * i + 1] = bf16_hi(u[i]);
  }
}

// Eight e2m1 codes in a word: a code of magnitude 0 loses its sign bit.
__device__ __forceinline__ uint32_t clear_negative_zero(uint32_t w) {
  const uint32_t m = w & 0x77777777u;
  const uint32_t nz = (m | (m >> 1) | (m >> 2)) & 0x11111111u;  // bit 0 of each nibble: magnitude != 0
  return m | (w & (nz << 3));
}

__device__ __forceinline__ int64_t sf_offset(int64_t r, int64_t j, int64_t kt_count) {
  return ((r >> 7) * kt_count + (j >> 4)) * 2048 + ((j >> 2) & 3) * 512 + (r & 31) * 16 + ((r >> 5) & 3) * 4 +
         (j & 3);
}

// One warp per row (rows up to the padded count; padding rows only write
// zero scales).  The quantised row is x, or u = x * gamma when a gain vector
// is given (the RMSNorm gain, applied without rounding u to bf16).  Pass 1:
// the row's amax (and, when rstd is given, sum x^2 for 1 / rms(x)).  Pass 2,
// lane per 16-element block: the block's e4m3 scale and sixteen e2m1 codes.
template <bool GAMMA, bool RSTD>
__global__ void __launch_bounds__(256) quantize_nvfp4_rows_kernel(const __nv_bfloat16* __restrict__ X, int64_t ldx,
                                                                  int64_t M, int64_t K, uint8_t* __restrict__ Q,
                                                                  uint8_t* __restrict__ SF,
                                                                  float* __restrict__ scale, int64_t rows_pad,
                                                                  int64_t kt_count, const float* __restrict__ gamma,
                                                                  float* __restrict__ rstd, float eps) {
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  const int64_t nb = K / 16, nb_pad = kt_count * 16;
  for (int64_t r = static_cast<int64_t>(blockIdx.x) * (blockDim.x >> 5) + (threadIdx.x >> 5); r < rows_pad;
       r += warps) {
    if (r >= M) {
      for (int64_t j = lane; j < nb_pad; j += 32) SF[sf_offset(r, j, kt_count)] = 0;
      continue;
    }
    const __nv_bfloat16* row = X + r * ldx;
    float amax = 0.f, ss = 0.f;
#pragma unroll 4
    for (int64_t j = lane; j < nb; j += 32) {
      float x[16];
      load_block16(row, j, x);
      if constexpr (RSTD) {
#pragma unroll
        for (int i = 0; i < 16; ++i) ss = fmaf(x[i], x[i], ss);
      }
      if constexpr (GAMMA) apply_gamma(gamma, j, x);
#pragma unroll
      for (int i = 0; i < 16; ++i) amax = fmaxf(amax, fabsf(x[i]));
    }
#pragma unroll
    for (int o = 16; o; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if constexpr (RSTD) {
#pragma unroll
      for (int o = 16; o; o >>= 1) ss += __shfl_xor_sync(0xffffffffu, ss, o);
      if (lane == 0) rstd[r] = 1.f / sqrtf(ss / static_cast<float>(K) + eps);
    }
    const float s = amax > 0.f ? __fdiv_rn(amax, 2688.0f) : 1.0f;
    if (lane == 0) scale[r] = s;
    const float t = __fmul_rn(6.0f, s);
#pragma unroll 2
    for (int64_t j = lane; j < nb_pad; j += 32) {
      uint32_t sfb = 0;
      if (j < nb) {
        float x[16];
        load_block16(row, j, x);
        if constexpr (GAMMA) apply_gamma(gamma, j, x);
        float bmax = 0.f;
#pragma unroll
        for (int i = 0; i < 16; ++i) bmax = fmaxf(bmax, fabsf(x[i]));
        const float sf_f = fminf(__fdiv_rn(bmax, t), 448.0f);
        sfb = __nv_cvt_float_to_fp8(sf_f, __NV_SATFINITE, __NV_E4M3);
        const float denom = __fmul_rn(e4m3_value(sfb), s);
        uint32_t lo = 0, hi = 0;
        if (denom > 0.f) {
          // one division per block: the elements are scaled by its reciprocal
          const float inv = fminf(__fdiv_rn(1.0f, denom), 3.40282347e38f);
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            // element 2i in the low nibble, 2i + 1 in the high nibble
            const uint32_t c2 = __nv_cvt_float2_to_fp4x2(
                make_float2(__fmul_rn(x[2 * i], inv), __fmul_rn(x[2 * i + 1], inv)), __NV_E2M1, cudaRoundNearest);
            if (i < 4)
              lo |= (c2 & 0xFFu) << (8 * i);
            else
              hi |= (c2 & 0xFFu) << (8 * (i - 4));
          }
          lo = clear_negative_zero(lo);
          hi = clear_negative_zero(hi);
        }
        *reinterpret_cast<uint2*>(Q + r * (K / 2) + j * 8) = make_uint2(lo, hi);
      }
      SF[sf_offset(r, j, kt_count)] = static_cast<uint8_t>(sfb);
    }
  }
}

// Stores a warp's 32 rows x 16 columns as bf16 (thread `lane` passes the 16
// values of row row0 + lane, columns col0 ..) through the warp's 1 KB buffer:
// 16-byte chunk p of row r sits at r * 32 + ((p ^ ((r >> 2) & 1)) * 16), so
// the row-wise writes cover all banks once per 8 lanes and the reads take a
// contiguous 512 bytes; each global store then covers 16 rows x 32
// contiguous bytes.  Rows >= M and columns >= N are not written (N is a
// multiple of 8).  Called by all 32 lanes.
__device__ __forceinline__ void f4_store_bf16x16(uint8_t* stage, __nv_bfloat16* base, int64_t ld, int row0, int M,
                                                 int col0, int N, const float* v, bool stream) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int p = 0; p < 2; ++p) {
    const uint4 w = make_uint4(pack_bf16x2(v[p * 8 + 0], v[p * 8 + 1]), pack_bf16x2(v[p * 8 + 2], v[p * 8 + 3]),
                               pack_bf16x2(v[p * 8 + 4], v[p * 8 + 5]), pack_bf16x2(v[p * 8 + 6], v[p * 8 + 7]));
    *reinterpret_cast<uint4*>(stage + lane * 32 + ((p ^ ((lane >> 2) & 1)) * 16)) = w;
  }
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const int r = i * 16 + (lane >> 1), p = lane & 1;
    const uint4 w = *reinterpret_cast<const uint4*>(stage + r * 32 + ((p ^ ((r >> 2) & 1)) * 16));
    const int row = row0 + r, col = col0 + p * 8;
    if (row < M && col < N) {
      __nv_bfloat16* dst = base + static_cast<int64_t>(row) * ld + col;
      if (stream)
        asm volatile("st.global.cs.v4.u32 [%0], {%1, %2, %3, %4};" ::"l"(dst), "r"(w.x), "r"(w.y), "r"(w.z),
                     "r"(w.w)
                     : "memory");
      else
        *reinterpret_cast<uint4*>(dst) = w;
    }
  }
  __syncwarp();
}
__device__ __forceinline__ void f4_store_bf16x32(uint8_t* stage, __nv_bfloat16* base, int64_t ld, int row0, int M,
                                                 int col0, int N, const float* v, bool stream) {
  f4_store_bf16x16(stage, base, ld, row0, M, col0, N, v, stream);
  f4_store_bf16x16(stage, base, ld, row0, M, col0 + 16, N, v + 16, stream);
}

// The epilogue, one warp's share: 32 rows (TMEM lane quarter q) x 128
// accumulator columns (half h of the tile).  With one accumulator in TMEM
// the next tile's MMAs wait for it, so the warp first pulls its columns
// into registers and frees the accumulator, then scales, applies the map
// and stores while the next tile's mainloop runs.
//   KIND 0: y = rs_i * cs_j * acc (+ R), columns nb*256 + h*128 + [0, 128);
//   KIND 1: g = rs_i * cg_j * acc_gate, u = rs_i * cu_j * acc_up,
//           H = silu(g) * u, columns nb*128 + h*64 + [0, 64)
//   (rs = token scale x optional RMSNorm row factor; cs, cg, cu the
//   weights' row scales), as EpiPlain / EpiSwiglu do for the other kernels.
template <int KIND, bool PAIR = false>
__device__ __forceinline__ void f4_epilogue(const EpiArgs& e, const TileInfo& t, int h, uint64_t* tfull,
                                            uint32_t parity, uint64_t* tempty, volatile int* abort_flag,
                                            uint64_t timeout_ns, uint32_t sleep_ns, bool& aborted) {
  const int lane = threadIdx.x & 31;
  const int row = t.row;
  const bool rv = row < t.M;
  const int row0 = row - lane;
  float v[128];
  if (!mbar_wait_bounded(tfull, parity, abort_flag, t.status, timeout_ns, sleep_ns)) {
    aborted = true;
    return;
  }
  tc_fence_after();
  __syncwarp();
#pragma unroll
  for (int c = 0; c < 4; ++c) {
    // KIND 0: columns h*128 + 32c; KIND 1: gate h*64 + 32c (c < 2), up 128 + h*64 + 32(c-2)
    const uint32_t col = KIND == 0 ? h * 128 + 32 * c : (c < 2 ? h * 64 + 32 * c : 128 + h * 64 + 32 * (c - 2));
    tmem_ld32(t.taddr + col, *reinterpret_cast<float(*)[32]>(v + 32 * c));
  }
  tc_fence_before();
  __syncwarp();
  if (lane == 0) {
    if constexpr (PAIR)
      mbar_arrive_cluster(mapa_shared(tempty, 0));  // the pair's accumulator barrier is in the even CTA
    else
      mbar_arrive(tempty);
  }
  auto* D = static_cast<__nv_bfloat16*>(e.D);
  if constexpr (KIND == 0) {
    const float rs = (e.row_scale && rv) ? e.row_scale[row] : 1.f;
#pragma unroll
    for (int c = 0; c < 4; ++c) {
      const int col0 = t.nb * 256 + h * 128 + 32 * c;
      if (col0 >= t.N) break;
      float* x = v + 32 * c;
      if (rv) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int cc = col0 + g * 8;
          if (cc < t.N) {
            float s8[8];
            if (e.col_scale) {
              load_f32x8(e.col_scale + cc, s8);
            } else {
#pragma unroll
              for (int i = 0; i < 8; ++i) s8[i] = 1.f;
            }
#pragma unroll
            for (int i = 0; i < 8; ++i) x[g * 8 + i] = x[g * 8 + i] * rs * s8[i];
            if (e.aux0) {
              float r8[8];
              load_bf16x8(e.aux0 + static_cast<int64_t>(row) * e.ld_aux0 + cc, r8);
#pragma unroll
              for (int i = 0; i < 8; ++i) x[g * 8 + i] += r8[i];
            }
          }
        }
      }
      f4_store_bf16x32(t.stage, D, e.ldd, row0, t.M, col0, t.N, x, e.st_stream);
    }
  } else {
    const float rs =
        ((e.row_scale && rv) ? e.row_scale[row] : 1.f) * ((e.row_scale2 && rv) ? e.row_scale2[row] : 1.f);
#pragma unroll
    for (int c = 0; c < 2; ++c) {
      const int col0 = t.nb * 128 + h * 64 + 32 * c;
      if (col0 >= t.N) break;
      float* g = v + 32 * c;
      float* u = v + 64 + 32 * c;
      if (rv) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int cc = col0 + q * 8;
          float cg[8], cu[8];
          if (e.col_scale && cc < t.N) {
            load_f32x8(e.col_scale + cc, cg);
            load_f32x8(e.col_scale2 + cc, cu);
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            g[q * 8 + i] *= rs;
            u[q * 8 + i] *= rs;
            if (e.col_scale && cc < t.N) {
              g[q * 8 + i] *= cg[i];
              u[q * 8 + i] *= cu[i];
            }
          }
        }
      }
      if (e.out1) f4_store_bf16x32(t.stage, e.out1, e.ld_out1, row0, t.M, col0, t.N, g, e.st_stream);
      if (e.out2) f4_store_bf16x32(t.stage, e.out2, e.ld_out2, row0, t.M, col0, t.N, u, e.st_stream);
#pragma unroll
      for (int i = 0; i < 32; ++i) g[i] = g[i] / (1.f + __expf(-g[i])) * u[i];
      f4_store_bf16x32(t.stage, D, e.ldd, row0, t.M, col0, t.N, g, e.st_stream);
    }
  }
}

// KIND 0: EpiPlain (B = one weight, 256 columns); 1: EpiSwiglu (B = 128 gate
// + 128 up rows of two weights).  CG: 1, or 4 CTAs on four adjacent 128-row
// blocks sharing the B tile: each loads a 64-row quarter of B and a quarter
// of its block scales and multicasts them to all four, so every SM stages
// 27 KB of its own per k-slice instead of 54 KB.  The MMAs stay per CTA
// (cta_group::1); a stage is released when all four CTAs' MMAs are done
// with it (each commit arrives on the stage barrier of every CTA).
template <int KIND, int CG>
__global__ void __launch_bounds__(F4_THREADS, 1)
    coda_gemm_nvfp4_kernel(const __grid_constant__ CUtensorMap mA, const __grid_constant__ CUtensorMap mB0,
                           const __grid_constant__ CUtensorMap mB1, const GemmArgs args, const Nvfp4Scales sc) {
  static_assert(CG == 1 || CG == 2 || CG == 4, "cluster size");
  constexpr int S = F4_STAGES;
  constexpr bool MC = CG > 1;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* tiles = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * F4_STAGE_BYTES);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 1;
  uint64_t* drain = tempty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint8_t* epi_stage = smem + S * F4_STAGE_BYTES + F4_BAR_BYTES;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = MC ? cluster_ctarank() : 0u;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], CG);  // one commit from each CTA reading the stage's B quarters
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, F4_EW);
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mA);
    tma_prefetch_desc(&mB0);
    if (args.b_dual) tma_prefetch_desc(&mB1);
  }
  if (warp == 1) {
    tmem_alloc<false>(tmem_slot, F4_TMEM_COLS);
    tmem_relinquish<false>();
  }
  tc_fence_before();
  __syncthreads();
  if constexpr (MC) cluster_sync();  // peer barriers initialised before any multicast lands
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int num_kb = args.kb0;
  const int cluster_id = static_cast<int>(blockIdx.x) / CG;
  const int num_clusters = static_cast<int>(gridDim.x) / CG;
  bool aborted = false;

  if (warp == 0) {
    // ------------------------------------------------------------ producer
    const uint32_t el = elect_one();
    uint32_t it = 0;
    for (int u = cluster_id; u < args.num_units && !aborted; u += num_clusters) {
      int mbc, nb, nlen, chunk;
      unit_coords(args, u, mbc, nb, nlen, chunk);
      const int mb = mbc * CG + static_cast<int>(rank);
      for (int kb = 0; kb < num_kb; ++kb, ++it) {
        const int s = it % S;
        if (!mbar_wait_bounded(&empty[s], ((it / S) & 1) ^ 1, abort_flag, args.status, args.timeout_ns,
                               args.producer_sleep_ns)) {
          aborted = true;
          break;
        }
        mbar_arrive_expect_tx(&full[s], F4_STAGE_BYTES, el);
        uint8_t* sa = tiles + s * F4_STAGE_BYTES;
        uint8_t* sb = sa + F4_A_BYTES;
        uint8_t* sfa = sb + F4_B_BYTES;
        uint8_t* sfb = sfa + F4_SFA_BYTES;
        const int x = kb * 128;  // bytes of codes = 256 elements
        tma_load_2d(sa, &mA, &full[s], x, mb * BM, el);
        bulk_load(sfa, sc.a + (static_cast<int64_t>(mb) * sc.kt + kb) * 2048, 2048, &full[s], el);
        // B rows of the tile: [256 rows of B] or [128 gate | 128 up]; their
        // scales: two 2 KB groups (row blocks 2nb, 2nb + 1, or gate nb, up nb)
        const uint8_t* sf0 = args.b_dual ? sc.b0 + (static_cast<int64_t>(nb) * sc.kt + kb) * 2048
                                         : sc.b0 + (static_cast<int64_t>(2 * nb) * sc.kt + kb) * 2048;
        const uint8_t* sf1 = args.b_dual ? sc.b1 + (static_cast<int64_t>(nb) * sc.kt + kb) * 2048
                                         : sc.b0 + (static_cast<int64_t>(2 * nb + 1) * sc.kt + kb) * 2048;
        if constexpr (MC) {
          // piece r (of CG) of the tile's B rows and of their 4 KB of
          // scales, to every CTA of the cluster
          constexpr int P = F4_BN / CG;               // rows per piece
          constexpr uint32_t PS = F4_SFB_BYTES / CG;  // scale bytes per piece
          constexpr uint16_t ALL = (1u << CG) - 1;
          const int r = static_cast<int>(rank);
          const int tr = r * P;                       // first tile row of the piece
          const CUtensorMap* mb_map = (args.b_dual && tr >= F4_BN / 2) ? &mB1 : &mB0;
          const int row = args.b_dual ? nb * (F4_BN / 2) + tr % (F4_BN / 2) : nb * F4_BN + tr;
          tma_load_2d_mc(sb + tr * 128, mb_map, &full[s], x, row, ALL, el);
          const uint32_t so = r * PS;
          bulk_load_mc(sfb + so, (so >= 2048 ? sf1 : sf0) + so % 2048, PS, &full[s], ALL, el);
        } else {
          if (args.b_dual) {
            tma_load_2d(sb, &mB0, &full[s], x, nb * (F4_BN / 2), el);
            tma_load_2d(sb + (F4_BN / 2) * 128, &mB1, &full[s], x, nb * (F4_BN / 2), el);
          } else {
            tma_load_2d(sb, &mB0, &full[s], x, nb * F4_BN, el);
          }
          bulk_load(sfb, sf0, 2048, &full[s], el);
          bulk_load(sfb + 2048, sf1, 2048, &full[s], el);
        }
      }
    }
    if (aborted) {
      const uint32_t first = it > static_cast<uint32_t>(S) ? it - S : 0;
      for (uint32_t j = first; j < it; ++j) mbar_wait_drain(&full[j % S], (j / S) & 1, 200000000ull);
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ scale copies + MMA issuer
    const uint32_t el = elect_one();
    uint32_t it = 0, t = 0;
    bool issued = false;
    const uint32_t idesc = args.idesc;
    for (int u = cluster_id; u < args.num_units && !aborted; u += num_clusters, ++t) {
      if (!mbar_wait_bounded(tempty, (t & 1) ^ 1, abort_flag, args.status, args.timeout_ns)) {
        aborted = true;
        break;
      }
      tc_fence_after();
      for (int kb = 0; kb < num_kb; ++kb, ++it) {
        const int s = it % S;
        if (!mbar_wait_bounded(&full[s], (it / S) & 1, abort_flag, args.status, args.timeout_ns)) {
          aborted = true;
          break;
        }
        tc_fence_after();
        const uint32_t sa = smem_u32(tiles + s * F4_STAGE_BYTES);
        const uint32_t sb = sa + F4_A_BYTES;
        const uint32_t sfa = sb + F4_B_BYTES;
        const uint32_t sfb = sfa + F4_SFA_BYTES;
        const uint32_t slot = tmem_base + F4_SF_COL0 + static_cast<uint32_t>(s) * F4_SF_SLOT_COLS;
        // A: one 512-byte group per 64-element step -> 4 columns each;
        // B: two 128-row halves per step -> 8 columns each (rows 0-127, then 128-255)
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          tmem_cp_32x128_x4(slot + g * 4, sdesc_plain(sfa + g * 512, 128, 128), el);
          tmem_cp_32x128_x4(slot + 16 + g * 8, sdesc_plain(sfb + g * 512, 128, 128), el);
          tmem_cp_32x128_x4(slot + 16 + g * 8 + 4, sdesc_plain(sfb + 2048 + g * 512, 128, 128), el);
        }
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          // 64 e2m1 elements = 32 bytes of each 128-byte swizzled row
          const uint64_t ad = sdesc_sw128(sa + g * 32, 16, 1024);
          const uint64_t bd = sdesc_sw128(sb + g * 32, 16, 1024);
          umma_nvfp4(tmem_base, ad, bd, idesc, slot + g * 4, slot + 16 + g * 8, (kb | g) != 0, el);
        }
        issued = true;
        if constexpr (MC)
          umma_commit_mc(&empty[s], static_cast<uint16_t>((1u << CG) - 1), el);
        else
          umma_commit(&empty[s], el);
      }
      if (aborted) break;
      umma_commit(tfull, el);
    }
    if (aborted && issued) {
      umma_commit(drain, el);
      mbar_wait_drain(drain, 0, 200000000ull);
    }
  } else {
    // ------------------------------------------------------------ epilogue
    // warps 2-5 take the first half of the tile's columns, 6-9 the second
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    uint32_t t = 0;
    for (int u = cluster_id; u < args.num_units && !aborted; u += num_clusters, ++t) {
      int mbc, nb, nlen, chunk;
      unit_coords(args, u, mbc, nb, nlen, chunk);
      const int mb = mbc * CG + static_cast<int>(rank);
      TileInfo ti;
      ti.mb = mb;
      ti.nb = nb;
      ti.unit_chunk = chunk;
      ti.row = mb * BM + q * 32 + lane;
      ti.M = args.M;
      ti.N = args.N;
      ti.status = args.status;
      ti.stage = epi_stage + (warp - 2) * F4_EPI_WARP_BYTES;
      ti.taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      f4_epilogue<KIND>(args.e, ti, h, tfull, t & 1, tempty, abort_flag, args.timeout_ns, args.epilogue_sleep_ns,
                        aborted);
    }
  }

  tc_fence_before();
  __syncthreads();
  if constexpr (MC) cluster_sync();  // no CTA leaves while a peer may still write or signal it
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc<false>(tmem_base, F4_TMEM_COLS);
  }
}

// Grid: one CTA (CG = 1) or one 4-CTA cluster per unit up to the resident
// limit; the first call on a device sets the shared-memory limit and looks
// up the resident-cluster count.
template <int KIND, int CG>
cudaError_t launch_nvfp4(int num_units, int sms, cudaStream_t s, const CUtensorMap* m, const GemmArgs& a,
                         const Nvfp4Scales& sc) {
  static std::mutex init;
  static std::atomic<bool> attr_done[64];
  static std::atomic<int> max_clusters[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  auto kern = coda_gemm_nvfp4_kernel<KIND, CG>;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(F4_THREADS);
  cfg.dynamicSmemBytes = F4_SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = CG;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (!attr_done[dev].load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(init);
    if (!attr_done[dev].load(std::memory_order_relaxed)) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(F4_SMEM));
      if (e != cudaSuccess) return e;
      int n = sms;
      if (CG > 1) {
        cfg.gridDim = dim3(static_cast<unsigned>(sms - sms % CG));
        e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
        if (e != cudaSuccess) return e;
        if (n <= 0) return cudaErrorInvalidConfiguration;
      }
      max_clusters[dev].store(n, std::memory_order_relaxed);
      attr_done[dev].store(true, std::memory_order_release);
    }
  }
  const int resident = max_clusters[dev].load(std::memory_order_relaxed);
  cfg.gridDim = dim3(static_cast<unsigned>(CG * std::min(num_units, resident)));
  note_launch();
  e = cudaLaunchKernelEx(&cfg, kern, m[0], m[1], m[2], a, sc);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

// ------------------------------------------------------------------ CTA pairs
// The same GEMM on CTA pairs (tcgen05 cta_group::2): a cluster of two CTAs on
// adjacent 128-row blocks computes a 256 x 256 tile; each CTA stages its own
// 128 rows of A and its own 128 of the 256 B rows (the MMA reads the other
// half from the peer), its rows' block scales, and the scales of all 256 B
// rows (each CTA loads one half and multicasts it to both).  The scales
// travel through 2-D tensor maps (rows of 256 bytes, 8-row boxes = one 2 KB
// group), so that both CTAs' copies complete on the leader's barrier.  The
// leader (even CTA) moves the scales into TMEM with tcgen05.cp.cta_group::2
// (each CTA from its own shared memory into its own TMEM) and issues the
// MMAs; both CTAs run the epilogue on their own 128 rows.  A stage is 38 KB
// (five fit) for the same tensor work per CTA as a 54 KB single-CTA stage.
constexpr uint32_t P4_A_BYTES = BM * 128;
constexpr uint32_t P4_B_BYTES = (F4_BN / 2) * 128;
constexpr uint32_t P4_SFA_BYTES = 2048;
constexpr uint32_t P4_SFB_BYTES = 4096;
constexpr uint32_t P4_STAGE_BYTES = P4_A_BYTES + P4_B_BYTES + P4_SFA_BYTES + P4_SFB_BYTES;
constexpr int P4_STAGES = 5;
constexpr uint32_t P4_SF_SLOT_COLS = 48;
constexpr uint32_t P4_SMEM = 1024 + P4_STAGES * P4_STAGE_BYTES + F4_BAR_BYTES + F4_EPI_BYTES;
// bytes landing per stage, counted on the leader's barrier: A, B and A's
// scales from both CTAs, and both 2 KB halves of B's scales in both CTAs
constexpr uint32_t P4_TX = 2 * (P4_A_BYTES + P4_B_BYTES + P4_SFA_BYTES) + 2 * P4_SFB_BYTES;
static_assert(P4_STAGE_BYTES % 1024 == 0, "stages keep 1024-byte alignment");
static_assert(P4_SMEM <= 232448, "shared memory per CTA");
static_assert(F4_SF_COL0 + P4_STAGES * P4_SF_SLOT_COLS <= F4_TMEM_COLS, "TMEM columns");

__device__ __forceinline__ void tmem_cp_32x128_x4_pair(uint32_t taddr, uint64_t sdesc, uint32_t p) {
  asm volatile(
      "{\n\t.reg .pred P;\n\tsetp.ne.b32 P, %2, 0;\n\t"
      "@P tcgen05.cp.cta_group::2.32x128b.warpx4 [%0], %1;\n\t}" ::"r"(taddr),
      "l"(sdesc), "r"(p)
      : "memory");
}

__device__ __forceinline__ void umma_nvfp4_pair(uint32_t d_tmem, uint64_t adesc, uint64_t bdesc, uint32_t idesc,
                                                uint32_t sfa_tmem, uint32_t sfb_tmem, uint32_t accumulate,
                                                uint32_t p) {
  asm volatile(
      "{\n\t.reg .pred A, P;\n\t"
      "setp.ne.b32 A, %6, 0;\n\t"
      "setp.ne.b32 P, %7, 0;\n\t"
      "@P tcgen05.mma.cta_group::2.kind::mxf4nvf4.block_scale.scale_vec::4X [%0], %1, %2, %3, [%4], [%5], A;\n\t}" ::
          "r"(d_tmem),
      "l"(adesc), "l"(bdesc), "r"(idesc), "r"(sfa_tmem), "r"(sfb_tmem), "r"(accumulate), "r"(p)
      : "memory");
}

template <int KIND>
__global__ void __launch_bounds__(F4_THREADS, 1)
    coda_gemm_nvfp4_pair_kernel(const __grid_constant__ CUtensorMap mA, const __grid_constant__ CUtensorMap mB0,
                                const __grid_constant__ CUtensorMap mB1, const __grid_constant__ CUtensorMap mSA,
                                const __grid_constant__ CUtensorMap mSB0, const __grid_constant__ CUtensorMap mSB1,
                                const GemmArgs args, const Nvfp4Scales sc) {
  constexpr int S = P4_STAGES;
  extern __shared__ uint8_t smem_raw[];
  uint8_t* smem = reinterpret_cast<uint8_t*>((reinterpret_cast<uintptr_t>(smem_raw) + 1023) & ~uintptr_t(1023));
  uint8_t* tiles = smem;
  uint64_t* full = reinterpret_cast<uint64_t*>(smem + S * P4_STAGE_BYTES);
  uint64_t* empty = full + S;
  uint64_t* tfull = empty + S;
  uint64_t* tempty = tfull + 1;
  uint64_t* drain = tempty + 1;
  uint32_t* tmem_slot = reinterpret_cast<uint32_t*>(drain + 1);
  volatile int* abort_flag = reinterpret_cast<volatile int*>(tmem_slot + 1);
  uint8_t* epi_stage = smem + S * P4_STAGE_BYTES + F4_BAR_BYTES;

  const int warp = threadIdx.x >> 5;
  const int lane = threadIdx.x & 31;
  const uint32_t rank = cluster_ctarank();
  const bool leader = rank == 0;
  if (threadIdx.x == 0) {
    for (int s = 0; s < S; ++s) {
      mbar_init(&full[s], 1);
      mbar_init(&empty[s], 1);
    }
    mbar_init(tfull, 1);
    mbar_init(tempty, 2 * F4_EW);  // every epilogue warp of both CTAs
    mbar_init(drain, 1);
    *abort_flag = 0;
    fence_mbar_init();
  }
  if (warp == 0 && lane == 0) {
    tma_prefetch_desc(&mA);
    tma_prefetch_desc(&mB0);
    tma_prefetch_desc(&mSA);
    tma_prefetch_desc(&mSB0);
    if (args.b_dual) {
      tma_prefetch_desc(&mB1);
      tma_prefetch_desc(&mSB1);
    }
  }
  if (warp == 1) {
    tmem_alloc<true>(tmem_slot, F4_TMEM_COLS);
    tmem_relinquish<true>();
  }
  tc_fence_before();
  __syncthreads();
  cluster_sync();  // the leader's barriers are initialised before the peer signals them
  tc_fence_after();
  const uint32_t tmem_base = *tmem_slot;
  const int num_kb = args.kb0;
  const int cluster_id = static_cast<int>(blockIdx.x) / 2;
  const int num_clusters = static_cast<int>(gridDim.x) / 2;
  bool aborted = false;

  if (warp == 0) {
    // ------------------------------------------------------------ producer (both CTAs)
    const uint32_t el = elect_one();
    uint32_t it = 0;
    for (int u = cluster_id; u < args.num_units && !aborted; u += num_clusters) {
      int mbc, nb, nlen, chunk;
      unit_coords(args, u, mbc, nb, nlen, chunk);
      const int mb = mbc * 2 + static_cast<int>(rank);
      for (int kb = 0; kb < num_kb; ++kb, ++it) {
        const int s = it % S;
        if (!mbar_wait_bounded(&empty[s], ((it / S) & 1) ^ 1, abort_flag, args.status, args.timeout_ns,
                               args.producer_sleep_ns)) {
          aborted = true;
          break;
        }
        if (leader) mbar_arrive_expect_tx(&full[s], P4_TX, el);
        const uint32_t bar = mapa_shared(&full[s], 0);
        uint8_t* sa = tiles + s * P4_STAGE_BYTES;
        uint8_t* sb = sa + P4_A_BYTES;
        uint8_t* sfa = sb + P4_B_BYTES;
        uint8_t* sfb = sfa + P4_SFA_BYTES;
        const int x = kb * 128;
        tma_load_2d_pair(sa, &mA, bar, x, mb * BM, el);
        if (args.b_dual)
          tma_load_2d_pair(sb, rank ? &mB1 : &mB0, bar, x, nb * (F4_BN / 2), el);
        else
          tma_load_2d_pair(sb, &mB0, bar, x, nb * F4_BN + static_cast<int>(rank) * (F4_BN / 2), el);
        tma_load_2d_pair(sfa, &mSA, bar, 0, 8 * (mb * static_cast<int>(sc.kt) + kb), el);
        // B's scales: this CTA loads the group of its own B rows into slot
        // `rank` of both CTAs' scale area
        const int cb = args.b_dual ? nb * static_cast<int>(sc.kt) + kb
                                   : (2 * nb + static_cast<int>(rank)) * static_cast<int>(sc.kt) + kb;
        tma_load_2d_pair_mc(sfb + rank * 2048, (args.b_dual && rank) ? &mSB1 : &mSB0, bar, 0, 8 * cb, 0x3, el);
      }
    }
    if (aborted) {
      if (leader) {
        const uint32_t first = it > static_cast<uint32_t>(S) ? it - S : 0;
        for (uint32_t j = first; j < it; ++j) mbar_wait_drain(&full[j % S], (j / S) & 1, 200000000ull);
      } else {
        const uint64_t t0 = globaltimer_ns();
        while (globaltimer_ns() - t0 < 2000000ull) {
        }
      }
    }
  } else if (warp == 1) {
    // ------------------------------------------------------------ scale copies + MMA issuer (leader)
    if (leader) {
      const uint32_t el = elect_one();
      uint32_t it = 0, t = 0;
      bool issued = false;
      const uint32_t idesc = args.idesc;
      for (int u = cluster_id; u < args.num_units && !aborted; u += num_clusters, ++t) {
        if (!mbar_wait_bounded(tempty, (t & 1) ^ 1, abort_flag, args.status, args.timeout_ns)) {
          aborted = true;
          break;
        }
        tc_fence_after();
        for (int kb = 0; kb < num_kb; ++kb, ++it) {
          const int s = it % S;
          if (!mbar_wait_bounded(&full[s], (it / S) & 1, abort_flag, args.status, args.timeout_ns)) {
            aborted = true;
            break;
          }
          tc_fence_after();
          const uint32_t sa = smem_u32(tiles + s * P4_STAGE_BYTES);
          const uint32_t sb = sa + P4_A_BYTES;
          const uint32_t sfa = sb + P4_B_BYTES;
          const uint32_t sfb = sfa + P4_SFA_BYTES;
          const uint32_t slot = tmem_base + F4_SF_COL0 + static_cast<uint32_t>(s) * P4_SF_SLOT_COLS;
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            tmem_cp_32x128_x4_pair(slot + g * 4, sdesc_plain(sfa + g * 512, 128, 128), el);
            tmem_cp_32x128_x4_pair(slot + 16 + g * 8, sdesc_plain(sfb + g * 512, 128, 128), el);
            tmem_cp_32x128_x4_pair(slot + 16 + g * 8 + 4, sdesc_plain(sfb + 2048 + g * 512, 128, 128), el);
          }
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            const uint64_t ad = sdesc_sw128(sa + g * 32, 16, 1024);
            const uint64_t bd = sdesc_sw128(sb + g * 32, 16, 1024);
            umma_nvfp4_pair(tmem_base, ad, bd, idesc, slot + g * 4, slot + 16 + g * 8, (kb | g) != 0, el);
          }
          issued = true;
          umma_commit_pair_mc(&empty[s], 0x3, el);
        }
        if (aborted) break;
        umma_commit_pair_mc(tfull, 0x3, el);
      }
      if (aborted && issued) {
        umma_commit_pair(drain, el);
        mbar_wait_drain(drain, 0, 200000000ull);
      }
    }
  } else {
    // ------------------------------------------------------------ epilogue (both CTAs)
    const int q = warp & 3;
    const int h = (warp - 2) >> 2;
    uint32_t t = 0;
    for (int u = cluster_id; u < args.num_units && !aborted; u += num_clusters, ++t) {
      int mbc, nb, nlen, chunk;
      unit_coords(args, u, mbc, nb, nlen, chunk);
      const int mb = mbc * 2 + static_cast<int>(rank);
      TileInfo ti;
      ti.mb = mb;
      ti.nb = nb;
      ti.unit_chunk = chunk;
      ti.row = mb * BM + q * 32 + lane;
      ti.M = args.M;
      ti.N = args.N;
      ti.status = args.status;
      ti.stage = epi_stage + (warp - 2) * F4_EPI_WARP_BYTES;
      ti.taddr = tmem_base + (static_cast<uint32_t>(q * 32) << 16);
      f4_epilogue<KIND, true>(args.e, ti, h, tfull, t & 1, tempty, abort_flag, args.timeout_ns,
                              args.epilogue_sleep_ns, aborted);
    }
  }

  tc_fence_before();
  __syncthreads();
  cluster_sync();  // no CTA leaves while its peer may still write or signal it
  tc_fence_after();
  if (warp == 1) {
    __syncwarp();
    tmem_dealloc<true>(tmem_base, F4_TMEM_COLS);
  }
}

template <int KIND>
cudaError_t launch_nvfp4_pair(int num_units, int sms, cudaStream_t s, const CUtensorMap* m, const GemmArgs& a,
                              const Nvfp4Scales& sc) {
  static std::mutex init;
  static std::atomic<bool> attr_done[64];
  static std::atomic<int> max_clusters[64];
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  auto kern = coda_gemm_nvfp4_pair_kernel<KIND>;
  cudaLaunchConfig_t cfg = {};
  cfg.blockDim = dim3(F4_THREADS);
  cfg.dynamicSmemBytes = P4_SMEM;
  cfg.stream = s;
  cudaLaunchAttribute attr[1];
  attr[0].id = cudaLaunchAttributeClusterDimension;
  attr[0].val.clusterDim.x = 2;
  attr[0].val.clusterDim.y = 1;
  attr[0].val.clusterDim.z = 1;
  cfg.attrs = attr;
  cfg.numAttrs = 1;
  if (!attr_done[dev].load(std::memory_order_acquire)) {
    std::lock_guard<std::mutex> lock(init);
    if (!attr_done[dev].load(std::memory_order_relaxed)) {
      e = cudaFuncSetAttribute(kern, cudaFuncAttributeMaxDynamicSharedMemorySize, static_cast<int>(P4_SMEM));
      if (e != cudaSuccess) return e;
      cfg.gridDim = dim3(static_cast<unsigned>(sms - sms % 2));
      int n = 0;
      e = cudaOccupancyMaxActiveClusters(&n, kern, &cfg);
      if (e != cudaSuccess) return e;
      if (n <= 0) return cudaErrorInvalidConfiguration;
      max_clusters[dev].store(n, std::memory_order_relaxed);
      attr_done[dev].store(true, std::memory_order_release);
    }
  }
  const int resident = max_clusters[dev].load(std::memory_order_relaxed);
  cfg.gridDim = dim3(static_cast<unsigned>(2 * std::min(num_units, resident)));
  note_launch();
  e = cudaLaunchKernelEx(&cfg, kern, m[0], m[1], m[2], m[3], m[4], m[5], a, sc);
  if (e != cudaSuccess) return e;
  return cudaGetLastError();
}

}  // namespace

uint32_t nvfp4_idesc() { return idesc_nvfp4(BM, F4_BN); }
uint32_t nvfp4_idesc_pair() { return idesc_nvfp4(2 * BM, F4_BN); }

// CTA pairs: CODA_NVFP4=pair in the environment selects them when there are
// at least two 128-row blocks.
bool nvfp4_pairs(int64_t M) {
  static const bool env = [] {
    const char* v = std::getenv("CODA_NVFP4");
    return v && std::strcmp(v, "pair") == 0;
  }();
  return env && M > BM;
}

cudaError_t launch_gemm_nvfp4_pair(int kind, int num_units, int sms, cudaStream_t s, const CUtensorMap* m,
                                   const GemmArgs& a, const Nvfp4Scales& sc) {
  return kind == 1 ? launch_nvfp4_pair<1>(num_units, sms, s, m, a, sc)
                   : launch_nvfp4_pair<0>(num_units, sms, s, m, a, sc);
}

// Variant: single CTAs by default; CODA_NVFP4=2 or 4 in the environment
// selects clusters of that many CTAs sharing the B tile (for comparisons)
// when there are at least as many 128-row blocks.
int nvfp4_cluster_size(int64_t M) {
  static const int env = [] {
    const char* v = std::getenv("CODA_NVFP4");
    const int c = v ? std::atoi(v) : 1;
    return c == 2 || c == 4 ? c : 1;
  }();
  return M > (env - 1) * BM ? env : 1;
}

cudaError_t launch_quantize_nvfp4_rows(const __nv_bfloat16* X, int64_t ldx, int64_t M, int64_t K, uint8_t* Q,
                                       uint8_t* SF, float* scale, int num_sms, cudaStream_t s, const float* gamma,
                                       float* rstd, float eps) {
  const int64_t rows_pad = (M + 511) / 512 * 512;
  const int64_t kt = (K + 255) / 256;
  const int64_t blocks = std::min<int64_t>((rows_pad + 7) / 8, static_cast<int64_t>(num_sms) * 8);
  const unsigned grid = static_cast<unsigned>(std::max<int64_t>(blocks, 1));
  note_launch();
  if (gamma && rstd)
    quantize_nvfp4_rows_kernel<true, true><<<grid, 256, 0, s>>>(X, ldx, M, K, Q, SF, scale, rows_pad, kt, gamma,
                                                                  rstd, eps);
  else if (gamma)
    quantize_nvfp4_rows_kernel<true, false><<<grid, 256, 0, s>>>(X, ldx, M, K, Q, SF, scale, rows_pad, kt, gamma,
                                                                   rstd, eps);
  else if (rstd)
    quantize_nvfp4_rows_kernel<false, true><<<grid, 256, 0, s>>>(X, ldx, M, K, Q, SF, scale, rows_pad, kt, gamma,
                                                                   rstd, eps);
  else
    quantize_nvfp4_rows_kernel<false, false><<<grid, 256, 0, s>>>(X, ldx, M, K, Q, SF, scale, rows_pad, kt, gamma,
                                                                    rstd, eps);
  return cudaGetLastError();
}

cudaError_t launch_gemm_plain_nvfp4(int cg, int num_units, int sms, cudaStream_t s, const CUtensorMap* m,
                                    const GemmArgs& a, const Nvfp4Scales& sc) {
  switch (cg) {
    case 1: return launch_nvfp4<0, 1>(num_units, sms, s, m, a, sc);
    case 2: return launch_nvfp4<0, 2>(num_units, sms, s, m, a, sc);
    case 4: return launch_nvfp4<0, 4>(num_units, sms, s, m, a, sc);
    default: return cudaErrorInvalidValue;
  }
}
cudaError_t launch_gemm_swiglu_nvfp4(int cg, int num_units, int sms, cudaStream_t s, const CUtensorMap* m,
                                     const GemmArgs& a, const Nvfp4Scales& sc) {
  switch (cg) {
    case 1: return launch_nvfp4<1, 1>(num_units, sms, s, m, a, sc);
    case 2: return launch_nvfp4<1, 2>(num_units, sms, s, m, a, sc);
    case 4: return launch_nvfp4<1, 4>(num_units, sms, s, m, a, sc);
    default: return cudaErrorInvalidValue;
  }
}

}  // namespace coda
