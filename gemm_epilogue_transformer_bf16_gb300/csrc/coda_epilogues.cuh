// Epilogue functors for coda_gemm_kernel.
//
// Each functor is one composition of the five epilogue primitive classes of
// "CODA: Rewriting Transformer Blocks as GEMM-Epilogue Programs" §3.1:
//   (1) element-wise / pairwise maps, (2) rank-1 vector loads/stores,
//   (3) rank-2 tile loads/stores, (4) tile row/column reductions to partials
//   merged by a small second kernel, (5) running state across tiles.
//
// Thread layout: epilogue thread = one output row of the 128-row tile
// (its TMEM lane); it walks the tile's columns 32 at a time.  Row reductions
// are therefore thread-local; column reductions use a warp reduce-scatter.
// All TMEM loads are executed by full warps (rows past M only mask their
// global accesses).  The large bf16 outputs leave through warp_store_bf16x32,
// which turns the warp's 32 rows x 32 columns into row-contiguous stores.
#pragma once
#include "coda_gemm.cuh"

namespace coda {

constexpr float LOG2E = 1.4426950408889634f;

__device__ __forceinline__ void load_f32x8(const float* p, float* o) {
  const float4 a = *reinterpret_cast<const float4*>(p);
  const float4 b = *reinterpret_cast<const float4*>(p + 4);
  o[0] = a.x; o[1] = a.y; o[2] = a.z; o[3] = a.w;
  o[4] = b.x; o[5] = b.y; o[6] = b.z; o[7] = b.w;
}
__device__ __forceinline__ void store_f32x8(float* p, const float* v) {
  *reinterpret_cast<float4*>(p) = make_float4(v[0], v[1], v[2], v[3]);
  *reinterpret_cast<float4*>(p + 4) = make_float4(v[4], v[5], v[6], v[7]);
}

// Stores a warp's 32 rows x 32 columns as bf16: thread `lane` passes the 32
// values of row row0 + lane, columns col0 .. col0 + 31.  The fragment goes
// through the warp's 2 KB shared-memory buffer -- 16-byte chunk p of row r
// sits at r * 64 + ((p ^ ((r >> 1) & 3)) * 16), so the row-wise writes and
// the column-wise reads are both free of bank conflicts -- and leaves as
// 16-byte stores that each cover 8 rows x 64 contiguous bytes (whole 32-byte
// sectors) instead of 32 rows x 16 bytes.  Rows >= M and columns >= N are
// not written (N is a multiple of 8).  Called by all 32 lanes.
// Same, from the 32 values already rounded and packed in pairs (pk[i] holds
// columns 2i and 2i + 1).
__device__ __forceinline__ void warp_store_bf16x32_packed(uint8_t* stage, __nv_bfloat16* base, int64_t ld, int row0,
                                                          int M, int col0, int N, const uint32_t* pk, bool stream) {
  const int lane = threadIdx.x & 31;
#pragma unroll
  for (int p = 0; p < 4; ++p) {
    const uint4 w = make_uint4(pk[p * 4 + 0], pk[p * 4 + 1], pk[p * 4 + 2], pk[p * 4 + 3]);
    *reinterpret_cast<uint4*>(stage + lane * 64 + ((p ^ ((lane >> 1) & 3)) * 16)) = w;
  }
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const int r = i * 8 + (lane >> 2), p = lane & 3;
    const uint4 w = *reinterpret_cast<const uint4*>(stage + r * 64 + ((p ^ ((r >> 1) & 3)) * 16));
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
__device__ __forceinline__ void warp_store_bf16x32(uint8_t* stage, __nv_bfloat16* base, int64_t ld, int row0,
                                                   int M, int col0, int N, const float* v, bool stream) {
  uint32_t pk[16];
#pragma unroll
  for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
  warp_store_bf16x32_packed(stage, base, ld, row0, M, col0, N, pk, stream);
}

// Reduce-scatter over the warp: on entry thread `lane` holds p[0..31] of its
// row; afterwards p[0] of lane L is the sum over the warp's 32 rows of column
// L.  Fixed order, so bitwise reproducible.
__device__ __forceinline__ void warp_colsum_partial(float* p, int lane) {
  __syncwarp();
#pragma unroll
  for (int i = 0; i < 16; ++i) {
    const bool hi = lane & 16;
    const float keep = hi ? p[i + 16] : p[i];
    const float send = hi ? p[i] : p[i + 16];
    p[i] = keep + __shfl_xor_sync(0xffffffffu, send, 16);
  }
#pragma unroll
  for (int i = 0; i < 8; ++i) {
    const bool hi = lane & 8;
    const float keep = hi ? p[i + 8] : p[i];
    const float send = hi ? p[i] : p[i + 8];
    p[i] = keep + __shfl_xor_sync(0xffffffffu, send, 8);
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    const bool hi = lane & 4;
    const float keep = hi ? p[i + 4] : p[i];
    const float send = hi ? p[i] : p[i + 4];
    p[i] = keep + __shfl_xor_sync(0xffffffffu, send, 4);
  }
#pragma unroll
  for (int i = 0; i < 2; ++i) {
    const bool hi = lane & 2;
    const float keep = hi ? p[i + 2] : p[i];
    const float send = hi ? p[i] : p[i + 2];
    p[i] = keep + __shfl_xor_sync(0xffffffffu, send, 2);
  }
  {
    const bool hi = lane & 1;
    const float keep = hi ? p[1] : p[0];
    const float send = hi ? p[0] : p[1];
    p[0] = keep + __shfl_xor_sync(0xffffffffu, send, 1);
  }
}

// The accumulator chunk of columns col0 .. col0 + 31, with the FP8 operand
// scales applied when SCALED: acc * acc_rs[row] * acc_cs[col] (columns >= N
// scaled by 0).  Without them it is tmem_ld32; each epilogue chooses SCALED
// once per tile.
template <bool SCALED>
__device__ __forceinline__ void tmem_ld32_acc_t(uint32_t taddr, float (&v)[32], const EpiArgs& e, int row, bool rv,
                                                int col0, int N) {
  tmem_ld32(taddr, v);
  if (SCALED) {
    const float rs = (e.acc_rs && rv) ? e.acc_rs[row] : 1.f;
#pragma unroll
    for (int g = 0; g < 4; ++g) {
      float s8[8];
      if (e.acc_cs && col0 + g * 8 < N) {
        load_f32x8(e.acc_cs + col0 + g * 8, s8);
      } else {
#pragma unroll
        for (int i = 0; i < 8; ++i) s8[i] = (col0 + g * 8 < N) ? 1.f : 0.f;
      }
#pragma unroll
      for (int i = 0; i < 8; ++i) v[g * 8 + i] *= rs * s8[i];
    }
  }
}

// ---------------------------------------------------------------------------
// PLAIN:  D = rs_i * cs_j * acc + aux0 (+ acc_in) - coef_i * aux1[g_i]
//             - coef2_i * aux3 - sum_{t in csr(i)} w_t * aux2[t]  (+ D if beta)
// optional row partial  sum_j D_ij^2  (of the stored, rounded values), and
// optional second output  out1 = bf16(D_ij * cs2_j)  (D as stored: the
// input of the next RMSNorm-reparameterised GEMM, x ⊙ gamma, written by the
// epilogue that produces x).
// Covers: plain store, residual add, RMSNorm row-scale (+ residual),
// accumulate, the residual + partial-RMS epilogue, dX - c*X of the
// RMSNorm-reparameterised backward, and the exact one-hot terms of the
// cross-entropy backward (g_i = label row gather; csr = tokens per label).
// ---------------------------------------------------------------------------
template <int BN>
struct EpiPlain {
  struct State {};
  static constexpr int RING = 1;  // the residual (aux0) can come through the TMA ring
  static __device__ __forceinline__ int chunks(const TileInfo& t) {
    return max(0, min(BN / 32, (t.N - t.nb * BN + 31) / 32));
  }
  static __device__ __forceinline__ void begin(State&, const EpiArgs&, const TileInfo&) {}
  static __device__ __forceinline__ void end(State&, const EpiArgs&, const TileInfo&) {}
  // Issued before the tile's accumulator is ready (while its mainloop still
  // runs).  With the ring, the first RING_SLOTS chunks of the warp's
  // residual rows are copied into shared memory; otherwise the thread's row
  // segments of the tile's input tiles are requested into L2, so the chunk
  // loop's loads wait on L2 rather than on DRAM once per chunk (the last
  // tile's epilogue has no mainloop to hide behind).
  static __device__ __forceinline__ void prefetch(const EpiArgs& e, const TileInfo& t) {
    if (e.ring) {
      const int n = min(chunks(t), RING_SLOTS);
      const uint32_t g0 = t.ring_cnt[0];
      const int row0 = t.row - static_cast<int>(threadIdx.x & 31);
      for (int c = 0; c < n; ++c) ring_issue(t, 1, g0 + c, t.nb * BN + c * 32, row0);
      __syncwarp();
      if ((threadIdx.x & 31) == 0) t.ring_cnt[0] = g0 + n;
      __syncwarp();
    }
    const int row = t.row;
    const int cbase = t.nb * BN;
    if (!e.aux_prefetch || row >= t.M || cbase >= t.N) return;
    const int cols = min(BN, t.N - cbase);
    const int64_t arow = e.gather_rows ? e.gather_rows[row] : row;
    if (e.aux0 && !e.ring) prefetch_l2_span(e.aux0 + static_cast<int64_t>(row) * e.ld_aux0 + cbase, cols * 2);
    if (e.acc_in) prefetch_l2_span(e.acc_in + static_cast<int64_t>(row) * e.ld_acc_in + cbase, cols * 4);
    if (e.row_coef && arow >= 0) prefetch_l2_span(e.aux1 + arow * e.ld_aux1 + cbase, cols * 2);
    if (e.row_coef2) prefetch_l2_span(e.aux3 + static_cast<int64_t>(row) * e.ld_aux3 + cbase, cols * 2);
    if (e.beta)
      prefetch_l2_span(static_cast<const uint8_t*>(e.D) + (static_cast<int64_t>(row) * e.ldd + cbase) * (e.d_f32 ? 4 : 2),
                       cols * (e.d_f32 ? 4 : 2));
  }
  // GEN = false compiles the chunk loop for the launches that need only the
  // row scale, the residual, the row partial sums and the second output (the
  // block's projections, the RMSNorm-linear forward): with one epilogue warp
  // per SM sub-partition, the other features' per-chunk tests cost as much
  // as the arithmetic they guard.
  // RES (lean loops only): the residual is absent (0), loaded into registers
  // (1) or read from the TMA ring (2).
  static __device__ __forceinline__ void tile(State& st, const EpiArgs& e, const TileInfo& t) {
    const bool gen = e.no_lean || e.col_scale || e.acc_in || e.row_coef || e.row_coef2 || e.csr_off || e.d_f32 ||
                     e.beta || e.gather_rows;
    if (gen)
      tile_impl<true, 1>(st, e, t);
    else if (!e.aux0)
      tile_impl<false, 0>(st, e, t);
    else if (e.ring)
      tile_impl<false, 2>(st, e, t);
    else
      tile_impl<false, 1>(st, e, t);
  }
  template <bool GEN, int RES>
  static __device__ __forceinline__ void tile_impl(State&, const EpiArgs& e, const TileInfo& t) {
    const bool has_res = GEN ? e.aux0 != nullptr : RES > 0;
    const int row = t.row;
    const bool rv = row < t.M;
    const float rs = (e.row_scale && rv) ? e.row_scale[row] : 1.f;
    const float rc = (GEN && e.row_coef && rv) ? e.row_coef[row] : 0.f;
    const float rc2 = (GEN && e.row_coef2 && rv) ? e.row_coef2[row] : 0.f;
    const int64_t arow = (GEN && e.gather_rows) ? (rv ? e.gather_rows[row] : -1) : row;
    int cb0 = 0, cb1 = 0;
    if (GEN && e.csr_off && rv) {
      cb0 = e.csr_off[row];
      cb1 = e.csr_off[row + 1];
    }
    float ss = 0.f;
    const int row0 = row - static_cast<int>(threadIdx.x & 31);
    // The residual tile (aux0) arrives either through the TMA ring (issued
    // RING_SLOTS chunks ahead, the first ones before the accumulator was
    // ready) or, without it, in registers one 32-column chunk ahead, so its
    // L2 round trip overlaps the previous chunk's math and stores.  Per-lane
    // loads of 32 different rows wait ~3000 cycles on a busy SM, longer than
    // a chunk's math and stores, which is what the ring removes.
    const int64_t aoff = static_cast<int64_t>(row) * e.ld_aux0;
    uint4 an[4];
    auto fetch = [&](int col0) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int cc = col0 + q * 8;
        an[q] = (rv && cc < t.N) ? *reinterpret_cast<const uint4*>(e.aux0 + aoff + cc) : make_uint4(0u, 0u, 0u, 0u);
      }
    };
    const bool use_ring = GEN ? e.ring != 0 : RES == 2;
    const int nch = chunks(t);
    uint32_t g_done = use_ring ? t.ring_cnt[1] : 0u, g_issued = use_ring ? t.ring_cnt[0] : 0u;
    if (has_res && !use_ring) fetch(t.nb * BN);
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      const int col0 = t.nb * BN + c;
      if (col0 >= t.N) break;
      uint4 ac[4];
      if (use_ring) {
        if (!ring_wait(t, g_done)) break;
#pragma unroll
        for (int q = 0; q < 4; ++q) ac[q] = ring_read(t, 1, g_done, 0, q);
        __syncwarp();
        ++g_done;
        if (c / 32 + RING_SLOTS < nch) {
          ring_issue(t, 1, g_issued, col0 + RING_SLOTS * 32, row0);
          ++g_issued;
        }
      } else {
#pragma unroll
        for (int q = 0; q < 4; ++q) ac[q] = an[q];
        if (has_res && c + 32 < BN) fetch(col0 + 32);
      }
      float v[32];
      __syncwarp();
      tmem_ld32(t.taddr + c, v);
      if (rv) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int cc = col0 + g * 8;
          float* x = v + g * 8;
          if (cc < t.N) {
#pragma unroll
            for (int i = 0; i < 8; ++i) x[i] *= rs;
            if (GEN && e.col_scale) {
              float s8[8];
              load_f32x8(e.col_scale + cc, s8);
#pragma unroll
              for (int i = 0; i < 8; ++i) x[i] *= s8[i];
            }
            if (has_res) {
              float r8[8];
              bf16x8_to_f32(ac[g], r8);
#pragma unroll
              for (int i = 0; i < 8; ++i) x[i] += r8[i];
            }
            if (GEN && e.acc_in) {
              float a8[8];
              load_f32x8(e.acc_in + static_cast<int64_t>(row) * e.ld_acc_in + cc, a8);
#pragma unroll
              for (int i = 0; i < 8; ++i) x[i] += a8[i];
            }
            if (GEN && e.row_coef && arow >= 0) {
              float r8[8];
              load_bf16x8(e.aux1 + arow * e.ld_aux1 + cc, r8);
#pragma unroll
              for (int i = 0; i < 8; ++i) x[i] -= rc * r8[i];
            }
            if (GEN && e.row_coef2) {
              float r8[8];
              load_bf16x8(e.aux3 + static_cast<int64_t>(row) * e.ld_aux3 + cc, r8);
#pragma unroll
              for (int i = 0; i < 8; ++i) x[i] -= rc2 * r8[i];
            }
            for (int j = cb0; GEN && j < cb1; ++j) {
              const int32_t t2 = e.csr_idx[j];
              const float w2 = e.csr_w[t2];
              float r8[8];
              load_bf16x8(e.aux2 + static_cast<int64_t>(t2) * e.ld_aux2 + cc, r8);
#pragma unroll
              for (int i = 0; i < 8; ++i) x[i] -= w2 * r8[i];
            }
            if (GEN && e.d_f32) {
              float* d = static_cast<float*>(e.D) + static_cast<int64_t>(row) * e.ldd + cc;
              if (e.beta) {
                float o8[8];
                load_f32x8(d, o8);
#pragma unroll
                for (int i = 0; i < 8; ++i) x[i] += o8[i];
              }
              store_f32x8(d, x);
              if (e.partials) {
#pragma unroll
                for (int i = 0; i < 8; ++i) ss += x[i] * x[i];
              }
            } else {
              if (GEN && e.beta) {
                float o8[8];
                load_bf16x8(static_cast<const __nv_bfloat16*>(e.D) + static_cast<int64_t>(row) * e.ldd + cc, o8);
#pragma unroll
                for (int i = 0; i < 8; ++i) x[i] += o8[i];
              }
            }
          }
        }
      }
      if (!GEN || !e.d_f32) {
        // Each output is rounded to bf16 once (packed in pairs); the row's
        // partial sum of squares and the second output read the rounded
        // values back from the packed words.
        uint32_t pk[16];
#pragma unroll
        for (int i = 0; i < 16; ++i) pk[i] = pack_bf16x2(v[2 * i], v[2 * i + 1]);
        if (e.partials && rv) {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            if (col0 + g * 8 < t.N) {
#pragma unroll
              for (int i = 0; i < 4; ++i) {
                const float lo = bf16_lo(pk[g * 4 + i]), hi = bf16_hi(pk[g * 4 + i]);
                ss += lo * lo;
                ss += hi * hi;
              }
            }
          }
        }
        warp_store_bf16x32_packed(t.stage, static_cast<__nv_bfloat16*>(e.D), e.ldd, row0, t.M, col0, t.N, pk,
                                  e.st_stream);
        if (e.out1) {
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            float s8[8];
            if (col0 + g * 8 < t.N)
              load_f32x8(e.col_scale2 + col0 + g * 8, s8);
            else
#pragma unroll
              for (int i = 0; i < 8; ++i) s8[i] = 0.f;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              v[g * 8 + 2 * i] = bf16_lo(pk[g * 4 + i]) * s8[2 * i];
              v[g * 8 + 2 * i + 1] = bf16_hi(pk[g * 4 + i]) * s8[2 * i + 1];
            }
          }
          warp_store_bf16x32(t.stage, e.out1, e.ld_out1, row0, t.M, col0, t.N, v, e.st_stream);
        }
      }
    }
    if (use_ring) {
      __syncwarp();
      if ((threadIdx.x & 31) == 0) {
        t.ring_cnt[0] = g_issued;
        t.ring_cnt[1] = g_done;
      }
      __syncwarp();
    }
    if (e.partials && rv) e.partials[static_cast<int64_t>(t.nb) * e.ld_part + row] = ss;
  }
};

// ---------------------------------------------------------------------------
// SWIGLU (pairwise map on co-resident gate/up accumulators):
//   accumulator columns [0, BN/2) = X Wg^T, [BN/2, BN) = X Wu^T for the same
//   output columns;  g = rs*acc_g, u = rs*acc_u, H = silu(g) * u.  With FP8
//   operands rs also carries the token scale and g, u the per-column weight
//   scales (col_scale, col_scale2).
//   Optionally stores g and u (bf16) for the backward.
// ---------------------------------------------------------------------------
// UP: TMEM column offset of the up half from the gate half (BN / 2 when the
// tile is [gate | up]; a kernel that hands each epilogue warp a column range
// of a wider tile passes the wider tile's half).
template <int BN, int UP = BN / 2>
struct EpiSwiglu {
  struct State {};
  static constexpr int HALF = BN / 2;
  static __device__ __forceinline__ void begin(State&, const EpiArgs&, const TileInfo&) {}
  static __device__ __forceinline__ void end(State&, const EpiArgs&, const TileInfo&) {}
  static __device__ __forceinline__ void prefetch(const EpiArgs&, const TileInfo&) {}
  // per-tile choice of loop: per-column scales (FP8 weights), stored g and u
  static __device__ __forceinline__ void tile(State& st, const EpiArgs& e, const TileInfo& t) {
    const bool gu = e.out1 && e.out2;
    if (e.col_scale) {
      if (gu)
        tile_impl<true, true>(st, e, t);
      else
        tile_impl<true, false>(st, e, t);
    } else {
      if (gu)
        tile_impl<false, true>(st, e, t);
      else
        tile_impl<false, false>(st, e, t);
    }
  }
  // GU: both g and u are stored (otherwise each only if its pointer is set)
  template <bool CS, bool GU>
  static __device__ __forceinline__ void tile_impl(State&, const EpiArgs& e, const TileInfo& t) {
    const int row = t.row;
    const bool rv = row < t.M;
    const float rs = ((e.row_scale && rv) ? e.row_scale[row] : 1.f) * ((e.row_scale2 && rv) ? e.row_scale2[row] : 1.f);
    const int row0 = row - static_cast<int>(threadIdx.x & 31);
#pragma unroll 1
    for (int c = 0; c < HALF; c += 32) {
      const int col0 = t.nb * HALF + c;
      if (col0 >= t.N) break;
      float g[32], u[32];
      __syncwarp();
      tmem_ld32(t.taddr + c, g);
      tmem_ld32(t.taddr + UP + c, u);
      if (rv) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          const int cc = col0 + q * 8;
          float cg[8], cu[8];
          if (CS && cc < t.N) {
            load_f32x8(e.col_scale + cc, cg);
            load_f32x8(e.col_scale2 + cc, cu);
          }
#pragma unroll
          for (int i = 0; i < 8; ++i) {
            g[q * 8 + i] *= rs;
            u[q * 8 + i] *= rs;
            if (CS && cc < t.N) {
              g[q * 8 + i] *= cg[i];
              u[q * 8 + i] *= cu[i];
            }
          }
        }
      }
      float h[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) h[i] = g[i] / (1.f + __expf(-g[i])) * u[i];
      auto* D = static_cast<__nv_bfloat16*>(e.D);
      warp_store_bf16x32(t.stage, D, e.ldd, row0, t.M, col0, t.N, h, e.st_stream);
      if (GU || e.out1) warp_store_bf16x32(t.stage, e.out1, e.ld_out1, row0, t.M, col0, t.N, g, e.st_stream);
      if (GU || e.out2) warp_store_bf16x32(t.stage, e.out2, e.ld_out2, row0, t.M, col0, t.N, u, e.st_stream);
    }
  }
};

// ---------------------------------------------------------------------------
// DSWIGLU on the dH = dY Wd GEMM: loads the saved g, u tiles (aux0, aux1),
//   dG = dH u s (1 + g (1 - s)),  dU = dH g s,   s = sigmoid(g)
// stores rs*dG (out1) and rs*dU (out2) -- the row-scaled gradients G' that
// the RMSNorm-reparameterised backward feeds to its GEMMs -- and, when
// `partials` is set, the row partial sum_j (dG g + dU u) that the RMSNorm
// backward coefficient needs.  out3 (optional) receives H = silu(g) u.
// ---------------------------------------------------------------------------
template <int BN>
struct EpiDSwiglu {
  struct State {};
  static __device__ __forceinline__ void begin(State&, const EpiArgs&, const TileInfo&) {}
  static __device__ __forceinline__ void end(State&, const EpiArgs&, const TileInfo&) {}
  static __device__ __forceinline__ void prefetch(const EpiArgs& e, const TileInfo& t) {
    const int cbase = t.nb * BN;
    if (!e.aux_prefetch || t.row >= t.M || cbase >= t.N) return;
    const int bytes = min(BN, t.N - cbase) * 2;
    prefetch_l2_span(e.aux0 + static_cast<int64_t>(t.row) * e.ld_aux0 + cbase, bytes);
    prefetch_l2_span(e.aux1 + static_cast<int64_t>(t.row) * e.ld_aux1 + cbase, bytes);
  }
  // The per-tile choice of loop (FP8 operand scales, the H output) keeps
  // feature tests out of the chunk loop.
  static __device__ __forceinline__ void tile(State& st, const EpiArgs& e, const TileInfo& t) {
    const bool scaled = e.acc_rs || e.acc_cs;
    if (e.out3) {
      if (scaled)
        tile_impl<true, true>(st, e, t);
      else
        tile_impl<false, true>(st, e, t);
    } else {
      if (scaled)
        tile_impl<true, false>(st, e, t);
      else
        tile_impl<false, false>(st, e, t);
    }
  }
  template <bool SCALED, bool OUT3>
  static __device__ __forceinline__ void tile_impl(State&, const EpiArgs& e, const TileInfo& t) {
    const int row = t.row;
    const bool rv = row < t.M;
    const float rs = (e.row_scale && rv) ? e.row_scale[row] : 1.f;
    float dot = 0.f;
    const int row0 = row - static_cast<int>(threadIdx.x & 31);
    // The thread's row segments of g and u for the whole tile were requested
    // into L2 by prefetch(), before the accumulator was ready, and each
    // 32-column chunk's g and u are loaded into registers one chunk ahead, so
    // that their latency overlaps the previous chunk's math and stores (at
    // K = 4096 one round trip per chunk made this epilogue longer than the
    // next tile's mainloop).
    const int cbase = t.nb * BN;
    const int64_t goff = static_cast<int64_t>(row) * e.ld_aux0;
    const int64_t uoff = static_cast<int64_t>(row) * e.ld_aux1;
    uint4 gn[4], un[4];  // the next chunk's g and u, raw bf16
    auto fetch = [&](int col0) {
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        const int cc = col0 + q * 8;
        if (rv && cc < t.N) {
          gn[q] = *reinterpret_cast<const uint4*>(e.aux0 + goff + cc);
          un[q] = *reinterpret_cast<const uint4*>(e.aux1 + uoff + cc);
        } else {
          gn[q] = make_uint4(0u, 0u, 0u, 0u);
          un[q] = make_uint4(0u, 0u, 0u, 0u);
        }
      }
    };
    fetch(cbase);
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      const int col0 = cbase + c;
      if (col0 >= t.N) break;
      uint4 gc[4], uc[4];
#pragma unroll
      for (int q = 0; q < 4; ++q) {
        gc[q] = gn[q];
        uc[q] = un[q];
      }
      if (c + 32 < BN) fetch(col0 + 32);
      float dh[32], du[32] = {}, h[32] = {};  // rows past M keep zeros (never stored)
      __syncwarp();
      tmem_ld32_acc_t<SCALED>(t.taddr + c, dh, e, row, rv, col0, t.N);
      if (rv) {
#pragma unroll
        for (int q = 0; q < 4; ++q) {
          if (col0 + q * 8 < t.N) {
            float g8[8], u8[8];
            bf16x8_to_f32(gc[q], g8);
            bf16x8_to_f32(uc[q], u8);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float s = __fdividef(1.f, 1.f + __expf(-g8[i]));  // sigmoid(g); 0 once exp overflows
              const float sg = g8[i] * s;
              const float d = dh[q * 8 + i];
              const float dg = d * u8[i] * s * (1.f + g8[i] * (1.f - s));
              const float dui = d * sg;
              h[q * 8 + i] = sg * u8[i];
              dot += dg * g8[i] + dui * u8[i];
              dh[q * 8 + i] = dg * rs;   // G'_g
              du[q * 8 + i] = dui * rs;  // G'_u
            }
          }
        }
      }
      warp_store_bf16x32(t.stage, e.out1, e.ld_out1, row0, t.M, col0, t.N, dh, e.st_stream);
      warp_store_bf16x32(t.stage, e.out2, e.ld_out2, row0, t.M, col0, t.N, du, e.st_stream);
      if (OUT3) warp_store_bf16x32(t.stage, e.out3, e.ld_out3, row0, t.M, col0, t.N, h, e.st_stream);
    }
    if (e.partials && rv) e.partials[static_cast<int64_t>(t.nb) * e.ld_part + row] = dot;
  }
};

// ---------------------------------------------------------------------------
// COLDOT (weight-gradient epilogue of the RMSNorm-reparameterised backward):
// the accumulator is dW'[n, k] (rows = weight output features), optionally
// minus the rows of aux2 listed for row n in the CSR (the exact one-hot term
// of a cross-entropy head):  v = acc - sum_{t in csr(n)} w_t aux2[t, k];
//   D = cs_k * v                  (dW = dW' diag(gamma))
//   column partial  sum_n aux0[n, k] * v[n, k]     (dgamma contribution)
// written per (m block, warp) to partials[(mb*4 + warp) * ld_part + k].
// ---------------------------------------------------------------------------
template <int BN>
struct EpiColDot {
  struct State {};
  static __device__ __forceinline__ void begin(State&, const EpiArgs&, const TileInfo&) {}
  static __device__ __forceinline__ void end(State&, const EpiArgs&, const TileInfo&) {}
  static __device__ __forceinline__ void prefetch(const EpiArgs&, const TileInfo&) {}
  static __device__ __forceinline__ void tile(State&, const EpiArgs& e, const TileInfo& t) {
    const int row = t.row;
    const bool rv = row < t.M;
    const int lane = threadIdx.x & 31;
    const int q = (threadIdx.x >> 5) & 3;
    int cb0 = 0, cb1 = 0;
    if (e.csr_off && rv) {
      cb0 = e.csr_off[row];
      cb1 = e.csr_off[row + 1];
    }
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      const int col0 = t.nb * BN + c;
      if (col0 >= t.N) break;
      float v[32];
      __syncwarp();
      tmem_ld32(t.taddr + c, v);
      float p[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) p[i] = 0.f;
      if (rv) {
        const int64_t off = static_cast<int64_t>(row);
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int cc = col0 + g * 8;
          if (cc < t.N) {
            float w8[8], s8[8];
            for (int j = cb0; j < cb1; ++j) {
              const int32_t t2 = e.csr_idx[j];
              const float w2 = e.csr_w[t2];
              float r8[8];
              load_bf16x8(e.aux2 + static_cast<int64_t>(t2) * e.ld_aux2 + cc, r8);
#pragma unroll
              for (int i = 0; i < 8; ++i) v[g * 8 + i] -= w2 * r8[i];
            }
            load_bf16x8(e.aux0 + off * e.ld_aux0 + cc, w8);
            if (e.col_scale) load_f32x8(e.col_scale + cc, s8);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              p[g * 8 + i] = v[g * 8 + i] * w8[i];
              if (e.col_scale) v[g * 8 + i] *= s8[i];
            }
          }
        }
      }
      warp_store_bf16x32(t.stage, static_cast<__nv_bfloat16*>(e.D), e.ldd, row - lane, t.M, col0, t.N, v,
                         e.st_stream);
      warp_colsum_partial(p, lane);
      // (a CTA pair's second M block can lie wholly past M: no partial row for it)
      if (e.partials && col0 + lane < t.N && t.mb * BM < t.M)
        e.partials[static_cast<int64_t>(t.mb * 4 + q) * e.ld_part + col0 + lane] = p[0];
    }
  }
};

// ---------------------------------------------------------------------------
// RMSDX (input gradient of an RMSNorm-reparameterised projection whose GEMM
// read u = x ⊙ gamma, gamma applied by the producing epilogue): the
// accumulator is D = G' W with the weight not folded, and
//   out = cs_k * D + aux0 - coef_i * aux1     (gamma D + dX_resid - c x)
//   column partial  sum_i aux1[i, k] * D[i, k]  (dgamma contribution)
// written per (m block, warp) to partials[(mb*4 + warp) * ld_part + k].
// ---------------------------------------------------------------------------
template <int BN>
struct EpiRmsDx {
  struct State {};
  static __device__ __forceinline__ void begin(State&, const EpiArgs&, const TileInfo&) {}
  static __device__ __forceinline__ void end(State&, const EpiArgs&, const TileInfo&) {}
  // the tile's rows of x (and dX_resid) into L2, and its slice of gamma
  // (read by every lane) into L1, before the accumulator is ready
  static __device__ __forceinline__ void prefetch(const EpiArgs& e, const TileInfo& t) {
    const int cbase = t.nb * BN;
    if (!e.aux_prefetch || cbase >= t.N) return;
    const int cols = min(BN, t.N - cbase);
    const int lane = threadIdx.x & 31;
    if (lane * 32 < cols) asm volatile("prefetch.global.L1 [%0];" ::"l"(e.col_scale + cbase + lane * 32));
    if (t.row >= t.M) return;
    prefetch_l2_span(e.aux1 + static_cast<int64_t>(t.row) * e.ld_aux1 + cbase, cols * 2);
    if (e.aux0) prefetch_l2_span(e.aux0 + static_cast<int64_t>(t.row) * e.ld_aux0 + cbase, cols * 2);
  }
  // The per-tile choice of loop (residual gradient present, FP8 operand
  // scales) keeps feature tests out of the chunk loop.
  static __device__ __forceinline__ void tile(State& st, const EpiArgs& e, const TileInfo& t) {
    const bool scaled = e.acc_rs || e.acc_cs;
    if (e.aux0) {
      if (scaled)
        tile_impl<true, true>(st, e, t);
      else
        tile_impl<true, false>(st, e, t);
    } else {
      if (scaled)
        tile_impl<false, true>(st, e, t);
      else
        tile_impl<false, false>(st, e, t);
    }
  }
  template <bool RESID, bool SCALED>
  static __device__ __forceinline__ void tile_impl(State&, const EpiArgs& e, const TileInfo& t) {
    const int row = t.row;
    const bool rv = row < t.M;
    const int lane = threadIdx.x & 31;
    const int q = (threadIdx.x >> 5) & 3;
    const float rc = (e.row_coef && rv) ? e.row_coef[row] : 0.f;
    // x (aux1) and dX_resid (aux0) are loaded one 32-column chunk ahead
    // (as the residual in EpiPlain)
    const int64_t xoff = static_cast<int64_t>(row) * e.ld_aux1, roff = static_cast<int64_t>(row) * e.ld_aux0;
    uint4 xn[4], rn[4];
    auto fetch = [&](int col0) {
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        const int cc = col0 + k * 8;
        const bool in = rv && cc < t.N;
        xn[k] = in ? *reinterpret_cast<const uint4*>(e.aux1 + xoff + cc) : make_uint4(0u, 0u, 0u, 0u);
        rn[k] = (in && RESID) ? *reinterpret_cast<const uint4*>(e.aux0 + roff + cc) : make_uint4(0u, 0u, 0u, 0u);
      }
    };
    fetch(t.nb * BN);
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      const int col0 = t.nb * BN + c;
      if (col0 >= t.N) break;
      uint4 xc[4], rcur[4];
#pragma unroll
      for (int k = 0; k < 4; ++k) {
        xc[k] = xn[k];
        rcur[k] = rn[k];
      }
      if (c + 32 < BN) fetch(col0 + 32);
      float v[32];
      __syncwarp();
      tmem_ld32_acc_t<SCALED>(t.taddr + c, v, e, row, rv, col0, t.N);
      float p[32];
#pragma unroll
      for (int i = 0; i < 32; ++i) p[i] = 0.f;
      if (rv) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int cc = col0 + g * 8;
          if (cc < t.N) {
            float x8[8], s8[8], r8[8];
            bf16x8_to_f32(xc[g], x8);
            load_f32x8(e.col_scale + cc, s8);
            if (RESID) bf16x8_to_f32(rcur[g], r8);
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float d = v[g * 8 + i];
              p[g * 8 + i] = x8[i] * d;
              float o = d * s8[i];
              if (RESID) o += r8[i];
              v[g * 8 + i] = o - rc * x8[i];
            }
          }
        }
      }
      warp_store_bf16x32(t.stage, static_cast<__nv_bfloat16*>(e.D), e.ldd, row - lane, t.M, col0, t.N, v,
                         e.st_stream);
      warp_colsum_partial(p, lane);
      if (e.partials && col0 + lane < t.N && t.mb * BM < t.M)
        e.partials[static_cast<int64_t>(t.mb * 4 + q) * e.ld_part + col0 + lane] = p[0];
    }
  }
};

// ---------------------------------------------------------------------------
// CE_LSE (state transition): logits tile z = X W^T never leaves the chip.
// Per row, a running (max, sum-exp) over the unit's consecutive vocab tiles;
// the target logit is written when the label falls in the tile; at the end of
// the unit (one vocab chunk) the state goes to partials[chunk][row] (float2).
// ---------------------------------------------------------------------------
template <int BN>
struct EpiCeLse {
  struct State {
    float m, s;
    int label;
  };
  static __device__ __forceinline__ void begin(State& st, const EpiArgs& e, const TileInfo& t) {
    st.m = -INFINITY;
    st.s = 0.f;
    st.label = t.row < t.M ? e.labels[t.row] : -1;
  }
  static __device__ __forceinline__ void end(State& st, const EpiArgs& e, const TileInfo& t) {
    if (t.row < t.M)
      reinterpret_cast<float2*>(e.partials)[static_cast<int64_t>(t.unit_chunk) * e.ld_part + t.row] =
          make_float2(st.m, st.s);
  }
  static __device__ __forceinline__ void prefetch(const EpiArgs&, const TileInfo&) {}
  // per-tile choice of loop: FP8 operand scales, row scale
  static __device__ __forceinline__ void tile(State& st, const EpiArgs& e, const TileInfo& t) {
    if (e.acc_rs || e.acc_cs) {
      if (e.row_scale)
        tile_impl<true, true>(st, e, t);
      else
        tile_impl<true, false>(st, e, t);
    } else {
      if (e.row_scale)
        tile_impl<false, true>(st, e, t);
      else
        tile_impl<false, false>(st, e, t);
    }
  }
  template <bool SCALED, bool ROWSCALE>
  static __device__ __forceinline__ void tile_impl(State& st, const EpiArgs& e, const TileInfo& t) {
    const bool rv = t.row < t.M;
    const float rs = (ROWSCALE && rv) ? e.row_scale[t.row] : 1.f;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      const int col0 = t.nb * BN + c;
      if (col0 >= t.N) break;
      float z[32];
      __syncwarp();
      tmem_ld32_acc_t<SCALED>(t.taddr + c, z, e, t.row, rv, col0, t.N);
      if (rv) {
        if (ROWSCALE) {
#pragma unroll
          for (int i = 0; i < 32; ++i) z[i] *= rs;
        }
        const int nvalid = min(32, t.N - col0);
        float mc = -INFINITY;
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (i < nvalid) mc = fmaxf(mc, z[i]);
        const float mn = fmaxf(st.m, mc);
        const float mb = mn * LOG2E;
        float sc = 0.f;
#pragma unroll
        for (int i = 0; i < 32; ++i)
          if (i < nvalid) sc += exp2f(fmaf(z[i], LOG2E, -mb));
        st.s = st.s * exp2f((st.m - mn) * LOG2E) + sc;
        st.m = mn;
        const int rel = st.label - col0;
        if (rel >= 0 && rel < nvalid) {
          float tv = 0.f;
#pragma unroll
          for (int i = 0; i < 32; ++i)
            if (i == rel) tv = z[i];
          e.target_logit[t.row] = tv;
        }
      }
    }
  }
};

// ---------------------------------------------------------------------------
// CE_DLOGITS (softmax part of softmax minus one-hot): recomputed logits z,
//   dZ = exp(z - lse_i) * w_i,  w_i = dloss / n_valid for a valid row, 0 for
//   an ignored (or out-of-range) label;  stored bf16.  With `onehot` set the
//   -w_i at the label column is included (the generic-descriptor form); the
//   named cross-entropy backward instead applies it exactly in fp32 in the
//   epilogues of the dX and dW GEMMs, so the large label element is never
//   rounded to bf16.
// With a row scale rs (the final RMSNorm folded into the LM head, z = rs*acc)
// the stored value is rs * dZ (the row-scaled gradient G' of the
// reparameterised backward), and for the RMSNorm backward coefficient the
// epilogue also emits row partials sum_j p_ij z_ij (partials[nb][row]) and
// the target logit z_{i,y_i} (target_logit).
// A launch may cover one slice of the vocabulary: its column 0 is vocabulary
// column col_base, and n_total is the vocabulary size that decides which
// labels are valid.
// ---------------------------------------------------------------------------
template <int BN>
struct EpiCeDlogits {
  struct State {};
  static __device__ __forceinline__ void begin(State&, const EpiArgs&, const TileInfo&) {}
  static __device__ __forceinline__ void end(State&, const EpiArgs&, const TileInfo&) {}
  static __device__ __forceinline__ void prefetch(const EpiArgs&, const TileInfo&) {}
  // The per-tile choice of loop (FP8 operand scales, the -w label term, the
  // target-logit output) keeps feature tests out of the per-element math.
  static __device__ __forceinline__ void tile(State& st, const EpiArgs& e, const TileInfo& t) {
    const int k = ((e.acc_rs || e.acc_cs) ? 4 : 0) | (e.onehot ? 2 : 0) | (e.target_logit ? 1 : 0);
    switch (k) {
      case 0: tile_impl<false, false, false>(st, e, t); break;
      case 1: tile_impl<false, false, true>(st, e, t); break;
      case 2: tile_impl<false, true, false>(st, e, t); break;
      case 3: tile_impl<false, true, true>(st, e, t); break;
      case 4: tile_impl<true, false, false>(st, e, t); break;
      case 5: tile_impl<true, false, true>(st, e, t); break;
      case 6: tile_impl<true, true, false>(st, e, t); break;
      default: tile_impl<true, true, true>(st, e, t); break;
    }
  }
  template <bool SCALED, bool ONEHOT, bool TARGET>
  static __device__ __forceinline__ void tile_impl(State&, const EpiArgs& e, const TileInfo& t) {
    const int row = t.row;
    const bool rv = row < t.M;
    int lab = -1;
    float w = 0.f, lse = 0.f;
    if (rv) {
      lab = e.labels[row];
      const int nv = *e.n_valid;
      const int64_t vocab = e.n_total ? e.n_total : t.N;
      const bool valid = lab != e.ignore_index && lab >= 0 && lab < vocab && nv > 0;
      w = valid ? e.dloss / static_cast<float>(nv) : 0.f;
      // the label's column within this launch (a slice of the vocabulary
      // starts at col_base); outside the launch it matches no column
      const int64_t rel = static_cast<int64_t>(lab) - e.col_base;
      lab = (valid && rel >= 0 && rel < t.N) ? static_cast<int>(rel) : -1;
      lse = e.lse[row];
    }
    const float rs = (e.row_scale && rv) ? e.row_scale[row] : 1.f;
    const float ws = w * rs;
    const float lb = lse * LOG2E;
    const int row0 = row - static_cast<int>(threadIdx.x & 31);
    float pz = 0.f;
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      const int col0 = t.nb * BN + c;
      if (col0 >= t.N) break;
      float z[32];
      __syncwarp();
      tmem_ld32_acc_t<SCALED>(t.taddr + c, z, e, row, rv, col0, t.N);
      if (rv) {
#pragma unroll
        for (int g = 0; g < 4; ++g) {
          const int cc = col0 + g * 8;
          if (cc < t.N) {
#pragma unroll
            for (int i = 0; i < 8; ++i) {
              const float zz = z[g * 8 + i] * rs;
              const float p = exp2f(fmaf(zz, LOG2E, -lb));
              z[g * 8 + i] = (p - (ONEHOT && cc + i == lab ? 1.f : 0.f)) * ws;
              pz += p * zz;
              if (TARGET && cc + i == lab) e.target_logit[row] = zz;
            }
          }
        }
      }
      warp_store_bf16x32(t.stage, static_cast<__nv_bfloat16*>(e.D), e.ldd, row0, t.M, col0, t.N, z, e.st_stream);
    }
    if (e.partials && rv) e.partials[static_cast<int64_t>(t.nb) * e.ld_part + row] = pz;
  }
};

// ---------------------------------------------------------------------------
// SIGMOID (element-wise gate): z = rs * acc, s = sigmoid(z).
//   mode 0:  D = s, or s * aux0 when a gated tensor Z = aux0 is given.
//   mode 1 (backward on recomputed z, dY = aux1):
//            out1 = dz = dY (* Z) * s (1 - s);   out2 = dZ = dY * s (if Z).
// ---------------------------------------------------------------------------
template <int BN>
struct EpiSigmoid {
  struct State {};
  static __device__ __forceinline__ void begin(State&, const EpiArgs&, const TileInfo&) {}
  static __device__ __forceinline__ void end(State&, const EpiArgs&, const TileInfo&) {}
  static __device__ __forceinline__ void prefetch(const EpiArgs&, const TileInfo&) {}
  // per-tile choice of loop: gated (Z = aux0), forward or backward, dZ output
  static __device__ __forceinline__ void tile(State& st, const EpiArgs& e, const TileInfo& t) {
    const bool gated = e.aux0 != nullptr;
    if (e.mode == 0)
      gated ? tile_impl<true, 0, false>(st, e, t) : tile_impl<false, 0, false>(st, e, t);
    else if (e.out2)
      gated ? tile_impl<true, 1, true>(st, e, t) : tile_impl<false, 1, true>(st, e, t);
    else
      gated ? tile_impl<true, 1, false>(st, e, t) : tile_impl<false, 1, false>(st, e, t);
  }
  template <bool GATED, int MODE, bool OUT2>
  static __device__ __forceinline__ void tile_impl(State&, const EpiArgs& e, const TileInfo& t) {
    const int row = t.row;
    const bool rv = row < t.M;
    const int row0 = row - static_cast<int>(threadIdx.x & 31);
    const float rs = (e.row_scale && rv) ? e.row_scale[row] : 1.f;
    const int64_t off = static_cast<int64_t>(row);
#pragma unroll 1
    for (int c = 0; c < BN; c += 32) {
      const int col0 = t.nb * BN + c;
      if (col0 >= t.N) break;
      float v[32], o2[32];
      __syncwarp();
      tmem_ld32(t.taddr + c, v);
#pragma unroll
      for (int g = 0; g < 4; ++g) {
        const int cc = col0 + g * 8;
        const bool in = rv && cc < t.N;
        float z8[8] = {}, dy[8] = {};
        if (GATED && in) load_bf16x8(e.aux0 + off * e.ld_aux0 + cc, z8);
        if (MODE == 1 && in) load_bf16x8(e.aux1 + off * e.ld_aux1 + cc, dy);
#pragma unroll
        for (int i = 0; i < 8; ++i) {
          const float sg = 1.f / (1.f + __expf(-v[g * 8 + i] * rs));
          if (MODE == 0) {
            v[g * 8 + i] = GATED ? sg * z8[i] : sg;
          } else {
            const float gg = GATED ? dy[i] * z8[i] : dy[i];
            v[g * 8 + i] = gg * sg * (1.f - sg);   // dz
            o2[g * 8 + i] = dy[i] * sg;             // dZ
          }
        }
      }
      if (MODE == 0)
        warp_store_bf16x32(t.stage, static_cast<__nv_bfloat16*>(e.D), e.ldd, row0, t.M, col0, t.N, v, e.st_stream);
      else
        warp_store_bf16x32(t.stage, e.out1, e.ld_out1, row0, t.M, col0, t.N, v, e.st_stream);
      if (MODE == 1 && OUT2) warp_store_bf16x32(t.stage, e.out2, e.ld_out2, row0, t.M, col0, t.N, o2, e.st_stream);
    }
  }
};

// ---------------------------------------------------------------------------
// QKNORM_ROPE (row scale + per-head RMSNorm + RoPE rotation, pairwise map):
// a BN = 256 tile holds two 128-wide heads of the fused [q | k | v]
// projection.  q/k heads: x = rs*acc, n = x * rsqrt(mean(x^2) + eps) * gamma,
// pairs (2i, 2i+1) rotated by the (cos, sin) of (pos, i); optional save of x
// (pre-norm, out1).  v heads: rs*acc stored as is.
// ---------------------------------------------------------------------------
// HALF: RoPE pairs (j, j + 64) of each head instead of interleaved pairs
// (2j, 2j + 1); the angle of pair j is the same in both.
template <int BN, bool HALF = false>
struct EpiQkRope {
  static_assert(BN % 128 == 0, "heads are 128 wide");
  struct State {};
  static __device__ __forceinline__ void begin(State&, const EpiArgs&, const TileInfo&) {}
  static __device__ __forceinline__ void end(State&, const EpiArgs&, const TileInfo&) {}
  // Before the accumulator is ready: the lane's row of the cos/sin table
  // (512 bytes at its position) into L2 and the two gains into L1.
  static __device__ __forceinline__ void prefetch(const EpiArgs& e, const TileInfo& t) {
    if (!e.aux_prefetch) return;
    const int lane = threadIdx.x & 31;
    if (lane < 4 && e.gamma_q) asm volatile("prefetch.global.L1 [%0];" ::"l"(e.gamma_q + lane * 32));
    else if (lane >= 4 && lane < 8 && e.gamma_k)
      asm volatile("prefetch.global.L1 [%0];" ::"l"(e.gamma_k + (lane - 4) * 32));
    if (t.row >= t.M) return;
    int pos = e.pos[t.row];
    pos = pos < 0 ? 0 : (pos >= e.max_pos ? e.max_pos - 1 : pos);
    prefetch_l2_span(e.cos_sin + static_cast<int64_t>(pos) * 64, 64 * 8);
  }
  // per-tile choice of loop: FP8 operand scales, saved pre-norm q|k (out1)
  static __device__ __forceinline__ void tile(State& st, const EpiArgs& e, const TileInfo& t) {
    const bool scaled = e.acc_rs || e.acc_cs;
    if (e.out1) {
      if (scaled)
        tile_impl<true, true>(st, e, t);
      else
        tile_impl<false, true>(st, e, t);
    } else {
      if (scaled)
        tile_impl<true, false>(st, e, t);
      else
        tile_impl<false, false>(st, e, t);
    }
  }
  // Outputs leave through the warp's transpose buffer (rows row0 .. row0 + 31
  // of a head's 128 columns); the cos/sin pairs are read 16 bytes at a time.
  template <bool SCALED, bool OUT1>
  static __device__ __forceinline__ void tile_impl(State&, const EpiArgs& e, const TileInfo& t) {
    constexpr int D = 128;
    const int row = t.row;
    const bool rv = row < t.M;
    const int row0 = row - static_cast<int>(threadIdx.x & 31);
    const float rs = (e.row_scale && rv) ? e.row_scale[row] : 1.f;
    int pos = 0;
    if (rv) {
      pos = e.pos[row];
      if (pos < 0 || pos >= e.max_pos) {
        if (t.status) atomicOr(t.status, CODA_DEV_POSITION_RANGE);
        pos = pos < 0 ? 0 : e.max_pos - 1;
      }
    }
    const float4* cs4 = reinterpret_cast<const float4*>(e.cos_sin + static_cast<int64_t>(pos) * (D / 2));
    const bool st = e.st_stream != 0;
#pragma unroll 1
    for (int hh = 0; hh < BN / D; ++hh) {
      const int head = t.nb * (BN / D) + hh;
      if (head * D >= t.N) break;
      const uint32_t tcol = t.taddr + hh * D;
      if (head >= e.n_q + e.n_kv) {
        __nv_bfloat16* vbase = e.V + (head - e.n_q - e.n_kv) * D;
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          float v[32];
          __syncwarp();
          tmem_ld32_acc_t<SCALED>(tcol + c, v, e, row, rv, head * D + c, t.N);
#pragma unroll
          for (int i = 0; i < 32; ++i) v[i] *= rs;
          warp_store_bf16x32(t.stage, vbase, e.ldv, row0, t.M, c, D, v, st);
        }
        continue;
      }
      const bool is_q = head < e.n_q;
      const float* gamma = is_q ? e.gamma_q : e.gamma_k;
      __nv_bfloat16* obase = is_q ? e.Q + head * D : e.Kh + (head - e.n_q) * D;
      const int64_t ldo = is_q ? e.ldq : e.ldk;
      float ss = 0.f;
#pragma unroll 1
      for (int c = 0; c < D; c += 32) {
        float v[32];
        __syncwarp();
        tmem_ld32_acc_t<SCALED>(tcol + c, v, e, row, rv, head * D + c, t.N);
#pragma unroll
        for (int i = 0; i < 32; ++i) {
          v[i] *= rs;
          ss += v[i] * v[i];
        }
        if (OUT1) warp_store_bf16x32(t.stage, e.out1 + head * D, e.ld_out1, row0, t.M, c, D, v, st);
      }
      const float rho = rsqrtf(ss * (1.f / D) + e.eps);
      const float sr = rs * rho;
      if constexpr (HALF) {
        // pair j = c + i of the first half with j + 64 of the second half
#pragma unroll 1
        for (int c = 0; c < D / 2; c += 32) {
          float v1[32], v2[32];
          __syncwarp();
          tmem_ld32_acc_t<SCALED>(tcol + c, v1, e, row, rv, head * D + c, t.N);
          tmem_ld32_acc_t<SCALED>(tcol + D / 2 + c, v2, e, row, rv, head * D + D / 2 + c, t.N);
          float g1[32], g2[32];
#pragma unroll
          for (int g = 0; g < 4; ++g) {
            load_f32x8(gamma + c + g * 8, g1 + g * 8);
            load_f32x8(gamma + D / 2 + c + g * 8, g2 + g * 8);
          }
#pragma unroll
          for (int i = 0; i < 32; i += 2) {
            const float4 r = cs4[(c + i) / 2];  // pairs c + i and c + i + 1
            const float a0 = v1[i] * sr * g1[i], b0 = v2[i] * sr * g2[i];
            const float a1 = v1[i + 1] * sr * g1[i + 1], b1 = v2[i + 1] * sr * g2[i + 1];
            v1[i] = a0 * r.x - b0 * r.y;
            v2[i] = a0 * r.y + b0 * r.x;
            v1[i + 1] = a1 * r.z - b1 * r.w;
            v2[i + 1] = a1 * r.w + b1 * r.z;
          }
          warp_store_bf16x32(t.stage, obase, ldo, row0, t.M, c, D, v1, st);
          warp_store_bf16x32(t.stage, obase, ldo, row0, t.M, D / 2 + c, D, v2, st);
        }
      } else {
#pragma unroll 1
        for (int c = 0; c < D; c += 32) {
          float v[32];
          __syncwarp();
          tmem_ld32_acc_t<SCALED>(tcol + c, v, e, row, rv, head * D + c, t.N);
          float gm[32];
#pragma unroll
          for (int g = 0; g < 4; ++g) load_f32x8(gamma + c + g * 8, gm + g * 8);
          float o[32];
#pragma unroll
          for (int i = 0; i < 16; i += 2) {
            const float4 r = cs4[(c / 2 + i) / 2];  // pairs c/2 + i and c/2 + i + 1
            const float a0 = v[2 * i] * sr * gm[2 * i], b0 = v[2 * i + 1] * sr * gm[2 * i + 1];
            const float a1 = v[2 * i + 2] * sr * gm[2 * i + 2], b1 = v[2 * i + 3] * sr * gm[2 * i + 3];
            o[2 * i] = a0 * r.x - b0 * r.y;
            o[2 * i + 1] = a0 * r.y + b0 * r.x;
            o[2 * i + 2] = a1 * r.z - b1 * r.w;
            o[2 * i + 3] = a1 * r.w + b1 * r.z;
          }
          warp_store_bf16x32(t.stage, obase, ldo, row0, t.M, c, D, o, st);
        }
      }
    }
  }
};

}  // namespace coda
