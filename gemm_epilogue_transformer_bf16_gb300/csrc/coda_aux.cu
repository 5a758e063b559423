// Auxiliary kernels around the GEMM-epilogue path: the "lightweight
// auxiliary kernels" that merge tile partials ("CODA: Rewriting Transformer
// Blocks as GEMM-Epilogue Programs" §3.1 class 4 and §3.2), the gamma fold of
// the §3.2.1 reparameterisation, and the memory-bound passes that have no
// producing GEMM here (row RMS of a block input, RMSNorm-backward pre-pass,
// QK-RMSNorm + RoPE backward).  All are HBM-bound: 16-byte vector accesses,
// warp-per-row for row work, grids sized to the SM count.
#include <cmath>
#include <cstdlib>
#include <mutex>

#include <cuda_fp8.h>

#include "coda_epilogues.cuh"
#include "coda_internal.h"

namespace coda {

__device__ __forceinline__ float warp_sum(float v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) v += __shfl_xor_sync(0xffffffffu, v, o);
  return v;
}

// ---------------------------------------------------------------- gamma fold
__global__ void fold_gamma_kernel(const __nv_bfloat16* __restrict__ W, const float* __restrict__ gamma,
                                  __nv_bfloat16* Wf, int64_t N, int64_t K) {
  griddep_launch_dependents();
  const int64_t total8 = N * K / 8;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total8;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t e = i * 8;
    const int64_t k = e % K;
    float w[8], g[8];
    load_bf16x8(W + e, w);
    load_f32x8(gamma + k, g);
#pragma unroll
    for (int j = 0; j < 8; ++j) w[j] *= g[j];
    store_bf16x8(Wf + e, w);
  }
}

cudaError_t launch_fold_gamma(const __nv_bfloat16* W, const float* gamma, __nv_bfloat16* Wf, int64_t N, int64_t K,
                              int num_sms, cudaStream_t s) {
  const int64_t total8 = N * K / 8;
  const int64_t blocks = std::min<int64_t>((total8 + 255) / 256, static_cast<int64_t>(num_sms) * 8);
  note_launch();
  fold_gamma_kernel<<<static_cast<unsigned>(std::max<int64_t>(blocks, 1)), 256, 0, s>>>(W, gamma, Wf, N, K);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- row rstd
// One warp per row: r = 1/sqrt(mean_k X^2 + eps); with gamma, in the same
// read, U = bf16(X ⊙ gamma) (the input of an RMSNorm-reparameterised GEMM
// whose row scale r is applied in its epilogue).
__global__ void row_rstd_kernel(const __nv_bfloat16* __restrict__ X, int64_t ldx, int64_t M, int64_t K, float eps,
                                float* rstd, const float* __restrict__ gamma, __nv_bfloat16* __restrict__ U,
                                int64_t ldu) {
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t row = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5; row < M; row += warps) {
    const __nv_bfloat16* x = X + row * ldx;
    float s = 0.f;
    for (int64_t k = lane * 8; k < K; k += 256) {
      float v[8];
      load_bf16x8(x + k, v);
#pragma unroll
      for (int j = 0; j < 8; ++j) s += v[j] * v[j];
      if (U) {
        float g[8];
        load_f32x8(gamma + k, g);
#pragma unroll
        for (int j = 0; j < 8; ++j) v[j] *= g[j];
        store_bf16x8(U + row * ldu + k, v);
      }
    }
    s = warp_sum(s);
    if (lane == 0) rstd[row] = 1.f / sqrtf(s / static_cast<float>(K) + eps);
  }
}

cudaError_t launch_row_rstd(const __nv_bfloat16* X, int64_t ldx, int64_t M, int64_t K, float eps, float* rstd,
                            int num_sms, cudaStream_t s, const float* gamma, __nv_bfloat16* U, int64_t ldu) {
  const int64_t blocks = std::min<int64_t>((M + 7) / 8, static_cast<int64_t>(num_sms) * 8);
  note_launch();
  row_rstd_kernel<<<static_cast<unsigned>(std::max<int64_t>(blocks, 1)), 256, 0, s>>>(X, ldx, M, K, eps, rstd, gamma,
                                                                                       U, ldu);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- combine row partials
__global__ void combine_rows_kernel(const float* __restrict__ p, int64_t ld, int nparts, int64_t M, float inv_k,
                                    float eps, const float* __restrict__ r, float* out, int mode) {
  griddep_launch_dependents();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < M;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float s = 0.f;
    for (int t = 0; t < nparts; ++t) s += p[t * ld + i];
    if (mode == 0) {
      out[i] = 1.f / sqrtf(s * inv_k + eps);
    } else {
      const float ri = r ? r[i] : 1.f;
      out[i] = ri * ri * s * inv_k;
    }
  }
}

cudaError_t launch_combine_rows(const float* p, int64_t ld, int nparts, int64_t M, float inv_k, float eps,
                                const float* r, float* out, int mode, cudaStream_t s) {
  const int64_t blocks = std::min<int64_t>((M + 255) / 256, 4096);
  note_launch();
  combine_rows_kernel<<<static_cast<unsigned>(std::max<int64_t>(blocks, 1)), 256, 0, s>>>(p, ld, nparts, M, inv_k,
                                                                                          eps, r, out, mode);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- RMSNorm-bwd pre-pass
// G' = bf16(r * G);  c_i = r_i^2 * sum_n G_in (Y - R)_in * inv_k, the row
// coefficient of the RMSNorm backward (inv_k = 1 / K of the projection)
__global__ void rms_bwd_prepass_kernel(const __nv_bfloat16* __restrict__ G, const __nv_bfloat16* __restrict__ Y,
                                       const __nv_bfloat16* __restrict__ R, const float* __restrict__ rstd,
                                       int64_t M, int64_t N, float inv_k, __nv_bfloat16* Gp, float* coef) {
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t row = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5; row < M; row += warps) {
    const float r = rstd[row];
    float s = 0.f;
    for (int64_t n = lane * 8; n < N; n += 256) {
      const int64_t o = row * N + n;
      float g[8], y[8], rr[8];
      load_bf16x8(G + o, g);
      load_bf16x8(Y + o, y);
      if (R) {
        load_bf16x8(R + o, rr);
      } else {
#pragma unroll
        for (int j = 0; j < 8; ++j) rr[j] = 0.f;
      }
#pragma unroll
      for (int j = 0; j < 8; ++j) {
        s += g[j] * (y[j] - rr[j]);
        g[j] *= r;
      }
      store_bf16x8(Gp + o, g);
    }
    s = warp_sum(s);
    if (lane == 0) coef[row] = r * r * s * inv_k;
  }
}

cudaError_t launch_rms_bwd_prepass(const __nv_bfloat16* G, const __nv_bfloat16* Y, const __nv_bfloat16* R,
                                   const float* rstd, int64_t M, int64_t N, float inv_k, __nv_bfloat16* Gp,
                                   float* coef, int num_sms, cudaStream_t s) {
  const int64_t blocks = std::min<int64_t>((M + 7) / 8, static_cast<int64_t>(num_sms) * 8);
  note_launch();
  rms_bwd_prepass_kernel<<<static_cast<unsigned>(std::max<int64_t>(blocks, 1)), 256, 0, s>>>(G, Y, R, rstd, M, N,
                                                                                             inv_k, Gp, coef);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- column sums
// out[k] = sum_r p[r*ld + k], fixed summation order (deterministic); columns
// from `split` on go to out2[k - split] instead (two vectors in one launch).
// Block = 32 columns x 32 row groups; row group g sums rows g, g+32, ...;
// the 32 group sums are then added in order.
__global__ void colsum_kernel(const float* __restrict__ p, int64_t nrows, int64_t ncols, int64_t ld, float* out,
                              int64_t split, float* out2) {
  griddep_launch_dependents();
  __shared__ float part[32][33];
  const int tx = threadIdx.x & 31, ty = threadIdx.x >> 5;
  const int64_t col = blockIdx.x * 32 + tx;
  float s = 0.f;
  if (col < ncols)
    for (int64_t r = ty; r < nrows; r += 32) s += p[r * ld + col];
  part[ty][tx] = s;
  __syncthreads();
  if (ty == 0 && col < ncols) {
    float t = 0.f;
    for (int g = 0; g < 32; ++g) t += part[g][tx];
    if (col < split)
      out[col] = t;
    else
      out2[col - split] = t;
  }
}

cudaError_t launch_colsum(const float* p, int64_t nrows, int64_t ncols, int64_t ld, float* out, cudaStream_t s,
                          int64_t split, float* out2) {
  if (split < 0 || !out2) split = ncols;
  note_launch();
  colsum_kernel<<<static_cast<unsigned>((ncols + 31) / 32), 1024, 0, s>>>(p, nrows, ncols, ld, out, split, out2);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- cross-entropy combine
// Merge the (max, sum-exp) partials of every vocab chunk into lse_i, form
// loss_i = lse_i - z_{i,y_i} for valid rows, and reduce (double, fixed
// order) into per-block sums; a one-block finaliser writes the mean.
__global__ void ce_combine_kernel(const float2* __restrict__ part, int64_t ld, int nchunks,
                                  const float* __restrict__ target, const int32_t* __restrict__ labels,
                                  int32_t ignore, int64_t M, int64_t V, float* lse_out, double* blk_loss,
                                  int* blk_cnt, int* status) {
  griddep_launch_dependents();
  __shared__ double sl[CE_COMBINE_THREADS];
  __shared__ int sc[CE_COMBINE_THREADS];
  double acc = 0.0;
  int cnt = 0;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < M;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    float m = -INFINITY;
    for (int c = 0; c < nchunks; ++c) m = fmaxf(m, part[c * ld + i].x);
    float s = 0.f;
    for (int c = 0; c < nchunks; ++c) {
      const float2 q = part[c * ld + i];
      s += q.y * expf(q.x - m);
    }
    const float lse = m + logf(s);
    lse_out[i] = lse;
    const int32_t y = labels[i];
    if (y != ignore) {
      if (y >= 0 && y < V) {
        acc += static_cast<double>(lse) - static_cast<double>(target[i]);
        ++cnt;
      } else if (status) {
        atomicOr(status, CODA_DEV_LABEL_RANGE);
      }
    }
  }
  sl[threadIdx.x] = acc;
  sc[threadIdx.x] = cnt;
  __syncthreads();
  for (int o = CE_COMBINE_THREADS / 2; o > 0; o >>= 1) {
    if (threadIdx.x < o) {
      sl[threadIdx.x] += sl[threadIdx.x + o];
      sc[threadIdx.x] += sc[threadIdx.x + o];
    }
    __syncthreads();
  }
  if (threadIdx.x == 0) {
    blk_loss[blockIdx.x] = sl[0];
    blk_cnt[blockIdx.x] = sc[0];
  }
}

__global__ void ce_finalize_kernel(const double* blk_loss, const int* blk_cnt, int nblk, float* loss_mean,
                                   int32_t* n_valid) {
  griddep_launch_dependents();
  if (threadIdx.x != 0) return;
  double s = 0.0;
  long long c = 0;
  for (int b = 0; b < nblk; ++b) {
    s += blk_loss[b];
    c += blk_cnt[b];
  }
  *loss_mean = static_cast<float>(c > 0 ? s / static_cast<double>(c) : NAN);
  *n_valid = static_cast<int32_t>(c);
}

cudaError_t launch_ce_combine(const float2* part, int64_t ld, int nchunks, const float* target,
                              const int32_t* labels, int32_t ignore, int64_t M, int64_t V, float* lse,
                              double* blk_loss, int* blk_cnt, int nblk, float* loss_mean, int32_t* n_valid,
                              int* status, cudaStream_t s) {
  note_launch();
  ce_combine_kernel<<<nblk, CE_COMBINE_THREADS, 0, s>>>(part, ld, nchunks, target, labels, ignore, M, V, lse,
                                                        blk_loss, blk_cnt, status);
  cudaError_t e = cudaGetLastError();
  if (e != cudaSuccess) return e;
  note_launch();
  ce_finalize_kernel<<<1, 32, 0, s>>>(blk_loss, blk_cnt, nblk, loss_mean, n_valid);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- CE backward one-hot terms
// Per row: w_i = dloss / n_valid and its label for a valid row (else 0, -1);
// and, for the dW GEMM, the tokens of every vocabulary row (counting sort by
// label: histogram, exclusive scan, scatter, then each bucket sorted by token
// index so that the epilogue's fp32 sums have a fixed order).
__global__ void ce_prep_kernel(const int32_t* __restrict__ labels, int32_t ignore, int64_t M, int64_t V,
                               const int32_t* __restrict__ n_valid, float dloss, const float* __restrict__ rstd,
                               float* wrow, int32_t* lrow, int32_t* counts) {
  griddep_launch_dependents();
  const int32_t nv = *n_valid;
  const float w = nv > 0 ? dloss / static_cast<float>(nv) : 0.f;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < M;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int32_t y = labels[i];
    const bool valid = y != ignore && y >= 0 && y < V && nv > 0;
    wrow[i] = valid ? (rstd ? w * rstd[i] : w) : 0.f;
    lrow[i] = valid ? y : -1;
    if (valid) atomicAdd(&counts[y], 1);
  }
}

// Exclusive scan of counts[0..V) into off[0..V] with one 1024-thread block.
__global__ void __launch_bounds__(1024) scan_counts_kernel(const int32_t* __restrict__ counts, int64_t V,
                                                           int32_t* off) {
  __shared__ int32_t part[1024];
  const int64_t per = (V + 1023) / 1024;
  const int64_t b = threadIdx.x * per, e = (b + per < V) ? b + per : V;
  int32_t s = 0;
  for (int64_t i = b; i < e; ++i) s += counts[i];
  part[threadIdx.x] = s;
  __syncthreads();
  for (int o = 1; o < 1024; o <<= 1) {  // Hillis-Steele inclusive scan of the 1024 partials
    const int32_t v = threadIdx.x >= o ? part[threadIdx.x - o] : 0;
    __syncthreads();
    part[threadIdx.x] += v;
    __syncthreads();
  }
  int32_t run = threadIdx.x ? part[threadIdx.x - 1] : 0;
  for (int64_t i = b; i < e; ++i) {
    off[i] = run;
    run += counts[i];
  }
  if (threadIdx.x == 1023) off[V] = part[1023];
}

__global__ void ce_fill_kernel(const int32_t* __restrict__ lrow, int64_t M, const int32_t* __restrict__ off,
                               int32_t* cursor, int32_t* idx) {
  griddep_launch_dependents();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < M;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int32_t y = lrow[i];
    if (y >= 0) idx[off[y] + atomicAdd(&cursor[y], 1)] = static_cast<int32_t>(i);
  }
}

__global__ void ce_sort_buckets_kernel(const int32_t* __restrict__ off, int64_t V, int32_t* idx) {
  griddep_launch_dependents();
  for (int64_t v = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; v < V;
       v += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int32_t b = off[v], e = off[v + 1];
    for (int32_t i = b + 1; i < e; ++i) {  // insertion sort; buckets hold a few tokens
      const int32_t key = idx[i];
      int32_t j = i - 1;
      while (j >= b && idx[j] > key) {
        idx[j + 1] = idx[j];
        --j;
      }
      idx[j + 1] = key;
    }
  }
}

cudaError_t launch_ce_onehot_prep(const int32_t* labels, int32_t ignore, int64_t M, int64_t V,
                                  const int32_t* n_valid, float dloss, const float* rstd, float* wrow, int32_t* lrow,
                                  int32_t* counts, int32_t* cursor, int32_t* off, int32_t* idx, cudaStream_t s) {
  cudaError_t e;
  if ((e = cudaMemsetAsync(counts, 0, sizeof(int32_t) * V, s)) != cudaSuccess) return e;
  if ((e = cudaMemsetAsync(cursor, 0, sizeof(int32_t) * V, s)) != cudaSuccess) return e;
  const unsigned mb = static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>((M + 255) / 256, 1024)));
  note_launch();
  ce_prep_kernel<<<mb, 256, 0, s>>>(labels, ignore, M, V, n_valid, dloss, rstd, wrow, lrow, counts);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch();
  scan_counts_kernel<<<1, 1024, 0, s>>>(counts, V, off);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch();
  ce_fill_kernel<<<mb, 256, 0, s>>>(lrow, M, off, cursor, idx);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  const unsigned vb = static_cast<unsigned>(std::max<int64_t>(1, std::min<int64_t>((V + 255) / 256, 1024)));
  note_launch();
  ce_sort_buckets_kernel<<<vb, 256, 0, s>>>(off, V, idx);
  return cudaGetLastError();
}

// RMSNorm-backward coefficient of a row-scaled cross-entropy head:
//   c_i = r_i * (r_i w_i) * (sum_t pz[t][i] - z_{i,y_i}) / K,
// i.e. r_i^2 * sum_j dZ_ij z_ij / K with dZ = (softmax - onehot) * w_i.
// Rows with w_i = 0 (ignored labels) get 0 without reading their target.
__global__ void ce_norm_coef_kernel(const float* __restrict__ pz, int64_t ld, int nparts,
                                    const float* __restrict__ target, const float* __restrict__ rstd,
                                    const float* __restrict__ rw, int64_t M, float inv_k, float* coef) {
  griddep_launch_dependents();
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < M;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float w = rw[i];
    if (w == 0.f) {
      coef[i] = 0.f;
      continue;
    }
    float s = 0.f;
    for (int t = 0; t < nparts; ++t) s += pz[t * ld + i];
    coef[i] = rstd[i] * w * (s - target[i]) * inv_k;
  }
}

cudaError_t launch_ce_norm_coef(const float* pz, int64_t ld, int nparts, const float* target, const float* rstd,
                                const float* rw, int64_t M, float inv_k, float* coef, cudaStream_t s) {
  const int64_t blocks = std::min<int64_t>((M + 255) / 256, 4096);
  note_launch();
  ce_norm_coef_kernel<<<static_cast<unsigned>(std::max<int64_t>(blocks, 1)), 256, 0, s>>>(pz, ld, nparts, target,
                                                                                          rstd, rw, M, inv_k, coef);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- division by a fixed scale
// x / s rounded to nearest (fp32) for one divisor and many dividends, by
// Markstein's correction (P. Markstein, "Computation of elementary functions
// on the IBM RISC System/6000 processor", IBM J. Res. Dev. 34(1), 1990): with
// y = RN(1/s), the first quotient q = RN(x y) is within an ulp of x / s, the
// residual x - s q is exact in one FMA, and RN(q + (x - s q) y) is the
// correctly rounded quotient, barring overflow and results below the normal
// range (a quantiser's quotients lie in [0, 448], and one below 2^-126 rounds
// to a zero code either way).  The quotient takes x's sign (s > 0), which
// also keeps -0 / s = -0.  Three FP32 operations per element instead of a
// full division; the GPU tests compare the codes bit for bit with the
// oracle's IEEE division.
struct DivBy {
  float s, y;
  __device__ __forceinline__ explicit DivBy(float s_) : s(s_), y(1.f / s_) {}  // RN(1/s): one IEEE division
  __device__ __forceinline__ float operator()(float x) const {
    const float q = x * y;
    return copysignf(fmaf(fmaf(-s, q, x), y, q), x);
  }
};

// Four e4m3 codes, a in the low byte: two paired conversions (nearest even,
// saturating to +-448) instead of four single ones and their byte shifts.
__device__ __forceinline__ uint32_t e4m3x4(float a, float b, float c, float d) {
  const uint32_t lo = __nv_cvt_float2_to_fp8x2(make_float2(a, b), __NV_SATFINITE, __NV_E4M3);
  const uint32_t hi = __nv_cvt_float2_to_fp8x2(make_float2(c, d), __NV_SATFINITE, __NV_E4M3);
  return lo | (hi << 16);
}

// ---------------------------------------------------------------- FP8 (e4m3) row quantisation
// Warp per row: scale = amax / 448 (fp32; 1 for an all-zero row), codes =
// e4m3(x / scale), fp32 division, round to nearest even, saturating.
__global__ void quantize_fp8_rows_kernel(const __nv_bfloat16* __restrict__ X, int64_t ldx, int64_t M, int64_t K,
                                         uint8_t* Xq, int64_t ldq, float* scale) {
  griddep_launch_dependents();
  const int lane = threadIdx.x & 31;
  const int64_t warps = static_cast<int64_t>(gridDim.x) * (blockDim.x >> 5);
  for (int64_t row = (blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x) >> 5; row < M; row += warps) {
    const __nv_bfloat16* x = X + row * ldx;
    float amax = 0.f;
    for (int64_t k = lane * 8; k < K; k += 256) {
      float v[8];
      load_bf16x8(x + k, v);
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[j]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    const float s = amax > 0.f ? amax / 448.f : 1.f;
    if (lane == 0) scale[row] = s;
    const DivBy div(s);
    uint8_t* q = Xq + row * ldq;
    for (int64_t k = lane * 8; k < K; k += 256) {
      float v[8];
      load_bf16x8(x + k, v);
      const uint32_t lo = e4m3x4(div(v[0]), div(v[1]), div(v[2]), div(v[3]));
      const uint32_t hi = e4m3x4(div(v[4]), div(v[5]), div(v[6]), div(v[7]));
      *reinterpret_cast<uint2*>(q + k) = make_uint2(lo, hi);
    }
  }
}

// Same rule, one block per row at a time: each row is brought into shared
// memory by one bulk copy (double-buffered: the next row's copy is issued
// before this row's work), so HBM reads every element once and the block's
// 256 threads find the amax and write the codes from shared memory.  The
// copy wait is bounded: a row whose bytes do not arrive within the limit
// gets a NaN scale (its codes are not written), which no valid row has.
constexpr int QROW_THREADS = 256;
constexpr size_t QROW_SMEM_MAX = 232448;  // the per-block dynamic shared-memory limit

__global__ void __launch_bounds__(QROW_THREADS) quantize_fp8_rows_smem_kernel(
    const __nv_bfloat16* __restrict__ X, int64_t ldx, int64_t M, int64_t K, uint8_t* Xq, int64_t ldq, float* scale,
    uint32_t row_bytes_padded, uint64_t timeout_ns) {
  extern __shared__ __align__(128) uint8_t qsm[];
  griddep_launch_dependents();
  auto buf = [&](int b) { return qsm + b * row_bytes_padded; };
  uint64_t* bar = reinterpret_cast<uint64_t*>(qsm + 2 * row_bytes_padded);
  float* red = reinterpret_cast<float*>(bar + 2);
  const int tid = threadIdx.x, lane = tid & 31, warp = tid >> 5;
  const uint32_t bytes = static_cast<uint32_t>(K * 2);
  if (tid == 0) {
    mbar_init(&bar[0], 1);
    mbar_init(&bar[1], 1);
    fence_mbar_init();
  }
  __syncthreads();
  griddep_wait();
  int64_t row = blockIdx.x;
  if (tid == 0 && row < M) {
    mbar_arrive_expect_tx(&bar[0], bytes, 1);
    bulk_load(buf(0), X + row * ldx, bytes, &bar[0], 1);
  }
  bool failed = false;
  uint32_t i = 0;
  for (; row < M; ++i, row += gridDim.x) {
    const int b = i & 1;
    const int64_t next = row + gridDim.x;
    if (tid == 0 && next < M && !failed) {  // the other buffer was released by the last iteration's barrier
      asm volatile("fence.proxy.async.shared::cta;" ::: "memory");
      mbar_arrive_expect_tx(&bar[b ^ 1], bytes, 1);
      bulk_load(buf(b ^ 1), X + next * ldx, bytes, &bar[b ^ 1], 1);
    }
    bool ok = false;
    if (!failed) {  // bounded wait for this row's bytes (every thread polls the barrier)
      ok = mbar_try_wait(smem_u32(&bar[b]), (i >> 1) & 1);
      const uint64_t t0 = globaltimer_ns();
      while (!ok && globaltimer_ns() - t0 < timeout_ns) ok = mbar_try_wait(smem_u32(&bar[b]), (i >> 1) & 1);
    }
    ok = __syncthreads_and(ok);
    if (!ok) {  // no more copies from this block; its remaining rows get NaN scales
      if (tid == 0) scale[row] = __int_as_float(0x7fc00000);
      if (!failed && tid == 0 && next < M) {  // the next row's copy was issued: let it land (bounded)
        const uint64_t t0 = globaltimer_ns();
        while (!mbar_try_wait(smem_u32(&bar[b ^ 1]), ((i + 1) >> 1) & 1) && globaltimer_ns() - t0 < timeout_ns) {
        }
      }
      failed = true;
      continue;
    }
    const __nv_bfloat16* x = reinterpret_cast<const __nv_bfloat16*>(buf(b));
    float amax = 0.f;
    for (int64_t k = tid * 8; k < K; k += QROW_THREADS * 8) {
      float v[8];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(x + k), v);
#pragma unroll
      for (int j = 0; j < 8; ++j) amax = fmaxf(amax, fabsf(v[j]));
    }
#pragma unroll
    for (int o = 16; o > 0; o >>= 1) amax = fmaxf(amax, __shfl_xor_sync(0xffffffffu, amax, o));
    if (lane == 0) red[warp] = amax;
    __syncthreads();
    amax = red[0];
#pragma unroll
    for (int w = 1; w < QROW_THREADS / 32; ++w) amax = fmaxf(amax, red[w]);
    const float sc = amax > 0.f ? amax / 448.f : 1.f;
    if (tid == 0) scale[row] = sc;
    const DivBy div(sc);
    uint8_t* q = Xq + row * ldq;
    for (int64_t k = tid * 8; k < K; k += QROW_THREADS * 8) {
      float v[8];
      bf16x8_to_f32(*reinterpret_cast<const uint4*>(x + k), v);
      const uint32_t lo = e4m3x4(div(v[0]), div(v[1]), div(v[2]), div(v[3]));
      const uint32_t hi = e4m3x4(div(v[4]), div(v[5]), div(v[6]), div(v[7]));
      *reinterpret_cast<uint2*>(q + k) = make_uint2(lo, hi);
    }
    __syncthreads();  // buffer b and red[] are free for the next rows
  }
  // every copy issued was waited for: the copy of row `next` is issued only
  // when that row belongs to this block's loop, which waits for it (or, after
  // a timeout, drains it above)
}

// ---------------------------------------------------------------- FP8 (e4m3) column quantisation
// The transposed K-major operand of a GEMM that contracts over X's rows:
// scale_c = max_r |x_rc| / 448 (1 for an all-zero column), out[c, r] =
// e4m3(x_rc / scale_c), for X [R, C] with an optional X2 [R2, C] stacked
// below it (rows R .. R + R2 - 1 of the column).  Three passes: column
// maxima (as float bits; non-negative floats order like their bit patterns)
// reduced with atomicMax into `scale`, maxima -> scales in place, then a
// 64 x 64 shared-memory transpose that writes 16-byte rows of codes.
__global__ void fp8_col_amax_kernel(const __nv_bfloat16* __restrict__ X, int64_t ldx, int64_t R,
                                    const __nv_bfloat16* __restrict__ X2, int64_t ldx2, int64_t R2, int64_t C,
                                    int rows_per_block, unsigned int* amax_bits) {
  griddep_launch_dependents();
  __shared__ float red[8][256];
  const int cg = threadIdx.x & 31, rp = threadIdx.x >> 5;  // 8 columns per thread, 8 row phases
  const int64_t c0 = blockIdx.x * 256 + cg * 8;
  const int64_t r_begin = static_cast<int64_t>(blockIdx.y) * rows_per_block;
  const int64_t r_end = min(R + R2, r_begin + rows_per_block);
  float m[8] = {0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f, 0.f};
  if (c0 < C) {
    // unrolled so that several independent 16-byte loads per thread are in flight
#pragma unroll 4
    for (int64_t r = r_begin + rp; r < r_end; r += 8) {
      const __nv_bfloat16* src = r < R ? X + r * ldx + c0 : X2 + (r - R) * ldx2 + c0;
      float v[8];
      load_bf16x8(src, v);
#pragma unroll
      for (int j = 0; j < 8; ++j) m[j] = fmaxf(m[j], fabsf(v[j]));
    }
  }
#pragma unroll
  for (int j = 0; j < 8; ++j) red[rp][cg * 8 + j] = m[j];
  __syncthreads();
  const int64_t c = blockIdx.x * 256 + threadIdx.x;
  if (c < C) {
    float t = 0.f;
#pragma unroll
    for (int k = 0; k < 8; ++k) t = fmaxf(t, red[k][threadIdx.x]);
    atomicMax(amax_bits + c, __float_as_uint(t));
  }
}

__global__ void fp8_amax_to_scale_kernel(float* scale, int64_t C) {
  griddep_launch_dependents();
  for (int64_t c = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; c < C;
       c += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const float a = __uint_as_float(reinterpret_cast<unsigned int*>(scale)[c]);
    scale[c] = a > 0.f ? a / 448.f : 1.f;
  }
}

// Each block takes a strip of 64 columns over a run of rows, 64 x 64 tiles
// at a time: the next tile's rows are loaded into registers while the
// current tile goes through the shared-memory transpose, and each thread
// keeps its column's divisor for the whole run.
__global__ void fp8_col_quant_kernel(const __nv_bfloat16* __restrict__ X, int64_t ldx, int64_t R,
                                     const __nv_bfloat16* __restrict__ X2, int64_t ldx2, int64_t R2, int64_t C,
                                     const float* __restrict__ scale, uint8_t* out, int64_t ldo, int rows_per_block) {
  griddep_launch_dependents();
  __shared__ float tile[64][65];
  const int64_t RT = R + R2;
  const int64_t c0 = static_cast<int64_t>(blockIdx.x) * 64;
  const int64_t r_begin = static_cast<int64_t>(blockIdx.y) * rows_per_block;
  const int64_t r_end = min(RT, r_begin + rows_per_block);
  // load role: 64 rows x 64 columns, 8 columns (16 bytes) per thread and step, two steps
  uint4 nxt[2];
  auto load = [&](int64_t r0) {
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = threadIdx.x + h * 256;
      const int64_t r = r0 + (i >> 3), c = c0 + (i & 7) * 8;
      nxt[h] = (r < r_end && c < C) ? *reinterpret_cast<const uint4*>(r < R ? X + r * ldx + c : X2 + (r - R) * ldx2 + c)
                                    : make_uint4(0u, 0u, 0u, 0u);
    }
  };
  // store role: output row c = c0 + t / 4 takes 16 rows of the tile as one 16-byte chunk
  const int cc = threadIdx.x >> 2, part = threadIdx.x & 3;
  const int64_t c = c0 + cc;
  const DivBy div(c < C ? scale[c] : 1.f);
  if (r_begin < r_end) load(r_begin);
  for (int64_t r0 = r_begin; r0 < r_end; r0 += 64) {
    __syncthreads();  // the previous tile's reads of `tile` are done
#pragma unroll
    for (int h = 0; h < 2; ++h) {
      const int i = threadIdx.x + h * 256;
      float v[8];
      bf16x8_to_f32(nxt[h], v);
#pragma unroll
      for (int j = 0; j < 8; ++j) tile[i >> 3][(i & 7) * 8 + j] = v[j];
    }
    __syncthreads();
    if (r0 + 64 < r_end) load(r0 + 64);  // in flight while this tile is converted and stored
    if (c < C) {
      uint32_t w[4];
#pragma unroll
      for (int j = 0; j < 4; ++j) {
        const int rr = part * 16 + 4 * j;
        w[j] = e4m3x4(div(tile[rr][cc]), div(tile[rr + 1][cc]), div(tile[rr + 2][cc]), div(tile[rr + 3][cc]));
      }
      const int64_t r = r0 + part * 16;
      if (r + 16 <= r_end) {
        *reinterpret_cast<uint4*>(out + c * ldo + r) = make_uint4(w[0], w[1], w[2], w[3]);
      } else {
        for (int j = 0; j < 16 && r + j < r_end; ++j)
          out[c * ldo + r + j] = static_cast<uint8_t>(w[j >> 2] >> (8 * (j & 3)));
      }
    }
  }
}

cudaError_t launch_quantize_fp8_cols(const __nv_bfloat16* X, int64_t ldx, int64_t R, const __nv_bfloat16* X2,
                                     int64_t ldx2, int64_t R2, int64_t C, uint8_t* out, int64_t ldo, float* scale,
                                     int num_sms, cudaStream_t s) {
  cudaError_t e = cudaMemsetAsync(scale, 0, sizeof(float) * C, s);
  if (e != cudaSuccess) return e;
  const int64_t RT = R + R2;
  const int64_t cblk = (C + 255) / 256;
  // about sixteen blocks per SM in all (eight resident), each over a run of
  // rows: enough loads in flight to stream X at HBM speed
  const int64_t want = std::max<int64_t>(1, (16 * static_cast<int64_t>(num_sms) + cblk - 1) / cblk);
  const int64_t rsplit = std::min<int64_t>(want, std::max<int64_t>(1, (RT + 63) / 64));
  const int rows = static_cast<int>((RT + rsplit - 1) / rsplit);
  note_launch();
  fp8_col_amax_kernel<<<dim3(static_cast<unsigned>(cblk), static_cast<unsigned>(rsplit)), 256, 0, s>>>(
      X, ldx, R, X2, ldx2, R2, C, rows, reinterpret_cast<unsigned int*>(scale));
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  note_launch();
  fp8_amax_to_scale_kernel<<<static_cast<unsigned>(std::min<int64_t>((C + 255) / 256, 1024)), 256, 0, s>>>(scale, C);
  if ((e = cudaGetLastError()) != cudaSuccess) return e;
  // the transposing pass: each block a 64-column strip over four 64-row
  // tiles.  Blocks stay short-lived: the pass often runs beside a
  // persistent GEMM on another stream, whose ~200 KB CTAs can take an SM
  // only when the blocks there finish (one strip per block over all rows
  // was faster alone, 160 against 190 us for 8192 x 28672, but slowed the
  // FP8 block's backward by 0.5 ms)
  const int64_t cq = (C + 63) / 64;
  const int qrows = 4 * 64;
  note_launch();
  fp8_col_quant_kernel<<<dim3(static_cast<unsigned>(cq), static_cast<unsigned>((RT + qrows - 1) / qrows)), 256, 0,
                         s>>>(X, ldx, R, X2, ldx2, R2, C, scale, out, ldo, qrows);
  return cudaGetLastError();
}

// CODA_QROW_SMEM=0 in the environment selects the warp-per-row quantiser
// (for comparisons).
static bool qrow_staged_enabled() {
  static const bool v = [] {
    const char* e = std::getenv("CODA_QROW_SMEM");
    return !(e && e[0] == '0');
  }();
  return v;
}

cudaError_t launch_quantize_fp8_rows(const __nv_bfloat16* X, int64_t ldx, int64_t M, int64_t K, uint8_t* Xq,
                                     int64_t ldq, float* scale, int num_sms, cudaStream_t s) {
  // rows staged in shared memory when two of them fit in a block's shared
  // memory and the bulk copies' addresses and sizes are 16-byte multiples;
  // otherwise a warp per row (which reads each row twice).  G' of the SwiGLU
  // MLP, 8192 x 57344 (one block per SM): 0.365 against 0.460 ms.
  const uint32_t rowp = static_cast<uint32_t>((K * 2 + 127) / 128 * 128);
  const size_t smem = 2 * static_cast<size_t>(rowp) + 2 * sizeof(uint64_t) + 8 * sizeof(float);
  const int per_sm = static_cast<int>(std::min<size_t>(8, (228 * 1024) / (smem + 1024)));
  const bool staged = K > 0 && K % 8 == 0 && ldx % 8 == 0 && (reinterpret_cast<uintptr_t>(X) & 15) == 0 &&
                      smem <= QROW_SMEM_MAX && per_sm >= 1 && M > 0 && qrow_staged_enabled();
  if (staged) {
    static std::mutex mu;
    static bool raised[64] = {};
    int dev = 0;
    cudaError_t e = cudaGetDevice(&dev);
    if (e != cudaSuccess) return e;
    if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
    {
      std::lock_guard<std::mutex> lock(mu);
      if (!raised[dev]) {
        e = cudaFuncSetAttribute(quantize_fp8_rows_smem_kernel, cudaFuncAttributeMaxDynamicSharedMemorySize,
                                 static_cast<int>(QROW_SMEM_MAX));
        if (e != cudaSuccess) return e;
        raised[dev] = true;
      }
    }
    const int64_t blocks = std::min<int64_t>(M, static_cast<int64_t>(num_sms) * per_sm);
    note_launch();
    quantize_fp8_rows_smem_kernel<<<static_cast<unsigned>(blocks), QROW_THREADS, smem, s>>>(
        X, ldx, M, K, Xq, ldq, scale, rowp, 1000000000ull);
    return cudaGetLastError();
  }
  const int64_t blocks = std::min<int64_t>((M + 7) / 8, static_cast<int64_t>(num_sms) * 8);
  note_launch();
  quantize_fp8_rows_kernel<<<static_cast<unsigned>(std::max<int64_t>(blocks, 1)), 256, 0, s>>>(X, ldx, M, K, Xq,
                                                                                               ldq, scale);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- bounded-wait self-test
// One thread waits on an mbarrier that nothing arrives on, through the same
// bounded wait the GEMM pipeline uses; after `limit_ns` the wait gives up and
// records CODA_DEV_TIMEOUT in the status word.  Shows on a live GPU that a
// stuck pipeline stage turns into a host-readable error, not a hang.
__global__ void selftest_wait_timeout_kernel(uint64_t limit_ns, int* status) {
  __shared__ uint64_t bar;
  __shared__ int abort_flag;
  if (threadIdx.x != 0) return;
  mbar_init(&bar, 1);
  abort_flag = 0;
  fence_mbar_init();
  mbar_wait_bounded(&bar, 0, &abort_flag, status, limit_ns);
}

cudaError_t launch_selftest_wait_timeout(uint64_t limit_ns, int* status, cudaStream_t s) {
  note_launch();
  selftest_wait_timeout_kernel<<<1, 32, 0, s>>>(limit_ns, status);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- RoPE table
__global__ void rope_table_kernel(double theta, int head_dim, int max_pos, float2* cs) {
  griddep_launch_dependents();
  const int half = head_dim / 2;
  const int64_t total = static_cast<int64_t>(max_pos) * half;
  for (int64_t i = blockIdx.x * static_cast<int64_t>(blockDim.x) + threadIdx.x; i < total;
       i += static_cast<int64_t>(gridDim.x) * blockDim.x) {
    const int64_t p = i / half;
    const int j = static_cast<int>(i - p * half);
    const double a = static_cast<double>(p) * pow(theta, -2.0 * j / head_dim);
    double sn, cn;
    sincos(a, &sn, &cn);
    cs[i] = make_float2(static_cast<float>(cn), static_cast<float>(sn));
  }
}

cudaError_t launch_rope_table(double theta, int head_dim, int max_pos, float2* cs, cudaStream_t s) {
  const int64_t total = static_cast<int64_t>(max_pos) * (head_dim / 2);
  const int64_t blocks = std::min<int64_t>((total + 255) / 256, 4096);
  note_launch();
  rope_table_kernel<<<static_cast<unsigned>(std::max<int64_t>(blocks, 1)), 256, 0, s>>>(theta, head_dim, max_pos,
                                                                                       cs);
  return cudaGetLastError();
}

// ---------------------------------------------------------------- QK-RMSNorm + RoPE backward
// Warp per token row; lane owns elements 4*lane .. 4*lane+3 of every
// 128-wide head, i.e. RoPE pairs 2*lane and 2*lane+1.  For each q/k head:
//   dn = RoPE^-1(dOut), n = x * rho (x = saved pre-norm head, rho =
//   rsqrt(mean x^2 + eps)), dgamma += dn*n, dq = rho (dn*g - n mean(n dn g)).
// v heads pass dV through.  Writes G' = r * [dq | dk | dv] (bf16), the row
// sum s_i = sum (dq x + dk k + dv v) and per-block dgamma_q | dgamma_k sums.
__device__ __forceinline__ void load_bf16x4(const __nv_bfloat16* p, float* o) {
  const uint2 q = *reinterpret_cast<const uint2*>(p);
  o[0] = bf16_lo(q.x);
  o[1] = bf16_hi(q.x);
  o[2] = bf16_lo(q.y);
  o[3] = bf16_hi(q.y);
}
__device__ __forceinline__ void store_bf16x4(__nv_bfloat16* p, const float* v) {
  uint2 q;
  q.x = pack_bf16x2(v[0], v[1]);
  q.y = pack_bf16x2(v[2], v[3]);
  *reinterpret_cast<uint2*>(p) = q;
}

// Four warp sums at once: the shuffles of the four chains interleave.
__device__ __forceinline__ void warp_sum4(float* v) {
#pragma unroll
  for (int o = 16; o > 0; o >>= 1) {
#pragma unroll
    for (int j = 0; j < 4; ++j) v[j] += __shfl_xor_sync(0xffffffffu, v[j], o);
  }
}

// HALF: RoPE pairs (j, j + 64) of each head (lanes l and l + 16 hold the
// two elements of a pair) instead of interleaved pairs (2j, 2j + 1).
// A warp owns one token row and takes its heads four at a time: the four
// heads' gradient and saved-input loads are issued together, and their
// per-head reductions run as interleaved shuffle chains, so each warp keeps
// 2 KB of loads in flight instead of 512 bytes.  With rstd given, the row
// coefficient c_i = r_i^2 * sum_j dq_ij x_ij * inv_k of the input RMSNorm's
// backward is written to coef (no separate combine pass).
template <bool HALF>
__global__ void __launch_bounds__(QK_BWD_WARPS * 32)
    qk_bwd_kernel(const __nv_bfloat16* __restrict__ dQ, const __nv_bfloat16* __restrict__ dK,
                  const __nv_bfloat16* __restrict__ dV, const __nv_bfloat16* __restrict__ qk_save,
                  const __nv_bfloat16* __restrict__ Vs, const float* __restrict__ gq, const float* __restrict__ gk,
                  const int32_t* __restrict__ pos, const float2* __restrict__ cs, int max_pos, float eps, int n_q,
                  int n_kv, const float* __restrict__ rstd, int64_t M, float inv_k, __nv_bfloat16* Gp,
                  float* coef, float* dgam_part, int* status) {
  griddep_launch_dependents();
  constexpr int D = 128;
  constexpr int HG = 4;  // heads per group
  __shared__ float red[QK_BWD_WARPS][2 * D];
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int64_t ldq = static_cast<int64_t>(n_q) * D, ldkv = static_cast<int64_t>(n_kv) * D;
  const int64_t ldsave = ldq + ldkv, ldg = ldq + 2 * ldkv;
  const int nqk = n_q + n_kv;
  float aq[4] = {0.f, 0.f, 0.f, 0.f}, ak[4] = {0.f, 0.f, 0.f, 0.f};
  float g_q[4], g_k[4];
  {
    const float4 a = *reinterpret_cast<const float4*>(gq + 4 * lane);
    const float4 b = *reinterpret_cast<const float4*>(gk + 4 * lane);
    g_q[0] = a.x; g_q[1] = a.y; g_q[2] = a.z; g_q[3] = a.w;
    g_k[0] = b.x; g_k[1] = b.y; g_k[2] = b.z; g_k[3] = b.w;
  }
  const int64_t nwarps = static_cast<int64_t>(gridDim.x) * QK_BWD_WARPS;
  for (int64_t row = static_cast<int64_t>(blockIdx.x) * QK_BWD_WARPS + w; row < M; row += nwarps) {
    int p = pos[row];
    if (p < 0 || p >= max_pos) {
      if (lane == 0 && status) atomicOr(status, CODA_DEV_POSITION_RANGE);
      p = p < 0 ? 0 : max_pos - 1;
    }
    const float2 c0 = cs[static_cast<int64_t>(p) * (D / 2) + 2 * lane];
    const float2 c1 = cs[static_cast<int64_t>(p) * (D / 2) + 2 * lane + 1];
    // half-split: this lane's elements 4 (lane % 16) + i of a half, angles j = 4 (lane % 16) + i
    float2 ch[4];
    if constexpr (HALF) {
#pragma unroll
      for (int i = 0; i < 4; ++i) ch[i] = cs[static_cast<int64_t>(p) * (D / 2) + 4 * (lane & 15) + i];
    }
    const float r = rstd ? rstd[row] : 1.f;
    float s = 0.f;
    for (int h0 = 0; h0 < nqk; h0 += HG) {
      float d[HG][4], x[HG][4];
#pragma unroll
      for (int j = 0; j < HG; ++j) {
        const int h = h0 + j;
        if (h < nqk) {
          const __nv_bfloat16* src = h < n_q ? dQ + row * ldq + h * D : dK + row * ldkv + (h - n_q) * D;
          load_bf16x4(src + 4 * lane, d[j]);
          load_bf16x4(qk_save + row * ldsave + h * D + 4 * lane, x[j]);
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) d[j][i] = x[j][i] = 0.f;
        }
      }
      float rho[HG];
#pragma unroll
      for (int j = 0; j < HG; ++j)
        rho[j] = x[j][0] * x[j][0] + x[j][1] * x[j][1] + x[j][2] * x[j][2] + x[j][3] * x[j][3];
      warp_sum4(rho);
      float n[HG][4], dng[HG][4], t[HG];
#pragma unroll
      for (int j = 0; j < HG; ++j) {
        rho[j] = rsqrtf(rho[j] * (1.f / D) + eps);
        const bool is_q = h0 + j < n_q;
        float dn[4];
#pragma unroll
        for (int i = 0; i < 4; ++i) n[j][i] = x[j][i] * rho[j];
        if constexpr (HALF) {
          // inverse rotation of (first half, second half) element pairs; the
          // partner sits in lane l ^ 16 at the same index
          const bool second = lane >= 16;
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float dp = __shfl_xor_sync(0xffffffffu, d[j][i], 16);
            dn[i] = second ? -dp * ch[i].y + d[j][i] * ch[i].x : d[j][i] * ch[i].x + dp * ch[i].y;
          }
        } else {
          // inverse rotation of pairs (0,1) with c0 and (2,3) with c1
          dn[0] = d[j][0] * c0.x + d[j][1] * c0.y;
          dn[1] = -d[j][0] * c0.y + d[j][1] * c0.x;
          dn[2] = d[j][2] * c1.x + d[j][3] * c1.y;
          dn[3] = -d[j][2] * c1.y + d[j][3] * c1.x;
        }
        t[j] = 0.f;
        if (h0 + j < nqk) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            const float gg = is_q ? g_q[i] : g_k[i];
            if (is_q)
              aq[i] += dn[i] * n[j][i];
            else
              ak[i] += dn[i] * n[j][i];
            dng[j][i] = dn[i] * gg;
            t[j] += n[j][i] * dng[j][i];
          }
        } else {
#pragma unroll
          for (int i = 0; i < 4; ++i) dng[j][i] = 0.f;
        }
      }
      warp_sum4(t);
#pragma unroll
      for (int j = 0; j < HG; ++j) {
        const int h = h0 + j;
        if (h < nqk) {
          float dq[4];
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            dq[i] = rho[j] * (dng[j][i] - n[j][i] * t[j] * (1.f / D));
            s += dq[i] * x[j][i];
            dq[i] *= r;
          }
          store_bf16x4(Gp + row * ldg + h * D + 4 * lane, dq);
        }
      }
    }
    for (int h0 = 0; h0 < n_kv; h0 += HG) {
      float d[HG][4], v[HG][4];
#pragma unroll
      for (int j = 0; j < HG; ++j) {
        if (h0 + j < n_kv) {
          load_bf16x4(dV + row * ldkv + (h0 + j) * D + 4 * lane, d[j]);
          load_bf16x4(Vs + row * ldkv + (h0 + j) * D + 4 * lane, v[j]);
        }
      }
#pragma unroll
      for (int j = 0; j < HG; ++j) {
        if (h0 + j < n_kv) {
#pragma unroll
          for (int i = 0; i < 4; ++i) {
            s += d[j][i] * v[j][i];
            d[j][i] *= r;
          }
          store_bf16x4(Gp + row * ldg + ldsave + (h0 + j) * D + 4 * lane, d[j]);
        }
      }
    }
    s = warp_sum(s);
    if (lane == 0 && coef) coef[row] = r * r * s * inv_k;
  }
#pragma unroll
  for (int i = 0; i < 4; ++i) {
    red[w][4 * lane + i] = aq[i];
    red[w][D + 4 * lane + i] = ak[i];
  }
  __syncthreads();
  for (int j = threadIdx.x; j < 2 * D; j += blockDim.x) {
    float t = 0.f;
    for (int ww = 0; ww < QK_BWD_WARPS; ++ww) t += red[ww][j];
    dgam_part[static_cast<int64_t>(blockIdx.x) * 2 * D + j] = t;
  }
}

// The same map with its rows staged by bulk copies.  One persistent block
// per SM: a producer warp copies each token row's tensors -- dQ, dK, the
// saved pre-norm q|k, dV, V (each contiguous within the row) and the row's
// (cos, sin) table entry -- into a ring of shared-memory stages with
// cp.async.bulk, counted on the stage's "full" barrier; 18 compute warps
// take the row's heads (warp w: heads w, w + 18, ..., four at a time: the
// 64 + 8 q and k heads of a 70B-width block are one group of four per
// warp), store G' and arrive on the stage's "empty" barrier with their
// partial of the RMSNorm coefficient sum; the producer adds the partials
// when it reuses the stage (or at the end) and writes c for that row.  The
// copies keep a whole ring of rows in flight per SM, which a warp per row
// with register loads cannot.  Every wait is bounded (CODA_DEV_TIMEOUT).
// (8 compute warps, three groups each with a quarter of the slots idle:
// 84 us for 4096 such rows; 9: 74 us; 18: 62 us at 96 registers; 24 and
// more spill.)
constexpr int QKT_WARPS = 18;

template <bool HALF>
__global__ void __launch_bounds__((QKT_WARPS + 1) * 32, 1)
    qk_bwd_tma_kernel(const __nv_bfloat16* __restrict__ dQ, const __nv_bfloat16* __restrict__ dK,
                      const __nv_bfloat16* __restrict__ dV, const __nv_bfloat16* __restrict__ qk_save,
                      const __nv_bfloat16* __restrict__ Vs, const float* __restrict__ gq,
                      const float* __restrict__ gk, const int32_t* __restrict__ pos, const float2* __restrict__ cs,
                      int max_pos, float eps, int n_q, int n_kv, const float* __restrict__ rstd, int64_t M,
                      float inv_k, __nv_bfloat16* Gp, float* coef, float* dgam_part, int* status, int stages,
                      uint64_t timeout_ns) {
  griddep_launch_dependents();
  constexpr int D = 128;
  constexpr int HG = 4;
  extern __shared__ __align__(128) uint8_t qkt_smem[];
  __shared__ float red[QKT_WARPS][2 * D];
  __shared__ float part[8][QKT_WARPS];  // per stage (at most 8), per compute warp: partial of sum dq x
  __shared__ uint64_t full[8], empty[8];
  __shared__ int abort_flag;
  const int lane = threadIdx.x & 31, w = threadIdx.x >> 5;
  const int nqk = n_q + n_kv;
  const int64_t ldq = static_cast<int64_t>(n_q) * D, ldkv = static_cast<int64_t>(n_kv) * D;
  const int64_t ldsave = ldq + ldkv, ldg = ldq + 2 * ldkv;
  // stage layout (bytes): header {pos, r}, dQ, dK, saved q|k, dV, V, (cos, sin)[64]
  const uint32_t o_dq = 16, o_dk = o_dq + static_cast<uint32_t>(n_q) * 2 * D;
  const uint32_t o_sv = o_dk + static_cast<uint32_t>(n_kv) * 2 * D;
  const uint32_t o_dv = o_sv + static_cast<uint32_t>(nqk) * 2 * D;
  const uint32_t o_v = o_dv + static_cast<uint32_t>(n_kv) * 2 * D;
  const uint32_t o_cs = o_v + static_cast<uint32_t>(n_kv) * 2 * D;
  const uint32_t stage_bytes = o_cs + (D / 2) * 8;
  const uint32_t tx_bytes = stage_bytes - 16;
  if (threadIdx.x == 0) {
    for (int i = 0; i < stages; ++i) {
      mbar_init(&full[i], 1);
      mbar_init(&empty[i], QKT_WARPS);
    }
    abort_flag = 0;
    fence_mbar_init();
  }
  __syncthreads();
  const int64_t G = gridDim.x;
  if (w == QKT_WARPS) {
    // ------------------------------------------------------------ producer
    const uint32_t el = elect_one();
    const int lane_p = threadIdx.x & 31;
    int64_t it = 0;
    bool ok = true;
    // the positions and row factors of the block's next 32 rows, one per
    // lane, read by the whole warp at once (a row's cos/sin copy needs its
    // position: read row by row, each waited a global round trip)
    int pos_v = 0;
    float r_v = 1.f;
    for (int64_t row = blockIdx.x; row < M; row += G, ++it) {
      const int st = static_cast<int>(it % stages);
      const uint32_t ph = static_cast<uint32_t>((it / stages) & 1);
      if ((it & 31) == 0) {
        const int64_t rl = row + static_cast<int64_t>(lane_p) * G;
        pos_v = rl < M ? pos[rl] : 0;
        r_v = (rstd && rl < M) ? rstd[rl] : 1.f;
      }
      uint8_t* sb = qkt_smem + static_cast<size_t>(st) * stage_bytes;
      if (it >= stages) {
        if (!mbar_wait_bounded(&empty[st], ph ^ 1, &abort_flag, status, timeout_ns)) {
          ok = false;
          break;
        }
        if (el && coef) {  // the row that used this stage before (its r is in the stage header)
          const int64_t prev = row - static_cast<int64_t>(stages) * G;
          float t = 0.f;
          for (int k = 0; k < QKT_WARPS; ++k) t += part[st][k];
          const float r = reinterpret_cast<const float*>(sb)[1];
          coef[prev] = r * r * t * inv_k;
        }
      }
      int p = __shfl_sync(0xffffffffu, pos_v, static_cast<int>(it & 31));
      const float rrow = __shfl_sync(0xffffffffu, r_v, static_cast<int>(it & 31));
      if (p < 0 || p >= max_pos) {
        if (el && status) atomicOr(status, CODA_DEV_POSITION_RANGE);
        p = p < 0 ? 0 : max_pos - 1;
      }
      if (el) {
        reinterpret_cast<int*>(sb)[0] = p;
        reinterpret_cast<float*>(sb)[1] = rrow;
      }
      mbar_arrive_expect_tx(&full[st], tx_bytes, el);
      // (no copy of an empty range: a model without q or kv heads)
      const uint32_t el_q = n_q > 0 ? el : 0u, el_kv = n_kv > 0 ? el : 0u;
      bulk_load(sb + o_dq, dQ + row * ldq, static_cast<uint32_t>(ldq) * 2, &full[st], el_q);
      bulk_load(sb + o_dk, dK + row * ldkv, static_cast<uint32_t>(ldkv) * 2, &full[st], el_kv);
      bulk_load(sb + o_sv, qk_save + row * ldsave, static_cast<uint32_t>(ldsave) * 2, &full[st], el);
      bulk_load(sb + o_dv, dV + row * ldkv, static_cast<uint32_t>(ldkv) * 2, &full[st], el_kv);
      bulk_load(sb + o_v, Vs + row * ldkv, static_cast<uint32_t>(ldkv) * 2, &full[st], el_kv);
      bulk_load(sb + o_cs, cs + static_cast<int64_t>(p) * (D / 2), (D / 2) * 8, &full[st], el);
    }
    if (ok) {
      // the last rows of each stage: wait for their consumers, then write c
      const int64_t n_it = it;
      for (int64_t j = n_it > stages ? n_it - stages : 0; j < n_it; ++j) {
        const int st = static_cast<int>(j % stages);
        if (!mbar_wait_bounded(&empty[st], static_cast<uint32_t>((j / stages) & 1), &abort_flag, status,
                               timeout_ns))
          break;
        if (el && coef) {
          const int64_t row = blockIdx.x + j * G;
          float t = 0.f;
          for (int k = 0; k < QKT_WARPS; ++k) t += part[st][k];
          const float r = reinterpret_cast<const float*>(qkt_smem + static_cast<size_t>(st) * stage_bytes)[1];
          coef[row] = r * r * t * inv_k;
        }
      }
    } else {
      // let every issued copy land before the block's shared memory is released
      for (int64_t j = it > stages ? it - stages : 0; j < it; ++j)
        mbar_wait_drain(&full[j % stages], static_cast<uint32_t>((j / stages) & 1), 200000000ull);
    }
  } else {
    // ------------------------------------------------------------ compute warps
    float aq[4] = {0.f, 0.f, 0.f, 0.f}, ak[4] = {0.f, 0.f, 0.f, 0.f};
    float g_q[4], g_k[4];
    {
      const float4 a = *reinterpret_cast<const float4*>(gq + 4 * lane);
      const float4 b = *reinterpret_cast<const float4*>(gk + 4 * lane);
      g_q[0] = a.x; g_q[1] = a.y; g_q[2] = a.z; g_q[3] = a.w;
      g_k[0] = b.x; g_k[1] = b.y; g_k[2] = b.z; g_k[3] = b.w;
    }
    int64_t it = 0;
    for (int64_t row = blockIdx.x; row < M; row += G, ++it) {
      const int st = static_cast<int>(it % stages);
      if (!mbar_wait_bounded(&full[st], static_cast<uint32_t>((it / stages) & 1), &abort_flag, status,
                             timeout_ns))
        break;
      const uint8_t* sb = qkt_smem + static_cast<size_t>(st) * stage_bytes;
      const float r = reinterpret_cast<const float*>(sb)[1];
      const float2* css = reinterpret_cast<const float2*>(sb + o_cs);
      const float2 c0 = css[2 * lane], c1 = css[2 * lane + 1];
      float2 ch[4];
      if constexpr (HALF) {
#pragma unroll
        for (int i = 0; i < 4; ++i) ch[i] = css[4 * (lane & 15) + i];
      }
      float s = 0.f;
      for (int k0 = 0; w + k0 * QKT_WARPS < nqk; k0 += HG) {
        float d[HG][4], x[HG][4];
#pragma unroll
        for (int j = 0; j < HG; ++j) {
          const int h = w + (k0 + j) * QKT_WARPS;
          if (h < nqk) {
            const uint8_t* src = h < n_q ? sb + o_dq + h * 2 * D : sb + o_dk + (h - n_q) * 2 * D;
            const uint2 dr = *reinterpret_cast<const uint2*>(src + 8 * lane);
            const uint2 xr = *reinterpret_cast<const uint2*>(sb + o_sv + h * 2 * D + 8 * lane);
            d[j][0] = bf16_lo(dr.x); d[j][1] = bf16_hi(dr.x); d[j][2] = bf16_lo(dr.y); d[j][3] = bf16_hi(dr.y);
            x[j][0] = bf16_lo(xr.x); x[j][1] = bf16_hi(xr.x); x[j][2] = bf16_lo(xr.y); x[j][3] = bf16_hi(xr.y);
          } else {
#pragma unroll
            for (int i = 0; i < 4; ++i) d[j][i] = x[j][i] = 0.f;
          }
        }
        float rho[HG];
#pragma unroll
        for (int j = 0; j < HG; ++j)
          rho[j] = x[j][0] * x[j][0] + x[j][1] * x[j][1] + x[j][2] * x[j][2] + x[j][3] * x[j][3];
        warp_sum4(rho);
        float t[HG];
#pragma unroll
        for (int j = 0; j < HG; ++j) {
          const int h = w + (k0 + j) * QKT_WARPS;
          rho[j] = rsqrtf(rho[j] * (1.f / D) + eps);
          float dn[4];
          if constexpr (HALF) {
            // inverse rotation of (first half, second half) element pairs; the
            // partner sits in lane l ^ 16 at the same index
            const bool second = lane >= 16;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float dp = __shfl_xor_sync(0xffffffffu, d[j][i], 16);
              dn[i] = second ? -dp * ch[i].y + d[j][i] * ch[i].x : d[j][i] * ch[i].x + dp * ch[i].y;
            }
          } else {
            dn[0] = d[j][0] * c0.x + d[j][1] * c0.y;
            dn[1] = -d[j][0] * c0.y + d[j][1] * c0.x;
            dn[2] = d[j][2] * c1.x + d[j][3] * c1.y;
            dn[3] = -d[j][2] * c1.y + d[j][3] * c1.x;
          }
          t[j] = 0.f;
          if (h < nqk) {
            const bool is_q = h < n_q;
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float n = x[j][i] * rho[j];
              if (is_q)
                aq[i] += dn[i] * n;
              else
                ak[i] += dn[i] * n;
              d[j][i] = dn[i] * (is_q ? g_q[i] : g_k[i]);  // dn * gamma
              t[j] += n * d[j][i];
            }
          }
        }
        warp_sum4(t);
#pragma unroll
        for (int j = 0; j < HG; ++j) {
          const int h = w + (k0 + j) * QKT_WARPS;
          if (h < nqk) {
            float dq[4];
#pragma unroll
            for (int i = 0; i < 4; ++i) {
              const float n = x[j][i] * rho[j];
              dq[i] = rho[j] * (d[j][i] - n * t[j] * (1.f / D));
              s += dq[i] * x[j][i];
              dq[i] *= r;
            }
            store_bf16x4(Gp + row * ldg + h * D + 4 * lane, dq);
          }
        }
      }
      for (int h = w; h < n_kv; h += QKT_WARPS) {
        const uint2 dr = *reinterpret_cast<const uint2*>(sb + o_dv + h * 2 * D + 8 * lane);
        const uint2 vr = *reinterpret_cast<const uint2*>(sb + o_v + h * 2 * D + 8 * lane);
        float d[4] = {bf16_lo(dr.x), bf16_hi(dr.x), bf16_lo(dr.y), bf16_hi(dr.y)};
        const float v[4] = {bf16_lo(vr.x), bf16_hi(vr.x), bf16_lo(vr.y), bf16_hi(vr.y)};
#pragma unroll
        for (int i = 0; i < 4; ++i) {
          s += d[i] * v[i];
          d[i] *= r;
        }
        store_bf16x4(Gp + row * ldg + ldsave + h * D + 4 * lane, d);
      }
      s = warp_sum(s);
      __syncwarp();
      if (lane == 0) {
        part[st][w] = s;
        mbar_arrive(&empty[st]);  // this warp's reads of the stage are done
      }
    }
#pragma unroll
    for (int i = 0; i < 4; ++i) {
      red[w][4 * lane + i] = aq[i];
      red[w][D + 4 * lane + i] = ak[i];
    }
  }
  __syncthreads();
  for (int j = threadIdx.x; j < 2 * D; j += blockDim.x) {
    float t = 0.f;
    for (int ww = 0; ww < QKT_WARPS; ++ww) t += red[ww][j];
    dgam_part[static_cast<int64_t>(blockIdx.x) * 2 * D + j] = t;
  }
}

// Bytes of one stage of qk_bwd_tma_kernel and the stages that fit.
uint32_t qk_bwd_stage_bytes(int n_q, int n_kv) {
  return 16 + static_cast<uint32_t>(2 * n_q + 4 * n_kv) * 2 * 128 + 64 * 8;
}
int qk_bwd_tma_stages(int n_q, int n_kv) {
  const uint32_t b = qk_bwd_stage_bytes(n_q, n_kv);
  const int st = static_cast<int>(std::min<uint32_t>(4u, (200u * 1024u) / b));
  return st >= 2 ? st : 0;
}

cudaError_t launch_qk_bwd_tma(const __nv_bfloat16* dQ, const __nv_bfloat16* dK, const __nv_bfloat16* dV,
                              const __nv_bfloat16* qk_save, const __nv_bfloat16* V, const float* gq,
                              const float* gk, const int32_t* pos, const float2* cs, int max_pos, float eps, int n_q,
                              int n_kv, const float* rstd, int64_t M, float inv_k, __nv_bfloat16* Gp, float* coef,
                              float* dgam_part, int nblk, int* status, cudaStream_t s, bool rope_half,
                              uint64_t timeout_ns) {
  const int stages = qk_bwd_tma_stages(n_q, n_kv);
  if (stages == 0) return cudaErrorInvalidValue;
  const size_t smem = static_cast<size_t>(stages) * qk_bwd_stage_bytes(n_q, n_kv);
  auto k = rope_half ? qk_bwd_tma_kernel<true> : qk_bwd_tma_kernel<false>;
  // the shared-memory limit, raised once per device and variant to the
  // largest ring any call may use
  static std::mutex mu;
  static bool raised[64][2] = {};
  int dev = 0;
  cudaError_t e = cudaGetDevice(&dev);
  if (e != cudaSuccess) return e;
  if (dev < 0 || dev >= 64) return cudaErrorInvalidDevice;
  {
    std::lock_guard<std::mutex> lock(mu);
    if (!raised[dev][rope_half]) {
      e = cudaFuncSetAttribute(k, cudaFuncAttributeMaxDynamicSharedMemorySize, 200 * 1024);
      if (e != cudaSuccess) return e;
      raised[dev][rope_half] = true;
    }
  }
  note_launch();
  k<<<nblk, (QKT_WARPS + 1) * 32, smem, s>>>(dQ, dK, dV, qk_save, V, gq, gk, pos, cs, max_pos, eps, n_q, n_kv, rstd,
                                             M, inv_k, Gp, coef, dgam_part, status, stages, timeout_ns);
  return cudaGetLastError();
}

cudaError_t launch_qk_bwd(const __nv_bfloat16* dQ, const __nv_bfloat16* dK, const __nv_bfloat16* dV,
                          const __nv_bfloat16* qk_save, const __nv_bfloat16* V, const float* gq, const float* gk,
                          const int32_t* pos, const float2* cs, int max_pos, float eps, int n_q, int n_kv,
                          const float* rstd, int64_t M, float inv_k, __nv_bfloat16* Gp, float* coef,
                          float* dgam_part, int nblk, int* status, cudaStream_t s, bool rope_half) {
  note_launch();
  if (rope_half)
    qk_bwd_kernel<true><<<nblk, QK_BWD_WARPS * 32, 0, s>>>(dQ, dK, dV, qk_save, V, gq, gk, pos, cs, max_pos, eps,
                                                           n_q, n_kv, rstd, M, inv_k, Gp, coef, dgam_part, status);
  else
    qk_bwd_kernel<false><<<nblk, QK_BWD_WARPS * 32, 0, s>>>(dQ, dK, dV, qk_save, V, gq, gk, pos, cs, max_pos, eps,
                                                            n_q, n_kv, rstd, M, inv_k, Gp, coef, dgam_part, status);
  return cudaGetLastError();
}

}  // namespace coda
