// Internal launcher declarations shared by the host library's translation
// units.  Not part of the public ABI (see include/coda.h).
#pragma once
#include <cstdint>
#include <cuda.h>
#include <cuda_bf16.h>
#include <cuda_runtime.h>

#include "coda_gemm.cuh"

namespace coda {

enum class EpiKind : int { Plain = 0, Swiglu, DSwiglu, QkRope, CeLse, CeDlogits, ColDot, Sigmoid, RmsDx };

// Counts a kernel launch issued by this library (every launch site calls it
// just before its launch); coda_launch_count returns the process-wide total.
void note_launch();

// Tensor maps in the order A0, B0, A1, B1.  `cg` is the cluster size: 1
// (single CTAs), 2 (a cta_group::2 pair) or 4 (two pairs sharing B by TMA
// multicast); the launcher sizes the persistent grid.
cudaError_t launch_gemm_plain(int num_units, int sms, int cg, cudaStream_t s, const CUtensorMap* m,
                               const GemmArgs& a);
cudaError_t launch_gemm_swiglu(int num_units, int sms, int cg, cudaStream_t s, const CUtensorMap* m,
                               const GemmArgs& a);
cudaError_t launch_gemm_dswiglu(int num_units, int sms, int cg, cudaStream_t s, const CUtensorMap* m,
                               const GemmArgs& a);
cudaError_t launch_gemm_qkrope(int num_units, int sms, int cg, cudaStream_t s, const CUtensorMap* m,
                               const GemmArgs& a);
cudaError_t launch_gemm_qkrope_half(int num_units, int sms, int cg, cudaStream_t s, const CUtensorMap* m,
                                    const GemmArgs& a);
cudaError_t launch_gemm_celse(int num_units, int sms, int cg, cudaStream_t s, const CUtensorMap* m,
                               const GemmArgs& a);
cudaError_t launch_gemm_cedlogits(int num_units, int sms, int cg, cudaStream_t s, const CUtensorMap* m,
                               const GemmArgs& a);
cudaError_t launch_gemm_sigmoid(int num_units, int sms, int cg, cudaStream_t s, const CUtensorMap* m,
                                const GemmArgs& a);
cudaError_t launch_gemm_plain_fp8(int num_units, int sms, int cg, cudaStream_t s, const CUtensorMap* m,
                                  const GemmArgs& a);
cudaError_t launch_gemm_swiglu_fp8(int num_units, int sms, int cg, cudaStream_t s, const CUtensorMap* m,
                                   const GemmArgs& a);
cudaError_t launch_gemm_qkrope_fp8(int num_units, int sms, int cg, cudaStream_t s, const CUtensorMap* m,
                                   const GemmArgs& a);
cudaError_t launch_gemm_qkrope_half_fp8(int num_units, int sms, int cg, cudaStream_t s, const CUtensorMap* m,
                                        const GemmArgs& a);
cudaError_t launch_gemm_celse_fp8(int num_units, int sms, int cg, cudaStream_t s, const CUtensorMap* m,
                                  const GemmArgs& a);
cudaError_t launch_gemm_cedlogits_fp8(int num_units, int sms, int cg, cudaStream_t s, const CUtensorMap* m,
                                      const GemmArgs& a);
cudaError_t launch_gemm_dswiglu_fp8(int num_units, int sms, int cg, cudaStream_t s, const CUtensorMap* m,
                                    const GemmArgs& a);
cudaError_t launch_gemm_rmsdx_fp8(int num_units, int sms, int cg, cudaStream_t s, const CUtensorMap* m,
                                  const GemmArgs& a);
cudaError_t launch_gemm_rmsdx(int num_units, int sms, int cg, cudaStream_t s, const CUtensorMap* m,
                              const GemmArgs& a);
cudaError_t launch_gemm_coldot(int num_units, int sms, int cg, cudaStream_t s, const CUtensorMap* m,
                               const GemmArgs& a);

// NVFP4 operands (coda_nvfp4.cu): e2m1 codes in tensor maps m[0] (A), m[1]
// (B, or the gate half when a.b_dual), m[2] (the up half); the e4m3 block
// scales in the tensor-core order described there.
struct Nvfp4Scales {
  const uint8_t* a;   // A's block scales
  const uint8_t* b0;  // B's (gate weight's) block scales
  const uint8_t* b1;  // up weight's block scales (b_dual)
  int64_t kt;         // k tiles of 256 elements
};
uint32_t nvfp4_idesc();
// Cluster size of the NVFP4 kernel for M rows: 1 (single CTAs), 2 or 4
// (CTAs sharing B; each copies 256 / cg rows of the B tile, so the B tensor
// maps must have boxes of that many rows).
int nvfp4_cluster_size(int64_t M);
// CTA pairs (cta_group::2, 256 x 256 tiles) for M rows; then the tensor maps
// are A, B0, B1 with 128-row boxes and the block scales of A, B0, B1 as 2-D
// byte maps [bytes / 256, 256] with 8-row boxes (one 2 KB group).
bool nvfp4_pairs(int64_t M);
uint32_t nvfp4_idesc_pair();
cudaError_t launch_gemm_nvfp4_pair(int kind, int num_units, int sms, cudaStream_t s, const CUtensorMap* m,
                                   const GemmArgs& a, const Nvfp4Scales& sc);
// gamma (optional): quantise x * gamma (fp32 products); rstd (optional):
// also write 1 / sqrt(mean(x^2) + eps) per row.
cudaError_t launch_quantize_nvfp4_rows(const __nv_bfloat16* X, int64_t ldx, int64_t M, int64_t K, uint8_t* Q,
                                       uint8_t* SF, float* scale, int num_sms, cudaStream_t s,
                                       const float* gamma = nullptr, float* rstd = nullptr, float eps = 0.f);
cudaError_t launch_gemm_plain_nvfp4(int cg, int num_units, int sms, cudaStream_t s, const CUtensorMap* m,
                                    const GemmArgs& a, const Nvfp4Scales& sc);
cudaError_t launch_gemm_swiglu_nvfp4(int cg, int num_units, int sms, cudaStream_t s, const CUtensorMap* m,
                                     const GemmArgs& a, const Nvfp4Scales& sc);

// auxiliary kernels (coda_aux.cu)
cudaError_t launch_fold_gamma(const __nv_bfloat16* W, const float* gamma, __nv_bfloat16* Wf, int64_t N, int64_t K,
                              int num_sms, cudaStream_t s);
cudaError_t launch_row_rstd(const __nv_bfloat16* X, int64_t ldx, int64_t M, int64_t K, float eps, float* rstd,
                            int num_sms, cudaStream_t s, const float* gamma = nullptr, __nv_bfloat16* U = nullptr,
                            int64_t ldu = 0);
// mode 0: out = 1/sqrt(sum_t p[t] * inv_k + eps);  mode 1: out = r^2 * sum_t p[t] * inv_k
cudaError_t launch_combine_rows(const float* p, int64_t ld, int nparts, int64_t M, float inv_k, float eps,
                                const float* r, float* out, int mode, cudaStream_t s);
// G' = bf16(r G) and the RMSNorm-backward row coefficient c = r^2 sum G (Y - R) * inv_k
cudaError_t launch_rms_bwd_prepass(const __nv_bfloat16* G, const __nv_bfloat16* Y, const __nv_bfloat16* R,
                                   const float* rstd, int64_t M, int64_t N, float inv_k, __nv_bfloat16* Gp,
                                   float* coef, int num_sms, cudaStream_t s);
// column sums; with out2, columns from `split` on go to out2
cudaError_t launch_colsum(const float* p, int64_t nrows, int64_t ncols, int64_t ld, float* out, cudaStream_t s,
                          int64_t split = -1, float* out2 = nullptr);
cudaError_t launch_ce_combine(const float2* part, int64_t ld, int nchunks, const float* target,
                              const int32_t* labels, int32_t ignore, int64_t M, int64_t V, float* lse,
                              double* blk_loss, int* blk_cnt, int nblk, float* loss_mean, int32_t* n_valid,
                              int* status, cudaStream_t s);
cudaError_t launch_ce_onehot_prep(const int32_t* labels, int32_t ignore, int64_t M, int64_t V,
                                  const int32_t* n_valid, float dloss, const float* rstd, float* wrow, int32_t* lrow,
                                  int32_t* counts, int32_t* cursor, int32_t* off, int32_t* idx, cudaStream_t s);
cudaError_t launch_ce_norm_coef(const float* pz, int64_t ld, int nparts, const float* target, const float* rstd,
                                const float* rw, int64_t M, float inv_k, float* coef, cudaStream_t s);
cudaError_t launch_quantize_fp8_rows(const __nv_bfloat16* X, int64_t ldx, int64_t M, int64_t K, uint8_t* Xq,
                                     int64_t ldq, float* scale, int num_sms, cudaStream_t s);
// e4m3 codes of the transpose of X [R, C] (with X2 [R2, C] stacked below, or
// NULL): out [C, R + R2] (row stride ldo), per-column scales [C].
cudaError_t launch_quantize_fp8_cols(const __nv_bfloat16* X, int64_t ldx, int64_t R, const __nv_bfloat16* X2,
                                     int64_t ldx2, int64_t R2, int64_t C, uint8_t* out, int64_t ldo, float* scale,
                                     int num_sms, cudaStream_t s);
cudaError_t launch_selftest_wait_timeout(uint64_t limit_ns, int* status, cudaStream_t s);
cudaError_t launch_rope_table(double theta, int head_dim, int max_pos, float2* cs, cudaStream_t s);
cudaError_t launch_qk_bwd(const __nv_bfloat16* dQ, const __nv_bfloat16* dK, const __nv_bfloat16* dV,
                          const __nv_bfloat16* qk_save, const __nv_bfloat16* V, const float* gq, const float* gk,
                          const int32_t* pos, const float2* cs, int max_pos, float eps, int n_q, int n_kv,
                          const float* rstd, int64_t M, float inv_k, __nv_bfloat16* Gp, float* coef,
                          float* dgam_part, int nblk, int* status, cudaStream_t s, bool rope_half = false);

// The same map with its rows staged in shared memory by bulk copies (one
// persistent block per SM, nblk <= the SM count); qk_bwd_tma_stages() is 0
// when a row's tensors are too large for two stages, and then only
// launch_qk_bwd applies.
int qk_bwd_tma_stages(int n_q, int n_kv);
cudaError_t launch_qk_bwd_tma(const __nv_bfloat16* dQ, const __nv_bfloat16* dK, const __nv_bfloat16* dV,
                              const __nv_bfloat16* qk_save, const __nv_bfloat16* V, const float* gq,
                              const float* gk, const int32_t* pos, const float2* cs, int max_pos, float eps, int n_q,
                              int n_kv, const float* rstd, int64_t M, float inv_k, __nv_bfloat16* Gp, float* coef,
                              float* dgam_part, int nblk, int* status, cudaStream_t s, bool rope_half,
                              uint64_t timeout_ns);

constexpr int QK_BWD_WARPS = 8;
constexpr int CE_COMBINE_THREADS = 256;

}  // namespace coda
