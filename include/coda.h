/*
 * coda.h -- C ABI of libcoda.so: bf16 GEMMs whose output tiles are
 * transformed on chip by composable epilogue primitives, and the transformer
 * operators built from them (GB300 / sm_103a).
 *
 * Source of the method: "CODA: Rewriting Transformer Blocks as GEMM-Epilogue
 * Programs" (arXiv 2605.19269): §2.2 (GEMM mainloop + epilogue, locality
 * constraint), §3.1 (the five epilogue primitive classes), §3.2 (h = xW,
 * y[i,j] = f_ij(tile)), §3.2.1 (GEMM-residual-RMSNorm-GEMM reparameterisation
 * y = RMSNorm(xW0 + z, gamma) W1 = (r (xW0 + z) ⊙ gamma) W1, Fig. 4); the
 * functional operator names linear_swiglu, linear_cross_entropy and
 * linear_qknorm_rope come from the x-tip guide "CODA: 把 Transformer Block
 * 重写成 GEMM-Epilogue 程序" (section 核验过程 / 使用 Functional API).
 *
 * Conventions shared by every call
 * --------------------------------
 *  - All tensor pointers are DEVICE pointers owned by the caller.  The
 *    library never allocates or frees device memory.  Calls that need scratch
 *    take a caller-allocated workspace `ws` of at least the size returned by
 *    the matching *_workspace_size() query; its first 256 bytes hold the
 *    device status word (zero it once, e.g. with coda_reset_status, before
 *    first use).
 *  - Calls are asynchronous on `stream` (a cudaStream_t; NULL = legacy
 *    default stream).  They return after enqueueing.  A GEMM may run part of
 *    its tiles on a second, library-created non-blocking stream (one per
 *    device and caller stream, kept for the process), forked from and joined
 *    back to `stream` with events inside the call: work the caller enqueues
 *    on `stream` afterwards is ordered after all of it.
 *  - Calls can be captured into a CUDA graph (stream capture); the forks and
 *    joins above, and those of the optional side streams, become graph
 *    edges.  The first call of each kind on a device (which sets kernel
 *    attributes and creates the library's streams) and the first call on
 *    each capture stream must run outside a capture.
 *  - Matrices are row-major with a leading dimension (row stride) given in
 *    ELEMENTS.  Weights use the nn.Linear layout [out_features, in_features].
 *  - bf16 tensors are passed as uint16_t bit patterns (coda_bf16).  All
 *    fp32 -> bf16 conversions round to nearest even.  Accumulation is fp32.
 *  - Alignment: every tensor pointer 16-byte aligned, every leading dimension
 *    a multiple of 8 elements, feature dimensions (N, K, I, V, hidden) a
 *    multiple of 8.  M (tokens) is arbitrary.
 *  - Errors detected on the host are returned before anything is enqueued:
 *    CODA_ERR_INVALID_ARG, CODA_ERR_ALIGNMENT, CODA_ERR_UNSUPPORTED,
 *    CODA_ERR_WORKSPACE.  CODA_ERR_CUDA reports a failed launch.  Errors
 *    found on the device (a bounded wait that ran out, a label or position
 *    out of range) set bits of the workspace status word; read them with
 *    coda_get_status().
 *  - M == 0 (no rows) is a valid no-op.
 */
#ifndef CODA_H
#define CODA_H

#include <stddef.h>
#include <stdint.h>

#ifdef __cplusplus
extern "C" {
#endif

typedef uint16_t coda_bf16;
typedef void* coda_stream;

typedef enum coda_status {
  CODA_OK = 0,
  CODA_ERR_INVALID_ARG = 1,    /* null required pointer, negative size, bad enum */
  CODA_ERR_ALIGNMENT = 2,      /* pointer not 16-byte aligned or ld % 8 != 0 */
  CODA_ERR_UNSUPPORTED = 3,    /* shape or option combination not implemented */
  CODA_ERR_WORKSPACE = 4,      /* ws NULL or ws_bytes below the queried size */
  CODA_ERR_CUDA = 5,           /* a CUDA runtime call or launch failed */
  CODA_ERR_TIMEOUT = 6,        /* device: a bounded pipeline wait ran out */
  CODA_ERR_LABEL_RANGE = 7,    /* device: label outside [0,V) and != ignore_index */
  CODA_ERR_POSITION_RANGE = 8  /* device: RoPE position outside [0, max_pos) */
} coda_status;

/* Operand storage order of a GEMM operand. */
enum { CODA_K_MAJOR = 0, CODA_MN_MAJOR = 1 };
/* Output element type. */
enum { CODA_BF16 = 0, CODA_F32 = 1 };

/* Epilogue map selected in coda_epilogue_desc.map (§3.1 classes 1-5). */
enum {
  CODA_MAP_NONE = 0,         /* D = rs*cs*acc + aux_in[0] - row_coef*aux_in[1] (+D if beta); optional row sum-of-squares partials */
  CODA_MAP_SWIGLU = 1,       /* H = silu(rs*X B^T) * (rs*X B2^T); aux_out[0], aux_out[1] save g, u */
  CODA_MAP_DSWIGLU = 2,      /* acc = dH; aux_in = g, u; aux_out[0..2] = rs*dG, rs*dU, H; partials = row sum(dG g + dU u) */
  CODA_MAP_QKNORM_ROPE = 3,  /* per-head RMSNorm + RoPE of q/k heads, v pass-through; aux_out[0] saves pre-norm q|k */
  CODA_MAP_CE_LSE = 4,       /* online (max, sum-exp) per row over vocab tiles + target logit; D unused */
  CODA_MAP_CE_DLOGITS = 5,   /* D = (softmax(acc) - onehot) * dloss / n_valid */
  CODA_MAP_COLDOT = 6,       /* D = cs*acc; partials = column sums of aux_in[0]*acc per 32-row group */
  CODA_MAP_SIGMOID = 7,      /* D = sigmoid(rs*acc) (* aux_in[0] when given) */
  CODA_MAP_DSIGMOID = 8      /* recomputed z = rs*acc, dY = aux_in[1]: aux_out[0] = dY (*aux_in[0]) s(1-s), aux_out[1] = dY s */
};

/* RoPE pairing of a head's elements (the pages leave the convention open;
 * both are supported): CODA_ROPE_INTERLEAVED rotates pairs (2j, 2j+1),
 * CODA_ROPE_HALF rotates pairs (j, j + head_dim/2); pair j's angle is
 * pos * theta^(-2j/head_dim) in both. */
typedef enum coda_rope_pairing { CODA_ROPE_INTERLEAVED = 0, CODA_ROPE_HALF = 1 } coda_rope_pairing;

/*
 * Epilogue descriptor: which primitives run on each output tile before it is
 * written ("CODA" §3.1: element-wise/pairwise maps, rank-1 vector loads,
 * rank-2 tile loads/stores, tile reductions to partials, running state).
 * Unused pointers must be NULL, unused integers 0.
 */
typedef struct coda_epilogue_desc {
  int32_t map;                   /* CODA_MAP_* */
  const float* row_scale;        /* [M] fp32 per-row factor rs (e.g. 1/rms) or NULL */
  const float* col_scale;        /* [N] fp32 per-column factor cs (e.g. gamma) or NULL */
  const coda_bf16* aux_in[2];    /* rank-2 tile loads, [M, N] bf16 row-major */
  int64_t ld_aux_in[2];
  const float* row_coef;         /* [M] fp32: MAP_NONE subtracts row_coef[i]*aux_in[1][i,j] */
  coda_bf16* aux_out[3];         /* rank-2 tile stores, [M, N] bf16 row-major */
  int64_t ld_aux_out[3];
  float* partials;               /* reduction partials (layout per map, see coda_gemm_epilogue) */
  int64_t ld_partials;           /* elements between partial rows (>= M for row partials, >= N for column partials) */
  int32_t beta;                  /* 1: accumulate into D (D += result) */
  const coda_bf16* B2;           /* MAP_SWIGLU: second weight [N, K] (K-major) */
  int64_t ldb2;
  const coda_bf16* A2;           /* concatenated K: second (A2, B2) pair, same major-ness as A, B */
  int64_t lda2;
  int64_t K2;                    /* contraction length of the second pair (0 = none) */
  /* cross-entropy */
  const int32_t* labels;         /* [M] */
  int32_t ignore_index;
  const float* lse;              /* [M] saved log-sum-exp (CE_DLOGITS) */
  const int32_t* n_valid;        /* device int32: number of non-ignored rows (CE_DLOGITS) */
  float dloss;                   /* upstream gradient of the mean loss (CE_DLOGITS) */
  float* target_logit;           /* [M] fp32 out (CE_LSE) */
  int32_t vocab_tiles_per_unit;  /* CE_LSE: 256-wide vocab tiles per running-state chunk (0 = 16) */
  /* QK-RMSNorm + RoPE */
  const int32_t* positions;      /* [M] */
  const float* cos_sin;          /* [max_pos, head_dim/2, 2] fp32 table from coda_rope_table */
  int32_t max_pos;
  int32_t n_q_heads, n_kv_heads, head_dim;
  float eps;
  const float* gamma_q;          /* [head_dim] */
  const float* gamma_k;          /* [head_dim] */
  coda_bf16* Q;                  /* [M, n_q*head_dim] */
  coda_bf16* K;                  /* [M, n_kv*head_dim] */
  coda_bf16* V;                  /* [M, n_kv*head_dim] */
  int32_t rope_pairing;          /* coda_rope_pairing (0 = interleaved) */
  /* Operand type.  CODA_OPERAND_E4M3: A, B (and A2, B2) are e4m3 bytes,
   * K-major, K a multiple of 16, and the accumulator is dequantised as
   * acc[i, j] * acc_row_scale[i] * acc_col_scale[j] (each NULL = 1) before
   * the map runs -- the two operands' per-row scales of
   * coda_quantize_fp8_rows / coda_quantize_fp8_cols.  MAP_NONE and
   * MAP_SWIGLU take those scales in row_scale / col_scale instead. */
  int32_t operand_type;          /* CODA_OPERAND_BF16 (0) or CODA_OPERAND_E4M3 (1) */
  const float* acc_row_scale;    /* [M] or NULL */
  const float* acc_col_scale;    /* [N] or NULL */
} coda_epilogue_desc;

/* Operand element type of coda_epilogue_desc.operand_type. */
enum { CODA_OPERAND_BF16 = 0, CODA_OPERAND_E4M3 = 1 };

/* ------------------------------------------------------------------------
 * Library / device status
 * --------------------------------------------------------------------- */

/* Version string of the library. */
const char* coda_version(void);

/* Number of kernels this library has launched in the calling process, on
 * every device and stream, since it was loaded (a host-side counter: each
 * launch site counts its launch as it issues it; failed launches included,
 * driver memsets and copies not).  Read it before and after a region to
 * count that region's launches.  Never fails. */
uint64_t coda_launch_count(void);

/* Human-readable name of a status code. */
const char* coda_status_string(int status);

/* Synchronises `stream`, then maps the device status word at the start of
 * `ws` to a coda_status (CODA_OK if no device error bit is set).  The word is
 * sticky: it keeps its bits until coda_reset_status(). */
int coda_get_status(const void* ws, coda_stream stream);

/* Enqueues a clear of the device status word (asynchronous). */
int coda_reset_status(void* ws, coda_stream stream);

/* Failure-path self-test: enqueues one thread that waits, through the same
 * bounded mbarrier wait every GEMM pipeline stage uses, on a barrier that
 * nothing arrives on.  After limit_us microseconds (1 .. 1e6) the wait gives
 * up and sets the timeout bit of the status word in `ws` (256 bytes), so a
 * following coda_get_status returns CODA_ERR_TIMEOUT and the CUDA context
 * stays usable.  No kernel traps or spins without a limit. */
int coda_selftest_wait_timeout(uint32_t limit_us, void* ws, coda_stream stream);

/* ------------------------------------------------------------------------
 * Generic GEMM + epilogue ("CODA" §3.2: h = xW, y[i,j] = f_ij(h tile))
 *
 *   acc[m, n] = sum_k A(m, k) * B(n, k)   (+ the A2/B2 pair when K2 > 0)
 *   D = epilogue(acc)                      (desc->map, see CODA_MAP_*)
 *
 * A: a_major == CODA_K_MAJOR -> A is [M, K] with row stride lda;
 *    CODA_MN_MAJOR -> A is stored [K, M] with row stride lda.
 * B: b_major == CODA_K_MAJOR -> B is [N, K] (nn.Linear weight);
 *    CODA_MN_MAJOR -> B is stored [K, N].
 * D: [M, N] row-major, d_dtype CODA_BF16 or CODA_F32 (F32 only for MAP_NONE).
 * Partials layouts: MAP_NONE / MAP_DSWIGLU row partials [ceil(N/256), ld] fp32;
 * MAP_CE_LSE (max, sumexp) float2 [ceil(ceil(N/256)/tiles_per_unit), ld];
 * MAP_COLDOT column partials [4*ceil(M/128), ld].
 * MAP_SWIGLU: N is the output width; B and B2 are the gate and up weights.
 * Workspace: coda_gemm_epilogue_workspace_size() bytes (the status word).
 * ---------------------------------------------------------------------- */
size_t coda_gemm_epilogue_workspace_size(void);
int coda_gemm_epilogue(const coda_epilogue_desc* desc,
                       const coda_bf16* A, int64_t lda, int a_major,
                       const coda_bf16* B, int64_t ldb, int b_major,
                       void* D, int64_t ldd, int d_dtype,
                       int64_t M, int64_t N, int64_t K,
                       void* ws, size_t ws_bytes, coda_stream stream);

/* ------------------------------------------------------------------------
 * RMSNorm pieces ("CODA" §3.2.1)
 * --------------------------------------------------------------------- */

/* gamma fold: Wf[n, k] = bf16(gamma[k] * W[n, k]).  W, Wf: [N, K] bf16
 * (may alias for an in-place fold); gamma: [K] fp32.  This is the
 * "⊙ gamma moves into W1" step of the §3.2.1 equation; run once per weight
 * version. */
int coda_fold_gamma(const coda_bf16* W, const float* gamma, coda_bf16* Wf,
                    int64_t N, int64_t K, coda_stream stream);

/* r[i] = 1/sqrt(mean_k X[i,k]^2 + eps) for X [M, K] bf16 (row stride ldx):
 * the per-row inverse RMS factor r of §3.2.1 for an input that no upstream
 * GEMM epilogue produced. */
int coda_rms_rstd(const coda_bf16* X, int64_t ldx, int64_t M, int64_t K, float eps,
                  float* rstd, coda_stream stream);

/* RMSNorm prepass for an input no upstream GEMM epilogue produced:
 *   rstd[i] = 1/sqrt(mean_k X[i,k]^2 + eps),   U[i, k] = bf16(X[i,k] * gamma[k])
 * in one read of X [M, K] bf16 (row stride ldx).  U [M, K] bf16 (row stride
 * ldu) is the input of the RMSNorm-reparameterised GEMM that applies rstd in
 * its epilogue (§3.2.1: the gamma multiply is block-local and the row factor
 * r moves to the end of the next GEMM).  gamma [K] fp32.  All pointers
 * required, 16-byte aligned. */
int coda_rmsnorm_scale(const coda_bf16* X, int64_t ldx, int64_t M, int64_t K, float eps, const float* gamma,
                       float* rstd, coda_bf16* U, int64_t ldu, coda_stream stream);

/* RoPE table: cos_sin[p, j] = (cos a, sin a), a = p * theta^(-2j/head_dim),
 * j < head_dim/2, p < max_pos; computed in fp64, stored fp32.  Interleaved
 * pair convention (2j, 2j+1). */
int coda_rope_table(float theta, int32_t head_dim, int32_t max_pos, float* cos_sin,
                    coda_stream stream);

/* ------------------------------------------------------------------------
 * RMSNorm-reparameterised projection + residual (§3.2.1, second GEMM)
 *
 *   Y = R + r ⊙ (X Wf^T),   Wf = W diag(gamma) (coda_fold_gamma),
 *   which equals R + RMSNorm(X, gamma) W^T.
 * X [M, K], Wf [N, K], R [M, N] (or NULL), Y [M, N] bf16.
 * rstd_in: [M] fp32 r from an upstream epilogue, or NULL -> r is computed
 * from X (eps) and also written to rstd_out (required then).
 * ---------------------------------------------------------------------- */
size_t coda_rmsnorm_linear_workspace_size(int64_t M, int64_t N, int64_t K);
int coda_rmsnorm_linear(const coda_bf16* X, const float* rstd_in, const coda_bf16* Wf,
                        const coda_bf16* R, float eps, float* rstd_out, coda_bf16* Y,
                        int64_t M, int64_t N, int64_t K, void* ws, size_t ws_bytes, coda_stream stream);

/* Backward of coda_rmsnorm_linear for upstream gradient dY [M, N]:
 *   G' = r ⊙ dY,  c_i = r_i^2 sum_n dY_in (Y - R)_in / K,  D = G' W,
 *   dX = gamma ⊙ D - c ⊙ X,  dW = (G'^T X) diag(gamma),
 *   dgamma_k = sum_i X_ik D_ik   (column partials of the dX epilogue).
 *   (dR = dY: no copy is made.)
 * Inputs: X [M,K], W [N,K] (not folded), gamma [K], rstd [M], Y and R [M,N]
 * (R may be NULL = zero).  Outputs: dX [M,K], dW [N,K] bf16, dgamma [K] fp32.
 * The pages state only that this backward keeps the GEMM-epilogue form; the
 * formulas are the chain rule of the §3.2.1 equation, and they hold whether
 * the forward folded gamma into W or applied it to the GEMM input.
 * side_stream (optional, may be NULL): a second stream on which the dW GEMM
 * runs beside c -> dX (ordered by events the call records; the call returns
 * with `stream` waiting for both).  Both use the one workspace. */
size_t coda_rmsnorm_linear_bwd_workspace_size(int64_t M, int64_t N, int64_t K);
int coda_rmsnorm_linear_bwd(const coda_bf16* dY, const coda_bf16* X, const coda_bf16* W, const float* gamma,
                            const float* rstd, const coda_bf16* Y, const coda_bf16* R,
                            coda_bf16* dX, coda_bf16* dW, float* dgamma,
                            int64_t M, int64_t N, int64_t K, void* ws, size_t ws_bytes, coda_stream stream,
                            coda_stream side_stream);

/* ------------------------------------------------------------------------
 * Projection + residual (§3.2.1, first GEMM: "xW0 + z")
 *
 *   Y = R + X W^T    X [M, K], W [N, K], R [M, N] (NULL = 0), Y [M, N].
 * rstd_out (optional, [M]): the epilogue also emits per-tile partial sums of
 * squares of Y, merged by a small second kernel into
 * rstd_out[i] = 1/sqrt(mean_n Y_in^2 + eps): the row factor r the next
 * RMSNorm-reparameterised projection applies in its epilogue.
 * gamma_next [N] fp32 and U_out [M, N] bf16 (optional, both or neither): the
 * epilogue also writes U_out = bf16(Y ⊙ gamma_next), Y as stored -- the
 * "⊙ gamma" of §3.2.1 applied where it is block-local, so the next GEMM
 * reads U with its weight unfolded.
 * ---------------------------------------------------------------------- */
size_t coda_linear_residual_workspace_size(int64_t M, int64_t N, int64_t K);
int coda_linear_residual(const coda_bf16* X, const coda_bf16* W, const coda_bf16* R,
                         coda_bf16* Y, float eps, float* rstd_out, const float* gamma_next, coda_bf16* U_out,
                         int64_t M, int64_t N, int64_t K, void* ws, size_t ws_bytes, coda_stream stream);

/* Backward: dX = dY W [M, K], dW = dY^T X [N, K]; dR = dY (no copy). */
size_t coda_linear_residual_bwd_workspace_size(int64_t M, int64_t N, int64_t K);
int coda_linear_residual_bwd(const coda_bf16* dY, const coda_bf16* X, const coda_bf16* W,
                             coda_bf16* dX, coda_bf16* dW,
                             int64_t M, int64_t N, int64_t K, void* ws, size_t ws_bytes, coda_stream stream);

/* ------------------------------------------------------------------------
 * linear_swiglu (x-tip guide functional API; "CODA" §3.1 class 1 pairwise
 * SwiGLU gate)
 *
 *   g = r ⊙ (X Wg^T),  u = r ⊙ (X Wu^T),  H = silu(g) ⊙ u
 * X [M, K]; Wg, Wu [I, K] (pass gamma-folded weights with rstd for the
 * RMSNorm-reparameterised MLP input); rstd [M] or NULL (r = 1);
 * H [M, I]; g_save, u_save [M, I] or NULL.
 * ---------------------------------------------------------------------- */
size_t coda_linear_swiglu_workspace_size(int64_t M, int64_t I, int64_t K);
int coda_linear_swiglu(const coda_bf16* X, const float* rstd, const coda_bf16* Wg, const coda_bf16* Wu,
                       coda_bf16* H, coda_bf16* g_save, coda_bf16* u_save,
                       int64_t M, int64_t I, int64_t K, void* ws, size_t ws_bytes, coda_stream stream);

/* Backward of the SwiGLU MLP sublayer  Y = Xres + silu(g) u Wd^T  with
 * g, u = r ⊙ (X ⊙ gamma) [Wg; Wu]^T (linear_swiglu on the gain-scaled input,
 * or on X with gamma folded into Wg, Wu -- the gradients are the same):
 *   dH = dY Wd (GEMM) -> dSwiGLU epilogue -> G' = r ⊙ [dG | dU];
 *   D = G' [Wg; Wu]  (one GEMM over K = 2I),
 *   dX = gamma ⊙ D - c ⊙ X + dX_resid  with the dgamma_k = sum_i X_ik D_ik
 *   column partials in its epilogue;
 *   dWd = dY^T H;  dWg = (G'_g^T X) diag(gamma), dWu likewise.
 * With rstd == NULL there is no RMSNorm (r = 1, c = 0, gamma ignored,
 * dX = D + dX_resid, dgamma untouched).
 * Inputs: dY [M,K]; X [M,K]; rstd [M]|NULL; gamma [K]|NULL; Wg, Wu [I,K]
 * (not folded); Wd [K,I]; g, u, H [M,I] saved by the forward; dX_resid
 * [M,K]|NULL (gradient of the residual stream, added to dX).
 * Outputs: dX [M,K], dWg, dWu [I,K], dWd [K,I] bf16; dgamma [K] fp32|NULL.
 * side_stream (optional, may be NULL): a second stream on which dWd, dWg
 * and dWu run beside the dH -> dX chain (ordered by events the call
 * records; the call returns with `stream` waiting for both chains).  The
 * call's kernels on either stream use the one workspace. */
size_t coda_linear_swiglu_bwd_workspace_size(int64_t M, int64_t I, int64_t K);
int coda_linear_swiglu_bwd(const coda_bf16* dY, const coda_bf16* X, const float* rstd, const float* gamma,
                           const coda_bf16* Wg, const coda_bf16* Wu, const coda_bf16* Wd, const coda_bf16* g,
                           const coda_bf16* u, const coda_bf16* H, const coda_bf16* dX_resid,
                           coda_bf16* dX, coda_bf16* dWg, coda_bf16* dWu, coda_bf16* dWd, float* dgamma,
                           int64_t M, int64_t I, int64_t K, void* ws, size_t ws_bytes, coda_stream stream,
                           coda_stream side_stream);

/* ------------------------------------------------------------------------
 * linear_qknorm_rope (x-tip guide functional API): RMSNorm-reparameterised
 * fused QKV projection with per-head QK-RMSNorm and RoPE in the epilogue.
 *
 *   [q | k | v] = r ⊙ (X W^T),   which is RMSNorm(x, gamma_in) W_qkv^T when
 *   either X = x ⊙ gamma_in (coda_rmsnorm_scale) and W = W_qkv, or X = x and
 *   W = W_qkv diag(gamma_in) (coda_fold_gamma);
 *   Q_h = RoPE(RMSNorm_d(q_h) ⊙ gamma_q, pos),  K_h likewise, V = v.
 * head_dim must be 128.  Column order of W rows: n_q q heads, then
 * n_kv k heads, then n_kv v heads.  X [M, Kdim]; W [(n_q+2n_kv)*128, Kdim];
 * rstd [M] (NULL: r = 1); gamma_q, gamma_k [128]; pos [M] int32 in
 * [0, max_pos); cos_sin from coda_rope_table; rope_pairing a
 * coda_rope_pairing (the kernel is compiled for each).  Outputs Q [M, n_q*128],
 * K, V [M, n_kv*128]; qk_save [M, (n_q+n_kv)*128] pre-norm q|k or NULL.
 * ---------------------------------------------------------------------- */
size_t coda_linear_qknorm_rope_workspace_size(int64_t M, int64_t Kdim, int32_t n_q, int32_t n_kv, int32_t head_dim);
int coda_linear_qknorm_rope(const coda_bf16* X, const float* rstd, const coda_bf16* W,
                            const float* gamma_q, const float* gamma_k, const int32_t* pos,
                            const float* cos_sin, int32_t max_pos, float eps,
                            int32_t n_q, int32_t n_kv, int32_t head_dim, int32_t rope_pairing,
                            coda_bf16* Q, coda_bf16* K, coda_bf16* V, coda_bf16* qk_save,
                            int64_t M, int64_t Kdim, void* ws, size_t ws_bytes, coda_stream stream);

/* Backward: given dQ, dK, dV (gradients of the attention inputs), the saved
 * pre-norm q|k (qk_save) and V:
 *   per head  dn = RoPE^-1(dQ_h),  dq = rho (dn⊙gamma - n mean(n ⊙ dn⊙gamma)),
 *   dgamma_q = sum dn ⊙ n;  dv = dV;  then the RMSNorm-reparameterised
 *   projection backward with G' = r ⊙ [dq | dk | dv] and D = G' W_qkv:
 *   dX = gamma_in ⊙ D - c ⊙ X + dX_resid with the dgamma_in_k =
 *   sum_i X_ik D_ik column partials in its epilogue,
 *   dW_qkv = (G'^T X) diag(gamma_in).  W_qkv is not folded.
 * rstd/gamma_in may be NULL (no input RMSNorm: dX = D + dX_resid).
 * Outputs: dX [M, Kdim], dW_qkv [(n_q+2n_kv)*128, Kdim] bf16; dgamma_in [Kdim],
 * dgamma_q, dgamma_k [128] fp32. */
size_t coda_linear_qknorm_rope_bwd_workspace_size(int64_t M, int64_t Kdim, int32_t n_q, int32_t n_kv,
                                                  int32_t head_dim);
int coda_linear_qknorm_rope_bwd(const coda_bf16* dQ, const coda_bf16* dK, const coda_bf16* dV,
                                const coda_bf16* qk_save, const coda_bf16* V,
                                const float* gamma_q, const float* gamma_k, const int32_t* pos,
                                const float* cos_sin, int32_t max_pos, float eps,
                                int32_t n_q, int32_t n_kv, int32_t head_dim, int32_t rope_pairing,
                                const coda_bf16* X, const float* rstd, const float* gamma_in,
                                const coda_bf16* W_qkv, const coda_bf16* dX_resid,
                                coda_bf16* dX, coda_bf16* dW_qkv, float* dgamma_in,
                                float* dgamma_q, float* dgamma_k,
                                int64_t M, int64_t Kdim, void* ws, size_t ws_bytes, coda_stream stream);

/* ------------------------------------------------------------------------
 * linear_cross_entropy (x-tip guide functional API; "CODA" §3.1 class 5:
 * running max / sum-exp state for online log-sum-exp and cross-entropy).
 * Logits z = X W^T are never written to memory.
 *
 *   lse_i = log sum_j exp(z_ij),  loss_i = lse_i - z_{i,y_i},
 *   loss_mean = sum over rows with y_i != ignore_index / n_valid
 *   (NaN when n_valid == 0).
 * X [M, K]; W [V, K]; labels [M] int32.  Outputs (device): loss_mean [1]
 * fp32, lse [M] fp32 (saved for the backward), n_valid [1] int32.  A label
 * outside [0, V) other than ignore_index sets CODA_ERR_LABEL_RANGE in the
 * status word; the row is then treated as ignored.
 * ---------------------------------------------------------------------- */
size_t coda_linear_cross_entropy_workspace_size(int64_t M, int64_t V, int64_t K);
int coda_linear_cross_entropy(const coda_bf16* X, const coda_bf16* W, const int32_t* labels,
                              int32_t ignore_index, float* loss_mean, float* lse, int32_t* n_valid,
                              int64_t M, int64_t V, int64_t K, void* ws, size_t ws_bytes, coda_stream stream);

/* ------------------------------------------------------------------------
 * linear_sigmoid (x-tip guide functional API; the pages give only the name).
 * Reading: a linear layer with an element-wise sigmoid ("CODA" §3.1 class 1),
 * optionally gating a second tensor:
 *   Y = sigmoid(X W^T)            (Z == NULL)
 *   Y = sigmoid(X W^T) ⊙ Z        (Z [M, N] bf16)
 * X [M, K], W [N, K], Y [M, N] bf16.
 * ---------------------------------------------------------------------- */
size_t coda_linear_sigmoid_workspace_size(int64_t M, int64_t N, int64_t K);
int coda_linear_sigmoid(const coda_bf16* X, const coda_bf16* W, const coda_bf16* Z, coda_bf16* Y, int64_t M,
                        int64_t N, int64_t K, void* ws, size_t ws_bytes, coda_stream stream);

/* Backward for upstream gradient dY [M, N]: the logits are recomputed by the
 * GEMM and the epilogue forms dz = dY (⊙ Z) ⊙ s (1 - s) (staged bf16 in the
 * workspace) and dZ = dY ⊙ s; then dX = dz W [M, K] and dW = dz^T X [N, K].
 * dZ is required when Z is given, ignored otherwise. */
size_t coda_linear_sigmoid_bwd_workspace_size(int64_t M, int64_t N, int64_t K);
int coda_linear_sigmoid_bwd(const coda_bf16* dY, const coda_bf16* X, const coda_bf16* W, const coda_bf16* Z,
                            coda_bf16* dX, coda_bf16* dW, coda_bf16* dZ, int64_t M, int64_t N, int64_t K, void* ws,
                            size_t ws_bytes, coda_stream stream);

/* ------------------------------------------------------------------------
 * FP8 (e4m3) operands: the same mainloop with tcgen05 kind::f8f6f4 and the
 * same epilogues.  The pages motivate fusion by low-precision GEMMs ("CODA"
 * §1: FP8 / FP4 make the materialised tensors' cost more important) but give
 * no quantisation recipe; this library uses per-row scales:
 *   scale_i = max_k |x_ik| / 448 (fp32; 1 for an all-zero row),
 *   q_ik = e4m3(x_ik / scale_i)  (fp32 division, round to nearest even,
 *   saturating), x ~= q * scale.
 * Activations are scaled per token, weights per output channel.  FP8
 * operands are K-major with K a multiple of 16 (16-byte rows).
 * ---------------------------------------------------------------------- */

/* X [M, K] bf16 (row stride ldx) -> Xq [M, K] e4m3 bytes (row stride K),
 * scale [M] fp32. */
int coda_quantize_fp8_rows(const coda_bf16* X, int64_t ldx, int64_t M, int64_t K, uint8_t* Xq, float* scale,
                           coda_stream stream);

/* Y = R + (sx ⊙ Xq)(sw ⊙ Wq)^T: Xq [M, K], sx [M], Wq [N, K], sw [N],
 * R [M, N] bf16 or NULL, Y [M, N] bf16. */
size_t coda_linear_fp8_workspace_size(int64_t M, int64_t N, int64_t K);
int coda_linear_fp8(const uint8_t* Xq, const float* sx, const uint8_t* Wq, const float* sw, const coda_bf16* R,
                    coda_bf16* Y, int64_t M, int64_t N, int64_t K, void* ws, size_t ws_bytes, coda_stream stream);

/* linear_swiglu on e4m3 operands: g = r ⊙ (sx ⊙ Xq)(sg ⊙ Wgq)^T,
 * u = r ⊙ (sx ⊙ Xq)(su ⊙ Wuq)^T, H = silu(g) ⊙ u.  rstd [M] or NULL (r = 1,
 * the RMSNorm-reparameterised input when given with gamma-folded weights);
 * Wgq, Wuq [I, K]; sg, su [I]; H, g_save, u_save [M, I] bf16. */
size_t coda_linear_swiglu_fp8_workspace_size(int64_t M, int64_t I, int64_t K);
int coda_linear_swiglu_fp8(const uint8_t* Xq, const float* sx, const float* rstd, const uint8_t* Wgq,
                           const float* sg, const uint8_t* Wuq, const float* su, coda_bf16* H, coda_bf16* g_save,
                           coda_bf16* u_save, int64_t M, int64_t I, int64_t K, void* ws, size_t ws_bytes,
                           coda_stream stream);

/* X [R, C] bf16 (row stride ldx), with X2 [R2, C] (row stride ldx2) stacked
 * below it when given -> XTq [C, R + R2] e4m3 (row stride ldo >= R + R2, a
 * multiple of 16), scale [C] fp32: scale_c = max over the column of |x| /
 * 448, codes of x / scale_c (the row rule along columns).  This is the
 * K-major operand of a GEMM that contracts over X's rows, e.g. the W^T of a
 * backward GEMM dX = G W: coda_quantize_fp8_cols(W) gives W^T quantised per
 * input feature.  C % 8 == 0 and (R + R2) % 16 == 0.  `scale` also serves as
 * scratch for the column maxima (no workspace). */
int coda_quantize_fp8_cols(const coda_bf16* X, int64_t ldx, int64_t R, const coda_bf16* X2, int64_t ldx2,
                           int64_t R2, int64_t C, uint8_t* XTq, int64_t ldo, float* scale, coda_stream stream);

/* linear_qknorm_rope on e4m3 operands: [q | k | v] = r ⊙ ((sx ⊙ Xq)(sw ⊙ Wq)^T),
 * then per head RMSNorm + RoPE as in coda_linear_qknorm_rope (same layouts,
 * gains, positions, table, pairing and outputs).  Xq [M, Kdim], sx [M],
 * Wq [(n_q+2n_kv)*128, Kdim], sw [(n_q+2n_kv)*128]; Kdim % 16 == 0. */
size_t coda_linear_qknorm_rope_fp8_workspace_size(int64_t M, int64_t Kdim, int32_t n_q, int32_t n_kv,
                                                  int32_t head_dim);
int coda_linear_qknorm_rope_fp8(const uint8_t* Xq, const float* sx, const float* rstd, const uint8_t* Wq,
                                const float* sw, const float* gamma_q, const float* gamma_k, const int32_t* pos,
                                const float* cos_sin, int32_t max_pos, float eps, int32_t n_q, int32_t n_kv,
                                int32_t head_dim, int32_t rope_pairing, coda_bf16* Q, coda_bf16* K, coda_bf16* V,
                                coda_bf16* qk_save, int64_t M, int64_t Kdim, void* ws, size_t ws_bytes,
                                coda_stream stream);

/* linear_cross_entropy on e4m3 operands: z = (sx ⊙ Xq)(sw ⊙ Wq)^T, then the
 * online log-sum-exp and loss of coda_linear_cross_entropy (same outputs and
 * label rules).  Xq [M, K], sx [M], Wq [V, K], sw [V]; K % 16 == 0. */
size_t coda_linear_cross_entropy_fp8_workspace_size(int64_t M, int64_t V, int64_t K);
int coda_linear_cross_entropy_fp8(const uint8_t* Xq, const float* sx, const uint8_t* Wq, const float* sw,
                                  const int32_t* labels, int32_t ignore_index, float* loss_mean, float* lse,
                                  int32_t* n_valid, int64_t M, int64_t V, int64_t K, void* ws, size_t ws_bytes,
                                  coda_stream stream);

/* Its backward: the softmax gradient dZ = (softmax(z) - onehot) * dloss /
 * n_valid at the logits z of the e4m3 operands (recomputed, by vocabulary
 * slices as in coda_linear_cross_entropy_bwd), then dX = dZ W and
 * dW = dZ^T X in bf16 GEMMs with the bf16 operands X [M, K], W [V, K]
 * (softmax probabilities of a 128k vocabulary lie far below e4m3's range,
 * so the gradient GEMMs keep dZ in bf16). */
size_t coda_linear_cross_entropy_bwd_fp8_workspace_size(int64_t M, int64_t V, int64_t K);
int coda_linear_cross_entropy_bwd_fp8(const uint8_t* Xq, const float* sx, const uint8_t* Wq, const float* sw,
                                      const coda_bf16* X, const coda_bf16* W, const int32_t* labels,
                                      int32_t ignore_index, const float* lse, const int32_t* n_valid, float dloss,
                                      coda_bf16* dX, coda_bf16* dW, int64_t M, int64_t V, int64_t K, void* ws,
                                      size_t ws_bytes, coda_stream stream);

/* The first GEMM of the SwiGLU MLP backward on e4m3 operands, with the
 * dSwiGLU pairwise map in its epilogue:
 *   dH = (sdy ⊙ dYq)(swd ⊙ WdTq)^T   (dY Wd; WdTq = coda_quantize_fp8_cols(Wd)),
 *   dG = dH ⊙ u ⊙ silu'(g),  dU = dH ⊙ silu(g),
 *   Gp [M, 2I] = r ⊙ [dG | dU] bf16 (r = rstd, or 1 when NULL),
 *   row_out [M] fp32 (or NULL): with rstd the RMSNorm-backward coefficient
 *   c_i = r_i^2 sum_j (dG g + dU u)_ij / K that the dX GEMM
 *   (coda_rmsnorm_linear_dx_fp8) takes as coef; without rstd the sum itself;
 *   H [M, I] = silu(g) ⊙ u (or NULL).
 * dYq [M, K], sdy [M], WdTq [I, K], swd [I]; g, u [M, I] the forward's saved
 * projections; K % 16 == 0. */
size_t coda_linear_dswiglu_fp8_workspace_size(int64_t M, int64_t I, int64_t K);
int coda_linear_dswiglu_fp8(const uint8_t* dYq, const float* sdy, const uint8_t* WdTq, const float* swd,
                            const coda_bf16* g, const coda_bf16* u, const float* rstd, coda_bf16* Gp, float* row_out,
                            coda_bf16* H, int64_t M, int64_t I, int64_t K, void* ws, size_t ws_bytes,
                            coda_stream stream);

/* The input gradient of an RMSNorm-reparameterised projection
 * y = r ⊙ ((X ⊙ gamma) W^T) on e4m3 operands, with the RMSNorm backward in
 * its epilogue:
 *   D = (sg ⊙ Gq)(sw ⊙ WTq)^T   (G' W; WTq = coda_quantize_fp8_cols(W)),
 *   dX = gamma ⊙ D - coef ⊙ X (+ dX_resid),  dgamma_k = sum_i X_ik D_ik.
 * Gq [M, N] (G' = r ⊙ G quantised per row), sg [M], WTq [K, N], sw [K],
 * X [M, K], gamma [K], coef [M] (c_i = r_i^2 sum_n G_in y_in / K),
 * dX_resid [M, K] or NULL; outputs dX [M, K] bf16, dgamma [K] fp32.
 * N % 16 == 0. */
size_t coda_rmsnorm_linear_dx_fp8_workspace_size(int64_t M, int64_t N, int64_t K);
int coda_rmsnorm_linear_dx_fp8(const uint8_t* Gq, const float* sg, const uint8_t* WTq, const float* sw,
                               const coda_bf16* X, const float* gamma, const float* coef, const coda_bf16* dX_resid,
                               coda_bf16* dX, float* dgamma, int64_t M, int64_t N, int64_t K, void* ws,
                               size_t ws_bytes, coda_stream stream);

/* The backward of linear_qknorm_rope with both of its GEMMs on e4m3
 * operands.  The per-head map (RoPE^-1, QK-RMSNorm backward, dgamma_q,
 * dgamma_k) and the RMSNorm coefficient c are those of
 * coda_linear_qknorm_rope_bwd and write G' = r ⊙ [dq | dk | dv] in bf16
 * into the workspace; G' is then quantised per row (Gq, sg) and per column
 * (GTq, sgT) into the workspace, and
 *   D  = (sg ⊙ Gq)(sw ⊙ WTq)^T          (G' W_qkv; WTq = coda_quantize_fp8_cols(W_qkv)),
 *   dX = gamma_in ⊙ D - c ⊙ X + dX_resid,  dgamma_in_k = sum_i X_ik D_ik
 *        (without rstd: dX = D + dX_resid),
 *   dW_qkv = (sgT ⊙ GTq)(su ⊙ UTq)^T     (G'^T U; UTq = coda_quantize_fp8_cols(U)),
 * where U is the forward GEMM's input: U = X ⊙ gamma_in (the U of
 * coda_rmsnorm_scale) with the input RMSNorm, X without it, so that
 * G'^T U = (G'^T X) diag(gamma_in).  Arguments as in
 * coda_linear_qknorm_rope_bwd, with W_qkv replaced by WTq [Kdim, N] uint8
 * (row stride N = (n_q+2n_kv)*128), sw [Kdim], and the codes of U by
 * UTq [Kdim, M] uint8 (row stride M), su [Kdim].  M % 16 == 0 (the dW GEMM
 * contracts over the tokens); CODA_ERR_UNSUPPORTED otherwise. */
size_t coda_linear_qknorm_rope_bwd_fp8_workspace_size(int64_t M, int64_t Kdim, int32_t n_q, int32_t n_kv,
                                                      int32_t head_dim);
int coda_linear_qknorm_rope_bwd_fp8(const coda_bf16* dQ, const coda_bf16* dK, const coda_bf16* dV,
                                    const coda_bf16* qk_save, const coda_bf16* V, const float* gamma_q,
                                    const float* gamma_k, const int32_t* pos, const float* cos_sin, int32_t max_pos,
                                    float eps, int32_t n_q, int32_t n_kv, int32_t head_dim, int32_t rope_pairing,
                                    const coda_bf16* X, const float* rstd, const float* gamma_in,
                                    const uint8_t* WTq, const float* sw, const uint8_t* UTq, const float* su,
                                    const coda_bf16* dX_resid, coda_bf16* dX, coda_bf16* dW_qkv, float* dgamma_in,
                                    float* dgamma_q, float* dgamma_k, int64_t M, int64_t Kdim, void* ws,
                                    size_t ws_bytes, coda_stream stream);

/* ------------------------------------------------------------------------
 * NVFP4 operands: 4-bit e2m1 elements, one e4m3 scale per 16 consecutive
 * elements along K, an fp32 scale per row; the GEMM runs on tcgen05.mma
 * kind::mxf4nvf4 (block-scaled) with the same epilogues.  The pages name
 * FP4 beside FP8 as the formats that make the GEMMs fast and the data
 * movement around them dominant ("CODA: Rewriting Transformer Blocks as
 * GEMM-Epilogue Programs", §1; the news flash on it) and give no recipe:
 * this is NVIDIA's NVFP4 block format with the second-level scale per row.
 *
 * Quantisation of row x (each step one fp32 operation):
 *   s = amax(x) / 2688 (= 6 * 448; 1 for a zero row);
 *   per block of 16: sf = e4m3(bmax / (6 s)), nearest even, <= 448;
 *   inv = min(1 / (sf s), FLT_MAX), one per block;
 *   code = e2m1(x inv), nearest even, saturating at +-6; 0 when sf s = 0;
 *   x ~= e2m1(code) * sf * s.
 * Layouts:
 *   Xq     [rows, K/2] bytes, contiguous: element 2j in the low nibble of byte
 *          j, 2j+1 in the high nibble; e2m1 = bit 3 sign, bits 0-2 index of
 *          the magnitude in {0, 0.5, 1, 1.5, 2, 3, 4, 6}; no negative zero.
 *   scale  [rows] fp32.
 *   sf     coda_nvfp4_scale_bytes(rows, K) bytes, the order the tensor core
 *          reads: the scale of row r, 16-element block j sits at byte
 *            ((r/128) * KT + j/16) * 2048 + ((j/4) % 4) * 512
 *            + (r % 32) * 16 + ((r % 128) / 32) * 4 + j % 4
 *          with KT = ceil(K / 256); rows are padded to a multiple of 512 and
 *          blocks to KT * 16, the padding holding zero scales.
 * Requirements: K % 32 == 0; Xq, sf 16-byte aligned; N (I) % 8 == 0.  */
size_t coda_nvfp4_scale_bytes(int64_t rows, int64_t K);
int coda_quantize_nvfp4_rows(const coda_bf16* X, int64_t ldx, int64_t M, int64_t K, uint8_t* Xq, uint8_t* sf,
                             float* scale, coda_stream stream);

/* The RMSNorm input stage of an NVFP4 projection in one pass over X: the
 * codes, block scales and row scales of u = x ⊙ gamma (fp32 products, not
 * rounded to bf16) as coda_quantize_nvfp4_rows writes them, and, when rstd
 * is not NULL, rstd = 1 / sqrt(mean(x^2) + eps) per row — the row factor r
 * of the RMSNorm reparameterisation ("CODA: Rewriting Transformer Blocks as
 * GEMM-Epilogue Programs", §3.2.1), applied by the next GEMM's epilogue
 * (coda_linear_swiglu_nvfp4's rstd).  gamma [K] fp32, 16-byte aligned. */
int coda_rmsnorm_scale_nvfp4(const coda_bf16* X, int64_t ldx, int64_t M, int64_t K, float eps, const float* gamma,
                             float* rstd, uint8_t* Xq, uint8_t* sf, float* scale, coda_stream stream);

/* Y = R + (sx ⊙ deq(Xq, sfx))(sw ⊙ deq(Wq, sfw))^T: X side [M, K], W side
 * [N, K] (as quantised by coda_quantize_nvfp4_rows), R [M, N] bf16 or NULL,
 * Y [M, N] bf16. */
size_t coda_linear_nvfp4_workspace_size(int64_t M, int64_t N, int64_t K);
int coda_linear_nvfp4(const uint8_t* Xq, const uint8_t* sfx, const float* sx, const uint8_t* Wq, const uint8_t* sfw,
                      const float* sw, const coda_bf16* R, coda_bf16* Y, int64_t M, int64_t N, int64_t K, void* ws,
                      size_t ws_bytes, coda_stream stream);

/* linear_swiglu on NVFP4 operands: g = r ⊙ X̂ Ŵgᵀ, u = r ⊙ X̂ Ŵuᵀ,
 * H = silu(g) ⊙ u with X̂ = sx ⊙ deq(Xq, sfx) and likewise for the weights
 * ([I, K] each); rstd [M] or NULL (r = 1); H, g_save, u_save [M, I] bf16
 * (g_save, u_save may be NULL). */
size_t coda_linear_swiglu_nvfp4_workspace_size(int64_t M, int64_t I, int64_t K);
int coda_linear_swiglu_nvfp4(const uint8_t* Xq, const uint8_t* sfx, const float* sx, const float* rstd,
                             const uint8_t* Wgq, const uint8_t* sfg, const float* sg, const uint8_t* Wuq,
                             const uint8_t* sfu, const float* su, coda_bf16* H, coda_bf16* g_save,
                             coda_bf16* u_save, int64_t M, int64_t I, int64_t K, void* ws, size_t ws_bytes,
                             coda_stream stream);

/* ------------------------------------------------------------------------
 * Final RMSNorm -> LM head -> cross-entropy ("CODA" §3.2.1, third site of
 * the GEMM-residual-RMSNorm-GEMM pattern: final down-projection -> residual
 * -> final RMSNorm -> language-model head)
 *
 *   z = r ⊙ (X Wf^T),  Wf = W diag(gamma) (coda_fold_gamma),
 *   which equals RMSNorm(X, gamma) W^T; then the cross-entropy of
 *   coda_linear_cross_entropy.  rstd [M] comes from the producing epilogue
 *   (coda_linear_residual's rstd_out) or coda_rms_rstd.  The workspace and the
 *   outputs are those of coda_linear_cross_entropy (lse is that of z).
 * ---------------------------------------------------------------------- */
size_t coda_rmsnorm_linear_cross_entropy_workspace_size(int64_t M, int64_t V, int64_t K);
int coda_rmsnorm_linear_cross_entropy(const coda_bf16* X, const float* rstd, const coda_bf16* Wf,
                                      const int32_t* labels, int32_t ignore_index, float* loss_mean, float* lse,
                                      int32_t* n_valid, int64_t M, int64_t V, int64_t K, void* ws, size_t ws_bytes,
                                      coda_stream stream);

/* Backward for upstream gradient dloss of the mean loss.  With
 * G = dZ = (softmax(z) - onehot) * dloss / n_valid and G' = r ⊙ G:
 *   dX = G' Wf - c ⊙ X (+ dX_resid),  c_i = r_i^2 sum_v G_iv z_iv / K,
 *   dW = (G'^T X) diag(gamma),  dgamma_k = sum_v W_vk (G'^T X)_vk.
 * The one-hot part of G' is applied exactly in fp32 (row gather of Wf for dX,
 * a label -> token list for dW); only r * softmax * w is staged in bf16, one
 * vocabulary slice of 16384 columns at a time, as in
 * coda_linear_cross_entropy_bwd (workspace of order M x min(V, 16384)).
 * Inputs: X [M,K] (the un-normalised residual stream), rstd [M], gamma [K],
 * W and Wf [V,K], labels [M], lse [M] and n_valid from the forward,
 * dX_resid [M,K] or NULL.  Outputs: dX [M,K], dW [V,K] bf16, dgamma [K] fp32. */
size_t coda_rmsnorm_linear_cross_entropy_bwd_workspace_size(int64_t M, int64_t V, int64_t K);
int coda_rmsnorm_linear_cross_entropy_bwd(const coda_bf16* X, const float* rstd, const float* gamma,
                                          const coda_bf16* W, const coda_bf16* Wf, const int32_t* labels,
                                          int32_t ignore_index, const float* lse, const int32_t* n_valid, float dloss,
                                          const coda_bf16* dX_resid, coda_bf16* dX, coda_bf16* dW, float* dgamma,
                                          int64_t M, int64_t V, int64_t K, void* ws, size_t ws_bytes,
                                          coda_stream stream);

/* Variant of coda_linear_cross_entropy that allocates nothing and takes no
 * workspace, for callers that cannot obtain device memory: a plugin or
 * callback inside a host application that owns all device memory and passes
 * it only input and output buffers, or a latency-critical loop that must not
 * call cudaMalloc because it may synchronise the device.  The paper has no
 * counterpart; this is an interface convenience of this library.
 *
 * Same arguments and results as coda_linear_cross_entropy, minus ws.  Its
 * scratch is a fixed device array inside libcoda.so of
 * coda_noalloc_scratch_bytes() bytes (8 MiB), held by every GPU that loads the
 * library until the process exits; a problem whose
 * coda_linear_cross_entropy_workspace_size(M, V, K) exceeds it is rejected
 * with CODA_ERR_WORKSPACE before anything is enqueued (at V = 128256 that is
 * M above about 32,000 tokens).  The first call on a device looks up the
 * array's device address (set-up, once per device, with that device
 * current); make that first call before any stream capture.  The address
 * is kept until the process exits: after cudaDeviceReset on a device the
 * library's device image is loaded again elsewhere, so do not call this
 * entry point on that device after a reset (the regular
 * coda_linear_cross_entropy with a workspace has no such limit).  Every call
 * shares the array, so calls that overlap on the GPU (different streams or
 * threads) race and must be serialised by the caller.
 * status_out (optional device int32) receives this call's device status word:
 * 0 if no device error, otherwise the bits that coda_get_status maps (2 = a
 * label out of range, 1 = a pipeline wait timed out). */
size_t coda_noalloc_scratch_bytes(void);
int coda_linear_cross_entropy_noalloc(const coda_bf16* X, const coda_bf16* W, const int32_t* labels,
                                      int32_t ignore_index, float* loss_mean, float* lse, int32_t* n_valid,
                                      int32_t* status_out, int64_t M, int64_t V, int64_t K, coda_stream stream);

/* Backward for upstream gradient dloss of the mean loss:
 *   dZ = (softmax(z) - onehot(y)) * dloss / n_valid (0 on ignored rows),
 *   dX = dZ W [M, K], dW = dZ^T X [V, K] (bf16).
 * lse and n_valid are the forward's outputs (device pointers).  The
 * gradient of the whole logit matrix is never held: the vocabulary is taken
 * in slices of 16384 columns, and for each slice dZ_s is recomputed from
 * X W_s^T into the workspace (bf16, two buffers of M x 16384), dX += dZ_s W_s
 * is summed in fp32 (an M x K buffer) and dW_s = dZ_s^T X written; the
 * one-hot part is applied exactly in fp32 by the dX and dW epilogues.  The
 * workspace therefore grows as M x min(V, 16384) (about 0.6 GB at
 * M = 8192, K = 2048), not as M x V.  The dX and dW GEMMs of each slice run
 * on two helper streams forked from and joined back to `stream` (created on
 * the first call; the call is CUDA-graph capturable once that first call
 * has run outside the capture). */
size_t coda_linear_cross_entropy_bwd_workspace_size(int64_t M, int64_t V, int64_t K);
int coda_linear_cross_entropy_bwd(const coda_bf16* X, const coda_bf16* W, const int32_t* labels,
                                  int32_t ignore_index, const float* lse, const int32_t* n_valid,
                                  float dloss, coda_bf16* dX, coda_bf16* dW,
                                  int64_t M, int64_t V, int64_t K, void* ws, size_t ws_bytes,
                                  coda_stream stream);

#ifdef __cplusplus
}
#endif

#endif /* CODA_H */
