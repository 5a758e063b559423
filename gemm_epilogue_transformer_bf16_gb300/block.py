"""The non-attention transformer block as a sequence of GEMM-epilogue calls.

Forward ("CODA: Rewriting Transformer Blocks as GEMM-Epilogue Programs"
§3.2.1, sites 1 and 2 of the GEMM-residual-RMSNorm-GEMM pattern).  The
residual add and the "⊙ gamma" of RMSNorm(y, gamma) are block-local, so the
epilogue that produces y applies them; the row factor r = 1/rms(y) needs a
whole row and moves to the epilogue of the next GEMM:

  rms0   r0 = 1/rms(x0), u0 = x0 ⊙ gamma_attn  (x0 has no producing GEMM here)
  qkv    Q, K, V = QKnorm+RoPE epilogue of r0 ⊙ (u0 Wqkv^T)
         [attention itself is out of scope: its output A is an input]
  oproj  x1 = x0 + A Wo^T; the epilogue also writes u1 = x1 ⊙ gamma_mlp and
         partial sums of squares -> r1
  gateup H = silu(r1 ⊙ u1 Wg^T) ⊙ (r1 ⊙ u1 Wu^T)         (SwiGLU epilogue)
  down   x2 = x1 + H Wd^T                                  (residual epilogue)

Backward (given dx2 and the attention-input gradients dQ, dK, dV):

  mlp    dSwiGLU epilogue on dH = dx2 Wd -> G'; dx1 = gamma ⊙ (G' [Wg; Wu])
         - c ⊙ x1 + dx2 with the dgamma_mlp column partials in its epilogue;
         dWg, dWu = (G'^T x1) diag(gamma) (column-scale epilogue); dWd = dx2^T H
  oproj  dA = dx1 Wo, dWo = dx1^T A
  qkv    QK-norm+RoPE backward map, then the same RMSNorm-reparameterised
         backward for dx0 = dx1 + qkv branch, dWqkv, dgamma_attn;
         dgamma_q, dgamma_k

With ``fold_weights=True`` the forward instead folds gamma into the weights
(W' = W diag(gamma), once per step since the weights change every step) and
its GEMMs read x; the backward is the same either way.

Every step is a libcoda.so call; buffers and workspaces are allocated once,
so a step launches only the library's kernels.  With ``concurrent`` (the
default) the forward's QKV branch (row RMS of x0, QKV projection; with
folded weights also the Wqkv fold) runs on a second stream beside the
O-projection (and the MLP weights' folds that follow it, which share SMs
with the tensor-bound GEMM).  With ``concurrent_bwd`` the backward does the
same (the O-projection backward beside the QKV backward, the MLP's
weight-gradient GEMMs beside its dH -> dX chain); it is off by default:
two persistent GEMMs started together split the SMs by whichever places its
CTAs first, and in a loop of steps the backward ran 1 % slower that way than
on one stream.  The gate/up and down GEMMs run alone.
"""
from __future__ import annotations

import torch

from . import (K_MAJOR, MN_MAJOR, EpilogueDesc, fold_gamma, gemm_epilogue, linear_cross_entropy,
               linear_cross_entropy_bwd, linear_dswiglu_fp8, linear_fp8, linear_qknorm_rope, linear_qknorm_rope_bwd,
               linear_qknorm_rope_bwd_fp8, linear_qknorm_rope_fp8, linear_residual, linear_residual_bwd, linear_swiglu, linear_swiglu_bwd,
               linear_swiglu_fp8, load, quantize_fp8_cols, quantize_fp8_rows, rms_rstd, rmsnorm_linear_dx_fp8,
               rmsnorm_scale, rope_table, workspace)


class Block:
    def __init__(self, shape, weights, device="cuda", concurrent=True, fold_weights=False, concurrent_bwd=False):
        self.s = s = shape
        self.w = weights
        self.concurrent = concurrent
        self.concurrent_bwd = concurrent and concurrent_bwd
        self.fold_weights = fold_weights
        lib = load()
        T, Hd, I, d = s.tokens, s.hidden, s.inter, s.head_dim
        nqkv = s.qkv_out
        bf = dict(dtype=torch.bfloat16, device=device)
        f32 = dict(dtype=torch.float32, device=device)
        e = torch.empty
        if fold_weights:
            self.Wqkv_f = e(nqkv, Hd, **bf)
            self.Wg_f = e(I, Hd, **bf)
            self.Wu_f = e(I, Hd, **bf)
        else:
            self.U0 = e(T, Hd, **bf)
            self.U1 = e(T, Hd, **bf)
        self.cos_sin = rope_table(s.theta, d, s.seq_len, device=device)
        self.rstd0 = e(T, **f32)
        self.rstd1 = e(T, **f32)
        self.fwd = {"Q": e(T, s.n_q * d, **bf), "K": e(T, s.n_kv * d, **bf), "V": e(T, s.n_kv * d, **bf),
                    "qk_save": e(T, (s.n_q + s.n_kv) * d, **bf)}
        self.x1 = e(T, Hd, **bf)
        self.x2 = e(T, Hd, **bf)
        self.H = e(T, I, **bf)
        self.g = e(T, I, **bf)
        self.u = e(T, I, **bf)
        self.dx1 = e(T, Hd, **bf)
        self.grads_mlp = {"dX": self.dx1, "dWg": e(I, Hd, **bf), "dWu": e(I, Hd, **bf), "dWd": e(Hd, I, **bf),
                          "dgamma": e(Hd, **f32)}
        self.grads_o = {"dX": e(T, s.n_q * d, **bf), "dW": e(Hd, s.n_q * d, **bf)}
        self.grads_qkv = {"dX": e(T, Hd, **bf), "dW": e(nqkv, Hd, **bf), "dgamma_in": e(Hd, **f32),
                          "dgamma_q": e(d, **f32), "dgamma_k": e(d, **f32)}
        need = max(
            lib.coda_linear_qknorm_rope_workspace_size(T, Hd, s.n_q, s.n_kv, d),
            lib.coda_linear_residual_workspace_size(T, Hd, s.n_q * d),
            lib.coda_linear_swiglu_workspace_size(T, I, Hd),
            lib.coda_linear_residual_workspace_size(T, Hd, I),
            lib.coda_linear_swiglu_bwd_workspace_size(T, I, Hd),
            lib.coda_linear_residual_bwd_workspace_size(T, Hd, s.n_q * d),
            lib.coda_linear_qknorm_rope_bwd_workspace_size(T, Hd, s.n_q, s.n_kv, d),
        )
        self.ws = workspace(need, device)
        # second stream and its own workspace (calls on different streams must
        # not share scratch)
        self.s2 = torch.cuda.Stream(device=device) if concurrent else None
        self.ws2 = workspace(need, device) if concurrent else self.ws

    # Stages as the step's CUDA events delimit them on the main stream, and the
    # kernels each launches (library calls are fixed sequences).  "pre" is the
    # row RMS + QKV branch beside the O-projection (with the folds when the
    # weights are folded); "attn_bwd" the O-projection backward beside the
    # QKV backward.
    # kernels per stage without the second slices of split GEMM launches
    # (bench.py counts the launches themselves with coda_launch_count)
    LAUNCHES = {"pre": 4, "gateup": 1, "down": 1, "mlp_bwd": 7, "attn_bwd": 7}
    LAUNCHES_FOLDED = {"pre": 7, "gateup": 1, "down": 1, "mlp_bwd": 7, "attn_bwd": 7}

    def launches(self):
        return self.LAUNCHES_FOLDED if self.fold_weights else self.LAUNCHES

    def gemm_flops(self):
        """Algorithmic GEMM FLOPs (2*M*N*K) of each stage of one step."""
        s = self.s
        T, Hd, I, a = s.tokens, s.hidden, s.inter, s.n_q * s.head_dim
        q = s.qkv_out
        return {"pre": 2 * T * Hd * q + 2 * T * a * Hd, "gateup": 4 * T * Hd * I, "down": 2 * T * I * Hd,
                "mlp_bwd": 2 * (2 * T * Hd * I) + 2 * (4 * T * Hd * I), "attn_bwd": 4 * T * a * Hd + 4 * T * Hd * q}

    def _side(self):
        """Context running calls on the second stream (or the main one)."""
        if self.s2 is None:
            return _NullCtx(), self.ws
        self.s2.wait_stream(torch.cuda.current_stream(self.s2.device))
        return torch.cuda.stream(self.s2), self.ws2

    def _join(self):
        if self.s2 is not None:
            torch.cuda.current_stream(self.s2.device).wait_stream(self.s2)

    # ------------------------------------------------------------------ forward
    def forward(self, x0, A, pos, mark=None):
        s, w = self.s, self.w
        mark = mark or (lambda name: None)
        ctx, ws2 = self._side()
        if self.fold_weights:
            with ctx:   # QKV branch: independent of the O-projection
                fold_gamma(w["Wqkv"], w["gamma_attn"], out=self.Wqkv_f)
                rms_rstd(x0, s.eps, out=self.rstd0)
                linear_qknorm_rope(x0, self.Wqkv_f, w["gamma_q"], w["gamma_k"], pos, self.cos_sin, s.n_q, s.n_kv,
                                   rstd=self.rstd0, eps=s.eps, head_dim=s.head_dim, out=self.fwd, ws=ws2)
            linear_residual(A, w["Wo"], x0, eps=s.eps, Y=self.x1, rstd_out=self.rstd1, ws=self.ws)
            # HBM-bound folds after the O-projection: they run beside the QKV
            # GEMM (their blocks use no shared memory and fit next to its CTAs)
            fold_gamma(w["Wg"], w["gamma_mlp"], out=self.Wg_f)
            fold_gamma(w["Wu"], w["gamma_mlp"], out=self.Wu_f)
            xin, Wg, Wu = self.x1, self.Wg_f, self.Wu_f
        else:
            with ctx:   # QKV branch: independent of the O-projection
                rmsnorm_scale(x0, w["gamma_attn"], s.eps, rstd=self.rstd0, U=self.U0)
                linear_qknorm_rope(self.U0, w["Wqkv"], w["gamma_q"], w["gamma_k"], pos, self.cos_sin, s.n_q,
                                   s.n_kv, rstd=self.rstd0, eps=s.eps, head_dim=s.head_dim, out=self.fwd, ws=ws2)
            linear_residual(A, w["Wo"], x0, eps=s.eps, Y=self.x1, rstd_out=self.rstd1, gamma_next=w["gamma_mlp"],
                            U_out=self.U1, ws=self.ws)
            xin, Wg, Wu = self.U1, w["Wg"], w["Wu"]
        self._join()
        mark("pre")
        linear_swiglu(xin, Wg, Wu, rstd=self.rstd1, H=self.H, g=self.g, u=self.u, ws=self.ws)
        mark("gateup")
        linear_residual(self.H, w["Wd"], self.x1, Y=self.x2, ws=self.ws)
        mark("down")
        return {"Q": self.fwd["Q"], "K": self.fwd["K"], "V": self.fwd["V"], "x1": self.x1, "x2": self.x2}

    # ------------------------------------------------------------------ backward
    def backward(self, x0, A, pos, dx2, dQ, dK, dV, mark=None):
        s, w = self.s, self.w
        mark = mark or (lambda name: None)
        side = self.s2 if self.concurrent_bwd else None
        linear_swiglu_bwd(dx2, self.x1, w["Wg"], w["Wu"], w["Wd"], self.g, self.u, self.H, rstd=self.rstd1,
                          gamma=w["gamma_mlp"], dX_resid=dx2, ws=self.ws, out=self.grads_mlp, side_stream=side)
        mark("mlp_bwd")
        ctx, ws2 = self._side() if self.concurrent_bwd else (_NullCtx(), self.ws)
        with ctx:   # both need only dx1
            linear_residual_bwd(self.dx1, A, w["Wo"], ws=ws2, out=self.grads_o)
        linear_qknorm_rope_bwd(dQ, dK, dV, self.fwd["qk_save"], self.fwd["V"], w["gamma_q"], w["gamma_k"], pos,
                               self.cos_sin, s.n_q, s.n_kv, x0, w["Wqkv"], rstd=self.rstd0,
                               gamma_in=w["gamma_attn"], dX_resid=self.dx1, eps=s.eps, head_dim=s.head_dim,
                               ws=self.ws, out=self.grads_qkv)
        self._join()
        mark("attn_bwd")
        return {"dx0": self.grads_qkv["dX"], "dA": self.grads_o["dX"], "dx1": self.dx1,
                "dWqkv": self.grads_qkv["dW"], "dWo": self.grads_o["dW"], "dWg": self.grads_mlp["dWg"],
                "dWu": self.grads_mlp["dWu"], "dWd": self.grads_mlp["dWd"],
                "dgamma_attn": self.grads_qkv["dgamma_in"], "dgamma_mlp": self.grads_mlp["dgamma"],
                "dgamma_q": self.grads_qkv["dgamma_q"], "dgamma_k": self.grads_qkv["dgamma_k"]}

    def step(self, x0, A, pos, dx2, dQ, dK, dV, mark=None):
        self.forward(x0, A, pos, mark)
        return self.backward(x0, A, pos, dx2, dQ, dK, dV, mark)


class BlockFP8:
    """The same block step with the GEMMs that have e4m3 instances on e4m3
    operands: the forward projections (QKV + QK-norm + RoPE, O-projection +
    residual, gate/up + SwiGLU, down + residual) and the input-gradient
    GEMMs of the MLP (dH with the dSwiGLU epilogue, dX with the
    RMSNorm-backward epilogue) and of the O-projection (dA).  Activations are
    quantised per token and weights per output row (forward) or per input
    column (backward, transposed by the column quantiser) every step, since
    the weights change every step.  With fp8_wgrad (the default) the weight
    gradients are e4m3 GEMMs as well: both operands quantised per column
    over the tokens by the transposing quantiser, dW = (G^T)_q (X^T)_q^T
    with the two column scales; and the QKV backward takes both of its GEMMs
    on e4m3 operands (linear_qknorm_rope_bwd_fp8: G' quantised per row for
    dx0 and per column for dWqkv, against W_qkv^T and the column codes of
    the forward's u0 = x0 ⊙ gamma_attn).  Without it the weight gradients
    and the whole QKV backward are bf16.  The O-projection's output x1 goes
    through the RMSNorm scale pass for r1 and u1 (the bf16 block gets them
    from its epilogue)."""

    def __init__(self, shape, weights, device="cuda", concurrent=True, fp8_wgrad=True):
        self.s = s = shape
        self.w = w = weights
        lib = load()
        T, Hd, I, d = s.tokens, s.hidden, s.inter, s.head_dim
        nqkv, a_in = s.qkv_out, s.n_q * s.head_dim
        bf = dict(dtype=torch.bfloat16, device=device)
        f32 = dict(dtype=torch.float32, device=device)
        u8 = dict(dtype=torch.uint8, device=device)
        e = torch.empty
        self.device = device

        def q(rows, cols):
            return (e(rows, cols, **u8), e(rows, **f32))
        # weights: forward (per output row) and backward (per input column, transposed)
        self.Wqkv_q, self.Wo_q, self.Wg_q, self.Wu_q, self.Wd_q = (q(nqkv, Hd), q(Hd, a_in), q(I, Hd), q(I, Hd),
                                                                   q(Hd, I))
        self.WdT_q, self.WguT_q, self.WoT_q = q(I, Hd), q(Hd, 2 * I), q(a_in, Hd)
        self.WqkvT_q = q(Hd, nqkv) if fp8_wgrad else None
        # activations
        self.U0, self.U1 = e(T, Hd, **bf), e(T, Hd, **bf)
        self.U0_q, self.A_q, self.U1_q, self.H_q = q(T, Hd), q(T, a_in), q(T, Hd), q(T, I)
        self.dx2_q, self.G_q, self.dx1_q = q(T, Hd), q(T, 2 * I), q(T, Hd)
        self.fp8_wgrad = fp8_wgrad
        if fp8_wgrad:  # transposed, per-column codes of the weight gradients' operands
            self.dx2T_q, self.HT_q, self.GT_q = q(Hd, T), q(I, T), q(2 * I, T)
            self.U1T_q, self.dx1T_q, self.AT_q = q(Hd, T), q(Hd, T), q(a_in, T)
            self.U0T_q = q(Hd, T)
        self.cos_sin = rope_table(s.theta, d, s.seq_len, device=device)
        self.rstd0, self.rstd1, self.coef1 = e(T, **f32), e(T, **f32), e(T, **f32)
        self.fwd = {"Q": e(T, s.n_q * d, **bf), "K": e(T, s.n_kv * d, **bf), "V": e(T, s.n_kv * d, **bf),
                    "qk_save": e(T, (s.n_q + s.n_kv) * d, **bf)}
        self.x1, self.x2 = e(T, Hd, **bf), e(T, Hd, **bf)
        self.H, self.g, self.u = e(T, I, **bf), e(T, I, **bf), e(T, I, **bf)
        self.Gp = e(T, 2 * I, **bf)
        self.dx1 = {"dX": e(T, Hd, **bf), "dgamma": e(Hd, **f32)}
        self.dA = e(T, a_in, **bf)
        self.dWgu = e(2 * I, Hd, **bf)   # dWg above dWu: one GEMM over G' = [G'_g | G'_u]
        self.dW = {"dWg": self.dWgu[:I], "dWu": self.dWgu[I:], "dWd": e(Hd, I, **bf), "dWo": e(Hd, a_in, **bf)}
        self.grads_qkv = {"dX": e(T, Hd, **bf), "dW": e(nqkv, Hd, **bf), "dgamma_in": e(Hd, **f32),
                          "dgamma_q": e(d, **f32), "dgamma_k": e(d, **f32)}
        need = max(lib.coda_linear_qknorm_rope_fp8_workspace_size(T, Hd, s.n_q, s.n_kv, d),
                   lib.coda_linear_fp8_workspace_size(T, Hd, a_in), lib.coda_linear_swiglu_fp8_workspace_size(T, I, Hd),
                   lib.coda_linear_dswiglu_fp8_workspace_size(T, I, Hd),
                   lib.coda_rmsnorm_linear_dx_fp8_workspace_size(T, 2 * I, Hd),
                   lib.coda_linear_qknorm_rope_bwd_workspace_size(T, Hd, s.n_q, s.n_kv, d),
                   lib.coda_linear_qknorm_rope_bwd_fp8_workspace_size(T, Hd, s.n_q, s.n_kv, d),
                   lib.coda_gemm_epilogue_workspace_size(), lib.coda_linear_fp8_workspace_size(Hd, I, T),
                   lib.coda_linear_fp8_workspace_size(2 * I, Hd, T), lib.coda_linear_fp8_workspace_size(Hd, a_in, T))
        self.ws = workspace(need, device)
        self.s2 = torch.cuda.Stream(device=device) if concurrent else None
        self.ws2 = workspace(need, device) if concurrent else self.ws

    # kernels per stage (coda_launch_count at 8192 tokens, hidden 8192, the
    # default launch switches)
    LAUNCHES = {"quant_w": 17, "fwd": 10, "bwd": 41}
    LAUNCHES_BF16_WGRAD = {"quant_w": 14, "fwd": 10, "bwd": 17}

    def launches(self):
        return self.LAUNCHES if self.fp8_wgrad else self.LAUNCHES_BF16_WGRAD

    def gemm_flops(self):
        return Block.gemm_flops(self)

    def _side(self):
        return Block._side(self)

    def _join(self):
        Block._join(self)

    def quantize_weights(self):
        """The step's e4m3 copies of the weights (they change every step)."""
        w = self.w
        for src, dst in ((w["Wqkv"], self.Wqkv_q), (w["Wo"], self.Wo_q), (w["Wg"], self.Wg_q), (w["Wu"], self.Wu_q),
                         (w["Wd"], self.Wd_q)):
            quantize_fp8_rows(src, Xq=dst[0], scale=dst[1])
        quantize_fp8_cols(w["Wd"], XTq=self.WdT_q[0], scale=self.WdT_q[1])
        quantize_fp8_cols(w["Wg"], w["Wu"], XTq=self.WguT_q[0], scale=self.WguT_q[1])
        quantize_fp8_cols(w["Wo"], XTq=self.WoT_q[0], scale=self.WoT_q[1])
        if self.fp8_wgrad:
            quantize_fp8_cols(w["Wqkv"], XTq=self.WqkvT_q[0], scale=self.WqkvT_q[1])

    def _wgrad(self, A, lda, B, ldb, D, M, N, K, col_scale=None, ws=None):
        """D [M, N] = A^T B (A stored [K, M], B stored [K, N]) in bf16, with an
        optional column scale: the weight-gradient GEMMs."""
        d = EpilogueDesc()
        if col_scale is not None:
            d.col_scale = col_scale.data_ptr()
        gemm_epilogue(d, A, B, D, M, N, K, a_major=MN_MAJOR, b_major=MN_MAJOR, lda=lda, ldb=ldb, ws=ws)

    def _wgrad_fp8(self, G, GT_q, X, XT_q, D, ws):
        """D [m, n] = G^T X over the tokens (G [T, m], X [T, n]) as an e4m3 GEMM
        on the column-quantised transposes."""
        quantize_fp8_cols(G, XTq=GT_q[0], scale=GT_q[1])
        quantize_fp8_cols(X, XTq=XT_q[0], scale=XT_q[1])
        linear_fp8(GT_q[0], GT_q[1], XT_q[0], XT_q[1], Y=D, ws=ws)

    def forward(self, x0, A, pos, mark=None):
        s, w = self.s, self.w
        mark = mark or (lambda name: None)
        self.quantize_weights()
        mark("quant_w")
        rmsnorm_scale(x0, w["gamma_attn"], s.eps, rstd=self.rstd0, U=self.U0)
        quantize_fp8_rows(self.U0, Xq=self.U0_q[0], scale=self.U0_q[1])
        linear_qknorm_rope_fp8(self.U0_q[0], self.U0_q[1], self.Wqkv_q[0], self.Wqkv_q[1], w["gamma_q"],
                               w["gamma_k"], pos, self.cos_sin, s.n_q, s.n_kv, rstd=self.rstd0, eps=s.eps,
                               head_dim=s.head_dim, out=self.fwd, ws=self.ws)
        quantize_fp8_rows(A, Xq=self.A_q[0], scale=self.A_q[1])
        linear_fp8(self.A_q[0], self.A_q[1], self.Wo_q[0], self.Wo_q[1], R=x0, Y=self.x1, ws=self.ws)
        rmsnorm_scale(self.x1, w["gamma_mlp"], s.eps, rstd=self.rstd1, U=self.U1)
        quantize_fp8_rows(self.U1, Xq=self.U1_q[0], scale=self.U1_q[1])
        linear_swiglu_fp8(self.U1_q[0], self.U1_q[1], self.Wg_q[0], self.Wg_q[1], self.Wu_q[0], self.Wu_q[1],
                          rstd=self.rstd1, H=self.H, g=self.g, u=self.u, ws=self.ws)
        quantize_fp8_rows(self.H, Xq=self.H_q[0], scale=self.H_q[1])
        linear_fp8(self.H_q[0], self.H_q[1], self.Wd_q[0], self.Wd_q[1], R=self.x1, Y=self.x2, ws=self.ws)
        mark("fwd")
        return {"Q": self.fwd["Q"], "K": self.fwd["K"], "V": self.fwd["V"], "x1": self.x1, "x2": self.x2}

    def backward(self, x0, A, pos, dx2, dQ, dK, dV, mark=None):
        s, w = self.s, self.w
        mark = mark or (lambda name: None)
        T, Hd, I, a_in = s.tokens, s.hidden, s.inter, s.n_q * s.head_dim
        quantize_fp8_rows(dx2, Xq=self.dx2_q[0], scale=self.dx2_q[1])
        linear_dswiglu_fp8(self.dx2_q[0], self.dx2_q[1], self.WdT_q[0], self.WdT_q[1], self.g, self.u,
                           rstd=self.rstd1, out={"Gp": self.Gp, "row": self.coef1, "H": None}, ws=self.ws)
        ctx, ws2 = self._side()
        with ctx:   # weight gradients of the MLP beside its input gradient
            if self.fp8_wgrad:
                self._wgrad_fp8(dx2, self.dx2T_q, self.H, self.HT_q, self.dW["dWd"], ws2)
                self._wgrad_fp8(self.Gp, self.GT_q, self.U1, self.U1T_q, self.dWgu, ws2)
                # the QKV backward's dW operand: u0 = x0 ⊙ gamma_attn per column
                quantize_fp8_cols(self.U0, XTq=self.U0T_q[0], scale=self.U0T_q[1])
            else:
                self._wgrad(dx2, Hd, self.H, I, self.dW["dWd"], Hd, I, T, ws=ws2)
                self._wgrad(self.Gp, 2 * I, self.U1, Hd, self.dW["dWg"], I, Hd, T, ws=ws2)
                # the up half of G' (a flat view from its first element; rows 2I apart)
                self._wgrad(self.Gp.view(-1)[I:], 2 * I, self.U1, Hd, self.dW["dWu"], I, Hd, T, ws=ws2)
        quantize_fp8_rows(self.Gp, Xq=self.G_q[0], scale=self.G_q[1])
        rmsnorm_linear_dx_fp8(self.G_q[0], self.G_q[1], self.WguT_q[0], self.WguT_q[1], self.x1, w["gamma_mlp"],
                              self.coef1, dX_resid=dx2, out=self.dx1, ws=self.ws)
        dx1 = self.dx1["dX"]
        quantize_fp8_rows(dx1, Xq=self.dx1_q[0], scale=self.dx1_q[1])
        linear_fp8(self.dx1_q[0], self.dx1_q[1], self.WoT_q[0], self.WoT_q[1], Y=self.dA, ws=self.ws)
        self._join()
        ctx, ws2 = self._side()
        with ctx:
            if self.fp8_wgrad:
                self._wgrad_fp8(dx1, self.dx1T_q, A, self.AT_q, self.dW["dWo"], ws2)
            else:
                self._wgrad(dx1, Hd, A, a_in, self.dW["dWo"], Hd, a_in, T, ws=ws2)
        if self.fp8_wgrad:
            linear_qknorm_rope_bwd_fp8(dQ, dK, dV, self.fwd["qk_save"], self.fwd["V"], w["gamma_q"], w["gamma_k"],
                                       pos, self.cos_sin, s.n_q, s.n_kv, self.WqkvT_q[0], self.WqkvT_q[1],
                                       self.U0T_q[0], self.U0T_q[1], X=x0, rstd=self.rstd0,
                                       gamma_in=w["gamma_attn"], dX_resid=dx1, eps=s.eps, head_dim=s.head_dim,
                                       ws=self.ws, out=self.grads_qkv)
        else:
            linear_qknorm_rope_bwd(dQ, dK, dV, self.fwd["qk_save"], self.fwd["V"], w["gamma_q"], w["gamma_k"], pos,
                                   self.cos_sin, s.n_q, s.n_kv, x0, w["Wqkv"], rstd=self.rstd0,
                                   gamma_in=w["gamma_attn"], dX_resid=dx1, eps=s.eps, head_dim=s.head_dim,
                                   ws=self.ws, out=self.grads_qkv)
        self._join()
        mark("bwd")
        return {"dx0": self.grads_qkv["dX"], "dA": self.dA, "dx1": dx1, "dWqkv": self.grads_qkv["dW"],
                "dWo": self.dW["dWo"], "dWg": self.dW["dWg"], "dWu": self.dW["dWu"], "dWd": self.dW["dWd"],
                "dgamma_attn": self.grads_qkv["dgamma_in"], "dgamma_mlp": self.dx1["dgamma"],
                "dgamma_q": self.grads_qkv["dgamma_q"], "dgamma_k": self.grads_qkv["dgamma_k"]}

    def step(self, x0, A, pos, dx2, dQ, dK, dV, mark=None):
        self.forward(x0, A, pos, mark)
        return self.backward(x0, A, pos, dx2, dQ, dK, dV, mark)


class _NullCtx:
    def __enter__(self):
        return None

    def __exit__(self, *a):
        return False


class LinearCE:
    """Linear + cross-entropy forward and backward with persistent buffers."""

    def __init__(self, M, V, K, device="cuda"):
        lib = load()
        self.out = {"loss": torch.empty(1, dtype=torch.float32, device=device),
                    "lse": torch.empty(M, dtype=torch.float32, device=device),
                    "n_valid": torch.empty(1, dtype=torch.int32, device=device)}
        self.grads = {"dX": torch.empty(M, K, dtype=torch.bfloat16, device=device),
                      "dW": torch.empty(V, K, dtype=torch.bfloat16, device=device)}
        self.ws = workspace(max(lib.coda_linear_cross_entropy_workspace_size(M, V, K),
                                lib.coda_linear_cross_entropy_bwd_workspace_size(M, V, K)), device)

    def step(self, X, W, labels, ignore_index=-100):
        linear_cross_entropy(X, W, labels, ignore_index, out=self.out, ws=self.ws)
        linear_cross_entropy_bwd(X, W, labels, self.out["lse"], self.out["n_valid"], 1.0, ignore_index,
                                 out=self.grads, ws=self.ws)
        return self.out, self.grads
