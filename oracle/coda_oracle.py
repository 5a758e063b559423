"""fp64 CPU oracle for the CODA GEMM-epilogue transformer operators.

TEST INFRASTRUCTURE ONLY.  Only ``tests/``, ``__graft_entry__.smoke()`` and
``bench.py``'s CPU-baseline / reference leg may import or call this module.
The product path (the CUDA library and its Python binding) never imports it,
and this module imports nothing from the product path.

What it computes: the *canonical, unfused* formula of every operator, in
float64 NumPy, on the exact values of the bf16/fp32/int32 inputs.  It does not
use the GEMM-epilogue reparameterisations (those are what the CUDA path does);
it has no intermediate bf16 rounding, no tiling and no fusion.  Backward passes
are the textbook chain rule of the canonical forward formulas, derived here
independently of the CUDA path's fused backward.

Sources (page titles, then section / equation / figure):
  [P1] "CODA: Rewriting Transformer Blocks as GEMM-Epilogue Programs"
       (HTML text of arXiv 2605.19269, Chinese translation).
  [P2] "CODA: new research optimizes Transformer training with GEMM-epilogue
       programming" (news flash, Filipino).
  [P3] "CODA: 把 Transformer Block 重写成 GEMM-Epilogue 程序 · 干货攻略"
       (x-tip guide).

Readings where the pages are silent (each is also listed in the design notes):
  * RMSNorm: rms(x) = sqrt(mean(x^2) + eps), eps inside the root.
  * RMSNorm gain gamma multiplies after normalising and before the next
    projection ([P1] §3.2.1 equation).
  * RoPE: interleaved pairs (2j, 2j+1), angle = pos * theta^(-2j/d),
    [a, b] -> [a cos - b sin, a sin + b cos]; no frequency scaling.
  * QK-RMSNorm: per head over head_dim, gains shared by all heads, applied
    before RoPE.
  * Cross-entropy: natural log, mean over rows whose label != ignore_index;
    all rows ignored gives NaN (0/0) and a zero gradient; a label outside
    [0, V) other than ignore_index is reported as a range error and its row
    counts as ignored.

Parity status: every function below is pinned by a test in
``tests/test_oracle_pins.py`` (identities, closed forms, library special
cases, finite differences); none is "parity unpinned".
"""
from __future__ import annotations

import numpy as np

__all__ = [
    "rms_inv", "rmsnorm", "rmsnorm_bwd",
    "rmsnorm_linear_fwd", "rmsnorm_linear_bwd",
    "linear_residual_fwd", "linear_residual_bwd",
    "silu", "silu_grad", "swiglu_fwd", "mlp_fwd", "mlp_bwd",
    "rope_angles", "rope", "rope_inv", "qk_rmsnorm_rope_fwd", "qk_rmsnorm_rope_bwd",
    "linear_cross_entropy_fwd", "linear_cross_entropy_bwd",
    "block_fwd", "block_bwd", "block_flops", "mlp_flops", "ce_flops",
    "gemm_epilogue_plain",
    "rmsnorm_linear_cross_entropy_fwd", "rmsnorm_linear_cross_entropy_bwd",
    "sigmoid", "linear_sigmoid_fwd", "linear_sigmoid_bwd",
    "E4M3_MAX", "quantize_fp8_rows", "linear_fp8_fwd", "swiglu_fp8_fwd",
    "quantize_fp8_cols", "linear_qknorm_rope_fp8_fwd", "linear_cross_entropy_fp8_fwd",
    "linear_cross_entropy_fp8_bwd", "dswiglu_fp8", "rmsnorm_linear_dx_fp8",
    "E2M1_MAX", "E2M1_GRID", "NVFP4_BLOCK", "e2m1_round", "e2m1_value", "quantize_nvfp4_rows",
    "rmsnorm_scale_nvfp4",
    "linear_nvfp4_fwd", "swiglu_nvfp4_fwd",
]


# ---------------------------------------------------------------------------
# the generic GEMM + element-wise / rank-1 / rank-2 epilogue
# ---------------------------------------------------------------------------

def gemm_epilogue_plain(A, B, row_scale=None, col_scale=None, aux0=None, row_coef=None, aux1=None,
                        D_old=None):
    """h = A B^T (A [M, K], B [N, K]); y_ij = rs_i cs_j h_ij + aux0_ij
    - coef_i aux1_ij (+ D_old_ij).  [P1] §3.2: GEMM h = xW followed by a
    tile-wise function y[i,j] = f_ij(h); the terms are the element-wise map,
    rank-1 vector loads and rank-2 tile loads of §3.1 classes 1-3, and the
    accumulation named in the abstract."""
    y = A @ B.T
    if row_scale is not None:
        y = y * np.asarray(row_scale)[:, None]
    if col_scale is not None:
        y = y * np.asarray(col_scale)[None, :]
    if aux0 is not None:
        y = y + aux0
    if row_coef is not None:
        y = y - np.asarray(row_coef)[:, None] * aux1
    if D_old is not None:
        y = y + D_old
    return y


# ---------------------------------------------------------------------------
# RMSNorm
# ---------------------------------------------------------------------------

def rms_inv(x, eps):
    """r = 1/rms(x) per row, rms(x) = sqrt(mean_k x_k^2 + eps).

    [P1] §3.2.1: r is the row-wise inverse RMS factor of the pattern's
    equation y = RMSNorm(xW0 + z, gamma) W1 = (r (xW0 + z) ⊙ gamma) W1.
    eps placement is a reading (inside the root)."""
    x = np.asarray(x, dtype=np.float64)
    return 1.0 / np.sqrt(np.mean(x * x, axis=-1) + eps)


def rmsnorm(x, gamma, eps):
    """RMSNorm(x, gamma) = (x * r) ⊙ gamma   ([P1] §3.2.1 equation)."""
    r = rms_inv(x, eps)
    return (x * r[..., None]) * gamma


def rmsnorm_bwd(x, gamma, eps, dy):
    """Gradient of y = (x r) ⊙ gamma w.r.t. x and gamma (chain rule).

    n = x r,  dn = dy ⊙ gamma,  dx = r (dn - n * mean_k(n ⊙ dn)),
    dgamma = sum over all leading axes of dy ⊙ n.
    The pages give no backward formula ([P2] only states that block-local
    forwards keep a GEMM-epilogue backward); this is the textbook derivative
    of the forward definition above."""
    r = rms_inv(x, eps)[..., None]
    n = x * r
    dn = dy * gamma
    dx = r * (dn - n * np.mean(n * dn, axis=-1, keepdims=True))
    dgamma = (dy * n).reshape(-1, x.shape[-1]).sum(axis=0)
    return dx, dgamma


# ---------------------------------------------------------------------------
# RMSNorm followed by a projection (+ residual)
# ---------------------------------------------------------------------------

def rmsnorm_linear_fwd(X, gamma, W, eps, R=None):
    """y = R + RMSNorm(X, gamma) W^T   with W stored [out, in].

    [P1] §3.2.1 equation (second GEMM of the GEMM-RMSNorm-GEMM pattern, the
    residual being the preceding stream).  Returns (y, r)."""
    a = rmsnorm(X, gamma, eps)
    y = a @ W.T
    if R is not None:
        y = y + R
    return y, rms_inv(X, eps)


def rmsnorm_linear_bwd(X, gamma, W, eps, G):
    """Backward of rmsnorm_linear_fwd for upstream gradient G.

    a = RMSNorm(X, gamma); y = a W^T + R.
    da = G W, dW = G^T a, then RMSNorm backward gives dX and dgamma; dR = G.
    (Chain rule of the canonical formula; no page prints it.)"""
    a = rmsnorm(X, gamma, eps)
    da = G @ W
    dW = G.T @ a
    dX, dgamma = rmsnorm_bwd(X, gamma, eps, da)
    return {"dX": dX, "dW": dW, "dgamma": dgamma, "dR": G}


# ---------------------------------------------------------------------------
# projection + residual (the first GEMM of the pattern)
# ---------------------------------------------------------------------------

def linear_residual_fwd(X, W, R, eps=1e-6):
    """u = X W^T + R, the "xW0 + z" of [P1] §3.2.1, and r = 1/rms(u), the
    row factor that the first GEMM's epilogue prepares (as partial sums of
    squares) for the next projection."""
    u = X @ W.T + R
    return u, rms_inv(u, eps)


def linear_residual_bwd(X, W, G):
    """dX = G W, dW = G^T X, dR = G (chain rule)."""
    return {"dX": G @ W, "dW": G.T @ X, "dR": G}


# ---------------------------------------------------------------------------
# SwiGLU, workloads 1 and 3
# ---------------------------------------------------------------------------

def silu(a):
    """silu(a) = a * sigmoid(a) = a / (1 + exp(-a)).  The SwiGLU gate of
    [P1] §3.1 class 1 (pairwise maps) and [P3]'s linear_swiglu example."""
    a = np.asarray(a, dtype=np.float64)
    return a / (1.0 + np.exp(-a))


def silu_grad(a):
    """d silu / da = s (1 + a (1 - s)), s = sigmoid(a)  (calculus)."""
    s = 1.0 / (1.0 + np.exp(-np.asarray(a, dtype=np.float64)))
    return s * (1.0 + a * (1.0 - s))


def swiglu_fwd(X, Wg, Wu):
    """H = silu(X Wg^T) ⊙ (X Wu^T); returns (H, g, u).  Workload 1."""
    g = X @ Wg.T
    u = X @ Wu.T
    return silu(g) * u, g, u


def mlp_fwd(X, Wg, Wu, Wd, R, gamma=None, eps=1e-6):
    """SwiGLU MLP sublayer: a = X (or RMSNorm(X, gamma) when gamma is given),
    g = a Wg^T, u = a Wu^T, H = silu(g) ⊙ u, y = R + H Wd^T.
    Returns a dict with y and the intermediates."""
    a = X if gamma is None else rmsnorm(X, gamma, eps)
    H, g, u = swiglu_fwd(a, Wg, Wu)
    y = R + H @ Wd.T
    return {"y": y, "H": H, "g": g, "u": u, "a": a}


def mlp_bwd(X, Wg, Wu, Wd, dY, gamma=None, eps=1e-6):
    """Backward of mlp_fwd (chain rule).  dR = dY is returned separately;
    dX is the gradient through the MLP branch only."""
    f = mlp_fwd(X, Wg, Wu, Wd, np.zeros_like(dY), gamma, eps)
    g, u, H, a = f["g"], f["u"], f["H"], f["a"]
    dH = dY @ Wd
    dWd = dY.T @ H
    dg = dH * u * silu_grad(g)
    du = dH * silu(g)
    da = dg @ Wg + du @ Wu
    out = {"dWd": dWd, "dWg": dg.T @ a, "dWu": du.T @ a, "dR": dY,
           "dH": dH, "dg": dg, "du": du}
    if gamma is None:
        out["dX"] = da
    else:
        out["dX"], out["dgamma"] = rmsnorm_bwd(X, gamma, eps, da)
    return out


# ---------------------------------------------------------------------------
# QK-RMSNorm + RoPE
# ---------------------------------------------------------------------------

def rope_angles(pos, head_dim, theta):
    """angle[t, j] = pos[t] * theta^(-2j/head_dim), j < head_dim/2 (reading)."""
    j = np.arange(head_dim // 2, dtype=np.float64)
    inv_freq = theta ** (-2.0 * j / head_dim)
    return np.asarray(pos, dtype=np.float64)[:, None] * inv_freq[None, :]


def rope(v, pos, theta, pairing="interleaved"):
    """Rotate pairs of v[t, head, d] by angle[t, j] = pos[t] * theta^(-2j/d):
    [a, b] -> [a cos - b sin, a sin + b cos].  pairing "interleaved": pair j
    is (2j, 2j+1); "half": pair j is (j, j + d/2) (the two halves of the
    head).  [P1] §3.1 class 1 names RoPE-style rotations as a pairwise map;
    the pairing convention is a reading, and both are supported."""
    d = v.shape[-1]
    ang = rope_angles(pos, d, theta)[:, None, :]
    c, s = np.cos(ang), np.sin(ang)
    out = np.empty_like(v)
    if pairing == "interleaved":
        a, b = v[..., 0::2], v[..., 1::2]
        out[..., 0::2] = a * c - b * s
        out[..., 1::2] = a * s + b * c
    elif pairing == "half":
        a, b = v[..., : d // 2], v[..., d // 2:]
        out[..., : d // 2] = a * c - b * s
        out[..., d // 2:] = a * s + b * c
    else:
        raise ValueError(pairing)
    return out


def rope_inv(v, pos, theta, pairing="interleaved"):
    """Rotation by the negative angle: the inverse (and transpose) of rope."""
    return rope(v, -np.asarray(pos, dtype=np.float64), theta, pairing)


def qk_rmsnorm_rope_fwd(q, gamma, pos, theta, eps, pairing="interleaved"):
    """q[t, head, d] -> RoPE(RMSNorm_d(q) ⊙ gamma, pos).  [P3]'s
    linear_qknorm_rope names the fused operator: per-head RMSNorm, then RoPE."""
    return rope(rmsnorm(q, gamma, eps), pos, theta, pairing)


def qk_rmsnorm_rope_bwd(q, gamma, pos, theta, eps, dout, pairing="interleaved"):
    """Backward: inverse rotation of the gradient, then per-head RMSNorm
    backward.  Returns (dq, dgamma)."""
    dn = rope_inv(dout, pos, theta, pairing)
    return rmsnorm_bwd(q, gamma, eps, dn)


# ---------------------------------------------------------------------------
# linear + cross-entropy
# ---------------------------------------------------------------------------

def _lse(z):
    m = z.max(axis=-1, keepdims=True)
    return (m + np.log(np.exp(z - m).sum(axis=-1, keepdims=True)))[..., 0]


def _ce_valid(labels, ignore_index, V):
    """Rows that enter the loss: label != ignore_index and 0 <= label < V.
    A label outside [0, V) other than ignore_index is a range error; the row
    counts as ignored (reading: the pages give no rule for bad labels)."""
    in_range = (labels >= 0) & (labels < V)
    valid = (labels != ignore_index) & in_range
    bad = (labels != ignore_index) & ~in_range
    return valid, bool(bad.any())


def linear_cross_entropy_fwd(X, W, labels, ignore_index=-100):
    """z = X W^T; lse_i = log sum_j exp(z_ij); loss_i = lse_i - z_{i, y_i};
    mean over rows with y_i != ignore_index and 0 <= y_i < V.

    [P1] §3.1 class 5 (running max / sum-exp state for online log-sum-exp and
    cross-entropy) and [P3]'s linear_cross_entropy.  Returns a dict with
    loss (scalar), lse [M], per-row loss [M] (0 on ignored rows), n_valid,
    and label_range_error (some label other than ignore_index lies outside
    [0, V); such rows count as ignored)."""
    labels = np.asarray(labels)
    z = X @ W.T
    lse = _lse(z)
    valid, bad = _ce_valid(labels, ignore_index, W.shape[0])
    rows = np.nonzero(valid)[0]
    per_row = np.zeros(X.shape[0])
    per_row[rows] = lse[rows] - z[rows, labels[rows]]
    n_valid = int(valid.sum())
    loss = per_row[rows].sum() / n_valid if n_valid > 0 else float("nan")
    return {"loss": loss, "lse": lse, "per_row": per_row, "n_valid": n_valid, "label_range_error": bad}


def linear_cross_entropy_bwd(X, W, labels, ignore_index=-100, dloss=1.0, vocab_rows=None):
    """dZ = (softmax(z) - onehot(y)) * dloss / n_valid on valid rows, 0 on
    ignored rows (label == ignore_index or outside [0, V)); dX = dZ W,
    dW = dZ^T X (chain rule).

    With vocab_rows (indices into the vocabulary) only those rows of dW are
    returned, as "dW_rows" = dZ[:, vocab_rows]^T X (the softmax still
    normalises over the whole vocabulary); dX is then not formed."""
    labels = np.asarray(labels)
    z = X @ W.T
    p = np.exp(z - _lse(z)[:, None])
    valid, _ = _ce_valid(labels, ignore_index, W.shape[0])
    rows = np.nonzero(valid)[0]
    n_valid = int(valid.sum())
    dZ = np.zeros_like(z)
    if n_valid > 0:
        dZ[rows] = p[rows]
        dZ[rows, labels[rows]] -= 1.0
        dZ *= dloss / n_valid
    if vocab_rows is not None:
        return {"dW_rows": dZ[:, np.asarray(vocab_rows)].T @ X}
    return {"dX": dZ @ W, "dW": dZ.T @ X, "dZ": dZ}


# ---------------------------------------------------------------------------
# linear + sigmoid (gate)
# ---------------------------------------------------------------------------

def sigmoid(a):
    """1 / (1 + exp(-a))."""
    return 1.0 / (1.0 + np.exp(-np.asarray(a, dtype=np.float64)))


def linear_sigmoid_fwd(X, W, Z=None):
    """y = sigmoid(X W^T), or sigmoid(X W^T) ⊙ Z when a gated tensor Z is given.
    [P3] names linear_sigmoid among the functional operators; reading: a
    linear layer with an element-wise sigmoid, optionally gating Z (the
    §3.1 class-1 element-wise / pairwise map)."""
    s = sigmoid(X @ W.T)
    return s if Z is None else s * Z


def linear_sigmoid_bwd(X, W, dY, Z=None):
    """Chain rule: dz = dY ⊙ (Z) ⊙ s (1 - s), dX = dz W, dW = dz^T X, and
    dZ = dY ⊙ s when Z is given."""
    s = sigmoid(X @ W.T)
    g = dY if Z is None else dY * Z
    dz = g * s * (1.0 - s)
    out = {"dX": dz @ W, "dW": dz.T @ X}
    if Z is not None:
        out["dZ"] = dY * s
    return out


# ---------------------------------------------------------------------------
# FP8 (e4m3) operands with per-row scales
# ---------------------------------------------------------------------------
# The pages motivate fusion by low-precision GEMMs (FP8 / FP4, [P1] §1 and
# [P2]); they give no quantisation recipe.  Reading: per-row (per token, per
# output channel) scales s = amax / 448 in fp32, codes q = e4m3(x / s) with
# the division in fp32, round to nearest even, saturating at +-448.  These
# are the decisions the kernel takes, in the kernel's precision (fp32), so
# the codes must match bit for bit.

E4M3_MAX = 448.0


def quantize_fp8_rows(X):
    """Returns (codes uint8 [M, K], values float64 [M, K] = e4m3(codes),
    scales float32 [M]); x ~= values * scale."""
    import torch
    x32 = np.asarray(X, dtype=np.float32)
    amax = np.max(np.abs(x32), axis=1) if x32.shape[1] else np.zeros(x32.shape[0], np.float32)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    v = np.clip((x32 / scale[:, None]).astype(np.float32), -E4M3_MAX, E4M3_MAX)
    q = torch.from_numpy(v).to(torch.float8_e4m3fn)
    return q.view(torch.uint8).numpy(), q.double().numpy(), scale


def linear_fp8_fwd(Xv, sx, Wv, sw, R=None, row_scale=None):
    """y = R + rs_i * (Xv_i sx_i) . (Wv_n sw_n): the plain linear of
    gemm_epilogue_plain on the dequantised operands."""
    A = Xv * np.asarray(sx, dtype=np.float64)[:, None]
    B = Wv * np.asarray(sw, dtype=np.float64)[:, None]
    return gemm_epilogue_plain(A, B, row_scale=row_scale, aux0=R)


def swiglu_fp8_fwd(Xv, sx, Wgv, sg, Wuv, su, row_scale=None):
    """swiglu_fwd on the dequantised operands, with the optional row factor r
    applied to g and u before the gate (as the RMSNorm-reparameterised
    gate/up projection does).  Returns (H, g, u)."""
    A = Xv * np.asarray(sx, dtype=np.float64)[:, None]
    if row_scale is not None:
        A = A * np.asarray(row_scale, dtype=np.float64)[:, None]
    return swiglu_fwd(A, Wgv * np.asarray(sg, dtype=np.float64)[:, None],
                      Wuv * np.asarray(su, dtype=np.float64)[:, None])



def quantize_fp8_cols(X):
    """Column quantiser, the row quantiser's rule along the other axis:
    scale_j = max_i |x_ij| / 448 (fp32; 1 for an all-zero column),
    q_ij = e4m3(x_ij / scale_j).  Returned transposed, as the K-major operand
    of a GEMM that contracts over X's rows: (codes uint8 [C, R] of X^T,
    values float64 [C, R], scales float32 [C]); x_ij ~= values[j, i] * scale_j."""
    import torch
    x32 = np.asarray(X, dtype=np.float32)
    amax = np.max(np.abs(x32), axis=0) if x32.shape[0] else np.zeros(x32.shape[1], np.float32)
    scale = np.where(amax > 0, amax / np.float32(E4M3_MAX), np.float32(1.0)).astype(np.float32)
    v = np.clip((x32 / scale[None, :]).astype(np.float32), -E4M3_MAX, E4M3_MAX)
    q = torch.from_numpy(np.ascontiguousarray(v.T)).to(torch.float8_e4m3fn)
    return q.view(torch.uint8).numpy(), q.double().numpy(), scale


def _deq(values, scales):
    """Dequantised operand: values * per-row scales."""
    return np.asarray(values, dtype=np.float64) * np.asarray(scales, dtype=np.float64)[:, None]


def linear_qknorm_rope_fp8_fwd(Xv, sx, Wv, sw, gamma_q, gamma_k, pos, theta, eps, n_q, n_kv, head_dim,
                               row_scale=None, pairing="interleaved"):
    """The QKV projection with QK-RMSNorm + RoPE on e4m3 operands:
    [q | k | v] = r ⊙ ((Xv sx)(Wv sw)^T) (r = 1 without row_scale), then per
    head Q = RoPE(RMSNorm_d(q) ⊙ gamma_q), K likewise, V = v ([P3]'s
    linear_qknorm_rope on the dequantised operands).  Returns Q, K, V and
    the pre-norm q|k, flattened per token."""
    qkv = gemm_epilogue_plain(_deq(Xv, sx), _deq(Wv, sw), row_scale=row_scale)
    d, M = head_dim, qkv.shape[0]
    q = _heads(qkv[:, : n_q * d], n_q, d)
    k = _heads(qkv[:, n_q * d: (n_q + n_kv) * d], n_kv, d)
    Q = qk_rmsnorm_rope_fwd(q, gamma_q, pos, theta, eps, pairing)
    K = qk_rmsnorm_rope_fwd(k, gamma_k, pos, theta, eps, pairing)
    return {"Q": Q.reshape(M, -1), "K": K.reshape(M, -1), "V": qkv[:, (n_q + n_kv) * d:],
            "qk": qkv[:, : (n_q + n_kv) * d]}


def linear_cross_entropy_fp8_fwd(Xv, sx, Wv, sw, labels, ignore_index=-100):
    """linear_cross_entropy_fwd on the dequantised e4m3 operands."""
    return linear_cross_entropy_fwd(_deq(Xv, sx), _deq(Wv, sw), labels, ignore_index)


def linear_cross_entropy_fp8_bwd(Xv, sx, Wv, sw, X, W, labels, ignore_index=-100, dloss=1.0):
    """The softmax gradient dZ of linear_cross_entropy_bwd at the logits of
    the dequantised e4m3 operands, then dX = dZ W and dW = dZ^T X with the
    operands X, W of the two gradient GEMMs (bf16)."""
    dZ = linear_cross_entropy_bwd(_deq(Xv, sx), _deq(Wv, sw), labels, ignore_index, dloss)["dZ"]
    return {"dX": dZ @ W, "dW": dZ.T @ X, "dZ": dZ}


def dswiglu_fp8(dYv, sdy, WdTv, swd, g, u, row_scale=None):
    """The dSwiGLU map on the dH GEMM with e4m3 operands:
    dH = (dYv sdy)(WdTv swd)^T  (dY Wd with Wd^T quantised per unit),
    dG = dH ⊙ u ⊙ silu'(g),  dU = dH ⊙ silu(g)  (g, u the saved projections);
    returns G' = r ⊙ [dG | dU] ([M, 2I]; r = 1 without row_scale), the row
    sums dot_i = sum_j (dG g + dU u)_ij, with row_scale the RMSNorm-backward
    coefficient coef_i = r_i^2 dot_i / K (K = dY's width), H = silu(g) ⊙ u
    and dH.  (The chain rule of mlp_fwd's H = silu(g) u.)"""
    dH = _deq(dYv, sdy) @ _deq(WdTv, swd).T
    g = np.asarray(g, dtype=np.float64)
    u = np.asarray(u, dtype=np.float64)
    dG = dH * u * silu_grad(g)
    dU = dH * silu(g)
    r = np.ones(dH.shape[0]) if row_scale is None else np.asarray(row_scale, dtype=np.float64)
    dot = (dG * g + dU * u).sum(axis=1)
    coef = None if row_scale is None else r * r * dot / np.asarray(dYv).shape[1]
    return {"Gp": np.concatenate([dG, dU], axis=1) * r[:, None], "dot": dot, "coef": coef,
            "H": silu(g) * u, "dH": dH}


def rmsnorm_linear_dx_fp8(Gv, sgp, WTv, sw, X, gamma, coef, dX_resid=None):
    """The input gradient of an RMSNorm-reparameterised projection with e4m3
    operands: D = (Gv sgp)(WTv sw)^T (G' W with W^T quantised per input
    feature), dX = gamma ⊙ D - coef ⊙ X (+ dX_resid), dgamma_k = sum_i X_ik D_ik
    (the backward of y = r ⊙ ((X ⊙ gamma) W^T) written out by the chain
    rule; coef_i = r_i^2 sum_n G_in y_in / K comes from the caller)."""
    D = _deq(Gv, sgp) @ _deq(WTv, sw).T
    X = np.asarray(X, dtype=np.float64)
    dX = D * np.asarray(gamma, dtype=np.float64)[None, :] - np.asarray(coef, dtype=np.float64)[:, None] * X
    if dX_resid is not None:
        dX = dX + dX_resid
    return {"dX": dX, "dgamma": (X * D).sum(axis=0), "D": D}


def _bf16(x):
    """Round to bfloat16 (nearest even), returned as float64."""
    import torch
    return torch.from_numpy(np.asarray(x, dtype=np.float64)).to(torch.bfloat16).double().numpy()


def linear_qknorm_rope_fp8_bwd(dQ, dK, dV, qk_save, V, gamma_q, gamma_k, pos, theta, eps, n_q, n_kv, head_dim,
                               WTv, sw, UTv, su, X=None, row_scale=None, gamma_in=None, dX_resid=None,
                               pairing="interleaved"):
    """The backward of linear_qknorm_rope_fp8_fwd with both gradient GEMMs on
    e4m3 operands.  Per head the inverse rotation and the QK-RMSNorm backward
    (qk_rmsnorm_rope_bwd) at the saved pre-norm q|k give dq, dk; with dv = dV,
    G = [dq | dk | dv] is the gradient of the projection y = [q | k | v] and
    G' = r ⊙ G (r = 1 without row_scale).  Reading: G' is held in bf16 and
    quantised per row (for D = G' W) and per column (for dW = G'^T U) by the
    rules of quantize_fp8_rows / quantize_fp8_cols; W enters as W^T quantised
    per input feature (WTv, sw) and U, the forward GEMM's input (x ⊙ gamma_in
    with the input RMSNorm), likewise (UTv, su).  Then
        D = (G'_q)(W^T_q)^T,   dW = (G'^T_q)(U^T_q)^T,
        with row_scale: c_i = r_i^2 sum_n G_in y_in / K  (K = X's width),
        dX = gamma_in ⊙ D - c ⊙ X (+ dX_resid),  dgamma_in = sum_i X_i ⊙ D_i;
        without: dX = D (+ dX_resid)
    (the chain rule of y = r ⊙ ((X ⊙ gamma_in) W^T), as in
    rmsnorm_linear_dx_fp8)."""
    d = head_dim
    qk_save = np.asarray(qk_save, dtype=np.float64)
    M = qk_save.shape[0]
    q = _heads(qk_save[:, : n_q * d], n_q, d)
    k = _heads(qk_save[:, n_q * d:], n_kv, d)
    dq, dgq = qk_rmsnorm_rope_bwd(q, gamma_q, pos, theta, eps, _heads(dQ, n_q, d), pairing)
    dk, dgk = qk_rmsnorm_rope_bwd(k, gamma_k, pos, theta, eps, _heads(dK, n_kv, d), pairing)
    G = np.concatenate([dq.reshape(M, -1), dk.reshape(M, -1), np.asarray(dV, dtype=np.float64)], axis=1)
    r = np.ones(M) if row_scale is None else np.asarray(row_scale, dtype=np.float64)
    Gp = _bf16(G * r[:, None])
    _, gv, sg = quantize_fp8_rows(Gp)
    _, gtv, sgt = quantize_fp8_cols(Gp)
    D = _deq(gv, sg) @ _deq(WTv, sw).T
    out = {"Gr": G * r[:, None], "Gp": Gp, "D": D, "dgamma_q": dgq, "dgamma_k": dgk,
           "dW": _deq(gtv, sgt) @ _deq(UTv, su).T}
    if row_scale is None:
        dX = D
    else:
        Xf = np.asarray(X, dtype=np.float64)
        y = np.concatenate([qk_save, np.asarray(V, dtype=np.float64)], axis=1)
        coef = r * r * (G * y).sum(axis=1) / Xf.shape[1]
        dX = D * np.asarray(gamma_in, dtype=np.float64)[None, :] - coef[:, None] * Xf
        out["dgamma_in"] = (Xf * D).sum(axis=0)
        out["coef"] = coef
    out["dX"] = dX if dX_resid is None else dX + np.asarray(dX_resid, dtype=np.float64)
    return out


# ---------------------------------------------------------------------------
# NVFP4 operands: e2m1 elements, an e4m3 scale per 16 elements, fp32 row scale
# ---------------------------------------------------------------------------
# [P1] §1 and [P2] name FP4 beside FP8 as the formats that make the GEMMs
# fast and the data movement around them dominant; the pages give no recipe.
# Reading: NVIDIA's NVFP4 block format (4-bit e2m1 values, one e4m3 scale
# per 16 consecutive elements along K), with the second-level fp32 scale
# taken per row (token or output channel) as in the FP8 path.  Per row:
#
#   s      = amax(row) / (6 * 448)            (1 for an all-zero row)
#   for each block of 16 elements along K, with bmax = max |x| over it:
#   sf     = e4m3(bmax / (6 * s))             nearest even, saturating at 448
#   inv    = min(1 / (sf * s), FLT_MAX)       the block's reciprocal divisor
#   code_k = e2m1(x_k * inv)                  nearest even, saturating at +-6;
#            0 for the whole block when sf * s = 0
#   x_k   ~= e2m1(code_k) * sf * s
#
# Each quotient and product is a single fp32 operation: the codes and scales
# are integer decisions taken in the kernel's precision, so they must match
# bit for bit.  The elements are scaled by the block's reciprocal (one
# division per 16 elements); the cap keeps rows whose scales are far below
# the fp32 normal range finite.  A code of magnitude 0 carries no sign (-0 is
# written as +0).

E2M1_MAX = 6.0
# magnitudes of the e2m1 codes 0..7 (1 sign bit, 2 exponent bits with bias 1,
# 1 mantissa bit; exponent 0 holds 0 and the subnormal 0.5)
E2M1_GRID = np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])
NVFP4_BLOCK = 16
_NVFP4_SCALE_DIV = np.float32(E2M1_MAX * E4M3_MAX)   # 2688


def e2m1_round(v):
    """Values -> e2m1 codes (uint8: bit 3 sign, bits 0-2 magnitude index):
    the nearest grid magnitude, ties to the even index, |v| >= 6 -> 6."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    lo = np.clip(np.searchsorted(E2M1_GRID, a, side="right") - 1, 0, 7)
    hi = np.minimum(lo + 1, 7)
    d_lo = a - E2M1_GRID[lo]
    d_hi = E2M1_GRID[hi] - a
    up = (hi != lo) & ((d_hi < d_lo) | ((d_hi == d_lo) & (hi % 2 == 0)))
    idx = np.where(up, hi, lo).astype(np.uint8)
    neg = (np.asarray(v) < 0) & (idx > 0)
    return (idx | np.where(neg, 8, 0)).astype(np.uint8)


def e2m1_value(codes):
    c = np.asarray(codes, dtype=np.uint8)
    return np.where(c & 8, -1.0, 1.0) * E2M1_GRID[c & 7]


def quantize_nvfp4_rows(X):
    """Returns (codes uint8 [M, K], one e2m1 code per element; sf uint8
    [M, K/16], e4m3 block-scale codes; s float32 [M]; values float64 [M, K] =
    e2m1(code) * e4m3(sf), so that x ~= values * s).  K % 16 == 0."""
    import torch
    x32 = np.asarray(X, dtype=np.float32)
    M, K = x32.shape
    assert K % NVFP4_BLOCK == 0
    nb = K // NVFP4_BLOCK
    ax = np.abs(x32)
    amax = ax.max(axis=1) if K else np.zeros(M, np.float32)
    s = np.where(amax > 0, amax / _NVFP4_SCALE_DIV, np.float32(1.0)).astype(np.float32)
    bmax = ax.reshape(M, nb, NVFP4_BLOCK).max(axis=2) if K else np.zeros((M, 0), np.float32)
    t = (np.float32(E2M1_MAX) * s).astype(np.float32)
    sf_f = np.minimum((bmax / t[:, None]).astype(np.float32), np.float32(E4M3_MAX))
    sfq = torch.from_numpy(np.ascontiguousarray(sf_f)).to(torch.float8_e4m3fn)
    sf = sfq.view(torch.uint8).numpy().copy()
    sf_val = sfq.float().numpy()
    denom = (sf_val * s[:, None]).astype(np.float32)
    with np.errstate(divide="ignore", invalid="ignore", over="ignore"):
        inv = np.minimum(np.float32(1.0) / denom, np.finfo(np.float32).max).astype(np.float32)
        v = (x32 * np.repeat(inv, NVFP4_BLOCK, axis=1)).astype(np.float32)
    zero_block = np.repeat(denom == 0, NVFP4_BLOCK, axis=1)
    codes = np.where(zero_block, 0, e2m1_round(np.where(zero_block, 0, v))).astype(np.uint8)
    values = e2m1_value(codes) * np.repeat(sf_val.astype(np.float64), NVFP4_BLOCK, axis=1)
    return codes, sf, s, values


def rmsnorm_scale_nvfp4(X, gamma, eps):
    """The RMSNorm input stage of an NVFP4 projection ([P1] §3.2.1: the
    projection applies r to the product of x ⊙ gamma and W): the NVFP4
    quantisation of u = x ⊙ gamma, the products taken in fp32 and not
    rounded to bf16, and r = 1/rms(x).  Returns quantize_nvfp4_rows(u) + (r,)."""
    u = (np.asarray(X, dtype=np.float32) * np.asarray(gamma, dtype=np.float32)[None, :]).astype(np.float32)
    return quantize_nvfp4_rows(u) + (rms_inv(X, eps),)


def linear_nvfp4_fwd(Xv, sx, Wv, sw, R=None, row_scale=None):
    """The plain linear on dequantised NVFP4 operands: y = R + rs_i *
    (Xv_i sx_i) . (Wv_n sw_n), values from quantize_nvfp4_rows."""
    return linear_fp8_fwd(Xv, sx, Wv, sw, R=R, row_scale=row_scale)


def swiglu_nvfp4_fwd(Xv, sx, Wgv, sg, Wuv, su, row_scale=None):
    """swiglu_fwd on dequantised NVFP4 operands (row factor r applied to g
    and u before the gate).  Returns (H, g, u)."""
    return swiglu_fp8_fwd(Xv, sx, Wgv, sg, Wuv, su, row_scale=row_scale)


# ---------------------------------------------------------------------------
# final RMSNorm -> LM head -> cross-entropy (third site of the pattern)
# ---------------------------------------------------------------------------

def rmsnorm_linear_cross_entropy_fwd(X, gamma, W, labels, eps, ignore_index=-100):
    """z = RMSNorm(X, gamma) W^T followed by the mean cross-entropy.
    [P1] §3.2.1, third item of the pattern (final MLP down-projection ->
    residual -> final RMSNorm -> language-model head).  Returns the dict of
    linear_cross_entropy_fwd plus the row factor r."""
    f = linear_cross_entropy_fwd(rmsnorm(X, gamma, eps), W, labels, ignore_index)
    f["rstd"] = rms_inv(X, eps)
    return f


def rmsnorm_linear_cross_entropy_bwd(X, gamma, W, labels, eps, ignore_index=-100, dloss=1.0):
    """Backward (chain rule): the cross-entropy backward on a = RMSNorm(X),
    then the RMSNorm backward of its dX.  Returns dX, dW, dgamma."""
    a = rmsnorm(X, gamma, eps)
    b = linear_cross_entropy_bwd(a, W, labels, ignore_index, dloss)
    dX, dgamma = rmsnorm_bwd(X, gamma, eps, b["dX"])
    return {"dX": dX, "dW": b["dW"], "dgamma": dgamma}


# ---------------------------------------------------------------------------
# the non-attention transformer block
# ---------------------------------------------------------------------------

def _heads(t, n, d):
    return t.reshape(t.shape[0], n, d)


def block_fwd(p, n_q, n_kv, head_dim, theta, eps):
    """Pre-norm block without the attention core (its output A is an input):

      a0 = RMSNorm(x0, gamma_attn);  [q | k | v] = a0 Wqkv^T
      Q = RoPE(RMSNorm_head(q, gamma_q)), K likewise with gamma_k, V = v
      x1 = x0 + A Wo^T
      a1 = RMSNorm(x1, gamma_mlp);  g = a1 Wg^T, u = a1 Wu^T, H = silu(g) u
      x2 = x1 + H Wd^T

    The two GEMM-residual-RMSNorm-GEMM sites are [P1] §3.2.1 items 1 and 2.
    ``p`` maps names to float64 arrays (pos as integers)."""
    d = head_dim
    a0 = rmsnorm(p["x0"], p["gamma_attn"], eps)
    qkv = a0 @ p["Wqkv"].T
    q = _heads(qkv[:, : n_q * d], n_q, d)
    k = _heads(qkv[:, n_q * d: (n_q + n_kv) * d], n_kv, d)
    v = qkv[:, (n_q + n_kv) * d:]
    Q = qk_rmsnorm_rope_fwd(q, p["gamma_q"], p["pos"], theta, eps)
    K = qk_rmsnorm_rope_fwd(k, p["gamma_k"], p["pos"], theta, eps)
    x1 = p["x0"] + p["A"] @ p["Wo"].T
    m = mlp_fwd(x1, p["Wg"], p["Wu"], p["Wd"], x1, p["gamma_mlp"], eps)
    return {"Q": Q.reshape(Q.shape[0], -1), "K": K.reshape(K.shape[0], -1), "V": v,
            "x1": x1, "x2": m["y"], "H": m["H"], "g": m["g"], "u": m["u"],
            "q": q.reshape(q.shape[0], -1), "k": k.reshape(k.shape[0], -1)}


def block_bwd(p, n_q, n_kv, head_dim, theta, eps):
    """Backward of block_fwd given dx2 (gradient of x2) and dQ, dK, dV
    (gradients of the attention inputs, supplied because attention is out of
    scope).  Returns the gradients of x0, A, every weight and every gain."""
    d = head_dim
    f = block_fwd(p, n_q, n_kv, head_dim, theta, eps)
    # MLP sublayer: x2 = x1 + mlp(x1)
    mb = mlp_bwd(f["x1"], p["Wg"], p["Wu"], p["Wd"], p["dx2"], p["gamma_mlp"], eps)
    dx1 = p["dx2"] + mb["dX"]
    # attention output projection: x1 = x0 + A Wo^T
    dA = dx1 @ p["Wo"]
    dWo = dx1.T @ p["A"]
    # QKV projection with QK-RMSNorm + RoPE
    q = _heads(f["q"], n_q, d)
    k = _heads(f["k"], n_kv, d)
    dq, dgq = qk_rmsnorm_rope_bwd(q, p["gamma_q"], p["pos"], theta, eps, _heads(p["dQ"], n_q, d))
    dk, dgk = qk_rmsnorm_rope_bwd(k, p["gamma_k"], p["pos"], theta, eps, _heads(p["dK"], n_kv, d))
    dqkv = np.concatenate([dq.reshape(dq.shape[0], -1), dk.reshape(dk.shape[0], -1), p["dV"]], axis=1)
    a0 = rmsnorm(p["x0"], p["gamma_attn"], eps)
    da0 = dqkv @ p["Wqkv"]
    dWqkv = dqkv.T @ a0
    dx0_n, dga = rmsnorm_bwd(p["x0"], p["gamma_attn"], eps, da0)
    return {"dx0": dx1 + dx0_n, "dA": dA, "dx1": dx1, "dWqkv": dWqkv, "dWo": dWo,
            "dWg": mb["dWg"], "dWu": mb["dWu"], "dWd": mb["dWd"],
            "dgamma_attn": dga, "dgamma_mlp": mb["dgamma"], "dgamma_q": dgq, "dgamma_k": dgk,
            "dqkv": dqkv}


# ---------------------------------------------------------------------------
# algorithmic FLOP counts (2*M*N*K per GEMM; element-wise work not counted)
# ---------------------------------------------------------------------------

def mlp_flops(tokens, hidden, inter, backward=True):
    fwd = 2 * tokens * hidden * inter * 3
    return fwd + (2 * fwd if backward else 0)


def ce_flops(tokens, hidden, vocab, backward=True):
    fwd = 2 * tokens * hidden * vocab
    # backward recomputes the logits, then dX and dW
    return fwd + (3 * fwd if backward else 0)


def block_flops(tokens, hidden, qkv_out, attn_in, inter, backward=True):
    fwd = 2 * tokens * hidden * (qkv_out + 3 * inter) + 2 * tokens * attn_in * hidden
    return fwd + (2 * fwd if backward else 0)
