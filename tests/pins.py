"""Checks that pin the fp64 oracle to facts that do not come from the oracle.

Each ``check_*`` function takes the oracle module as an argument and returns
the largest relative discrepancy it found, so that ``test_oracle_pins`` can run
it on the real oracle (expects ~0) and on deliberately broken copies of it
(expects a large value).  The facts used are: identities and special cases the
pages state, closed forms from calculus, independent library routines
(torch float64 CPU ops) for special cases, and central finite differences.
"""
from __future__ import annotations

import math

import numpy as np
import torch
import torch.nn.functional as F

RNG = np.random.default_rng


def _rel(a, b):
    a = np.asarray(a, dtype=np.float64)
    b = np.asarray(b, dtype=np.float64)
    den = max(np.max(np.abs(b)), 1e-300)
    return float(np.max(np.abs(a - b)) / den)


def _fd_grad(fun, x, h=1e-6):
    """Central finite differences of scalar fun w.r.t. every entry of x."""
    g = np.zeros_like(x)
    it = np.nditer(x, flags=["multi_index"])
    for _ in it:
        i = it.multi_index
        old = x[i]
        x[i] = old + h
        fp = fun()
        x[i] = old - h
        fm = fun()
        x[i] = old
        g[i] = (fp - fm) / (2 * h)
    return g


# ---------------------------------------------------------------------------
# RMSNorm-reparameterised projection
# ---------------------------------------------------------------------------

def check_reparam_identity(o):
    """CODA §3.2.1 equation: RMSNorm(x, gamma) W = diag(r) x (diag(gamma) W)
    with r the per-row inverse RMS.  Written here in the reparameterised form
    (row scale applied after the product with the gamma-folded weight)."""
    r = RNG(1)
    X = r.standard_normal((3, 8))
    g = 1 + 0.1 * r.standard_normal(8)
    W = r.standard_normal((5, 8))          # stored [out, in]
    eps = 1e-6
    y, rinv = o.rmsnorm_linear_fwd(X, g, W, eps)
    rms = np.sqrt((X ** 2).sum(axis=1) / 8 + eps)
    Wfold = W * g[None, :]                 # diag(gamma) folded into the weight
    y_reparam = (X @ Wfold.T) / rms[:, None]
    return max(_rel(y, y_reparam), _rel(rinv, 1 / rms))


def check_rmsnorm_library(o):
    """gamma = 1, W = I, no residual reduces to torch's rms_norm (float64)."""
    r = RNG(2)
    X = r.standard_normal((4, 16)) * 3
    eps = 1e-6
    y, _ = o.rmsnorm_linear_fwd(X, np.ones(16), np.eye(16), eps)
    ref = F.rms_norm(torch.from_numpy(X), (16,), eps=eps).numpy()
    g = 1 + 0.1 * r.standard_normal(16)
    y2 = o.rmsnorm(X, g, eps)
    ref2 = F.rms_norm(torch.from_numpy(X), (16,), weight=torch.from_numpy(g), eps=eps).numpy()
    return max(_rel(y, ref), _rel(y2, ref2))


def check_rmsnorm_scale_invariance(o):
    """With eps = 0, RMSNorm(a x) = RMSNorm(x) for a > 0."""
    r = RNG(3)
    X = r.standard_normal((3, 8))
    g = 1 + 0.1 * r.standard_normal(8)
    W = r.standard_normal((5, 8))
    y1, _ = o.rmsnorm_linear_fwd(X, g, W, 0.0)
    y2, _ = o.rmsnorm_linear_fwd(7.5 * X, g, W, 0.0)
    return _rel(y1, y2)


def check_rmsnorm_linear_grad(o):
    """FD gradients of L = sum(G ⊙ y) for y = R + RMSNorm(X, gamma) W^T."""
    r = RNG(4)
    M, K, N = 3, 8, 5
    X = r.standard_normal((M, K))
    g = 1 + 0.1 * r.standard_normal(K)
    W = r.standard_normal((N, K))
    R = r.standard_normal((M, N))
    G = r.standard_normal((M, N))
    eps = 1e-6
    b = o.rmsnorm_linear_bwd(X, g, W, eps, G)

    def L():
        return float((G * o.rmsnorm_linear_fwd(X, g, W, eps, R)[0]).sum())
    errs = [_rel(b["dX"], _fd_grad(L, X)), _rel(b["dW"], _fd_grad(L, W)),
            _rel(b["dgamma"], _fd_grad(L, g))]
    fR = _fd_grad(L, R)
    errs.append(_rel(b["dR"], fR))
    return max(errs)


def check_linear_residual(o):
    """u = X W^T + R against torch's linear; r from partial sums of squares
    over column blocks (any split) equals r over the whole row."""
    r = RNG(5)
    X = r.standard_normal((4, 12))
    W = r.standard_normal((10, 12))
    R = r.standard_normal((4, 10))
    u, rinv = o.linear_residual_fwd(X, W, R, 1e-6)
    ref = F.linear(torch.from_numpy(X), torch.from_numpy(W)).numpy() + R
    parts = [np.sum(ref[:, a:b] ** 2, axis=1) for a, b in ((0, 3), (3, 7), (7, 10))]
    r_parts = 1 / np.sqrt(sum(parts[::-1]) / 10 + 1e-6)
    b = o.linear_residual_bwd(X, W, R)   # R as an arbitrary upstream gradient

    def L():
        return float((R * (X @ W.T)).sum())
    return max(_rel(u, ref), _rel(rinv, r_parts), _rel(b["dX"], _fd_grad(L, X)),
               _rel(b["dW"], _fd_grad(L, W)))


# ---------------------------------------------------------------------------
# SwiGLU
# ---------------------------------------------------------------------------

def check_silu_closed_forms(o):
    """silu(0) = 0, silu'(0) = 1/2, silu(a) -> a (a -> +inf), -> 0 (a -> -inf),
    silu = a*sigmoid(a) vs torch, silu_grad vs central differences."""
    errs = [abs(o.silu(0.0)), abs(o.silu_grad(0.0) - 0.5),
            abs(o.silu(40.0) - 40.0) / 40.0, abs(o.silu(-40.0)),
            abs(o.silu(1.0) - 1.0 / (1.0 + math.exp(-1.0)))]
    a = np.linspace(-8, 8, 41)
    errs.append(_rel(o.silu(a), F.silu(torch.from_numpy(a)).numpy()))
    h = 1e-6
    fd = (o.silu(a + h) - o.silu(a - h)) / (2 * h)
    errs.append(_rel(o.silu_grad(a), fd))
    return max(errs)


def check_swiglu_library(o):
    """H = silu(X Wg^T) ⊙ (X Wu^T) against torch linear/silu in float64."""
    r = RNG(6)
    X = r.standard_normal((5, 8))
    Wg = r.standard_normal((6, 8))
    Wu = r.standard_normal((6, 8))
    H, g, u = o.swiglu_fwd(X, Wg, Wu)
    tX = torch.from_numpy(X)
    ref = (F.silu(F.linear(tX, torch.from_numpy(Wg))) * F.linear(tX, torch.from_numpy(Wu))).numpy()
    return max(_rel(H, ref), _rel(g, X @ Wg.T), _rel(u, X @ Wu.T))


def check_mlp_special_cases(o):
    """Wd = 0 gives y = R; R = 0 and gamma absent gives y = H Wd^T with H from
    swiglu_fwd; gamma present equals feeding torch's rms_norm output."""
    r = RNG(7)
    X = r.standard_normal((3, 8))
    Wg, Wu = r.standard_normal((6, 8)), r.standard_normal((6, 8))
    Wd = r.standard_normal((8, 6))
    R = r.standard_normal((3, 8))
    g = 1 + 0.1 * r.standard_normal(8)
    e1 = _rel(o.mlp_fwd(X, Wg, Wu, np.zeros_like(Wd), R)["y"], R)
    H, _, _ = o.swiglu_fwd(X, Wg, Wu)
    e2 = _rel(o.mlp_fwd(X, Wg, Wu, Wd, np.zeros_like(R))["y"], H @ Wd.T)
    a = F.rms_norm(torch.from_numpy(X), (8,), weight=torch.from_numpy(g), eps=1e-6).numpy()
    H2, _, _ = o.swiglu_fwd(a, Wg, Wu)
    e3 = _rel(o.mlp_fwd(X, Wg, Wu, Wd, R, g, 1e-6)["y"], R + H2 @ Wd.T)
    return max(e1, e2, e3)


def check_mlp_grad(o, with_gamma):
    r = RNG(8 + int(with_gamma))
    M, K, I = 3, 6, 5
    X = r.standard_normal((M, K))
    Wg, Wu = r.standard_normal((I, K)), r.standard_normal((I, K))
    Wd = r.standard_normal((K, I))
    dY = r.standard_normal((M, K))
    g = 1 + 0.1 * r.standard_normal(K) if with_gamma else None
    b = o.mlp_bwd(X, Wg, Wu, Wd, dY, g, 1e-6)

    def L():
        return float((dY * o.mlp_fwd(X, Wg, Wu, Wd, np.zeros_like(dY), g, 1e-6)["y"]).sum())
    errs = [_rel(b["dX"], _fd_grad(L, X)), _rel(b["dWg"], _fd_grad(L, Wg)),
            _rel(b["dWu"], _fd_grad(L, Wu)), _rel(b["dWd"], _fd_grad(L, Wd))]
    if with_gamma:
        errs.append(_rel(b["dgamma"], _fd_grad(L, g)))
    return max(errs)


# ---------------------------------------------------------------------------
# RoPE and QK-RMSNorm
# ---------------------------------------------------------------------------

def check_rope_invariants(o):
    """Pair norms preserved; pos = 0 is the identity; <R_m q, R_n k> depends
    only on m - n; rope_inv undoes rope; one pair checked against the closed
    form rotation (angle = pos * theta^(-2j/d))."""
    r = RNG(10)
    d, theta = 8, 10000.0
    v = r.standard_normal((4, 3, d))
    pos = np.array([0, 1, 5, 17])
    w = o.rope(v, pos, theta)
    e = [_rel(np.hypot(w[..., 0::2], w[..., 1::2]), np.hypot(v[..., 0::2], v[..., 1::2]))]
    e.append(_rel(w[0], v[0]))
    e.append(_rel(o.rope_inv(w, pos, theta), v))
    q = r.standard_normal((1, 1, d))
    k = r.standard_normal((1, 1, d))
    dots = []
    for m, n in ((3, 1), (10, 8), (102, 100)):
        dots.append(float((o.rope(q, [m], theta) * o.rope(k, [n], theta)).sum()))
    e.append(abs(dots[0] - dots[1]) / abs(dots[0]) + abs(dots[0] - dots[2]) / abs(dots[0]))
    # pair j = 1 of head_dim 8 at pos 3: angle 3 * 10000^(-1/4) = 0.3 rad
    unit = np.zeros((1, 1, d))
    unit[0, 0, 2] = 1.0
    w1 = o.rope(unit, [3], theta)[0, 0]
    e.append(abs(w1[2] - math.cos(0.3)) + abs(w1[3] - math.sin(0.3)) + np.abs(np.delete(w1, [2, 3])).sum())
    return max(e)


def check_rope_half(o):
    """Half-split pairing: (1) equals the interleaved rotation after moving
    element j to 2j and j + d/2 to 2j + 1 (and back); (2) pair j = 1 of
    head_dim 8 at pos 3 rotates elements 1 and 5 by 0.3 rad, nothing else
    moves; (3) pair norms are preserved and rope_inv undoes it; (4) the
    pairing name is checked."""
    r = RNG(13)
    d, theta = 8, 10000.0
    v = r.standard_normal((4, 3, d))
    pos = np.array([0, 1, 5, 17])
    perm = np.empty(d, dtype=int)                 # interleaved position of each half-split element
    perm[: d // 2] = 2 * np.arange(d // 2)
    perm[d // 2:] = 2 * np.arange(d // 2) + 1
    vi = np.empty_like(v)
    vi[..., perm] = v
    w = o.rope(v, pos, theta, "half")
    e = [_rel(w, o.rope(vi, pos, theta)[..., perm])]
    unit = np.zeros((1, 1, d))
    unit[0, 0, 1] = 1.0
    w1 = o.rope(unit, [3], theta, "half")[0, 0]
    e.append(abs(w1[1] - math.cos(0.3)) + abs(w1[5] - math.sin(0.3)) + np.abs(np.delete(w1, [1, 5])).sum())
    e.append(_rel(np.hypot(w[..., : d // 2], w[..., d // 2:]), np.hypot(v[..., : d // 2], v[..., d // 2:])))
    e.append(_rel(o.rope_inv(w, pos, theta, "half"), v))
    try:
        o.rope(v, pos, theta, "other")
        e.append(1.0)
    except ValueError:
        pass
    return max(e)


def check_qknorm_closed_form(o):
    """gamma = 1 and pos = 0: each head of the output has mean square
    ms / (ms + eps) where ms is the head's input mean square."""
    r = RNG(11)
    q = r.standard_normal((3, 4, 8)) * 0.01
    eps = 1e-4
    out = o.qk_rmsnorm_rope_fwd(q, np.ones(8), np.zeros(3), 500000.0, eps)
    ms = np.mean(q * q, axis=-1)
    return _rel(np.mean(out * out, axis=-1), ms / (ms + eps))


def check_qknorm_grad(o, pairing="interleaved"):
    r = RNG(12)
    q = r.standard_normal((3, 2, 8))
    g = 1 + 0.1 * r.standard_normal(8)
    pos = np.array([0, 7, 300])
    dout = r.standard_normal(q.shape)
    dq, dg = o.qk_rmsnorm_rope_bwd(q, g, pos, 500000.0, 1e-6, dout, pairing)

    def L():
        return float((dout * o.qk_rmsnorm_rope_fwd(q, g, pos, 500000.0, 1e-6, pairing)).sum())
    return max(_rel(dq, _fd_grad(L, q)), _rel(dg, _fd_grad(L, g)))


# ---------------------------------------------------------------------------
# linear + cross-entropy
# ---------------------------------------------------------------------------

def check_ce_uniform(o):
    """All-equal logits (W = 0) give loss = ln V exactly; V = 128256 is the
    unembedding size of the linear-CE workload."""
    V = 128256
    X = np.ones((2, 4))
    W = np.zeros((V, 4))
    f = o.linear_cross_entropy_fwd(X, W, np.array([0, V - 1]))
    return max(abs(f["loss"] - math.log(V)) / math.log(V), _rel(f["lse"], [math.log(V)] * 2),
               abs(math.log(V) - 11.761783545564427))


def check_ce_library(o):
    """Against torch cross_entropy(ignore_index=-100) in float64; one dominant
    logit gives loss -> 0; gradient rows sum to zero; ignored rows have zero
    gradient; n_valid is an exact count; FD gradients of the mean loss, and
    of dloss times it for an upstream gradient dloss = -1.75."""
    r = RNG(13)
    M, K, V = 6, 5, 11
    X = r.standard_normal((M, K))
    W = r.standard_normal((V, K))
    lab = np.array([0, 10, -100, 3, -100, 7])
    f = o.linear_cross_entropy_fwd(X, W, lab)
    z = torch.from_numpy(X @ W.T)
    ref = F.cross_entropy(z, torch.from_numpy(lab).long(), ignore_index=-100).item()
    ref_rows = F.cross_entropy(z, torch.from_numpy(lab).long(), ignore_index=-100, reduction="none").numpy()
    e = [abs(f["loss"] - ref) / abs(ref), _rel(f["per_row"], ref_rows), abs(f["n_valid"] - 4),
         _rel(f["lse"], torch.logsumexp(z, dim=1).numpy())]
    b = o.linear_cross_entropy_bwd(X, W, lab)
    e.append(float(np.max(np.abs(b["dZ"].sum(axis=1)))))
    e.append(float(np.max(np.abs(b["dZ"][[2, 4]]))))

    def L():
        return o.linear_cross_entropy_fwd(X, W, lab)["loss"]
    e += [_rel(b["dX"], _fd_grad(L, X)), _rel(b["dW"], _fd_grad(L, W))]
    # an upstream gradient dloss != 1 scales the gradient of the mean loss
    b2 = o.linear_cross_entropy_bwd(X, W, lab, dloss=-1.75)
    e += [_rel(b2["dX"], _fd_grad(lambda: -1.75 * L(), X)), _rel(b2["dW"], _fd_grad(lambda: -1.75 * L(), W))]
    Wd = np.zeros((V, K))
    Wd[3] = 100.0
    Xd = np.ones((1, K))
    e.append(o.linear_cross_entropy_fwd(Xd, Wd, np.array([3]))["loss"])
    return max(e)


def check_ce_lse_merge(o):
    """Per-chunk (max, sum-exp) states over any split of the vocabulary,
    merged as m = max_c m_c, s = sum_c s_c exp(m_c - m), give the full-row
    lse = m + log s of the oracle: the state the online-LSE epilogue carries
    and its combine pass merges."""
    r = RNG(16)
    M, K, V = 4, 6, 23
    X = r.standard_normal((M, K)) * 3
    W = r.standard_normal((V, K))
    lab = np.array([0, 5, 22, 11])
    full = o.linear_cross_entropy_fwd(X, W, lab)["lse"]
    e = []
    for cuts in ([7, 15], [1, 2, 3, 20], [11]):
        m = np.full(M, -np.inf)
        acc = np.zeros(M)
        for lo, hi in zip([0] + cuts, cuts + [V]):
            z = X @ W[lo:hi].T                      # the chunk's logits
            mc = z.max(axis=1)
            sc = np.exp(z - mc[:, None]).sum(axis=1)
            mn = np.maximum(m, mc)
            acc = acc * np.exp(m - mn) + sc * np.exp(mc - mn)
            m = mn
        e.append(_rel(m + np.log(acc), full))
    return max(e)


def check_ce_all_ignored(o):
    """Every row ignored: loss = 0/0 = NaN (torch's mean reduction), zero grad."""
    r = RNG(14)
    X = r.standard_normal((3, 4))
    W = r.standard_normal((7, 4))
    lab = np.array([-100, -100, -100])
    f = o.linear_cross_entropy_fwd(X, W, lab)
    b = o.linear_cross_entropy_bwd(X, W, lab)
    ok = math.isnan(f["loss"]) and f["n_valid"] == 0 and not np.any(b["dX"]) and not np.any(b["dW"])
    return 0.0 if ok else 1.0


def check_ce_bad_labels(o):
    """Labels outside [0, V) other than -100 (a negative one and two at or
    above V) count as ignored and raise the range flag: loss, per-row loss
    and n_valid equal torch cross_entropy(ignore_index=-100) on the labels
    with the bad ones replaced by -100; the gradient equals finite
    differences of that loss and is zero on the bad rows; the flag is off
    when every label is valid or ignored."""
    r = RNG(17)
    M, K, V = 7, 5, 9
    X = r.standard_normal((M, K))
    W = r.standard_normal((V, K))
    lab = np.array([2, -5, V, -100, 0, V + 3, V - 1])
    clean = np.where((lab >= 0) & (lab < V), lab, -100)
    f = o.linear_cross_entropy_fwd(X, W, lab)
    z = torch.from_numpy(X @ W.T)
    ref = F.cross_entropy(z, torch.from_numpy(clean).long(), ignore_index=-100).item()
    ref_rows = F.cross_entropy(z, torch.from_numpy(clean).long(), ignore_index=-100, reduction="none").numpy()
    e = [abs(f["loss"] - ref) / abs(ref), _rel(f["per_row"], ref_rows), abs(f["n_valid"] - 3),
         0.0 if f["label_range_error"] is True else 1.0]
    b = o.linear_cross_entropy_bwd(X, W, lab)
    e.append(float(np.max(np.abs(b["dZ"][[1, 2, 3, 5]]))))

    def L():
        return o.linear_cross_entropy_fwd(X, W, lab)["loss"]
    e += [_rel(b["dX"], _fd_grad(L, X)), _rel(b["dW"], _fd_grad(L, W))]
    e.append(0.0 if o.linear_cross_entropy_fwd(X, W, clean)["label_range_error"] is False else 1.0)
    return max(e)


def check_ce_dw_rows(o):
    """dW restricted to a few vocabulary rows equals those rows of finite
    differences of the mean loss in W (the softmax still normalises over
    the whole vocabulary), also when the rows are summed over token blocks
    with dloss = the block's valid count / the total valid count."""
    r = RNG(18)
    M, K, V = 8, 4, 13
    X = r.standard_normal((M, K))
    W = r.standard_normal((V, K))
    lab = np.array([0, 12, -100, 5, 5, 7, -100, 12])
    ids = np.array([0, 5, 9, 12])

    def L():
        return o.linear_cross_entropy_fwd(X, W, lab)["loss"]
    fd = _fd_grad(L, W)[ids]
    e = [_rel(o.linear_cross_entropy_bwd(X, W, lab, vocab_rows=ids)["dW_rows"], fd)]
    nv = int((lab != -100).sum())
    acc = np.zeros((len(ids), K))
    for lo, hi in ((0, 3), (3, 8)):
        lb = lab[lo:hi]
        acc += o.linear_cross_entropy_bwd(X[lo:hi], W, lb, dloss=int((lb != -100).sum()) / nv,
                                          vocab_rows=ids)["dW_rows"]
    e.append(_rel(acc, fd))
    return max(e)


# ---------------------------------------------------------------------------
# the block
# ---------------------------------------------------------------------------

def tiny_block(seed=15, n_q=2, n_kv=1, d=4, h=8, inter=6, tokens=3):
    r = RNG(seed)
    qkv = (n_q + 2 * n_kv) * d
    p = {
        "x0": r.standard_normal((tokens, h)), "Wqkv": r.standard_normal((qkv, h)) * 0.5,
        "Wo": r.standard_normal((h, n_q * d)) * 0.5, "Wg": r.standard_normal((inter, h)) * 0.5,
        "Wu": r.standard_normal((inter, h)) * 0.5, "Wd": r.standard_normal((h, inter)) * 0.5,
        "gamma_attn": 1 + 0.1 * r.standard_normal(h), "gamma_mlp": 1 + 0.1 * r.standard_normal(h),
        "gamma_q": 1 + 0.1 * r.standard_normal(d), "gamma_k": 1 + 0.1 * r.standard_normal(d),
        "A": r.standard_normal((tokens, n_q * d)), "dx2": r.standard_normal((tokens, h)),
        "dQ": r.standard_normal((tokens, n_q * d)), "dK": r.standard_normal((tokens, n_kv * d)),
        "dV": r.standard_normal((tokens, n_kv * d)), "pos": np.arange(tokens) * 5 + 1,
    }
    return p, dict(n_q=n_q, n_kv=n_kv, head_dim=d, theta=10000.0, eps=1e-6)


def check_block_special_cases(o):
    """Structure of the block ([P1] §3.2.1 sites 1 and 2): with Wd = 0 the
    output is x0 + A Wo^T (torch linear); with A = 0 the MLP sees x0 and
    x2 - x0 equals the MLP branch computed from torch rms_norm/linear/silu;
    V is the plain projection of RMSNorm(x0); with gamma_q = 1 and pos = 0
    every Q head has mean square ms/(ms+eps); Q and K are RoPE of the q and
    k slices normalised per head by torch rms_norm with their own gains."""
    p, cfg = tiny_block()
    e = []
    q = dict(p)
    q["Wd"] = np.zeros_like(p["Wd"])
    f = o.block_fwd(q, **cfg)
    ref = p["x0"] + F.linear(torch.from_numpy(p["A"]), torch.from_numpy(p["Wo"])).numpy()
    e.append(_rel(f["x2"], ref))
    e.append(_rel(f["x1"], ref))
    q = dict(p)
    q["A"] = np.zeros_like(p["A"])
    f = o.block_fwd(q, **cfg)
    t = torch.from_numpy
    a1 = F.rms_norm(t(p["x0"]), (8,), weight=t(p["gamma_mlp"]), eps=cfg["eps"])
    br = F.linear(F.silu(F.linear(a1, t(p["Wg"]))) * F.linear(a1, t(p["Wu"])), t(p["Wd"])).numpy()
    e.append(_rel(f["x2"] - p["x0"], br))
    a0 = F.rms_norm(t(p["x0"]), (8,), weight=t(p["gamma_attn"]), eps=cfg["eps"])
    qkv = F.linear(a0, t(p["Wqkv"])).numpy()
    e.append(_rel(f["V"], qkv[:, 12:]))
    q = dict(p)
    q["gamma_q"] = np.ones(4)
    q["pos"] = np.zeros(3, dtype=np.int64)
    f = o.block_fwd(q, **cfg)
    qh = qkv[:, :8].reshape(3, 2, 4)
    ms = np.mean(qh ** 2, axis=-1)
    e.append(_rel(np.mean(f["Q"].reshape(3, 2, 4) ** 2, axis=-1), ms / (ms + cfg["eps"])))
    # Q and K at general gains and positions: the q and k column slices of
    # the projection, each head normalised by torch rms_norm with its own
    # gain (gamma_q for Q, gamma_k for K), then the (separately pinned) RoPE
    f = o.block_fwd(p, **cfg)
    for name, cols, heads, gain in (("Q", slice(0, 8), 2, "gamma_q"), ("K", slice(8, 12), 1, "gamma_k")):
        hn = F.rms_norm(t(qkv[:, cols].reshape(3, heads, 4)), (4,), weight=t(p[gain]), eps=cfg["eps"]).numpy()
        ref = o.rope(hn, p["pos"], cfg["theta"]).reshape(3, -1)
        e.append(_rel(f[name], ref))
    return max(e)


def check_block_grad(o):
    """FD gradients of L = <dx2, x2> + <dQ, Q> + <dK, K> + <dV, V>."""
    p, cfg = tiny_block()
    b = o.block_bwd(p, **cfg)

    def L():
        f = o.block_fwd(p, **cfg)
        return float((p["dx2"] * f["x2"]).sum() + (p["dQ"] * f["Q"]).sum()
                     + (p["dK"] * f["K"]).sum() + (p["dV"] * f["V"]).sum())
    pairs = [("dx0", "x0"), ("dA", "A"), ("dWqkv", "Wqkv"), ("dWo", "Wo"), ("dWg", "Wg"),
             ("dWu", "Wu"), ("dWd", "Wd"), ("dgamma_attn", "gamma_attn"),
             ("dgamma_mlp", "gamma_mlp"), ("dgamma_q", "gamma_q"), ("dgamma_k", "gamma_k")]
    return max(_rel(b[g], _fd_grad(L, p[x])) for g, x in pairs)


def check_gemm_epilogue_bruteforce(o):
    """Triple loop over (i, j, k) in plain Python on a tiny problem."""
    r = RNG(16)
    M, N, K = 3, 4, 5
    A, B = r.standard_normal((M, K)), r.standard_normal((N, K))
    rs, cs = r.standard_normal(M), r.standard_normal(N)
    a0, a1, d0 = r.standard_normal((M, N)), r.standard_normal((M, N)), r.standard_normal((M, N))
    coef = r.standard_normal(M)
    got = o.gemm_epilogue_plain(A, B, rs, cs, a0, coef, a1, d0)
    ref = np.zeros((M, N))
    for i in range(M):
        for j in range(N):
            acc = 0.0
            for k in range(K):
                acc += A[i, k] * B[j, k]
            ref[i, j] = rs[i] * cs[j] * acc + a0[i, j] - coef[i] * a1[i, j] + d0[i, j]
    plain = o.gemm_epilogue_plain(A, B)
    ref2 = np.array([[sum(A[i, k] * B[j, k] for k in range(K)) for j in range(N)] for i in range(M)])
    return max(_rel(got, ref), _rel(plain, ref2))


def check_rmsnorm_ce_library(o):
    """gamma = 1: the loss equals torch's cross_entropy of torch rms_norm's
    output times W^T (float64), ignore_index = -100."""
    r = RNG(17)
    X = r.standard_normal((5, 8)) * 2
    W = r.standard_normal((9, 8))
    lab = np.array([0, 8, -100, 4, 2])
    f = o.rmsnorm_linear_cross_entropy_fwd(X, np.ones(8), W, lab, 1e-6)
    a = F.rms_norm(torch.from_numpy(X), (8,), eps=1e-6)
    ref = F.cross_entropy(F.linear(a, torch.from_numpy(W)), torch.from_numpy(lab).long(), ignore_index=-100).item()
    return max(abs(f["loss"] - ref) / abs(ref), _rel(f["rstd"], 1 / np.sqrt((X ** 2).mean(axis=1) + 1e-6)))


def check_rmsnorm_ce_grad(o):
    """FD gradients of dloss times the mean loss (dloss = 0.6, the upstream
    gradient) w.r.t. X, W and gamma."""
    r = RNG(18)
    X = r.standard_normal((4, 6))
    W = r.standard_normal((7, 6))
    g = 1 + 0.1 * r.standard_normal(6)
    lab = np.array([1, -100, 6, 0])
    b = o.rmsnorm_linear_cross_entropy_bwd(X, g, W, lab, 1e-6, dloss=0.6)

    def L():
        return 0.6 * o.rmsnorm_linear_cross_entropy_fwd(X, g, W, lab, 1e-6)["loss"]
    return max(_rel(b["dX"], _fd_grad(L, X)), _rel(b["dW"], _fd_grad(L, W)), _rel(b["dgamma"], _fd_grad(L, g)))


def check_linear_sigmoid(o):
    """sigmoid(0) = 1/2, sigmoid(a) + sigmoid(-a) = 1, vs torch sigmoid/linear
    in float64, and FD gradients (with and without the gated tensor)."""
    r = RNG(19)
    X = r.standard_normal((4, 6))
    W = r.standard_normal((5, 6))
    Z = r.standard_normal((4, 5))
    dY = r.standard_normal((4, 5))
    a = np.linspace(-6, 6, 13)
    e = [abs(o.sigmoid(0.0) - 0.5), float(np.max(np.abs(o.sigmoid(a) + o.sigmoid(-a) - 1.0)))]
    ref = torch.sigmoid(F.linear(torch.from_numpy(X), torch.from_numpy(W))).numpy()
    e += [_rel(o.linear_sigmoid_fwd(X, W), ref), _rel(o.linear_sigmoid_fwd(X, W, Z), ref * Z)]
    for gated in (False, True):
        zz = Z if gated else None
        b = o.linear_sigmoid_bwd(X, W, dY, zz)

        def L():
            return float((dY * o.linear_sigmoid_fwd(X, W, zz)).sum())
        e += [_rel(b["dX"], _fd_grad(L, X)), _rel(b["dW"], _fd_grad(L, W))]
        if gated:
            e.append(_rel(b["dZ"], _fd_grad(L, Z)))
    return max(e)


def _e4m3_table():
    """All finite e4m3 codes and their values, decoded from the format's
    definition (1 sign, 4 exponent bits with bias 7, 3 mantissa bits,
    subnormals at exponent 0, code 0x7f / 0xff = NaN)."""
    codes, vals = [], []
    for c in range(256):
        if c & 0x7F == 0x7F:
            continue
        sgn = -1.0 if c & 0x80 else 1.0
        e, m = (c >> 3) & 0xF, c & 0x7
        v = (m / 8.0) * 2.0 ** -6 if e == 0 else (1 + m / 8.0) * 2.0 ** (e - 7)
        codes.append(c)
        vals.append(sgn * v)
    return np.array(codes, dtype=np.uint8), np.array(vals)


def check_fp8_quantizer(o):
    """(1) every finite e4m3 value, in a row whose max is 448 (scale 1),
    quantises to its own code; (2) |q s - x| <= 2^-4 |x| in the normal range
    and <= 2^-10 s below it; (3) each row's max maps to +-448 exactly;
    (4) a zero row gives zero codes and scale 1; (5) monotone."""
    codes, vals = _e4m3_table()
    row = np.concatenate([vals, [448.0]])[None, :]
    qc, qv, sc = o.quantize_fp8_rows(row)
    e = [float(np.any(qc[0, :-1] != codes)), abs(float(sc[0]) - 1.0), _rel(qv[0, :-1], vals)]
    r = RNG(20)
    X = r.standard_normal((6, 300)) * np.array([1e-3, 1, 30, 1e4, 0.5, 7])[:, None]
    qc, qv, sc = o.quantize_fp8_rows(X)
    deq = qv * sc[:, None].astype(np.float64)
    ax = np.abs(X)
    normal = ax / sc[:, None] >= 2.0 ** -6
    err = np.abs(deq - X)
    rel_normal = float(np.max(np.where(normal, err / np.maximum(ax, 1e-300), 0.0)))
    abs_sub = float(np.max(np.where(normal, 0.0, err / sc[:, None])))
    e.append(0.0 if rel_normal <= 2.0 ** -4 * (1 + 1e-6) else 1.0)   # half an ulp of a 3-bit mantissa
    e.append(0.0 if abs_sub <= 2.0 ** -10 * (1 + 1e-6) else 1.0)     # half the subnormal spacing 2^-9
    e.append(float(np.max(np.abs(np.abs(qv).max(axis=1) - 448.0))))
    qc0, qv0, sc0 = o.quantize_fp8_rows(np.zeros((1, 5)))
    e.append(float(np.any(qv0 != 0)) + abs(float(sc0[0]) - 1.0))
    xs = np.sort(r.standard_normal(500))[None, :]
    e.append(float(np.any(np.diff(o.quantize_fp8_rows(xs)[1][0]) < 0)))
    return max(e)


def check_fp8_linear(o):
    """With operands already e4m3 values and row maxima 448 (scales 1), the
    FP8 linear and SwiGLU equal the bf16 definitions exactly."""
    codes, vals = _e4m3_table()
    r = RNG(21)
    pick = lambda shape: vals[r.integers(0, len(vals), size=shape)] * (2.0 ** -6)
    X = pick((4, 16))
    Wg, Wu = pick((6, 16)), pick((6, 16))
    X[:, 0], Wg[:, 0], Wu[:, 0] = 448.0 * 2.0 ** -6, 448.0 * 2.0 ** -6, 448.0 * 2.0 ** -6
    _, xv, sx = o.quantize_fp8_rows(X)
    _, gv, sg = o.quantize_fp8_rows(Wg)
    _, uv, su = o.quantize_fp8_rows(Wu)
    H, g, u = o.swiglu_fp8_fwd(xv, sx, gv, sg, uv, su)
    H0, g0, u0 = o.swiglu_fwd(X, Wg, Wu)
    y = o.linear_fp8_fwd(xv, sx, gv, sg)
    return max(_rel(H, H0), _rel(g, g0), _rel(u, u0), _rel(y, X @ Wg.T))


def check_fp8_cols_quantizer(o):
    """The column quantiser is the row quantiser of the transpose, bit for
    bit (codes, values, scales), and each column's maximum maps to +-448."""
    r = RNG(24)
    X = r.standard_normal((37, 24)) * np.array([1e-3, 1, 30, 1e4] * 6)[None, :]
    X[:, 5] = 0.0
    qc, qv, sc = o.quantize_fp8_cols(X)
    rc, rv, rs = o.quantize_fp8_rows(np.ascontiguousarray(X.T))
    e = [float(np.any(qc != rc)), float(np.any(sc != rs)), float(np.max(np.abs(qv - rv)))]
    nz = np.abs(X).max(axis=0) > 0
    e.append(float(np.max(np.abs(np.abs(qv[nz]).max(axis=1) - 448.0))))
    return max(e)


def _e4m3_exact(r, shape, vals):
    """Exact e4m3 values times 2^-6 with one 448 * 2^-6 per row, so that the
    row quantiser's scale is exactly 2^-6 and every code is exact."""
    X = vals[r.integers(0, len(vals), size=shape)] * (2.0 ** -6)
    X[:, 0] = 448.0 * 2.0 ** -6
    return X


def check_fp8_epilogue_ops(o):
    """With exact e4m3 operands, the FP8 operators equal the bf16 definitions:
    QKV + QK-norm + RoPE equals qk_rmsnorm_rope_fwd of the projection heads;
    the cross-entropy forward equals torch cross_entropy and the backward
    equals linear_cross_entropy_bwd (dX, dW with the same operands); the
    dSwiGLU map equals mlp_bwd's dg, du (and G' carries the row factor), and
    its row dot equals r dL/dr by finite differences; the RMSNorm input
    gradient equals rmsnorm_linear_bwd's dX and dgamma."""
    codes, vals = _e4m3_table()
    vals = vals[np.abs(vals) <= 448.0]
    r = RNG(25)
    e = []
    # QKV + QK-norm + RoPE (2 q heads, 1 kv head of 8)
    d, n_q, n_kv, M, K = 8, 2, 1, 3, 16
    X = _e4m3_exact(r, (M, K), vals)
    W = _e4m3_exact(r, ((n_q + 2 * n_kv) * d, K), vals)
    _, xv, sx = o.quantize_fp8_rows(X)
    _, wv, sw = o.quantize_fp8_rows(W)
    gq, gk = 1 + 0.1 * r.standard_normal(d), 1 + 0.1 * r.standard_normal(d)
    pos, rs = np.array([0, 5, 9]), np.array([0.5, 2.0, 1.25])
    f = o.linear_qknorm_rope_fp8_fwd(xv, sx, wv, sw, gq, gk, pos, 1e4, 1e-6, n_q, n_kv, d, row_scale=rs)
    qkv = (X @ W.T) * rs[:, None]
    Qr = o.qk_rmsnorm_rope_fwd(qkv[:, : n_q * d].reshape(M, n_q, d), gq, pos, 1e4, 1e-6).reshape(M, -1)
    Kr = o.qk_rmsnorm_rope_fwd(qkv[:, n_q * d: (n_q + n_kv) * d].reshape(M, n_kv, d), gk, pos, 1e4,
                               1e-6).reshape(M, -1)
    e += [_rel(f["Q"], Qr), _rel(f["K"], Kr), _rel(f["V"], qkv[:, (n_q + n_kv) * d:])]
    # cross-entropy forward and backward
    M, K, V = 5, 16, 9
    X = _e4m3_exact(r, (M, K), vals)
    W = _e4m3_exact(r, (V, K), vals)
    lab = np.array([0, 8, -100, 3, 3])
    _, xv, sx = o.quantize_fp8_rows(X)
    _, wv, sw = o.quantize_fp8_rows(W)
    fce = o.linear_cross_entropy_fp8_fwd(xv, sx, wv, sw, lab)
    ref = F.cross_entropy(torch.from_numpy(X @ W.T), torch.from_numpy(lab).long(), ignore_index=-100).item()
    e.append(abs(fce["loss"] - ref) / abs(ref))
    bce = o.linear_cross_entropy_fp8_bwd(xv, sx, wv, sw, X, W, lab, dloss=0.7)
    b0 = o.linear_cross_entropy_bwd(X, W, lab, dloss=0.7)
    e += [_rel(bce["dX"], b0["dX"]), _rel(bce["dW"], b0["dW"])]
    # dSwiGLU on the dH GEMM
    M, Hd, I = 3, 16, 6
    X = r.standard_normal((M, Hd))
    Wg, Wu = r.standard_normal((I, Hd)) * 0.4, r.standard_normal((I, Hd)) * 0.4
    Wd = _e4m3_exact(r, (I, Hd), vals).T.copy()          # Wd [Hd, I]; its transpose exact per unit row
    dY = _e4m3_exact(r, (M, Hd), vals)
    fm = o.mlp_fwd(X, Wg, Wu, Wd, np.zeros((M, Hd)))
    _, dyv, sdy = o.quantize_fp8_rows(dY)
    _, wdv, swd = o.quantize_fp8_rows(np.ascontiguousarray(Wd.T))
    rr = np.array([0.5, 1.0, 3.0])
    ds = o.dswiglu_fp8(dyv, sdy, wdv, swd, fm["g"], fm["u"], row_scale=rr)
    mb = o.mlp_bwd(X, Wg, Wu, Wd, dY)
    e += [_rel(ds["Gp"][:, :I], mb["dg"] * rr[:, None]), _rel(ds["Gp"][:, I:], mb["du"] * rr[:, None]),
          _rel(ds["H"], fm["H"])]

    def L(t):
        return float((dY * o.mlp_fwd(t * X, Wg, Wu, Wd, np.zeros((M, Hd)))["y"]).sum(axis=1)[i_row])
    h = 1e-6
    for i_row in range(M):
        e.append(abs((L(1 + h) - L(1 - h)) / (2 * h) - ds["dot"][i_row]) / max(abs(ds["dot"][i_row]), 1e-12))
    # the MLP's input-gradient chain through the input RMSNorm: the dSwiGLU
    # map's coefficient and G' fed to the RMSNorm input gradient (operands
    # given as values with unit scales) equal mlp_bwd's dX and dgamma
    M, Hd, I = 3, 16, 6
    x = r.standard_normal((M, Hd))
    gam = 1 + 0.1 * r.standard_normal(Hd)
    Wg, Wu = r.standard_normal((I, Hd)) * 0.4, r.standard_normal((I, Hd)) * 0.4
    Wd, dY = r.standard_normal((Hd, I)) * 0.3, r.standard_normal((M, Hd))
    fm = o.mlp_fwd(x, Wg, Wu, Wd, np.zeros((M, Hd)), gam, 1e-6)
    rx = o.rms_inv(x, 1e-6)
    ds = o.dswiglu_fp8(dY, np.ones(M), Wd.T, np.ones(I), fm["g"], fm["u"], row_scale=rx)
    dxr = o.rmsnorm_linear_dx_fp8(ds["Gp"], np.ones(M), np.hstack([Wg.T, Wu.T]), np.ones(Hd), x, gam, ds["coef"])
    mb = o.mlp_bwd(x, Wg, Wu, Wd, dY, gam, 1e-6)
    e += [_rel(dxr["dX"], mb["dX"]), _rel(dxr["dgamma"], mb["dgamma"])]
    # RMSNorm-reparameterised input gradient
    M, K, N = 4, 16, 8
    X = r.standard_normal((M, K))
    gam = 1 + 0.1 * r.standard_normal(K)
    W = _e4m3_exact(r, (K, N), vals).T.copy()              # W [N, K]; W^T [K, N] exact per row
    Gp = _e4m3_exact(r, (M, N), vals)                       # G' = r G, exact
    rstd = o.rms_inv(X, 1e-6)
    G = Gp / rstd[:, None]
    y, _ = o.rmsnorm_linear_fwd(X, gam, W, 1e-6)
    coef = rstd ** 2 * (G * y).sum(axis=1) / K
    _, gv, sg = o.quantize_fp8_rows(Gp)
    _, wtv, swt = o.quantize_fp8_rows(np.ascontiguousarray(W.T))
    dx = o.rmsnorm_linear_dx_fp8(gv, sg, wtv, swt, X, gam, coef)
    b = o.rmsnorm_linear_bwd(X, gam, W, 1e-6, G)
    e += [_rel(dx["dX"], b["dX"]), _rel(dx["dgamma"], b["dgamma"])]
    return max(e)


def _bf16_t(x):
    """bf16 rounding through torch (nearest even), as float64."""
    return torch.from_numpy(np.asarray(x, dtype=np.float64)).to(torch.bfloat16).double().numpy()


def check_fp8_qkv_bwd(o):
    """The QKV + QK-norm + RoPE backward on e4m3 operands.
    (1) dQ = dK = 0 and operands every quantiser takes exactly: token rows
    X_i = +-1/r_i with r = (1, 1/2, 1/4), so that at eps = 0 the input
    RMSNorm factor is exactly r_i and the columns of U = X ⊙ gamma are
    exact; W^T rows exact; dV of e4m3 values of magnitude >= 2^-4 (or 0)
    times 2^-6 with 448 * 2^-6 on its first row and column, so that
    G' = r ⊙ [0 | 0 | dV] is exact per row and per column.  Then dX, dW and
    dgamma_in equal rmsnorm_linear_bwd (G = [0 | 0 | dV]); without the input
    RMSNorm, dX = G W + dX_resid and dW = G^T X (X column-exact).
    (2) General dQ, dK, dV (QK eps 0.5, so the q and k terms of c count):
    G' equals r ⊙ block_bwd's dqkv rounded to bf16; dgamma_q and dgamma_k
    equal block_bwd's; c_i equals r_i^2 dL/dt / K for L(t) = <dQ, Q> +
    <dK, K> + <dV, V> at token i's projection scaled by t (finite
    differences); and D = G'_q W, dW = G'^T_q U lie within the e4m3
    rounding bound of G' (half a step: 2^-4 |g| in the normal range,
    2^-10 s below it, s the scale of g's row of G' or G'^T) around G' W and
    G'^T U, row by row, with one token's gradients 10^-6 of the others' (the
    other axis's scales would flush them to zero)."""
    codes, vals = _e4m3_table()
    vals = vals[(np.abs(vals) <= 448.0) & ((np.abs(vals) >= 2.0 ** -4) | (vals == 0))]
    rg = RNG(27)
    p, cfg = tiny_block(seed=16)
    n_q, n_kv, d, theta = cfg["n_q"], cfg["n_kv"], cfg["head_dim"], cfg["theta"]
    M, h = p["x0"].shape
    nqk, N = (n_q + n_kv) * d, (n_q + 2 * n_kv) * d
    r = np.array([1.0, 0.5, 0.25])
    X = np.where(rg.standard_normal((M, h)) < 0, -1.0, 1.0) / r[:, None]
    gam = p["gamma_attn"]
    W = _e4m3_exact(rg, (h, N), vals).T.copy()
    U = X * gam[None, :]
    _, wtv, sw = o.quantize_fp8_cols(W)
    _, utv, su = o.quantize_fp8_cols(U)
    gq, gk, pos = p["gamma_q"], p["gamma_k"], p["pos"]
    e = []
    # (1) exact operands
    y = o.rmsnorm(X, gam, 0.0) @ W.T
    dV = vals[rg.integers(0, len(vals), size=(M, n_kv * d))] * 2.0 ** -6
    dV[0, :] = np.where(rg.standard_normal(n_kv * d) < 0, -448.0, 448.0) * 2.0 ** -6
    dV[:, 0] = 448.0 * 2.0 ** -6
    zq, zk = np.zeros((M, n_q * d)), np.zeros((M, n_kv * d))
    G = np.hstack([zq, zk, dV])
    out = o.linear_qknorm_rope_fp8_bwd(zq, zk, dV, y[:, :nqk], y[:, nqk:], gq, gk, pos, theta, 1e-6, n_q, n_kv, d,
                                       wtv, sw, utv, su, X=X, row_scale=r, gamma_in=gam)
    b = o.rmsnorm_linear_bwd(X, gam, W, 0.0, G)
    e += [_rel(out["dX"], b["dX"]), _rel(out["dW"], b["dW"]), _rel(out["dgamma_in"], b["dgamma"])]
    X2 = _e4m3_exact(rg, (h, M), vals).T.copy()
    _, xtv, sx = o.quantize_fp8_cols(X2)
    R = rg.standard_normal((M, h))
    out = o.linear_qknorm_rope_fp8_bwd(zq, zk, dV, y[:, :nqk], y[:, nqk:], gq, gk, pos, theta, 1e-6, n_q, n_kv, d,
                                       wtv, sw, xtv, sx, dX_resid=R)
    e += [_rel(out["dX"], G @ W + R), _rel(out["dW"], G.T @ X2)]
    # (2) general gradients
    eps = 0.5
    rr = o.rms_inv(X, eps)
    y = o.rmsnorm(X, gam, eps) @ W.T
    # token 2's gradients 1e-6 of the others': quantised with the other
    # tokens' scale (per column) they would underflow, outside the bound
    tiny = np.array([1.0, 1.0, 1e-6])[:, None]
    dQ, dK, dV = p["dQ"] * tiny, p["dK"] * tiny, p["dV"] * tiny
    out = o.linear_qknorm_rope_fp8_bwd(dQ, dK, dV, y[:, :nqk], y[:, nqk:], gq, gk, pos, theta, eps, n_q, n_kv, d,
                                       wtv, sw, utv, su, X=X, row_scale=rr, gamma_in=gam)
    bb = o.block_bwd(dict(p, x0=X, Wqkv=W, gamma_attn=gam, dQ=dQ, dK=dK, dV=dV), n_q, n_kv, d, theta, eps)
    Gp = _bf16_t(bb["dqkv"] * rr[:, None])
    e += [_rel(out["Gp"], Gp), _rel(out["dgamma_q"], bb["dgamma_q"]), _rel(out["dgamma_k"], bb["dgamma_k"])]

    def L(i, t):
        yt = y.copy()
        yt[i] *= t
        Q = o.qk_rmsnorm_rope_fwd(yt[:, : n_q * d].reshape(M, n_q, d), gq, pos, theta, eps).reshape(M, -1)
        K = o.qk_rmsnorm_rope_fwd(yt[:, n_q * d: nqk].reshape(M, n_kv, d), gk, pos, theta, eps).reshape(M, -1)
        return float((dQ * Q).sum() + (dK * K).sum() + (dV * yt[:, nqk:]).sum())
    fd = np.array([(L(i, 1 + 1e-6) - L(i, 1 - 1e-6)) / 2e-6 for i in range(M)])
    e.append(_rel(out["coef"], rr ** 2 * fd / h))
    for got, A, B in ((out["D"], Gp, W), (out["dW"], Gp.T, U)):   # got ~ A B, A quantised per row
        s = np.abs(A).max(axis=1) / 448.0
        bound = (2.0 ** -4 * np.abs(A) + 2.0 ** -10 * s[:, None]) @ np.abs(B) * (1 + 1e-6)
        ex = np.maximum(np.abs(got - A @ B) - bound, 0.0).max(axis=1) / np.abs(A @ B).max(axis=1)
        e.append(float(ex.max()))
    return max(e)


def _e2m1_decode_table():
    """The 16 e2m1 codes decoded from the format's definition: bit 3 sign,
    bits 1-2 exponent with bias 1, bit 0 mantissa; exponent 0 is subnormal
    (mantissa x 0.5)."""
    out = []
    for c in range(16):
        sgn = -1.0 if c & 8 else 1.0
        e, m = (c >> 1) & 3, c & 1
        out.append(sgn * (m * 0.5 if e == 0 else (1 + m / 2.0) * 2.0 ** (e - 1)))
    return np.array(out)


def _e2m1_nearest_even(v):
    """Round to the e2m1 grid binade by binade: spacing 0.5 below 2, 1 in
    [2, 4), 2 in [4, 6]; np.round rounds halves to even multiples, which
    are the even codes; saturate at 6."""
    a = np.abs(np.asarray(v, dtype=np.float64))
    sp = np.where(a < 2, 0.5, np.where(a < 4, 1.0, 2.0))
    return np.sign(v) * np.minimum(np.round(a / sp) * sp, 6.0)


def check_e2m1(o):
    """(1) the oracle's decode of every code equals the format definition;
    (2) rounding equals the binade-wise nearest-even reference on random
    values and on every tie point, with saturation at +-6 and no negative
    zero codes."""
    e = [_rel(o.e2m1_value(np.arange(16)), _e2m1_decode_table())]
    r = RNG(30)
    ties = np.array([0.25, 0.75, 1.25, 1.75, 2.5, 3.5, 5.0])
    v = np.concatenate([r.uniform(-8, 8, 4000), ties, -ties, [0.0, 6.0, -6.0, 7.5, -1e9, 1e-9, -1e-9]])
    v = v.astype(np.float32)
    c = o.e2m1_round(v)
    e.append(float(np.max(np.abs(o.e2m1_value(c) - _e2m1_nearest_even(v)))))
    e.append(float(np.any((c & 7) == 0) and np.any(c[(c & 7) == 0] != 0)))
    return max(e)


def _nvfp4_exact_rows(r, rows, nblocks, row_pow2):
    """Rows whose NVFP4 quantisation is exact: each block is grid magnitudes
    (random signs, one entry at 6) times an e4m3 scale; block 0 carries
    6 * 448 so s = 1, times 2^row_pow2[i] per row.  Returns (X, codes,
    sf codes, s)."""
    ecodes, evals = _e4m3_table()
    pos = evals > 0
    ecodes, evals = ecodes[pos], evals[pos]
    grid = _e2m1_decode_table()[:8]
    X = np.zeros((rows, nblocks * 16))
    codes = np.zeros((rows, nblocks * 16), np.uint8)
    sfc = np.zeros((rows, nblocks), np.uint8)
    for i in range(rows):
        for b in range(nblocks):
            j = len(ecodes) - 1 if b == 0 else r.integers(0, len(ecodes))   # 448 in block 0
            idx = r.integers(0, 8, 16)
            idx[r.integers(0, 16)] = 7
            sgn = np.where(r.random(16) < 0.5, 8, 0) * (idx > 0)
            codes[i, b * 16:(b + 1) * 16] = idx | sgn
            X[i, b * 16:(b + 1) * 16] = np.where(sgn, -1.0, 1.0) * grid[idx] * evals[j]
            sfc[i, b] = ecodes[j]
    X *= (2.0 ** np.asarray(row_pow2, dtype=np.float64))[:, None]
    return X, codes, sfc, 2.0 ** np.asarray(row_pow2, dtype=np.float64)


def check_nvfp4_quantizer(o):
    """(1) rows built from grid values and e4m3 scales (s a power of two)
    quantise to exactly those codes, scales and s; (2) s = amax / 2688;
    every block scale is within half an e4m3 ulp of bmax / (6 s) (normal
    range); the largest element of each such block gets magnitude code 7;
    every element is within half a grid step of x / (sf s), times sf s;
    (3) a zero row gives s = 1 and zero scales and codes; (4) a block whose
    scale underflows e4m3 gets zero codes."""
    r = RNG(31)
    X, codes, sfc, s_exp = _nvfp4_exact_rows(r, 5, 6, [0, -6, 3, -20, 10])
    c, sf, s, vals = o.quantize_nvfp4_rows(X)
    e = [float(np.any(c != codes)), float(np.any(sf != sfc)), _rel(s, s_exp),
         _rel(vals * s[:, None], X)]
    Y = (r.standard_normal((6, 256)) * np.array([1e-3, 1, 30, 1e4, 0.5, 7])[:, None]).astype(np.float32)
    Y[2, 16:32] *= 1e-3                                     # a quiet block among loud ones
    c, sf, s, vals = o.quantize_nvfp4_rows(Y)
    amax = np.abs(Y).max(axis=1)
    q = amax.astype(np.float64) / 2688.0                     # s is this quotient rounded to fp32
    e.append(0.0 if np.all(np.abs(s - q) <= 2.0 ** -24 * q) else 1.0)
    ecodes, evals = _e4m3_table()
    lut = np.zeros(256)
    lut[ecodes] = evals
    sfv = lut[sf]
    bmax = np.abs(Y.astype(np.float64)).reshape(6, 16, 16).max(axis=2)
    target = bmax / (6.0 * s.astype(np.float64)[:, None])
    normal = target >= 2.0 ** -6
    e.append(0.0 if np.all(np.abs(sfv - target)[normal] <= 2.0 ** -4 * target[normal] * (1 + 1e-6)) else 1.0)
    mag = (c & 7).reshape(6, 16, 16)
    arg = np.abs(Y).reshape(6, 16, 16).argmax(axis=2)
    top = np.take_along_axis(mag, arg[..., None], axis=2)[..., 0]
    e.append(float(np.any(top[normal] != 7)))
    denom = np.repeat(sfv * s.astype(np.float64)[:, None], 16, axis=1)
    ok = denom > 0
    v = np.abs(Y.astype(np.float64))[ok] / denom[ok]
    half = np.where(v < 2, 0.25, np.where(v < 4, 0.5, 1.0))
    err = np.abs(vals * s[:, None] - Y)[ok]
    e.append(0.0 if np.all(err <= denom[ok] * np.maximum(half, v - 6.0) * (1 + 1e-6)) else 1.0)
    c0, sf0, s0, v0 = o.quantize_nvfp4_rows(np.zeros((1, 32)))
    e.append(float(np.any(c0) or np.any(sf0) or np.any(v0)) + abs(float(s0[0]) - 1.0))
    Z = np.zeros((1, 32), np.float32)
    Z[0, 0] = 2688.0
    Z[0, 16:] = 1e-7                                        # 1e-7 / 6 far below e4m3's 2^-9
    cz, sfz, _, _ = o.quantize_nvfp4_rows(Z)
    e.append(float(sfz[0, 1] != 0 or np.any(cz[0, 16:])))
    return max(e)


def check_nvfp4_linear(o):
    """With exactly representable operands, the NVFP4 linear and SwiGLU
    equal the bf16 definitions exactly."""
    r = RNG(32)
    X, *_ = _nvfp4_exact_rows(r, 4, 2, [-10, -13, -8, -18])
    Wg, *_ = _nvfp4_exact_rows(r, 5, 2, [-11, -10, -12, -11, -13])
    Wu, *_ = _nvfp4_exact_rows(r, 5, 2, [-12, -11, -10, -12, -11])
    _, _, sx, xv = o.quantize_nvfp4_rows(X)
    _, _, sg, gv = o.quantize_nvfp4_rows(Wg)
    _, _, su, uv = o.quantize_nvfp4_rows(Wu)
    H, g, u = o.swiglu_nvfp4_fwd(xv, sx, gv, sg, uv, su)
    H0, g0, u0 = o.swiglu_fwd(X, Wg, Wu)
    y = o.linear_nvfp4_fwd(xv, sx, gv, sg)
    return max(_rel(H, H0), _rel(g, g0), _rel(u, u0), _rel(y, X @ Wg.T))


def check_rmsnorm_scale_nvfp4(o):
    """(1) gamma = 2^k per column block: codes and block scales equal those
    of x alone and the row scales carry the factor exactly (products by a
    power of two are exact); (2) r is the RMSNorm of x, not of x ⊙ gamma,
    written out here: 1 / sqrt(mean(x^2) + eps)."""
    r = RNG(33)
    X = (r.standard_normal((5, 64)) * np.array([1e-2, 1, 3, 50, 0.2])[:, None]).astype(np.float32)
    e = []
    for k in (-3, 0, 5):
        g = np.full(64, 2.0 ** k)
        c, sf, s, v, rr = o.rmsnorm_scale_nvfp4(X, g, 1e-6)
        c0, sf0, s0, v0 = o.quantize_nvfp4_rows(X)
        e += [float(np.any(c != c0)), float(np.any(sf != sf0)), _rel(s, s0 * 2.0 ** k)]
    g = 1 + 0.3 * r.standard_normal(64)
    *_, rr = o.rmsnorm_scale_nvfp4(X, g, 1e-6)
    x64 = X.astype(np.float64)
    e.append(_rel(rr, 1.0 / np.sqrt((x64 * x64).mean(axis=1) + 1e-6)))
    return max(e)


def check_quantised_swiglu_row_factor(o):
    """The row factor of the quantised SwiGLU forward is the RMSNorm row
    factor, applied to the input before the gate: with exactly representable
    operands and r = 1/rms(X), swiglu_fp8_fwd and swiglu_nvfp4_fwd with
    row_scale r equal the SwiGLU-MLP forward with unit gain (RMSNorm first,
    then the gate) on the same operands."""
    codes, vals = _e4m3_table()
    r = RNG(41)
    pick = lambda shape: vals[r.integers(0, len(vals), size=shape)] * (2.0 ** -6)
    e = []
    X, Wg, Wu = pick((4, 16)), pick((6, 16)), pick((6, 16))
    X[:, 0], Wg[:, 0], Wu[:, 0] = 448.0 * 2.0 ** -6, 448.0 * 2.0 ** -6, 448.0 * 2.0 ** -6
    _, xv, sx = o.quantize_fp8_rows(X)
    _, gv, sg = o.quantize_fp8_rows(Wg)
    _, uv, su = o.quantize_fp8_rows(Wu)
    ref = o.mlp_fwd(X, Wg, Wu, np.zeros((16, 6)), np.zeros((4, 16)), gamma=np.ones(16), eps=1e-6)
    H, g, u = o.swiglu_fp8_fwd(xv, sx, gv, sg, uv, su, row_scale=o.rms_inv(X, 1e-6))
    e += [_rel(H, ref["H"]), _rel(g, ref["g"]), _rel(u, ref["u"])]
    X, *_ = _nvfp4_exact_rows(r, 4, 2, [-10, -13, -8, -18])
    Wg, *_ = _nvfp4_exact_rows(r, 5, 2, [-11, -10, -12, -11, -13])
    Wu, *_ = _nvfp4_exact_rows(r, 5, 2, [-12, -11, -10, -12, -11])
    _, _, sx, xv = o.quantize_nvfp4_rows(X)
    _, _, sg, gv = o.quantize_nvfp4_rows(Wg)
    _, _, su, uv = o.quantize_nvfp4_rows(Wu)
    K = X.shape[1]
    ref = o.mlp_fwd(X, Wg, Wu, np.zeros((K, 5)), np.zeros((4, K)), gamma=np.ones(K), eps=1e-6)
    H, g, u = o.swiglu_nvfp4_fwd(xv, sx, gv, sg, uv, su, row_scale=o.rms_inv(X, 1e-6))
    e += [_rel(H, ref["H"]), _rel(g, ref["g"]), _rel(u, ref["u"])]
    return max(e)


ALL_CHECKS = {
    "rmsnorm_scale_nvfp4": (check_rmsnorm_scale_nvfp4, 1e-12),
    "e2m1": (check_e2m1, 0.0),
    "nvfp4_quantizer": (check_nvfp4_quantizer, 1e-12),
    "nvfp4_linear": (check_nvfp4_linear, 1e-14),
    "fp8_quantizer": (check_fp8_quantizer, 1e-12),
    "fp8_linear": (check_fp8_linear, 1e-14),
    "fp8_cols_quantizer": (check_fp8_cols_quantizer, 0.0),
    "fp8_epilogue_ops": (check_fp8_epilogue_ops, 1e-7),
    "fp8_qkv_bwd": (check_fp8_qkv_bwd, 1e-6),
    "quantised_swiglu_row_factor": (check_quantised_swiglu_row_factor, 1e-12),
    "linear_sigmoid": (check_linear_sigmoid, 1e-7),
    "rmsnorm_ce_library": (check_rmsnorm_ce_library, 1e-12),
    "rmsnorm_ce_grad": (check_rmsnorm_ce_grad, 1e-7),
    "gemm_epilogue_bruteforce": (check_gemm_epilogue_bruteforce, 1e-13),
    "reparam_identity": (check_reparam_identity, 1e-13),
    "rmsnorm_library": (check_rmsnorm_library, 1e-13),
    "rmsnorm_scale_invariance": (check_rmsnorm_scale_invariance, 1e-13),
    "rmsnorm_linear_grad": (check_rmsnorm_linear_grad, 1e-7),
    "linear_residual": (check_linear_residual, 1e-7),
    "silu_closed_forms": (check_silu_closed_forms, 1e-7),
    "swiglu_library": (check_swiglu_library, 1e-13),
    "mlp_special_cases": (check_mlp_special_cases, 1e-12),
    "mlp_grad": (lambda o: check_mlp_grad(o, False), 1e-7),
    "mlp_grad_gamma": (lambda o: check_mlp_grad(o, True), 1e-7),
    "rope_invariants": (check_rope_invariants, 1e-12),
    "qknorm_closed_form": (check_qknorm_closed_form, 1e-12),
    "qknorm_grad": (check_qknorm_grad, 1e-7),
    "qknorm_grad_half_pairing": (lambda o: check_qknorm_grad(o, "half"), 1e-7),
    "rope_half": (check_rope_half, 1e-12),
    "ce_uniform": (check_ce_uniform, 1e-14),
    "ce_library": (check_ce_library, 1e-7),
    "ce_all_ignored": (check_ce_all_ignored, 0.5),
    "ce_bad_labels": (check_ce_bad_labels, 1e-7),
    "ce_dw_rows": (check_ce_dw_rows, 1e-7),
    "ce_lse_merge": (check_ce_lse_merge, 1e-14),
    "block_special_cases": (check_block_special_cases, 1e-12),
    "block_grad": (check_block_grad, 1e-7),
}
