"""GPU parity of the named operators (the hot-path rows) against the fp64
oracle on seeded synthetic inputs: full size where the oracle finishes in
seconds, scaled-down shapes with ragged tails otherwise."""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import coda_oracle as O
from parity import assert_bf16, assert_f32, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def coda():
    import gemm_epilogue_transformer_bf16_gb300 as c
    from gemm_epilogue_transformer_bf16_gb300 import _build
    _build.build()
    c.load()
    return c


def dev(d):
    return {k: v.to(DEV) for k, v in d.items()}


def f64(d):
    return {k: to_np(v) for k, v in d.items()}


# ---------------------------------------------------------------- linear + SwiGLU
@pytest.mark.parametrize("shape", [synth.SwigluShape(), synth.SwigluShape(200, 136, 264)])
def test_linear_swiglu(coda, shape):
    t = synth.make_swiglu(shape, seed=0)
    d, o = dev(t), f64(t)
    H, g, u = coda.linear_swiglu(d["X"], d["Wg"], d["Wu"])
    Hr, gr, ur = O.swiglu_fwd(o["X"], o["Wg"], o["Wu"])
    assert_bf16(H, Hr, "H")
    assert_bf16(g, gr, "g")
    assert_bf16(u, ur, "u")


# ---------------------------------------------------------------- RMSNorm-reparameterised projection
@pytest.mark.parametrize("shape", [synth.RmsLinearShape(), synth.RmsLinearShape(300, 264, 200)])
@pytest.mark.parametrize("side", [False, True])
def test_rmsnorm_linear_fwd_bwd(coda, shape, side):
    """Forward and backward; with `side` the dW GEMM runs on a second stream
    and the two backward GEMMs each take half of the grid."""
    t = synth.make_rms_linear(shape, seed=0)
    d, o = dev(t), f64(t)
    Wf = coda.fold_gamma(d["W"], d["gamma"])
    Y, rstd = coda.rmsnorm_linear(d["X"], Wf, R=d["R"], eps=shape.eps)
    yr, rr = O.rmsnorm_linear_fwd(o["X"], o["gamma"], o["W"], shape.eps, o["R"])
    assert_bf16(Y, yr, "Y")
    assert_f32(rstd, rr, "rstd")
    g = coda.rmsnorm_linear_bwd(d["G"], d["X"], d["W"], d["gamma"], rstd, Y, d["R"],
                                side_stream=torch.cuda.Stream() if side else None)
    torch.cuda.synchronize()
    b = O.rmsnorm_linear_bwd(o["X"], o["gamma"], o["W"], shape.eps, o["G"])
    assert_bf16(g["dX"], b["dX"], "dX")
    assert_bf16(g["dW"], b["dW"], "dW")
    assert_bf16(g["dgamma"], b["dgamma"], "dgamma")


@pytest.mark.parametrize("shape", [synth.RmsLinearShape(), synth.RmsLinearShape(300, 264, 200)])
def test_rmsnorm_linear_rstd_in(coda, shape):
    """The projection with a row factor computed beforehand (coda_rms_rstd,
    passed as rstd_in), the fold and the row RMS on two streams: the same Y as
    the oracle's RMSNorm-linear forward."""
    t = synth.make_rms_linear(shape, seed=0)
    d, o = dev(t), f64(t)
    side = torch.cuda.Stream()
    side.wait_stream(torch.cuda.current_stream())
    with torch.cuda.stream(side):
        Wf = coda.fold_gamma(d["W"], d["gamma"])
    r = coda.rms_rstd(d["X"], shape.eps)
    torch.cuda.current_stream().wait_stream(side)
    Y, r2 = coda.rmsnorm_linear(d["X"], Wf, R=d["R"], rstd_in=r, eps=shape.eps)
    torch.cuda.synchronize()
    assert r2 is r
    yr, rr = O.rmsnorm_linear_fwd(o["X"], o["gamma"], o["W"], shape.eps, o["R"])
    assert_f32(r, rr, "rstd")
    assert_bf16(Y, yr, "Y (rstd_in)")


def test_launch_count(coda):
    """coda_launch_count counts each kernel launch once: the gain fold and
    the row RMS are one kernel each."""
    t = synth.make_rms_linear(synth.RmsLinearShape(64, 128, 72), seed=3)
    d = dev(t)
    c0 = coda.launch_count()
    coda.fold_gamma(d["W"], d["gamma"])
    c1 = coda.launch_count()
    coda.rms_rstd(d["X"], 1e-6)
    c2 = coda.launch_count()
    torch.cuda.synchronize()
    assert (c1 - c0, c2 - c1) == (1, 1)


def test_fold_gamma_and_rstd(coda):
    t = synth.make_rms_linear(synth.RmsLinearShape(64, 128, 72), seed=3)
    d, o = dev(t), f64(t)
    Wf = coda.fold_gamma(d["W"], d["gamma"])
    assert_bf16(Wf, o["W"] * o["gamma"][None, :], "Wf")
    r = coda.rms_rstd(d["X"], 1e-6)
    assert_f32(r, O.rms_inv(o["X"], 1e-6), "rstd")


def test_rmsnorm_scale(coda):
    """One pass: r = 1/rms(X) and U = X ⊙ gamma (bit-exact: one bf16 rounding
    of an fp32 product of two exact values)."""
    t = synth.make_rms_linear(synth.RmsLinearShape(200, 128, 264), seed=5)
    d, o = dev(t), f64(t)
    r, U = coda.rmsnorm_scale(d["X"], d["gamma"], 1e-6)
    assert_f32(r, O.rms_inv(o["X"], 1e-6), "rstd")
    assert torch.equal(U, (d["X"].float() * d["gamma"][None, :]).to(torch.bfloat16)), "U = X * gamma"


@pytest.mark.parametrize("M,N,K", [(256, 512, 384), (300, 776, 136)])
def test_linear_residual_gamma_output(coda, M, N, K):
    """The producing epilogue's second output U = Y ⊙ gamma (Y as stored)."""
    X = synth.randn_bf16((M, K), 1.0, 1)
    W = synth.randn_bf16((N, K), 1 / math.sqrt(K), 2)
    R = synth.randn_bf16((M, N), 1.0, 3)
    gamma = synth.gain_f32(N, 4).to(DEV)
    U = torch.empty(M, N, dtype=torch.bfloat16, device=DEV)
    Y, r = coda.linear_residual(X.to(DEV), W.to(DEV), R.to(DEV), eps=1e-6, want_rstd=True, gamma_next=gamma,
                                U_out=U)
    ur, rr = O.linear_residual_fwd(to_np(X), to_np(W), to_np(R), 1e-6)
    assert_bf16(Y, ur, "Y")
    assert_f32(r, rr, "rstd from partials")
    assert torch.equal(U, (Y.float() * gamma[None, :]).to(torch.bfloat16)), "U = Y * gamma"


@pytest.mark.parametrize("shape", [synth.MlpShape(512, 512, 1408), synth.MlpShape(200, 264, 392)])
def test_mlp_bwd_gamma_in_epilogue(coda, shape):
    """RMSNorm -> SwiGLU MLP with the gain applied to the GEMM input
    (U = X ⊙ gamma, weights unfolded): forward and the backward whose dX
    epilogue emits the dgamma column partials."""
    t = synth.make_mlp(shape, seed=1)
    t["gamma"] = synth.gain_f32(shape.hidden, 8)
    d, o = dev(t), f64(t)
    eps = 1e-6
    r, U = coda.rmsnorm_scale(d["X"], d["gamma"], eps)
    H, g, u = coda.linear_swiglu(U, d["Wg"], d["Wu"], rstd=r)
    f = O.mlp_fwd(o["X"], o["Wg"], o["Wu"], o["Wd"], o["R"], o["gamma"], eps)
    assert_bf16(H, f["H"], "H")
    gr = coda.linear_swiglu_bwd(d["dY"], d["X"], d["Wg"], d["Wu"], d["Wd"], g, u, H, rstd=r, gamma=d["gamma"],
                                dX_resid=d["dY"])
    torch.cuda.synchronize()
    b = O.mlp_bwd(o["X"], o["Wg"], o["Wu"], o["Wd"], o["dY"], o["gamma"], eps)
    assert_bf16(gr["dX"], b["dX"] + o["dY"], "dX")
    for k in ("dWg", "dWu", "dWd", "dgamma"):
        assert_bf16(gr[k], b[k], k)


# ---------------------------------------------------------------- residual + partial RMS
@pytest.mark.parametrize("M,N,K", [(256, 512, 384), (300, 776, 136)])
def test_linear_residual_partial_rms(coda, M, N, K):
    X = synth.randn_bf16((M, K), 1.0, 1)
    W = synth.randn_bf16((N, K), 1 / math.sqrt(K), 2)
    R = synth.randn_bf16((M, N), 1.0, 3)
    Y, r = coda.linear_residual(X.to(DEV), W.to(DEV), R.to(DEV), eps=1e-6, want_rstd=True)
    ur, rr = O.linear_residual_fwd(to_np(X), to_np(W), to_np(R), 1e-6)
    assert_bf16(Y, ur, "u")
    assert_f32(r, rr, "rstd from partials")
    G = synth.randn_bf16((M, N), 1.0, 4)
    g = coda.linear_residual_bwd(G.to(DEV), X.to(DEV), W.to(DEV))
    b = O.linear_residual_bwd(to_np(X), to_np(W), to_np(G))
    assert_bf16(g["dX"], b["dX"], "dX")
    assert_bf16(g["dW"], b["dW"], "dW")


# ---------------------------------------------------------------- SwiGLU MLP (scaled)
@pytest.mark.parametrize("shape", [synth.MlpShape(512, 512, 1408), synth.MlpShape(200, 264, 392)])
def test_swiglu_mlp_fwd_bwd(coda, shape):
    t = synth.make_mlp(shape, seed=0)
    d, o = dev(t), f64(t)
    H, g, u = coda.linear_swiglu(d["X"], d["Wg"], d["Wu"])
    Y = coda.linear_residual(H, d["Wd"], d["R"])
    f = O.mlp_fwd(o["X"], o["Wg"], o["Wu"], o["Wd"], o["R"])
    assert_bf16(H, f["H"], "H")
    assert_bf16(Y, f["y"], "y")
    gr = coda.linear_swiglu_bwd(d["dY"], d["X"], d["Wg"], d["Wu"], d["Wd"], g, u, H)
    b = O.mlp_bwd(o["X"], o["Wg"], o["Wu"], o["Wd"], o["dY"])
    for k in ("dX", "dWg", "dWu", "dWd"):
        assert_bf16(gr[k], b[k], k)


# ---------------------------------------------------------------- linear + cross-entropy (scaled)
# The backward takes the vocabulary in slices of 16384 columns: one slice up
# to 16384, then several with a ragged last one; labels sit on both sides of
# the slice boundaries.
CE_SHAPES = [synth.CeShape(512, 256, 4000), synth.CeShape(300, 136, 8192), synth.CeShape(300, 136, 40008)]


def _ce_labels(t, vocab):
    lab = t["labels"].clone()
    lab[1] = 0
    lab[2] = vocab - 1
    if vocab > 16384:
        lab[3], lab[4], lab[5] = 16383, 16384, 32768 if vocab > 32768 else 16385
    t["labels"] = lab


@pytest.mark.parametrize("shape", CE_SHAPES)
def test_linear_cross_entropy(coda, shape):
    t = synth.make_ce(shape, seed=0)
    _ce_labels(t, shape.vocab)
    d, o = dev(t), f64(t)
    labels_np = t["labels"].numpy()
    out = coda.linear_cross_entropy(d["X"], d["W"], d["labels"])
    f = O.linear_cross_entropy_fwd(o["X"], o["W"], labels_np)
    assert coda.get_status(out["ws"]) == 0
    assert int(out["n_valid"].item()) == f["n_valid"]
    assert_f32(out["lse"], f["lse"], "lse")
    assert_f32(out["loss"], [f["loss"]], "loss")
    g = coda.linear_cross_entropy_bwd(d["X"], d["W"], d["labels"], out["lse"], out["n_valid"], 1.0)
    b = O.linear_cross_entropy_bwd(o["X"], o["W"], labels_np)
    assert_bf16(g["dX"], b["dX"], "dX")
    assert_bf16(g["dW"], b["dW"], "dW")


def test_cross_entropy_all_ignored_and_bad_label(coda):
    """All rows ignored: NaN loss, n_valid 0, the oracle's lse, zero
    gradients.  Labels outside [0, V) other than -100 (one negative, one at
    V + 5): CODA_ERR_LABEL_RANGE in the status word, and lse, loss, n_valid,
    dX and dW equal the oracle's, which counts those rows as ignored."""
    s = synth.CeShape(64, 128, 1024)
    t = synth.make_ce(s, seed=5)
    d, o = dev(t), f64(t)
    lab = torch.full((s.tokens,), -100, dtype=torch.int32)
    out = coda.linear_cross_entropy(d["X"], d["W"], lab.to(DEV))
    f = O.linear_cross_entropy_fwd(o["X"], o["W"], lab.numpy())
    assert math.isnan(out["loss"].item()) and math.isnan(f["loss"])
    assert int(out["n_valid"].item()) == f["n_valid"] == 0
    assert_f32(out["lse"], f["lse"], "lse (all ignored)")
    g = coda.linear_cross_entropy_bwd(d["X"], d["W"], lab.to(DEV), out["lse"], out["n_valid"], 1.0)
    assert not torch.any(g["dX"].float() != 0) and not torch.any(g["dW"].float() != 0)
    assert coda.get_status(out["ws"]) == 0
    lab2 = t["labels"].clone()
    lab2[3] = s.vocab + 5
    lab2[7] = -5
    lab2[11] = -100
    out2 = coda.linear_cross_entropy(d["X"], d["W"], lab2.to(DEV))
    assert coda.get_status(out2["ws"]) == 7   # CODA_ERR_LABEL_RANGE
    f2 = O.linear_cross_entropy_fwd(o["X"], o["W"], lab2.numpy())
    assert f2["label_range_error"]
    assert int(out2["n_valid"].item()) == f2["n_valid"] == int(((lab2 >= 0) & (lab2 < s.vocab)).sum())
    assert_f32(out2["lse"], f2["lse"], "lse")
    assert_f32(out2["loss"], [f2["loss"]], "loss")
    g2 = coda.linear_cross_entropy_bwd(d["X"], d["W"], lab2.to(DEV), out2["lse"], out2["n_valid"], 1.0)
    b2 = O.linear_cross_entropy_bwd(o["X"], o["W"], lab2.numpy())
    assert_bf16(g2["dX"], b2["dX"], "dX")
    assert_bf16(g2["dW"], b2["dW"], "dW")
    assert not torch.any(g2["dX"][[3, 7, 11]].float() != 0)


# ---------------------------------------------------------------- transformer block (scaled)
SMALL_BLOCK = synth.BlockShape(tokens=256, hidden=512, n_q=4, n_kv=2, head_dim=128, inter=1024, seq_len=128)
RAGGED_BLOCK = synth.BlockShape(tokens=200, hidden=264, n_q=2, n_kv=1, head_dim=128, inter=392, seq_len=64)


@pytest.mark.parametrize("fold_weights,concurrent_bwd", [(False, False), (True, False), (False, True)])
@pytest.mark.parametrize("shape", [SMALL_BLOCK, RAGGED_BLOCK])
def test_block_fwd_bwd(coda, shape, fold_weights, concurrent_bwd):
    """Both ways of applying the RMSNorm gains: in the producing epilogue
    (u = x ⊙ gamma, the default) and folded into the weights; and the
    backward on one stream (the default) or with its second stream."""
    from gemm_epilogue_transformer_bf16_gb300.block import Block
    t = synth.make_block(shape, seed=0)
    d, o = dev(t), f64(t)
    blk = Block(shape, d, fold_weights=fold_weights, concurrent_bwd=concurrent_bwd)
    f = blk.forward(d["x0"], d["A"], d["pos"])
    g = blk.backward(d["x0"], d["A"], d["pos"], d["dx2"], d["dQ"], d["dK"], d["dV"])
    torch.cuda.synchronize()
    assert coda.get_status(blk.ws) == 0
    cfg = dict(n_q=shape.n_q, n_kv=shape.n_kv, head_dim=shape.head_dim, theta=shape.theta, eps=shape.eps)
    rf = O.block_fwd(o, **cfg)
    for k in ("Q", "K", "V", "x1", "x2"):
        assert_bf16(f[k], rf[k], k)
    rb = O.block_bwd(o, **cfg)
    for k in ("dx0", "dA", "dx1", "dWqkv", "dWo", "dWg", "dWu", "dWd", "dgamma_attn", "dgamma_mlp",
              "dgamma_q", "dgamma_k"):
        assert_bf16(g[k], rb[k], k)


# ---------------------------------------------------------------- final RMSNorm -> LM head -> CE
@pytest.mark.parametrize("shape", [synth.CeShape(512, 256, 4000), synth.CeShape(300, 136, 8200),
                                   synth.CeShape(260, 128, 33000)])
def test_rmsnorm_linear_cross_entropy(coda, shape):
    t = synth.make_ce(shape, seed=0)
    _ce_labels(t, shape.vocab)
    t["gamma"] = synth.gain_f32(shape.hidden, 9)
    t["R"] = synth.randn_bf16((shape.tokens, shape.hidden), 1.0, 10)
    d, o = dev(t), f64(t)
    labels_np = t["labels"].numpy()
    eps = 1e-6
    Wf = coda.fold_gamma(d["W"], d["gamma"])
    r = coda.rms_rstd(d["X"], eps)
    out = coda.rmsnorm_linear_cross_entropy(d["X"], r, Wf, d["labels"])
    f = O.rmsnorm_linear_cross_entropy_fwd(o["X"], o["gamma"], o["W"], labels_np, eps)
    assert coda.get_status(out["ws"]) == 0
    assert int(out["n_valid"].item()) == f["n_valid"]
    assert_f32(r, f["rstd"], "rstd")
    assert_f32(out["lse"], f["lse"], "lse")
    assert_f32(out["loss"], [f["loss"]], "loss")
    g = coda.rmsnorm_linear_cross_entropy_bwd(d["X"], r, d["gamma"], d["W"], Wf, d["labels"], out["lse"],
                                              out["n_valid"], 1.0, dX_resid=d["R"])
    b = O.rmsnorm_linear_cross_entropy_bwd(o["X"], o["gamma"], o["W"], labels_np, eps)
    assert coda.get_status(g["ws"]) == 0
    assert_bf16(g["dX"], b["dX"] + o["R"], "dX (+ residual gradient)")
    assert_bf16(g["dW"], b["dW"], "dW")
    assert_bf16(g["dgamma"], b["dgamma"], "dgamma")


# ---------------------------------------------------------------- linear_sigmoid
@pytest.mark.parametrize("gated", [False, True])
@pytest.mark.parametrize("M,N,K", [(512, 768, 384), (300, 264, 200)])
def test_linear_sigmoid(coda, gated, M, N, K):
    X = synth.randn_bf16((M, K), 1.0, 1)
    W = synth.randn_bf16((N, K), 1 / math.sqrt(K), 2)
    Z = synth.randn_bf16((M, N), 1.0, 3) if gated else None
    dY = synth.randn_bf16((M, N), 1.0, 4)
    Zd = Z.to(DEV) if gated else None
    Y = coda.linear_sigmoid(X.to(DEV), W.to(DEV), Zd)
    Zo = to_np(Z) if gated else None
    assert_bf16(Y, O.linear_sigmoid_fwd(to_np(X), to_np(W), Zo), "Y")
    g = coda.linear_sigmoid_bwd(dY.to(DEV), X.to(DEV), W.to(DEV), Zd)
    b = O.linear_sigmoid_bwd(to_np(X), to_np(W), to_np(dY), Zo)
    assert_bf16(g["dX"], b["dX"], "dX")
    assert_bf16(g["dW"], b["dW"], "dW")
    if gated:
        assert_bf16(g["dZ"], b["dZ"], "dZ")


# ---------------------------------------------------------------- FP8 (e4m3) operands
@pytest.mark.parametrize("M,N,K", [(512, 768, 512), (300, 264, 208)])
def test_fp8_quantize_and_linear(coda, M, N, K):
    X = synth.randn_bf16((M, K), 1.0, 1)
    W = synth.randn_bf16((N, K), 1 / math.sqrt(K), 2)
    R = synth.randn_bf16((M, N), 1.0, 3)
    xq, sx = coda.quantize_fp8_rows(X.to(DEV))
    wq, sw = coda.quantize_fp8_rows(W.to(DEV))
    ocx, ovx, osx = O.quantize_fp8_rows(to_np(X))
    ocw, ovw, osw = O.quantize_fp8_rows(to_np(W))
    # the quantised codes and scales are decisions: bit-exact
    assert np.array_equal(xq.cpu().numpy(), ocx) and np.array_equal(wq.cpu().numpy(), ocw)
    assert np.array_equal(sx.cpu().numpy(), osx) and np.array_equal(sw.cpu().numpy(), osw)
    Y = coda.linear_fp8(xq, sx, wq, sw, R.to(DEV))
    assert_bf16(Y, O.linear_fp8_fwd(ovx, osx, ovw, osw, R=to_np(R)), "Y fp8")


@pytest.mark.parametrize("shape", [synth.MlpShape(512, 512, 1408), synth.MlpShape(300, 272, 392)])
def test_fp8_linear_swiglu(coda, shape):
    t = synth.make_mlp(shape, seed=0)
    d = dev(t)
    r = coda.rms_rstd(d["X"], 1e-6)
    xq, sx = coda.quantize_fp8_rows(d["X"])
    gq, sg = coda.quantize_fp8_rows(d["Wg"])
    uq, su = coda.quantize_fp8_rows(d["Wu"])
    H, g, u = coda.linear_swiglu_fp8(xq, sx, gq, sg, uq, su, rstd=r)
    _, ovx, osx = O.quantize_fp8_rows(to_np(t["X"]))
    _, ovg, osg = O.quantize_fp8_rows(to_np(t["Wg"]))
    _, ovu, osu = O.quantize_fp8_rows(to_np(t["Wu"]))
    Hr, gr, ur = O.swiglu_fp8_fwd(ovx, osx, ovg, osg, ovu, osu, row_scale=O.rms_inv(to_np(t["X"]), 1e-6))
    assert_bf16(H, Hr, "H fp8")
    assert_bf16(g, gr, "g fp8")
    assert_bf16(u, ur, "u fp8")


# ---------------------------------------------------------------- leading dimensions
def test_leading_dims_match_flat_calls(coda):
    """[batch, seq, features] operands give, bit for bit, the flat [tokens,
    features] results, reshaped to the caller's leading shape (the wrappers
    only change views; the kernels see the same rows)."""
    s = RAGGED_BLOCK
    B, S = 2, s.tokens // 2
    t = dev(synth.make_block(s, seed=11))
    x = t["x0"]
    x3 = x.view(B, S, -1)
    pos3 = t["pos"].view(B, S)
    cs = coda.rope_table(s.theta, s.head_dim, s.seq_len)

    def same(a, b, name):
        assert torch.equal(a.reshape(b.shape), b), f"{name}: the 3-D call differs from the flat one"

    r2, U2 = coda.rmsnorm_scale(x, t["gamma_attn"], s.eps)
    r3, U3 = coda.rmsnorm_scale(x3, t["gamma_attn"], s.eps)
    assert r3.shape == (B, S) and U3.shape == x3.shape
    same(r3, r2, "rstd")
    same(U3, U2, "U")

    q2 = coda.linear_qknorm_rope(U2, t["Wqkv"], t["gamma_q"], t["gamma_k"], t["pos"], cs, s.n_q, s.n_kv, rstd=r2)
    q3 = coda.linear_qknorm_rope(U3, t["Wqkv"], t["gamma_q"], t["gamma_k"], pos3, cs, s.n_q, s.n_kv, rstd=r3)
    for k in ("Q", "K", "V", "qk_save"):
        assert q3[k].shape[:2] == (B, S)
        same(q3[k], q2[k], k)

    A = t["A"]
    y2, ry2 = coda.linear_residual(A, t["Wo"], x, eps=s.eps, want_rstd=True)
    y3, ry3 = coda.linear_residual(A.view(B, S, -1), t["Wo"], x3, eps=s.eps, want_rstd=True)
    assert y3.shape == x3.shape and ry3.shape == (B, S)
    same(y3, y2, "Y")
    same(ry3, ry2, "rstd_out")

    H2, g2, u2 = coda.linear_swiglu(y2, t["Wg"], t["Wu"], rstd=ry2)
    H3, g3, u3 = coda.linear_swiglu(y3, t["Wg"], t["Wu"], rstd=ry3)
    assert H3.shape == (B, S, s.inter)
    for a, b, n in ((H3, H2, "H"), (g3, g2, "g"), (u3, u2, "u")):
        same(a, b, n)

    Z = H2[:, : s.hidden].contiguous()
    sg2 = coda.linear_sigmoid(H2, t["Wd"], Z)
    sg3 = coda.linear_sigmoid(H3, t["Wd"], Z.view(B, S, -1))
    assert sg3.shape == (B, S, s.hidden)
    same(sg3, sg2, "sigmoid")

    labels = (torch.arange(s.tokens, device=DEV, dtype=torch.int32) * 7) % s.inter
    labels[3] = -100
    W_head = t["Wg"]                                       # [inter, hidden]: a small vocabulary
    c2 = coda.linear_cross_entropy(x, W_head, labels)
    c3 = coda.linear_cross_entropy(x3, W_head, labels.view(B, S))
    assert c3["lse"].shape == (B, S)
    same(c3["lse"], c2["lse"], "lse")
    same(c3["loss"], c2["loss"], "loss")

    with pytest.raises(ValueError):
        coda.linear_swiglu(y3.transpose(0, 1), t["Wg"], t["Wu"])


# ---------------------------------------------------------------- QK-RMSNorm + RoPE, both pairings
@pytest.mark.parametrize("pairing", ["interleaved", "half"])
def test_linear_qknorm_rope_pairings(coda, pairing):
    """The fused QKV projection with per-head QK-RMSNorm and RoPE, forward and
    backward, for interleaved pairs (2j, 2j+1) and half-split pairs
    (j, j + 64), against the oracle composed from its RMSNorm, per-head
    QK-norm + RoPE and their backward passes (ragged token count)."""
    s = RAGGED_BLOCK
    t = synth.make_block(s, seed=21)
    d = dev(t)
    o = {k: to_np(v) for k, v in t.items()}
    cs = coda.rope_table(s.theta, s.head_dim, s.seq_len)
    r, U = coda.rmsnorm_scale(d["x0"], d["gamma_attn"], s.eps)
    out = coda.linear_qknorm_rope(U, d["Wqkv"], d["gamma_q"], d["gamma_k"], d["pos"], cs, s.n_q, s.n_kv, rstd=r,
                                  eps=s.eps, pairing=pairing)
    g = coda.linear_qknorm_rope_bwd(d["dQ"], d["dK"], d["dV"], out["qk_save"], out["V"], d["gamma_q"], d["gamma_k"],
                                    d["pos"], cs, s.n_q, s.n_kv, d["x0"], d["Wqkv"], rstd=r, gamma_in=d["gamma_attn"],
                                    eps=s.eps, pairing=pairing)
    M, D = s.tokens, s.head_dim
    xn = O.rmsnorm(o["x0"], o["gamma_attn"], s.eps)
    qkv = xn @ o["Wqkv"].T
    q = qkv[:, : s.n_q * D].reshape(M, s.n_q, D)
    k = qkv[:, s.n_q * D:(s.n_q + s.n_kv) * D].reshape(M, s.n_kv, D)
    pos = t["pos"].numpy()
    Qr = O.qk_rmsnorm_rope_fwd(q, o["gamma_q"], pos, s.theta, s.eps, pairing).reshape(M, -1)
    Kr = O.qk_rmsnorm_rope_fwd(k, o["gamma_k"], pos, s.theta, s.eps, pairing).reshape(M, -1)
    assert_bf16(out["Q"], Qr, f"Q ({pairing})")
    assert_bf16(out["K"], Kr, f"K ({pairing})")
    assert_bf16(out["V"], qkv[:, (s.n_q + s.n_kv) * D:], f"V ({pairing})")
    dq, dgq = O.qk_rmsnorm_rope_bwd(q, o["gamma_q"], pos, s.theta, s.eps, o["dQ"].reshape(M, s.n_q, D), pairing)
    dk, dgk = O.qk_rmsnorm_rope_bwd(k, o["gamma_k"], pos, s.theta, s.eps, o["dK"].reshape(M, s.n_kv, D), pairing)
    dqkv = np.concatenate([dq.reshape(M, -1), dk.reshape(M, -1), o["dV"]], axis=1)
    dx, dgin = O.rmsnorm_bwd(o["x0"], o["gamma_attn"], s.eps, dqkv @ o["Wqkv"])
    assert_bf16(g["dX"], dx, f"dX ({pairing})")
    assert_bf16(g["dW"], dqkv.T @ xn, f"dWqkv ({pairing})")
    # gain gradients are sums over tokens with cancellation: the RMS-relative rule, as for the block
    assert_bf16(g["dgamma_in"], dgin, f"dgamma_in ({pairing})")
    assert_bf16(g["dgamma_q"], dgq, f"dgamma_q ({pairing})")
    assert_bf16(g["dgamma_k"], dgk, f"dgamma_k ({pairing})")
