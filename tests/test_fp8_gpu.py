"""GPU parity of the FP8 (e4m3) instances of the epilogues against the fp64
oracle on the dequantised operands: QKV + QK-norm + RoPE (both pairings),
linear + cross-entropy forward and backward (vocabularies of one and of
three backward slices), dSwiGLU on the dH GEMM and the RMSNorm-reparameterised
input gradient, and the column quantiser that gives the backward GEMMs their
K-major transposed operands.

Quantisation codes and scales are decisions: the GPU quantisers are checked
bit for bit against the oracle's, and each operator then runs on the codes
that both sides computed from the same bf16 input.  Shapes span several
tiles with ragged tails."""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import coda_oracle as O
from parity import assert_bf16, assert_bf16_within, assert_f32, e4m3_step_allowance, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def coda():
    import gemm_epilogue_transformer_bf16_gb300 as c
    from gemm_epilogue_transformer_bf16_gb300 import _build
    _build.build()
    c.load()
    return c


def _rows(coda, X):
    """GPU row quantisation, checked bit for bit against the oracle's;
    returns (device codes, device scales, oracle values, oracle scales)."""
    q, s = coda.quantize_fp8_rows(X.to(DEV))
    oc, ov, osc = O.quantize_fp8_rows(to_np(X))
    assert np.array_equal(q.cpu().numpy(), oc) and np.array_equal(s.cpu().numpy(), osc)
    return q, s, ov, osc


def _cols(coda, X, X2=None):
    q, s = coda.quantize_fp8_cols(X.to(DEV), None if X2 is None else X2.to(DEV))
    full = to_np(X) if X2 is None else np.vstack([to_np(X), to_np(X2)])
    oc, ov, osc = O.quantize_fp8_cols(full)
    assert np.array_equal(q.cpu().numpy(), oc) and np.array_equal(s.cpu().numpy(), osc)
    return q, s, ov, osc


def _every_bf16(width, n_gains=16, seed=7):
    """Rows of bf16 values covering every finite bf16 magnitude up to a gain
    g, both signs, for n_gains random gains: each group of rows holds all
    finite patterns with |x| <= g (others zeroed) and starts with g itself, so
    every row's scale is g / 448 and every quotient x / s the codes need is
    taken.  Returns [rows, width] bf16."""
    bits = torch.arange(65536, dtype=torch.int32).to(torch.int16).view(torch.bfloat16).float()
    gains = (torch.rand(n_gains, generator=torch.Generator().manual_seed(seed)) * 2000 + 1e-3)
    rows = []
    for g in gains.to(torch.bfloat16).float():
        v = torch.where(torch.isfinite(bits) & (bits.abs() <= g), bits, torch.zeros_like(bits))
        v = v.view(-1, width).clone()
        v[:, 0] = g
        rows.append(v)
    return torch.cat(rows).to(torch.bfloat16)


@pytest.mark.parametrize("width", [8192, 32768])
def test_quantize_fp8_rows_every_bf16(coda, width):
    """The codes for every finite bf16 value at 16 scales, bit for bit against
    the oracle's IEEE division (8192-wide rows take the shared-memory staged
    quantiser, 32768-wide rows the warp-per-row one)."""
    _rows(coda, _every_bf16(width))


def test_quantize_fp8_cols_every_bf16(coda):
    """The same values through the column quantiser (the transpose: every
    column holds all finite bf16 values up to its gain)."""
    X = _every_bf16(8192, n_gains=4).t().contiguous()
    _cols(coda, X)


@pytest.mark.parametrize("R,R2,C", [(304, 0, 264), (256, 48, 520), (8192, 0, 128)])
def test_quantize_fp8_cols(coda, R, R2, C):
    X = synth.randn_bf16((R, C), 1.0, 31)
    X[:, 3] = 0                                   # an all-zero column: scale 1, zero codes
    X2 = synth.randn_bf16((R2, C), 3.0, 32) if R2 else None
    _cols(coda, X, X2)


@pytest.mark.parametrize("pairing", ["interleaved", "half"])
def test_linear_qknorm_rope_fp8(coda, pairing):
    M, Kd, n_q, n_kv, d = 300, 272, 2, 1, 128
    X = synth.randn_bf16((M, Kd), 1.0, 41)
    W = synth.randn_bf16(((n_q + 2 * n_kv) * d, Kd), 1 / math.sqrt(Kd), 42)
    gq, gk = synth.gain_f32(d, 43), synth.gain_f32(d, 44)
    rstd = (0.5 + torch.rand(M, generator=torch.Generator().manual_seed(45))).float()
    pos = (torch.arange(M, dtype=torch.int32) * 7) % 1024
    cs = coda.rope_table(500000.0, d, 1024)
    xq, sx, xv, osx = _rows(coda, X)
    wq, sw, wv, osw = _rows(coda, W)
    out = coda.linear_qknorm_rope_fp8(xq, sx, wq, sw, gq.to(DEV), gk.to(DEV), pos.to(DEV), cs, n_q, n_kv,
                                      rstd=rstd.to(DEV), pairing=pairing)
    f = O.linear_qknorm_rope_fp8_fwd(xv, osx, wv, osw, to_np(gq), to_np(gk), pos.numpy(), 500000.0, 1e-6, n_q,
                                     n_kv, d, row_scale=to_np(rstd), pairing=pairing)
    for k, ref in (("Q", f["Q"]), ("K", f["K"]), ("V", f["V"]), ("qk_save", f["qk"])):
        assert_bf16(out[k], ref, f"fp8 {k}")


@pytest.mark.parametrize("shape", [synth.CeShape(300, 144, 8200), synth.CeShape(260, 128, 40008)])
def test_linear_cross_entropy_fp8(coda, shape):
    t = synth.make_ce(shape, seed=4)
    lab = t["labels"].clone()
    lab[1], lab[2] = 0, shape.vocab - 1
    if shape.vocab > 16384:
        lab[3], lab[4] = 16383, 16384
    xq, sx, xv, osx = _rows(coda, t["X"])
    wq, sw, wv, osw = _rows(coda, t["W"])
    d = {k: v.to(DEV) for k, v in t.items()}
    out = coda.linear_cross_entropy_fp8(xq, sx, wq, sw, lab.to(DEV))
    f = O.linear_cross_entropy_fp8_fwd(xv, osx, wv, osw, lab.numpy())
    assert coda.get_status(out["ws"]) == 0
    assert int(out["n_valid"].item()) == f["n_valid"]
    assert_f32(out["lse"], f["lse"], "fp8 lse")
    assert_f32(out["loss"], [f["loss"]], "fp8 loss")
    g = coda.linear_cross_entropy_bwd_fp8(xq, sx, wq, sw, d["X"], d["W"], lab.to(DEV), out["lse"], out["n_valid"],
                                          0.8)
    b = O.linear_cross_entropy_fp8_bwd(xv, osx, wv, osw, to_np(t["X"]), to_np(t["W"]), lab.numpy(), dloss=0.8)
    assert coda.get_status(g["ws"]) == 0
    assert_bf16(g["dX"], b["dX"], "fp8 CE dX")
    assert_bf16(g["dW"], b["dW"], "fp8 CE dW")


def test_linear_dswiglu_fp8(coda):
    M, K, I = 300, 272, 392
    dY = synth.randn_bf16((M, K), 1.0, 51)
    Wd = synth.randn_bf16((K, I), 1 / math.sqrt(I), 52)
    g = synth.randn_bf16((M, I), 1.5, 53)
    u = synth.randn_bf16((M, I), 1.0, 54)
    rstd = (0.5 + torch.rand(M, generator=torch.Generator().manual_seed(55))).float()
    dyq, sdy, dyv, osdy = _rows(coda, dY)
    wdq, swd, wdv, oswd = _cols(coda, Wd)
    out = coda.linear_dswiglu_fp8(dyq, sdy, wdq, swd, g.to(DEV), u.to(DEV), rstd=rstd.to(DEV), want_H=True)
    r = O.dswiglu_fp8(dyv, osdy, wdv, oswd, to_np(g), to_np(u), row_scale=to_np(rstd))
    assert_bf16(out["Gp"], r["Gp"], "fp8 G' = r [dG | dU]")
    assert_bf16(out["H"], r["H"], "fp8 dSwiGLU H")
    assert_bf16(out["row"], r["coef"], "fp8 dSwiGLU RMSNorm coefficient")


def test_rmsnorm_linear_dx_fp8(coda):
    M, N, K = 300, 400, 272
    Gp = synth.randn_bf16((M, N), 1.0, 61)
    W = synth.randn_bf16((N, K), 1 / math.sqrt(K), 62)
    X = synth.randn_bf16((M, K), 1.0, 63)
    R = synth.randn_bf16((M, K), 1.0, 64)
    gam = synth.gain_f32(K, 65)
    coef = (0.1 * torch.randn(M, generator=torch.Generator().manual_seed(66))).float()
    gq, sg, gv, osg = _rows(coda, Gp)
    wq, sw, wv, osw = _cols(coda, W)
    out = coda.rmsnorm_linear_dx_fp8(gq, sg, wq, sw, X.to(DEV), gam.to(DEV), coef.to(DEV), dX_resid=R.to(DEV))
    r = O.rmsnorm_linear_dx_fp8(gv, osg, wv, osw, to_np(X), to_np(gam), to_np(coef), dX_resid=to_np(R))
    assert_bf16(out["dX"], r["dX"], "fp8 RMSNorm dX")
    assert_bf16(out["dgamma"], r["dgamma"], "fp8 RMSNorm dgamma")


@pytest.mark.parametrize("norm,pairing,shape", [(True, "interleaved", (304, 272, 2, 1)), (False, "half", (304, 272, 2, 1)),
                                                (True, "half", (160, 200, 4, 2))])
def test_linear_qknorm_rope_bwd_fp8(coda, norm, pairing, shape):
    """The QKV backward with both GEMMs on e4m3 operands: the per-head map
    into G' (in the workspace), G' quantised per row for dX and per column
    for dW, W^T and U^T given as column codes (checked bit for bit against
    the oracle's).  The saved q|k and v are seeded inputs (the backward is
    defined at any saved values).  G' is computed in fp32 by the kernel and
    in fp64 by the oracle, so at a bf16 rounding tie the two may round it
    differently and the e4m3 codes taken from it may differ by one step;
    the max-error bound of dX, dW and dgamma_in carries that admissible
    change through the GEMMs (parity.e4m3_step_allowance); dgamma_q and
    dgamma_k take no quantised operand and are held to the plain rule.
    304 tokens (two 128-token tiles and a ragged tail), 272 features, 2 q
    and 1 kv heads; and 160 tokens, 200 features, 4 q and 2 kv heads."""
    (M, Kd, n_q, n_kv), d = shape, 128
    N = (n_q + 2 * n_kv) * d
    qk = synth.randn_bf16((M, (n_q + n_kv) * d), 1.0, 71)
    V = synth.randn_bf16((M, n_kv * d), 1.0, 72)
    dQ = synth.randn_bf16((M, n_q * d), 1.0, 73)
    dK = synth.randn_bf16((M, n_kv * d), 1.0, 74)
    dV = synth.randn_bf16((M, n_kv * d), 1.0, 75)
    W = synth.randn_bf16((N, Kd), 1 / math.sqrt(Kd), 76)
    X = synth.randn_bf16((M, Kd), 1.0, 77)
    R = synth.randn_bf16((M, Kd), 1.0, 78)
    gin, gq, gk = synth.gain_f32(Kd, 79), synth.gain_f32(d, 80), synth.gain_f32(d, 81)
    rstd = (0.5 + torch.rand(M, generator=torch.Generator().manual_seed(82))).float() if norm else None
    pos = (torch.arange(M, dtype=torch.int32) * 7) % 1024
    U = (X.float() * gin[None, :]).to(torch.bfloat16) if norm else X    # the forward GEMM's input
    cs = coda.rope_table(500000.0, d, 1024)
    wtq, sw, wtv, osw = _cols(coda, W)
    utq, su, utv, osu = _cols(coda, U)
    dv = lambda t: None if t is None else t.to(DEV)
    ws = coda.workspace(coda.load().coda_linear_qknorm_rope_bwd_fp8_workspace_size(M, Kd, n_q, n_kv, d))
    g = coda.linear_qknorm_rope_bwd_fp8(dQ.to(DEV), dK.to(DEV), dV.to(DEV), qk.to(DEV), V.to(DEV), gq.to(DEV),
                                        gk.to(DEV), pos.to(DEV), cs, n_q, n_kv, wtq, sw, utq, su, X=dv(X),
                                        rstd=dv(rstd), gamma_in=dv(gin) if norm else None, dX_resid=R.to(DEV),
                                        eps=1e-6, pairing=pairing, ws=ws)
    torch.cuda.synchronize()
    assert coda.get_status(ws) == 0
    ref = O.linear_qknorm_rope_fp8_bwd(to_np(dQ), to_np(dK), to_np(dV), to_np(qk), to_np(V), to_np(gq), to_np(gk),
                                       pos.numpy(), 500000.0, 1e-6, n_q, n_kv, d, wtv, osw, utv, osu, X=to_np(X),
                                       row_scale=None if rstd is None else to_np(rstd),
                                       gamma_in=to_np(gin) if norm else None, dX_resid=to_np(R), pairing=pairing)
    a_d = e4m3_step_allowance(ref["Gr"]) @ np.abs(wtv * osw[:, None].astype(np.float64)).T
    a_w = e4m3_step_allowance(ref["Gr"].T) @ np.abs(utv * osu[:, None].astype(np.float64)).T
    a_x = a_d * np.abs(to_np(gin))[None, :] if norm else a_d
    assert_bf16_within(g["dX"], ref["dX"], a_x, f"fp8 QKV dX ({pairing})")
    assert_bf16_within(g["dW"], ref["dW"], a_w, f"fp8 QKV dW ({pairing})")
    if norm:
        assert_bf16_within(g["dgamma_in"], ref["dgamma_in"], (np.abs(to_np(X)) * a_d).sum(axis=0),
                           "fp8 QKV dgamma_in")
    assert_bf16(g["dgamma_q"], ref["dgamma_q"], "fp8 QKV dgamma_q")
    assert_bf16(g["dgamma_k"], ref["dgamma_k"], "fp8 QKV dgamma_k")


@pytest.mark.parametrize("fp8_wgrad,concurrent", [(True, True), (False, True), (True, False)])
def test_block_fp8_step(coda, fp8_wgrad, concurrent):
    """The block step with its forward projections and its MLP and
    O-projection input gradients on e4m3 operands (BlockFP8) -- and, with
    fp8_wgrad, the MLP and O-projection weight gradients on the
    column-quantised transposes of their operands -- against the
    fp64 oracle's bf16-free block on a ragged shape.  Each FP8 operator is
    checked exactly above on shared codes; here the quantisation of every
    activation and weight compounds (one e4m3 rounding is up to 2^-4 of a
    value, about 4 % RMS on a product of two quantised operands, and the
    chains run through two or three such GEMMs), so the bound is a relative
    Frobenius error of 0.15 per output: it catches wiring mistakes (a
    transposed operand, a wrong scale), which give errors of order one.
    Also on one stream (the default runs the weight gradients and their
    quantisers on a second one)."""
    from gemm_epilogue_transformer_bf16_gb300.block import BlockFP8
    shape = synth.BlockShape(tokens=256, hidden=512, n_q=4, n_kv=2, head_dim=128, inter=1024, seq_len=128)
    t = synth.make_block(shape, seed=0)
    d = {k: v.to(DEV) for k, v in t.items()}
    o = {k: (v.numpy() if v.dtype in (torch.int32, torch.int64) else to_np(v)) for k, v in t.items()}
    blk = BlockFP8(shape, d, fp8_wgrad=fp8_wgrad, concurrent=concurrent)
    f = blk.forward(d["x0"], d["A"], d["pos"])
    g = blk.backward(d["x0"], d["A"], d["pos"], d["dx2"], d["dQ"], d["dK"], d["dV"])
    torch.cuda.synchronize()
    assert coda.get_status(blk.ws) == 0 and coda.get_status(blk.ws2) == 0
    cfg = dict(n_q=shape.n_q, n_kv=shape.n_kv, head_dim=shape.head_dim, theta=shape.theta, eps=shape.eps)
    rf, rb = O.block_fwd(o, **cfg), O.block_bwd(o, **cfg)
    errs = {}
    for k, got, ref in [(k, f[k], rf[k]) for k in ("Q", "K", "V", "x1", "x2")] + \
            [(k, g[k], rb[k]) for k in ("dx0", "dA", "dx1", "dWqkv", "dWo", "dWg", "dWu", "dWd", "dgamma_attn",
                                        "dgamma_mlp", "dgamma_q", "dgamma_k")]:
        gv, rv = to_np(got), np.asarray(ref, dtype=np.float64)
        assert np.all(np.isfinite(gv)), k
        errs[k] = float(np.linalg.norm(gv - rv) / np.linalg.norm(rv))
    assert max(errs.values()) <= 0.15, errs
