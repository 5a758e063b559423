"""Full-size parity on the benchmark workloads (the SwiGLU MLP at hidden 4096,
linear + cross-entropy at vocabulary 128256, the block at hidden 8192 and the
FP8 / NVFP4 gate/up legs at its shape; the RMSNorm-linear workload runs in
full in test_ops_gpu.py), in the launch configuration bench.py times.

The fp64 oracle cannot evaluate these workloads whole in a test's time, so it
is evaluated exactly on samples:

  * row-local outputs (every forward output, dX, dA, dx0, dx1, lse) on sampled
    token rows -- the oracle run on those rows alone is exact for them;
  * weight gradients of the SwiGLU MLP on sampled intermediate units -- an
    MLP restricted to a subset of its intermediate units (rows of Wg, Wu,
    columns of Wd) has exactly those units' dWg, dWu rows and dWd columns;

and, where no exact sample is cheap, through properties that hold at any
size: dgamma_k * gamma_k = sum_n W_nk dW_nk for the RMSNorm-reparameterised
projections, mean loss = mean over valid rows of (lse_i - z_{i,y_i}), and the
columns of the cross-entropy dW summing to ~0 (softmax - onehot rows sum to 0).
"""
import math

import numpy as np
import pytest
import torch

import synth
from oracle import coda_oracle as O
from parity import assert_bf16, assert_f32, to_np

pytestmark = [pytest.mark.gpu, pytest.mark.slow]
DEV = "cuda"
N_ROWS = 48
N_UNITS = 24


@pytest.fixture(scope="module")
def coda():
    import gemm_epilogue_transformer_bf16_gb300 as c
    from gemm_epilogue_transformer_bf16_gb300 import _build
    _build.build()
    c.load()
    return c


def _units(n, k, seed):
    g = torch.Generator().manual_seed(seed)
    return torch.randperm(n, generator=g)[:k].sort().values.numpy()


def _at(t, idx, dim=0):
    """Rows (dim 0) or columns (dim 1) `idx` of a device tensor, on the host."""
    ix = torch.as_tensor(idx, dtype=torch.long, device=t.device)
    return t.index_select(dim, ix).cpu()


def _gamma_property(dgamma, gamma, pairs, name):
    """dgamma_k * gamma_k == sum over (W, dW) pairs of sum_n W_nk dW_nk."""
    lhs = to_np(dgamma) * to_np(gamma)
    rhs = sum((to_np(W) * to_np(dW)).sum(axis=0) for W, dW in pairs)
    assert_bf16(lhs, rhs, name)


# ---------------------------------------------------------------- SwiGLU MLP, hidden 4096
def test_mlp_fullsize(coda):
    s = synth.FULL["mlp"]
    t = synth.make_mlp(s, seed=0)
    d = {k: v.to(DEV) for k, v in t.items()}
    H, g, u = coda.linear_swiglu(d["X"], d["Wg"], d["Wu"])
    Y = coda.linear_residual(H, d["Wd"], d["R"])
    gr = coda.linear_swiglu_bwd(d["dY"], d["X"], d["Wg"], d["Wu"], d["Wd"], g, u, H)
    torch.cuda.synchronize()
    rows = synth.sample_rows(s.tokens, N_ROWS).numpy()
    o = {k: to_np(v) for k, v in t.items()}
    f = O.mlp_fwd(o["X"][rows], o["Wg"], o["Wu"], o["Wd"], o["R"][rows])
    assert_bf16(_at(H, rows), f["H"], "H rows")
    assert_bf16(_at(Y, rows), f["y"], "y rows")
    b = O.mlp_bwd(o["X"][rows], o["Wg"], o["Wu"], o["Wd"], o["dY"][rows])
    assert_bf16(_at(gr["dX"], rows), b["dX"], "dX rows")
    iu = _units(s.inter, N_UNITS, 7)
    bu = O.mlp_bwd(o["X"], o["Wg"][iu], o["Wu"][iu], o["Wd"][:, iu], o["dY"])
    assert_bf16(_at(gr["dWg"], iu), bu["dWg"], "dWg sampled units")
    assert_bf16(_at(gr["dWu"], iu), bu["dWu"], "dWu sampled units")
    assert_bf16(_at(gr["dWd"], iu, 1), bu["dWd"], "dWd sampled units")


# ---------------------------------------------------------------- linear + cross-entropy, vocabulary 128256
def test_cross_entropy_fullsize(coda):
    s = synth.FULL["linear_ce"]
    t = synth.make_ce(s, seed=0)
    d = {k: v.to(DEV) for k, v in t.items()}
    out = coda.linear_cross_entropy(d["X"], d["W"], d["labels"])
    g = coda.linear_cross_entropy_bwd(d["X"], d["W"], d["labels"], out["lse"], out["n_valid"], 1.0)
    torch.cuda.synchronize()
    assert coda.get_status(out["ws"]) == 0
    labels = t["labels"].numpy()
    n_valid = int((labels != s.ignore_index).sum())
    assert int(out["n_valid"].item()) == n_valid == s.tokens - math.floor(0.05 * s.tokens)
    rows = synth.sample_rows(s.tokens, N_ROWS).numpy()
    X, W = to_np(t["X"]), to_np(t["W"])
    f = O.linear_cross_entropy_fwd(X[rows], W, labels[rows])
    assert_f32(_at(out["lse"], rows), f["lse"], "lse rows")
    # the oracle's mean over the sample uses the sample's own count: rescale
    b = O.linear_cross_entropy_bwd(X[rows], W, labels[rows], dloss=f["n_valid"] / n_valid)
    assert_bf16(_at(g["dX"], rows), b["dX"], "dX rows")
    # mean loss vs lse (checked above on samples) and exact target logits
    valid = np.nonzero(labels != s.ignore_index)[0]
    z_t = np.einsum("ij,ij->i", X[valid], W[labels[valid]])
    mean = (to_np(out["lse"])[valid] - z_t).mean()
    assert_f32(out["loss"], [mean], "mean loss vs per-row lse")
    # rows of softmax - onehot sum to zero, so do the columns of dW
    dW = to_np(g["dW"])
    colsum = dW.sum(axis=0)
    scale = np.sqrt((dW ** 2).sum(axis=0))
    assert float(np.max(np.abs(colsum) / scale)) < 3e-2, "columns of dW do not sum to ~0"


# ---------------------------------------------------------------- block, hidden 8192 (the bench workload)
def test_block_fullsize(coda):
    from gemm_epilogue_transformer_bf16_gb300.block import Block
    s = synth.FULL["block"]
    t = synth.make_block(s, seed=0)
    d = {k: v.to(DEV) for k, v in t.items()}
    blk = Block(s, d)
    f = blk.forward(d["x0"], d["A"], d["pos"])
    gr = blk.backward(d["x0"], d["A"], d["pos"], d["dx2"], d["dQ"], d["dK"], d["dV"])
    torch.cuda.synchronize()
    assert coda.get_status(blk.ws) == 0
    rows = synth.sample_rows(s.tokens, N_ROWS).numpy()
    tok = {"x0", "A", "dx2", "dQ", "dK", "dV", "pos"}
    o = {k: (to_np(v)[rows] if k in tok else to_np(v)) for k, v in t.items()}
    o["pos"] = t["pos"].numpy()[rows]
    cfg = dict(n_q=s.n_q, n_kv=s.n_kv, head_dim=s.head_dim, theta=s.theta, eps=s.eps)
    rf = O.block_fwd(o, **cfg)
    for k in ("Q", "K", "V", "x1", "x2"):
        assert_bf16(_at(f[k], rows), rf[k], f"{k} rows")
    rb = O.block_bwd(o, **cfg)
    for k in ("dx0", "dA", "dx1"):
        assert_bf16(_at(gr[k], rows), rb[k], f"{k} rows")
    # MLP weight gradients on sampled intermediate units (needs x1 for all tokens)
    x1, _ = O.linear_residual_fwd(to_np(t["A"]), o["Wo"], to_np(t["x0"]))
    iu = _units(s.inter, N_UNITS, 11)
    bu = O.mlp_bwd(x1, o["Wg"][iu], o["Wu"][iu], o["Wd"][:, iu], to_np(t["dx2"]), o["gamma_mlp"], s.eps)
    assert_bf16(_at(gr["dWg"], iu), bu["dWg"], "dWg sampled units")
    assert_bf16(_at(gr["dWu"], iu), bu["dWu"], "dWu sampled units")
    assert_bf16(_at(gr["dWd"], iu, 1), bu["dWd"], "dWd sampled units")
    # gain gradients: consistency with the weight gradients at full size
    _gamma_property(gr["dgamma_mlp"], t["gamma_mlp"], [(t["Wg"], gr["dWg"]), (t["Wu"], gr["dWu"])],
                    "dgamma_mlp * gamma vs sum W dW")
    _gamma_property(gr["dgamma_attn"], t["gamma_attn"], [(t["Wqkv"], gr["dWqkv"])],
                    "dgamma_attn * gamma vs sum W dW")


# ---------------------------------------------------------------- low-precision gate/up legs (bench shape)
def _gateup_inputs():
    s = synth.FULL["block"]
    t = synth.make_block(s, seed=0)
    return s, t["x0"], t["Wg"], t["Wu"]


def test_fp8_gateup_fullsize(coda):
    """e4m3 gate/up + SwiGLU at the bench's shape (8192 x 2x28672 x 8192):
    quantisation is per row, so the oracle's codes for sampled token rows and
    sampled weight rows are exact, and so are the outputs at those entries."""
    s, x, Wg, Wu = _gateup_inputs()
    xq, sx = coda.quantize_fp8_rows(x.to(DEV))
    gq, sg = coda.quantize_fp8_rows(Wg.to(DEV))
    uq, su = coda.quantize_fp8_rows(Wu.to(DEV))
    H, g, u = coda.linear_swiglu_fp8(xq, sx, gq, sg, uq, su)
    torch.cuda.synchronize()
    rows = synth.sample_rows(s.tokens, N_ROWS).numpy()
    iu = _units(s.inter, 8 * N_UNITS, 11)
    ocx, ovx, osx = O.quantize_fp8_rows(to_np(x)[rows])
    ocg, ovg, osg = O.quantize_fp8_rows(to_np(Wg)[iu])
    ocu, ovu, osu = O.quantize_fp8_rows(to_np(Wu)[iu])
    assert np.array_equal(_at(xq, rows).numpy(), ocx) and np.array_equal(_at(gq, iu).numpy(), ocg)
    assert np.array_equal(_at(uq, iu).numpy(), ocu) and np.array_equal(_at(sx, rows).numpy(), osx)
    Hr, gr, ur = O.swiglu_fp8_fwd(ovx, osx, ovg, osg, ovu, osu)
    for name, got, ref in (("H", H, Hr), ("g", g, gr), ("u", u, ur)):
        assert_bf16(_at(_at(got, rows), iu, 1), ref, f"fp8 {name} sampled rows x units")


def test_nvfp4_gateup_fullsize(coda):
    """NVFP4 gate/up + SwiGLU at the bench's shape, checked the same way:
    codes and row scales of sampled rows bit for bit, outputs at sampled
    (token, unit) entries against the oracle on the dequantised operands."""
    s, x, Wg, Wu = _gateup_inputs()
    xq, sfx, sx = coda.quantize_nvfp4_rows(x.to(DEV))
    gq, sfg, sg = coda.quantize_nvfp4_rows(Wg.to(DEV))
    uq, sfu, su = coda.quantize_nvfp4_rows(Wu.to(DEV))
    H, g, u = coda.linear_swiglu_nvfp4(xq, sfx, sx, gq, sfg, sg, uq, sfu, su)
    torch.cuda.synchronize()
    rows = synth.sample_rows(s.tokens, N_ROWS).numpy()
    iu = _units(s.inter, 8 * N_UNITS, 12)

    def unpack(q):
        q = q.numpy()
        out = np.empty((q.shape[0], 2 * q.shape[1]), np.uint8)
        out[:, 0::2], out[:, 1::2] = q & 0xF, q >> 4
        return out
    cx, _, osx, ovx = O.quantize_nvfp4_rows(to_np(x)[rows])
    cg, _, osg, ovg = O.quantize_nvfp4_rows(to_np(Wg)[iu])
    cu, _, osu, ovu = O.quantize_nvfp4_rows(to_np(Wu)[iu])
    assert np.array_equal(unpack(_at(xq, rows)), cx) and np.array_equal(unpack(_at(gq, iu)), cg)
    assert np.array_equal(unpack(_at(uq, iu)), cu) and np.array_equal(_at(sx, rows).numpy(), osx)
    Hr, gr, ur = O.swiglu_nvfp4_fwd(ovx, osx, ovg, osg, ovu, osu)
    for name, got, ref in (("H", H, Hr), ("g", g, gr), ("u", u, ur)):
        assert_bf16(_at(_at(got, rows), iu, 1), ref, f"nvfp4 {name} sampled rows x units")
