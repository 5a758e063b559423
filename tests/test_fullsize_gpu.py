"""Full-size parity on the benchmark workloads (the SwiGLU MLP at hidden 4096,
linear + cross-entropy at vocabulary 128256, the block at hidden 8192 and the
FP8 / NVFP4 gate/up legs at its shape; the RMSNorm-linear workload runs in
full in test_ops_gpu.py), in the launch configuration bench.py times.

The fp64 oracle cannot evaluate the largest workloads whole in a test's
time, so it is evaluated exactly on samples or on sub-problems whose
outputs equal the full problem's:

  * row-local outputs (every forward output, dX, dA, dx0, dx1, lse) on sampled
    token rows -- the oracle run on those rows alone is exact for them; the
    cross-entropy lse and mean loss on every row, in row blocks;
  * weight gradients of the SwiGLU MLP on sampled intermediate units -- an
    MLP restricted to a subset of its intermediate units (rows of Wg, Wu,
    columns of Wd) has exactly those units' dWg, dWu rows and dWd columns;
  * the cross-entropy dW on sampled vocabulary rows (the softmax of every
    row normalised over the whole vocabulary, summed over token blocks);
  * the block's QKV-side gradients (dWqkv, dgamma_attn, dgamma_q, dgamma_k)
    whole: they depend on x0, the gains, Wqkv, pos and dQ, dK, dV only, so
    the oracle's block with the MLP cut to a few units and the attention
    output to one 128-wide slice has exactly the same ones;
  * dgamma_mlp whole, as the sum over blocks of intermediate units of the
    restricted MLPs' dgamma (the gain gradient is linear in the MLP's
    per-unit contributions).

dWo, a sum over every token of dx1 (which needs the whole MLP backward), is
checked through a property that holds at any size: dWo v = dx1^T (A v) for a
random vector v, with dx1 itself checked against the oracle on sampled rows.
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
MLP_UNIT_BLOCK = 4096


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
CE_ROW_BLOCK = 512


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
    X, W = to_np(t["X"]), to_np(t["W"])
    # vocabulary rows of dW: both ends, rows that are some token's label
    # (their one-hot term), and rows no label hits
    lab_ids = np.unique(labels[labels >= 0])
    pick = torch.randperm(len(lab_ids), generator=torch.Generator().manual_seed(21))[:14].numpy()
    ids = np.unique(np.concatenate([[0, s.vocab - 1], lab_ids[pick], _units(s.vocab, 16, 22)]))
    lse = np.empty(s.tokens)
    per_row = np.empty(s.tokens)
    dw_rows = np.zeros((len(ids), s.hidden))
    for lo in range(0, s.tokens, CE_ROW_BLOCK):
        sl = slice(lo, lo + CE_ROW_BLOCK)
        f = O.linear_cross_entropy_fwd(X[sl], W, labels[sl])
        lse[sl], per_row[sl] = f["lse"], f["per_row"]
        # the block's share of the mean: dloss = its valid count / the total
        dw_rows += O.linear_cross_entropy_bwd(X[sl], W, labels[sl], dloss=f["n_valid"] / n_valid,
                                              vocab_rows=ids)["dW_rows"]
    assert_f32(out["lse"], lse, "lse, every row")
    assert_f32(out["loss"], [per_row.sum() / n_valid], "mean loss")
    assert_bf16(_at(g["dW"], ids), dw_rows, f"dW, {len(ids)} sampled vocabulary rows")
    rows = synth.sample_rows(s.tokens, N_ROWS).numpy()
    f = O.linear_cross_entropy_fwd(X[rows], W, labels[rows])
    # the oracle's mean over the sample uses the sample's own count: rescale
    b = O.linear_cross_entropy_bwd(X[rows], W, labels[rows], dloss=f["n_valid"] / n_valid)
    assert_bf16(_at(g["dX"], rows), b["dX"], "dX rows")


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
    # dgamma_mlp: the sum over blocks of intermediate units of the restricted
    # MLPs' gain gradients
    dgm = np.zeros(s.hidden)
    for lo in range(0, s.inter, MLP_UNIT_BLOCK):
        c = slice(lo, lo + MLP_UNIT_BLOCK)
        dgm += O.mlp_bwd(x1, o["Wg"][c], o["Wu"][c], o["Wd"][:, c], to_np(t["dx2"]), o["gamma_mlp"],
                         s.eps)["dgamma"]
    assert_bf16(gr["dgamma_mlp"], dgm, "dgamma_mlp")
    del x1
    # QKV-side gradients whole: the oracle's block with every head, the MLP
    # cut to the sampled units and the attention output to one 128-wide
    # slice (neither enters dWqkv or the three gains)
    sub = {k: to_np(v) for k, v in t.items() if k not in ("Wg", "Wu", "Wd", "A", "Wo")}
    sub["pos"] = t["pos"].numpy()
    sub["Wg"], sub["Wu"], sub["Wd"] = o["Wg"][iu], o["Wu"][iu], o["Wd"][:, iu]
    sub["A"], sub["Wo"] = to_np(t["A"])[:, :128], o["Wo"][:, :128]
    rq = O.block_bwd(sub, **cfg)
    assert_bf16(gr["dWqkv"], rq["dWqkv"], "dWqkv, every row")
    for k in ("dgamma_attn", "dgamma_q", "dgamma_k"):
        assert_bf16(gr[k], rq[k], k)
    del sub, rq
    # dWo = dx1^T A: probed with a random vector against dx1 (checked above
    # on sampled rows)
    v = np.random.default_rng(23).standard_normal(s.n_q * s.head_dim)
    lhs = to_np(gr["dWo"]) @ v
    rhs = to_np(gr["dx1"]).T @ (to_np(t["A"]) @ v)
    assert_bf16(lhs, rhs, "dWo v vs dx1^T (A v)")


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
