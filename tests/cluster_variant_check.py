"""Run by test_cluster_variants_gpu.py in a fresh process (the cluster-size
switches are read once per process): a ragged transformer block forward and
backward, a SwiGLU MLP backward, an FP8 linear and a linear + residual whose
shape the launch policy runs as CTA pairs, and the RMSNorm-linear forward
and backward with its dW GEMM on a second stream (the two backward GEMMs
share the grid), against the fp64 oracle.
Exits non-zero on the first mismatch."""
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import synth  # noqa: E402
from oracle import coda_oracle as O  # noqa: E402
from parity import assert_bf16, assert_f32, to_np  # noqa: E402

import gemm_epilogue_transformer_bf16_gb300 as coda  # noqa: E402
from gemm_epilogue_transformer_bf16_gb300.block import Block  # noqa: E402


def f64(t):
    return {k: (v.numpy() if v.dtype in (torch.int32, torch.int64) else v.double().numpy()) for k, v in t.items()}


def main():
    coda.load()
    dev = "cuda"
    shape = synth.BlockShape(tokens=600, hidden=264, n_q=2, n_kv=1, head_dim=128, inter=392, seq_len=256)
    t = synth.make_block(shape, seed=3)
    d, o = {k: v.to(dev) for k, v in t.items()}, f64(t)
    blk = Block(shape, d)
    f = blk.forward(d["x0"], d["A"], d["pos"])
    g = blk.backward(d["x0"], d["A"], d["pos"], d["dx2"], d["dQ"], d["dK"], d["dV"])
    torch.cuda.synchronize()
    assert coda.get_status(blk.ws) == 0
    cfg = dict(n_q=shape.n_q, n_kv=shape.n_kv, head_dim=shape.head_dim, theta=shape.theta, eps=shape.eps)
    rf, rb = O.block_fwd(o, **cfg), O.block_bwd(o, **cfg)
    for k in ("Q", "K", "V", "x1", "x2"):
        assert_bf16(f[k], rf[k], k)
    for k in ("dx0", "dA", "dWqkv", "dWo", "dWg", "dWu", "dWd", "dgamma_attn", "dgamma_mlp", "dgamma_q",
              "dgamma_k"):
        assert_bf16(g[k], rb[k], k)
    # FP8 linear + residual on an M that spans several cluster sizes' tiles
    M, N, K = 700, 520, 256
    X = synth.randn_bf16((M, K), 1.0, 11).to(dev)
    W = synth.randn_bf16((N, K), 1 / 16, 12).to(dev)
    xq, sx = coda.quantize_fp8_rows(X)
    wq, sw = coda.quantize_fp8_rows(W)
    Y = coda.linear_fp8(xq, sx, wq, sw)
    torch.cuda.synchronize()
    _, ovx, osx = O.quantize_fp8_rows(to_np(X))
    _, ovw, osw = O.quantize_fp8_rows(to_np(W))
    assert_bf16(Y, O.linear_fp8_fwd(ovx, osx, ovw, osw), "fp8 Y")
    # linear + residual at 8192 x 4096: eight waves of two-pair units but
    # seven of CTA pairs, so the default launch policy runs it as pairs
    M, N, K = 8192, 4096, 128
    X = synth.randn_bf16((M, K), 1.0, 21)
    W = synth.randn_bf16((N, K), 1 / 12, 22)
    R = synth.randn_bf16((M, N), 1.0, 23)
    Y, r = coda.linear_residual(X.to(dev), W.to(dev), R.to(dev), eps=1e-6, want_rstd=True)
    torch.cuda.synchronize()
    ur, rr = O.linear_residual_fwd(to_np(X), to_np(W), to_np(R), 1e-6)
    assert_bf16(Y, ur, "8192x4096 Y")
    assert_f32(r, rr, "8192x4096 rstd")
    # RMSNorm-linear forward and backward, dW on a second stream
    rs = synth.RmsLinearShape(1000, 520, 264)
    tr = synth.make_rms_linear(rs, seed=5)
    dr, orr = {k: v.to(dev) for k, v in tr.items()}, f64(tr)
    Wf = coda.fold_gamma(dr["W"], dr["gamma"])
    Yr, rstd = coda.rmsnorm_linear(dr["X"], Wf, R=dr["R"], eps=rs.eps)
    side = torch.cuda.Stream()
    gr = coda.rmsnorm_linear_bwd(dr["G"], dr["X"], dr["W"], dr["gamma"], rstd, Yr, dr["R"], side_stream=side)
    torch.cuda.synchronize()
    yr_, _ = O.rmsnorm_linear_fwd(orr["X"], orr["gamma"], orr["W"], rs.eps, orr["R"])
    br = O.rmsnorm_linear_bwd(orr["X"], orr["gamma"], orr["W"], rs.eps, orr["G"])
    assert_bf16(Yr, yr_, "rmsnorm-linear Y")
    for k in ("dX", "dW", "dgamma"):
        assert_bf16(gr[k], br[k], "rmsnorm-linear " + k)
    print("ok")


if __name__ == "__main__":
    main()
