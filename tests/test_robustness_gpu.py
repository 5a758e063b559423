"""GPU robustness: determinism, device-side error reporting and empty inputs.

* Two runs of the fused block fwd+bwd give bit-identical outputs (every
  reduction -- tile partials, combines, column sums -- has a fixed order).
* A RoPE position outside the table sets CODA_ERR_POSITION_RANGE.
* A pipeline wait that nothing satisfies ends after its limit with
  CODA_ERR_TIMEOUT in the status word, and the context stays usable.
* Calls with no token rows succeed and write only what they must.
"""
import math

import pytest
import torch

import synth
from oracle import coda_oracle as O
from parity import assert_bf16, to_np

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def coda():
    import gemm_epilogue_transformer_bf16_gb300 as c
    from gemm_epilogue_transformer_bf16_gb300 import _build
    _build.build()
    c.load()
    return c


def test_block_bitwise_deterministic(coda):
    from gemm_epilogue_transformer_bf16_gb300.block import Block
    shape = synth.BlockShape(tokens=640, hidden=512, n_q=4, n_kv=2, head_dim=128, inter=1024, seq_len=256)
    t = synth.make_block(shape, seed=4)
    d = {k: v.to(DEV) for k, v in t.items()}
    runs = []
    for _ in range(2):
        blk = Block(shape, d)
        f = blk.forward(d["x0"], d["A"], d["pos"])
        g = blk.backward(d["x0"], d["A"], d["pos"], d["dx2"], d["dQ"], d["dK"], d["dV"])
        torch.cuda.synchronize()
        runs.append({k: v.clone() for k, v in {**f, **g}.items()})
    for k in runs[0]:
        assert torch.equal(runs[0][k], runs[1][k]), f"{k} differs between identical runs"


def test_position_out_of_range_sets_status(coda):
    shape = synth.BlockShape(tokens=128, hidden=256, n_q=2, n_kv=1, head_dim=128, inter=256, seq_len=64)
    t = synth.make_block(shape, seed=2)
    d = {k: v.to(DEV) for k, v in t.items()}
    cs = coda.rope_table(shape.theta, 128, shape.seq_len)
    pos = d["pos"].clone()
    pos[7] = shape.seq_len          # one past the table
    ws = coda.workspace(256)
    coda.linear_qknorm_rope(d["x0"], d["Wqkv"], d["gamma_q"], d["gamma_k"], pos, cs, shape.n_q, shape.n_kv, ws=ws)
    assert coda.get_status(ws) == 8      # CODA_ERR_POSITION_RANGE
    coda.reset_status(ws)
    coda.linear_qknorm_rope(d["x0"], d["Wqkv"], d["gamma_q"], d["gamma_k"], d["pos"], cs, shape.n_q, shape.n_kv,
                            ws=ws)
    assert coda.get_status(ws) == 0


def test_bounded_wait_reports_timeout_and_context_survives(coda):
    lib = coda.load()
    ws = coda.workspace(256)
    stream = torch.cuda.current_stream().cuda_stream
    assert lib.coda_selftest_wait_timeout(50_000, ws.data_ptr(), stream) == 0   # 50 ms limit
    assert coda.get_status(ws) == 6      # CODA_ERR_TIMEOUT
    assert lib.coda_selftest_wait_timeout(0, ws.data_ptr(), stream) == 1         # limit out of range
    coda.reset_status(ws)
    # the context still runs a fused GEMM correctly afterwards
    X = synth.randn_bf16((256, 256), 1.0, 1)
    Wg = synth.randn_bf16((512, 256), 1 / 16, 2)
    Wu = synth.randn_bf16((512, 256), 1 / 16, 3)
    H, _, _ = coda.linear_swiglu(X.to(DEV), Wg.to(DEV), Wu.to(DEV), ws=ws)
    assert coda.get_status(ws) == 0
    assert_bf16(H, O.swiglu_fwd(to_np(X), to_np(Wg), to_np(Wu))[0], "H after timeout")


def test_empty_token_batch(coda):
    K, N, V = 256, 512, 1000
    X = torch.empty(0, K, dtype=torch.bfloat16, device=DEV)
    W = synth.randn_bf16((N, K), 0.05, 1).to(DEV)
    Y = coda.linear_residual(X, W)
    assert Y.shape == (0, N)
    H, g, u = coda.linear_swiglu(X, W, W)
    assert H.shape == (0, N)
    Wv = synth.randn_bf16((V, K), 0.05, 2).to(DEV)
    lab = torch.empty(0, dtype=torch.int32, device=DEV)
    out = coda.linear_cross_entropy(X, Wv, lab)
    assert math.isnan(out["loss"].item()) and int(out["n_valid"].item()) == 0
    gr = coda.linear_cross_entropy_bwd(X, Wv, lab, out["lse"], out["n_valid"], 1.0)
    assert not torch.any(gr["dW"].float() != 0)


def test_mlp_backward_side_stream_matches_single_stream(coda):
    """The weight-gradient GEMMs on a second stream give the same bits."""
    M, I, K = 640, 512, 256
    dev = "cuda"
    X = synth.randn_bf16((M, K), 1.0, 71).to(dev)
    Wg = synth.randn_bf16((I, K), 1 / 16, 72).to(dev)
    Wu = synth.randn_bf16((I, K), 1 / 16, 73).to(dev)
    Wd = synth.randn_bf16((K, I), 1 / 16, 74).to(dev)
    dY = synth.randn_bf16((M, K), 1.0, 75).to(dev)
    gamma = synth.gain_f32(K, 76).to(dev)
    rstd = coda.rms_rstd(X, 1e-6)
    Wgf = coda.fold_gamma(Wg, gamma)
    Wuf = coda.fold_gamma(Wu, gamma)
    H, g, u = coda.linear_swiglu(X, Wgf, Wuf, rstd=rstd)
    one = coda.linear_swiglu_bwd(dY, X, Wg, Wu, Wd, g, u, H, rstd=rstd, gamma=gamma, dX_resid=dY)
    side = torch.cuda.Stream()
    two = coda.linear_swiglu_bwd(dY, X, Wg, Wu, Wd, g, u, H, rstd=rstd, gamma=gamma, dX_resid=dY,
                                 side_stream=side)
    torch.cuda.synchronize()
    for k in ("dX", "dWg", "dWu", "dWd", "dgamma"):
        assert torch.equal(one[k], two[k]), f"{k} differs with a side stream"


def test_rmsnorm_linear_backward_side_stream_matches_single_stream(coda):
    """dW on a second stream beside c -> dX gives the same bits, and so does a
    CUDA-graph replay of the forward + backward captured with that side stream
    (the call's fork and join become graph edges)."""
    M, N, K = 4096, 2048, 2048            # the RMSNorm-linear benchmark shape
    dev = "cuda"
    t = {k: v.to(dev) for k, v in synth.make_rms_linear(synth.RmsLinearShape(M, K, N), seed=9).items()}
    Wf = coda.fold_gamma(t["W"], t["gamma"])
    Y, r = coda.rmsnorm_linear(t["X"], Wf, t["R"], eps=1e-6)
    one = coda.rmsnorm_linear_bwd(t["G"], t["X"], t["W"], t["gamma"], r, Y, t["R"])
    side = torch.cuda.Stream()
    two = coda.rmsnorm_linear_bwd(t["G"], t["X"], t["W"], t["gamma"], r, Y, t["R"], side_stream=side)
    torch.cuda.synchronize()
    for k in ("dX", "dW", "dgamma"):
        assert torch.equal(one[k], two[k]), f"{k} differs with a side stream"
    lib = coda.load()
    ws1 = coda.workspace(lib.coda_rmsnorm_linear_workspace_size(M, N, K))
    ws2 = coda.workspace(lib.coda_rmsnorm_linear_bwd_workspace_size(M, N, K))
    Y2, r2 = torch.empty_like(Y), torch.empty_like(r)
    out = {k: torch.empty_like(v) for k, v in one.items()}

    def step():
        coda.fold_gamma(t["W"], t["gamma"], out=Wf)
        coda.rmsnorm_linear(t["X"], Wf, t["R"], eps=1e-6, rstd_out=r2, Y=Y2, ws=ws1)
        coda.rmsnorm_linear_bwd(t["G"], t["X"], t["W"], t["gamma"], r2, Y2, t["R"], ws=ws2, out=out,
                                side_stream=side)
    cap = torch.cuda.Stream()
    with torch.cuda.stream(cap):
        step()                              # first calls set up kernels and streams outside the capture
    torch.cuda.synchronize()
    g = torch.cuda.CUDAGraph()
    with torch.cuda.graph(g, stream=cap):
        step()
    for v in out.values():
        v.zero_()
    g.replay()
    torch.cuda.synchronize()
    assert torch.equal(Y2, Y) and torch.equal(r2, r)
    for k in ("dX", "dW", "dgamma"):
        assert torch.equal(out[k], one[k]), f"{k} differs in the graph replay"
    assert coda.get_status(ws1) == 0 and coda.get_status(ws2) == 0
