"""GPU parity of the NVFP4 path against the fp64 oracle: the quantiser's
codes, block scales (read back through the documented tensor-core order,
padding included) and row scales bit for bit; the block-scaled GEMMs with
the plain and SwiGLU epilogues against the oracle's linear on the
dequantised operands."""
import math

import numpy as np
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


def unpack_codes(q):
    q = q.cpu().numpy()
    out = np.empty((q.shape[0], 2 * q.shape[1]), np.uint8)
    out[:, 0::2] = q & 0xF
    out[:, 1::2] = q >> 4
    return out


def scale_offsets(M, K):
    """Byte offset of (row r, 16-element block j) in the block-scale buffer
    (the layout include/coda.h documents)."""
    kt = -(-K // 256)
    r = np.arange(M)[:, None]
    j = np.arange(K // 16)[None, :]
    return ((r // 128) * kt + j // 16) * 2048 + ((j // 4) % 4) * 512 + (r % 32) * 16 + ((r % 128) // 32) * 4 + j % 4


def check_quantised(coda, X, q, sf, s):
    """Bit-exact against the oracle; returns the oracle's (values, s)."""
    M, K = X.shape
    oc, osf, os_, ov = O.quantize_nvfp4_rows(to_np(X))
    assert np.array_equal(unpack_codes(q), oc), "e2m1 codes"
    assert np.array_equal(s.cpu().numpy(), os_), "row scales"
    buf = sf.cpu().numpy()
    assert buf.size == coda.load().coda_nvfp4_scale_bytes(M, K) == -(-M // 512) * 4 * -(-K // 256) * 2048
    off = scale_offsets(M, K)
    assert np.array_equal(buf[off], osf), "block scales"
    pad = np.ones(buf.size, bool)
    pad[off.ravel()] = False
    assert not np.any(buf[pad]), "padding scales must be zero"
    return ov, os_


@pytest.mark.parametrize("M,N,K", [(512, 768, 2048), (300, 264, 224), (4096, 2048, 512)])
def test_nvfp4_quantize_and_linear(coda, M, N, K):
    X = synth.randn_bf16((M, K), 1.0, 1)
    W = synth.randn_bf16((N, K), 1 / math.sqrt(K), 2)
    R = synth.randn_bf16((M, N), 1.0, 3)
    xq, sfx, sx = coda.quantize_nvfp4_rows(X.to(DEV))
    wq, sfw, sw = coda.quantize_nvfp4_rows(W.to(DEV))
    xv, osx = check_quantised(coda, X, xq, sfx, sx)
    wv, osw = check_quantised(coda, W, wq, sfw, sw)
    ws = coda.workspace(256)
    Y = coda.linear_nvfp4(xq, sfx, sx, wq, sfw, sw, R.to(DEV), ws=ws)
    assert coda.get_status(ws) == 0
    assert_bf16(Y, O.linear_nvfp4_fwd(xv, osx, wv, osw, R=to_np(R)), "Y nvfp4")
    Y0 = coda.linear_nvfp4(xq, sfx, sx, wq, sfw, sw)
    assert_bf16(Y0, O.linear_nvfp4_fwd(xv, osx, wv, osw), "Y nvfp4 without residual")


@pytest.mark.parametrize("shape", [synth.MlpShape(512, 512, 1408), synth.MlpShape(300, 288, 392)])
def test_nvfp4_linear_swiglu(coda, shape):
    t = synth.make_mlp(shape, seed=0)
    d = {k: v.to(DEV) for k, v in t.items()}
    r = coda.rms_rstd(d["X"], 1e-6)
    xq, sfx, sx = coda.quantize_nvfp4_rows(d["X"])
    gq, sfg, sg = coda.quantize_nvfp4_rows(d["Wg"])
    uq, sfu, su = coda.quantize_nvfp4_rows(d["Wu"])
    xv, osx = check_quantised(coda, t["X"], xq, sfx, sx)
    gv, osg = check_quantised(coda, t["Wg"], gq, sfg, sg)
    uv, osu = check_quantised(coda, t["Wu"], uq, sfu, su)
    H, g, u = coda.linear_swiglu_nvfp4(xq, sfx, sx, gq, sfg, sg, uq, sfu, su, rstd=r)
    Hr, gr, ur = O.swiglu_nvfp4_fwd(xv, osx, gv, osg, uv, osu, row_scale=O.rms_inv(to_np(t["X"]), 1e-6))
    assert_bf16(H, Hr, "H nvfp4")
    assert_bf16(g, gr, "g nvfp4")
    assert_bf16(u, ur, "u nvfp4")
    H2, _, _ = coda.linear_swiglu_nvfp4(xq, sfx, sx, gq, sfg, sg, uq, sfu, su, rstd=r, save=False)
    assert torch.equal(H2, H), "H without the saved g, u"


def test_nvfp4_special_rows(coda):
    """A zero row, a row with one loud element (its other blocks' scales
    underflow to zero codes) and exactly representable rows."""
    K = 256
    X = synth.randn_bf16((130, K), 1.0, 7)
    X[0] = 0
    X[1] = 1e-6
    X[1, 5] = 3000.0
    xq, sfx, sx = coda.quantize_nvfp4_rows(X.to(DEV))
    check_quantised(coda, X, xq, sfx, sx)


@pytest.mark.parametrize("variant", ["1", "2", "4", "pair"])
def test_nvfp4_kernel_variants(variant):
    """Each kernel variant (single CTAs, clusters of 2 or 4 CTAs sharing the
    B tile by multicast, CTA pairs) in a fresh process."""
    import os
    import subprocess
    import sys
    here = os.path.dirname(os.path.abspath(__file__))
    env = dict(os.environ, CODA_NVFP4=variant)
    r = subprocess.run([sys.executable, os.path.join(here, "nvfp4_variant_check.py")], env=env,
                       capture_output=True, text=True, timeout=600)
    assert r.returncode == 0 and r.stdout.strip().endswith("ok"), f"{variant}:\n{r.stdout[-2000:]}\n{r.stderr[-4000:]}"


@pytest.mark.parametrize("shape", [synth.MlpShape(512, 512, 1408), synth.MlpShape(300, 288, 392)])
def test_rmsnorm_scale_nvfp4_into_swiglu(coda, shape):
    """The fused RMSNorm input stage (r = 1/rms(x) and the NVFP4 codes of
    x ⊙ gamma in one pass) bit for bit against the oracle, then the NVFP4
    SwiGLU projection with r as its row factor."""
    t = synth.make_mlp(shape, seed=4)
    d = {k: v.to(DEV) for k, v in t.items()}
    gamma = synth.gain_f32(shape.hidden, 5)
    xq, sfx, sx, r = coda.rmsnorm_scale_nvfp4(d["X"], gamma.to(DEV), 1e-6)
    oc, osf, osx, ov, orr = O.rmsnorm_scale_nvfp4(to_np(t["X"]), gamma.numpy(), 1e-6)
    assert np.array_equal(unpack_codes(xq), oc), "codes of x * gamma"
    assert np.array_equal(sx.cpu().numpy(), osx), "row scales"
    assert np.array_equal(sfx.cpu().numpy()[scale_offsets(*t["X"].shape)], osf), "block scales"
    from parity import assert_f32
    assert_f32(r, orr, "rstd")
    gq, sfg, sg = coda.quantize_nvfp4_rows(d["Wg"])
    uq, sfu, su = coda.quantize_nvfp4_rows(d["Wu"])
    gv, osg = check_quantised(coda, t["Wg"], gq, sfg, sg)
    uv, osu = check_quantised(coda, t["Wu"], uq, sfu, su)
    H, g, u = coda.linear_swiglu_nvfp4(xq, sfx, sx, gq, sfg, sg, uq, sfu, su, rstd=r)
    Hr, gr, ur = O.swiglu_nvfp4_fwd(ov, osx, gv, osg, uv, osu, row_scale=orr)
    assert_bf16(H, Hr, "H (fused input stage)")
    assert_bf16(g, gr, "g (fused input stage)")
    assert_bf16(u, ur, "u (fused input stage)")
