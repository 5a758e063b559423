"""Run by test_nvfp4_gpu.py in a fresh process (the NVFP4 kernel variant is
read once per process from CODA_NVFP4, the cluster size): the
NVFP4 linear and SwiGLU at ragged sizes that leave CTAs of a cluster past
the last row block, against the fp64 oracle.  Exits non-zero on the first
mismatch."""
import math
import os
import sys

import torch

sys.path.insert(0, os.path.dirname(os.path.abspath(__file__)))
sys.path.insert(0, os.path.dirname(os.path.dirname(os.path.abspath(__file__))))

import synth  # noqa: E402
from oracle import coda_oracle as O  # noqa: E402
from parity import assert_bf16, to_np  # noqa: E402

import gemm_epilogue_transformer_bf16_gb300 as coda  # noqa: E402


def quant(X):
    q, sf, s = coda.quantize_nvfp4_rows(X.to("cuda"))
    _, _, os_, ov = O.quantize_nvfp4_rows(to_np(X))
    return (q, sf, s), (ov, os_)


def main():
    coda.load()
    M, N, K = 600, 520, 288
    X = synth.randn_bf16((M, K), 1.0, 21)
    W = synth.randn_bf16((N, K), 1 / math.sqrt(K), 22)
    R = synth.randn_bf16((M, N), 1.0, 23)
    xd, xo = quant(X)
    wd, wo = quant(W)
    ws = coda.workspace(256)
    Y = coda.linear_nvfp4(*xd, *wd, R.to("cuda"), ws=ws)
    torch.cuda.synchronize()
    assert coda.get_status(ws) == 0
    assert_bf16(Y, O.linear_nvfp4_fwd(*xo, *wo, R=to_np(R)), "nvfp4 Y")
    # more tiles than resident CTAs or clusters: each works through several
    M, N, K = 4096, 2048, 256
    X = synth.randn_bf16((M, K), 1.0, 27)
    W = synth.randn_bf16((N, K), 1 / math.sqrt(K), 28)
    xd, xo = quant(X)
    wd, wo = quant(W)
    Y = coda.linear_nvfp4(*xd, *wd, ws=ws)
    torch.cuda.synchronize()
    assert coda.get_status(ws) == 0
    assert_bf16(Y, O.linear_nvfp4_fwd(*xo, *wo), "nvfp4 Y, several tiles per CTA")
    M, I, K = 700, 392, 512
    X = synth.randn_bf16((M, K), 1.0, 24)
    Wg = synth.randn_bf16((I, K), 1 / math.sqrt(K), 25)
    Wu = synth.randn_bf16((I, K), 1 / math.sqrt(K), 26)
    xd, xo = quant(X)
    gd, go = quant(Wg)
    ud, uo = quant(Wu)
    H, g, u = coda.linear_swiglu_nvfp4(*xd, *gd, *ud, ws=ws)
    torch.cuda.synchronize()
    assert coda.get_status(ws) == 0
    Hr, gr, ur = O.swiglu_nvfp4_fwd(*xo, *go, *uo)
    assert_bf16(H, Hr, "nvfp4 H")
    assert_bf16(g, gr, "nvfp4 g")
    assert_bf16(u, ur, "nvfp4 u")
    print("ok")


if __name__ == "__main__":
    main()
