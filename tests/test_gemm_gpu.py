"""GPU parity of the generic GEMM + epilogue (coda_gemm_epilogue) against the
fp64 oracle: all four operand major-ness combinations, ragged M/N/K tails,
every option of the element-wise/rank-1/rank-2 epilogue, fp32 accumulate
(beta), row sum-of-squares partials and the concatenated-K second pair."""
import numpy as np
import pytest
import torch

from oracle import coda_oracle as O
from parity import assert_bf16, assert_f32, to_np
from synth import randn_bf16

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module")
def coda():
    import gemm_epilogue_transformer_bf16_gb300 as c
    from gemm_epilogue_transformer_bf16_gb300 import _build
    _build.build()
    c.load()
    return c


def _operand(t_mk, major):
    """Storage for an operand whose math shape is [rows, K]."""
    return t_mk.contiguous() if major == 0 else t_mk.t().contiguous()


@pytest.mark.parametrize("a_major", [0, 1])
@pytest.mark.parametrize("b_major", [0, 1])
@pytest.mark.parametrize("shape", [(256, 512, 256), (296, 264, 200), (128, 256, 64), (8, 16, 8)])
def test_plain_gemm_majorness(coda, a_major, b_major, shape):
    M, N, K = shape
    A = randn_bf16((M, K), 1.0, 11)
    B = randn_bf16((N, K), 1.0 / np.sqrt(K), 12)
    dev = "cuda"
    Ad = _operand(A, a_major).to(dev)
    Bd = _operand(B, b_major).to(dev)
    D = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    desc = coda.EpilogueDesc()
    ws = coda.gemm_epilogue(desc, Ad, Bd, D, M, N, K, a_major=a_major, b_major=b_major)
    torch.cuda.synchronize()
    assert coda.get_status(ws) == 0
    ref = O.gemm_epilogue_plain(to_np(A), to_np(B))
    assert_bf16(D, ref, f"D a_major={a_major} b_major={b_major} {shape}")


def test_plain_epilogue_options(coda):
    M, N, K = 300, 520, 328
    dev = "cuda"
    A = randn_bf16((M, K), 1.0, 21)
    B = randn_bf16((N, K), 1.0 / np.sqrt(K), 22)
    R = randn_bf16((M, N), 1.0, 23)
    X1 = randn_bf16((M, N), 1.0, 24)
    g = torch.Generator().manual_seed(25)
    rs = (torch.rand(M, generator=g) + 0.5).float()
    cs = (torch.rand(N, generator=g) + 0.5).float()
    coef = (torch.rand(M, generator=g) - 0.5).float()
    D0 = (torch.randn(M, N, generator=g)).float()
    Ad, Bd, Rd, X1d = A.to(dev), B.to(dev), R.to(dev), X1.to(dev)
    rsd, csd, coefd = rs.to(dev), cs.to(dev), coef.to(dev)
    part = torch.zeros(((N + 255) // 256) * M, dtype=torch.float32, device=dev)
    desc = coda.EpilogueDesc()
    desc.row_scale = rsd.data_ptr()
    desc.col_scale = csd.data_ptr()
    desc.aux_in[0] = Rd.data_ptr()
    desc.ld_aux_in[0] = N
    desc.aux_in[1] = X1d.data_ptr()
    desc.ld_aux_in[1] = N
    desc.row_coef = coefd.data_ptr()
    # bf16 output with row sum-of-squares partials
    D = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    desc.partials = part.data_ptr()
    desc.ld_partials = M
    coda.gemm_epilogue(desc, Ad, Bd, D, M, N, K)
    ref = O.gemm_epilogue_plain(to_np(A), to_np(B), to_np(rs), to_np(cs), to_np(R), to_np(coef), to_np(X1))
    assert_bf16(D, ref, "D (rs, cs, residual, coef)")
    ss = part.view(-1, M).sum(0)
    assert_f32(ss, (ref ** 2).sum(axis=1), "row sum of squares partials", tol=1e-2)
    # fp32 output accumulated into existing D (beta = 1)
    desc.partials = None
    desc.beta = 1
    Df = D0.to(dev)
    coda.gemm_epilogue(desc, Ad, Bd, Df, M, N, K)
    torch.cuda.synchronize()
    ref_f = O.gemm_epilogue_plain(to_np(A), to_np(B), to_np(rs), to_np(cs), to_np(R), to_np(coef), to_np(X1),
                                  to_np(D0))
    assert_bf16(Df, ref_f, "D fp32 beta accumulate")


@pytest.mark.parametrize("a_major,b_major", [(0, 0), (0, 1), (1, 1)])
def test_concatenated_k(coda, a_major, b_major):
    M, N, K1, K2 = 264, 256, 192, 136
    dev = "cuda"
    A1 = randn_bf16((M, K1), 1.0, 31)
    A2 = randn_bf16((M, K2), 1.0, 32)
    B1 = randn_bf16((N, K1), 0.1, 33)
    B2 = randn_bf16((N, K2), 0.1, 34)
    a1, a2 = _operand(A1, a_major).to(dev), _operand(A2, a_major).to(dev)
    b1, b2 = _operand(B1, b_major).to(dev), _operand(B2, b_major).to(dev)
    D = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    desc = coda.EpilogueDesc()
    desc.A2 = a2.data_ptr()
    desc.lda2 = K2 if a_major == 0 else M
    desc.B2 = b2.data_ptr()
    desc.ldb2 = K2 if b_major == 0 else N
    desc.K2 = K2
    coda.gemm_epilogue(desc, a1, b1, D, M, N, K1, a_major=a_major, b_major=b_major)
    torch.cuda.synchronize()
    ref = O.gemm_epilogue_plain(to_np(A1), to_np(B1)) + O.gemm_epilogue_plain(to_np(A2), to_np(B2))
    assert_bf16(D, ref, "concatenated K")


def test_large_k_many_tiles(coda):
    """Several waves of persistent tiles, K spanning many pipeline stages."""
    M, N, K = 1024, 2048, 2048
    dev = "cuda"
    A = randn_bf16((M, K), 1.0, 41)
    B = randn_bf16((N, K), 1.0 / np.sqrt(K), 42)
    D = torch.empty(M, N, dtype=torch.bfloat16, device=dev)
    ws = coda.gemm_epilogue(coda.EpilogueDesc(), A.to(dev), B.to(dev), D, M, N, K)
    assert coda.get_status(ws) == 0
    assert_bf16(D, O.gemm_epilogue_plain(to_np(A), to_np(B)), "D 1024x2048x2048")


@pytest.mark.parametrize("a_major,b_major", [(0, 0), (1, 1), (0, 1)])
@pytest.mark.parametrize("M", [129, 255, 257, 383, 511, 513, 700])
def test_cluster_boundaries_and_no_stray_writes(coda, a_major, b_major, M):
    """M around the single-CTA / CTA-pair / two-pair switch points (128, 256,
    512 rows), where the second pair of a 4-CTA cluster can lie partly or
    wholly past M.  D is a window of a larger buffer (row stride N + 24):
    every element outside the M x N window must keep its sentinel."""
    N, K = 264, 200
    dev = "cuda"
    A = randn_bf16((M, K), 1.0, 51)
    B = randn_bf16((N, K), 1.0 / np.sqrt(K), 52)
    full = torch.full((M + 40, N + 24), 7.0, dtype=torch.bfloat16, device=dev)
    # an MN-major A is [K, M] with its row stride padded to a multiple of 8
    # elements (16 bytes, the tensor-map stride rule)
    lda = None
    Ad = _operand(A, a_major)
    if a_major == 1:
        lda = (M + 7) // 8 * 8
        Ad = torch.zeros(K, lda, dtype=torch.bfloat16)
        Ad[:, :M] = A.t()
    # the output starts at full[0, 0] with row stride N + 24
    ws = coda.gemm_epilogue(coda.EpilogueDesc(), Ad.to(dev), _operand(B, b_major).to(dev), full,
                            M, N, K, a_major=a_major, b_major=b_major, lda=lda, ldd=N + 24)
    torch.cuda.synchronize()
    assert coda.get_status(ws) == 0
    assert_bf16(full[:M, :N], O.gemm_epilogue_plain(to_np(A), to_np(B)), f"D M={M}")
    assert bool((full[M:] == 7.0).all()), "write below row M"
    assert bool((full[:, N:] == 7.0).all()), "write right of column N"


@pytest.mark.parametrize("M", [257, 513, 700])
def test_swiglu_cluster_boundaries(coda, M):
    """The gate/up pair split across the CTAs of 2- and 4-CTA clusters."""
    I, K = 264, 200
    dev = "cuda"
    X = randn_bf16((M, K), 1.0, 61)
    Wg = randn_bf16((I, K), 1.0 / np.sqrt(K), 62)
    Wu = randn_bf16((I, K), 1.0 / np.sqrt(K), 63)
    H, g, u = coda.linear_swiglu(X.to(dev), Wg.to(dev), Wu.to(dev))
    torch.cuda.synchronize()
    ref = O.swiglu_fwd(to_np(X), to_np(Wg), to_np(Wu))
    assert_bf16(H, ref[0], f"H M={M}")


@pytest.mark.parametrize("a_major,b_major", [(0, 0), (1, 1), (0, 1)])
@pytest.mark.parametrize("M,N", [(500, 36 * 256 + 200), (300, 36 * 256 + 8)])
def test_split_launch_ragged(coda, a_major, b_major, M, N):
    """A GEMM that takes a split launch on a 152-SM GB300: one two-pair tile
    row and 37 N tiles -- 36 for the 36 resident 4-CTA clusters, the last,
    ragged tile for a CTA-pair kernel beside them (one wave instead of two).
    Parity, and nothing written outside the M x N window of a larger
    buffer."""
    K = 136
    dev = "cuda"
    A = randn_bf16((M, K), 1.0, 81)
    B = randn_bf16((N, K), 1.0 / np.sqrt(K), 82)
    full = torch.full((M + 24, N + 40), 7.0, dtype=torch.bfloat16, device=dev)
    lda = None
    Ad = _operand(A, a_major)
    if a_major == 1:
        lda = (M + 7) // 8 * 8
        Ad = torch.zeros(K, lda, dtype=torch.bfloat16)
        Ad[:, :M] = A.t()
    ws = coda.gemm_epilogue(coda.EpilogueDesc(), Ad.to(dev), _operand(B, b_major).to(dev), full, M, N, K,
                            a_major=a_major, b_major=b_major, lda=lda, ldd=N + 40)
    torch.cuda.synchronize()
    assert coda.get_status(ws) == 0
    assert_bf16(full[:M, :N], O.gemm_epilogue_plain(to_np(A), to_np(B)), f"D {M}x{N}")
    assert bool((full[M:] == 7.0).all()), "write below row M"
    assert bool((full[:, N:] == 7.0).all()), "write right of column N"


def test_split_launch_swiglu_and_partials(coda):
    """Split launches on the gate/up dual-B tile (I = 36 * 128 + 72: 37
    half-tiles) and on a residual epilogue whose row partials (the next
    RMSNorm's r) come from both slices."""
    M, I, K = 500, 36 * 128 + 72, 136
    dev = "cuda"
    X = randn_bf16((M, K), 1.0, 91)
    Wg = randn_bf16((I, K), 1.0 / np.sqrt(K), 92)
    Wu = randn_bf16((I, K), 1.0 / np.sqrt(K), 93)
    H, g, u = coda.linear_swiglu(X.to(dev), Wg.to(dev), Wu.to(dev))
    N = 36 * 256 + 200
    R = randn_bf16((M, N), 1.0, 94)
    W = randn_bf16((N, K), 1.0 / np.sqrt(K), 95)
    Y, r = coda.linear_residual(X.to(dev), W.to(dev), R.to(dev), eps=1e-6, want_rstd=True)
    torch.cuda.synchronize()
    ref = O.swiglu_fwd(to_np(X), to_np(Wg), to_np(Wu))
    assert_bf16(H, ref[0], "H")
    yr, rr = O.linear_residual_fwd(to_np(X), to_np(W), to_np(R), 1e-6)
    assert_bf16(Y, yr, "Y")
    assert_f32(r, rr, "rstd from both slices' partials")
