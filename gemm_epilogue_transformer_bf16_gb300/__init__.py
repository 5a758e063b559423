"""Python binding of libcoda.so (C ABI in include/coda.h).

Argument marshalling only: every step of every operator runs in the CUDA
kernels of libcoda.so.  PyTorch supplies device memory and the current
stream.  There is no CPU or PyTorch fallback: if the library is missing or a
tensor is not on a CUDA device, calls raise.

Function names mirror the C entry points without the ``coda_`` prefix.
Tensors must be contiguous, bf16 tensors ``torch.bfloat16``, vectors
``torch.float32``, labels/positions ``torch.int32``.  Workspaces are allocated
with torch (the library never allocates) unless the caller passes ``ws=``.
"""
from __future__ import annotations

import ctypes
import os

import torch

from ._build import LIB as _LIB_PATH

__all__ = [
    "load", "CodaError", "lib_path", "status_string", "get_status", "reset_status",
    "fold_gamma", "rms_rstd", "rmsnorm_scale", "rope_table", "gemm_epilogue", "EpilogueDesc",
    "rmsnorm_linear", "rmsnorm_linear_bwd", "linear_residual", "linear_residual_bwd",
    "linear_swiglu", "linear_swiglu_bwd", "linear_qknorm_rope", "linear_qknorm_rope_bwd",
    "ROPE_INTERLEAVED", "ROPE_HALF",
    "linear_cross_entropy", "linear_cross_entropy_bwd", "linear_cross_entropy_noalloc", "workspace",
    "rmsnorm_linear_cross_entropy", "rmsnorm_linear_cross_entropy_bwd", "rms_rstd",
    "linear_sigmoid", "linear_sigmoid_bwd", "quantize_fp8_rows", "linear_fp8", "linear_swiglu_fp8", "quantize_nvfp4_rows", "rmsnorm_scale_nvfp4", "linear_nvfp4",
    "linear_swiglu_nvfp4", "quantize_fp8_cols", "linear_qknorm_rope_fp8", "linear_cross_entropy_fp8",
    "linear_cross_entropy_bwd_fp8", "linear_dswiglu_fp8", "rmsnorm_linear_dx_fp8",
    "linear_qknorm_rope_bwd_fp8", "launch_count",
    "MAP_NONE", "MAP_SWIGLU", "MAP_DSWIGLU", "MAP_QKNORM_ROPE", "MAP_CE_LSE",
    "MAP_CE_DLOGITS", "MAP_COLDOT", "MAP_SIGMOID", "MAP_DSIGMOID", "K_MAJOR", "MN_MAJOR",
]

K_MAJOR, MN_MAJOR = 0, 1
BF16, F32 = 0, 1
(MAP_NONE, MAP_SWIGLU, MAP_DSWIGLU, MAP_QKNORM_ROPE, MAP_CE_LSE, MAP_CE_DLOGITS,
 MAP_COLDOT, MAP_SIGMOID, MAP_DSIGMOID) = range(9)

_P = ctypes.c_void_p
_I64 = ctypes.c_int64
_I32 = ctypes.c_int32
_F = ctypes.c_float
_SZ = ctypes.c_size_t

# name -> argtypes (restype int unless noted)
_SIGS = {
    "coda_version": ([], ctypes.c_char_p),
    "coda_launch_count": ([], ctypes.c_uint64),
    "coda_status_string": ([ctypes.c_int], ctypes.c_char_p),
    "coda_get_status": ([_P, _P], ctypes.c_int),
    "coda_reset_status": ([_P, _P], ctypes.c_int),
    "coda_selftest_wait_timeout": ([ctypes.c_uint32, _P, _P], ctypes.c_int),
    "coda_gemm_epilogue_workspace_size": ([], _SZ),
    "coda_gemm_epilogue": ([_P, _P, _I64, ctypes.c_int, _P, _I64, ctypes.c_int, _P, _I64, ctypes.c_int,
                            _I64, _I64, _I64, _P, _SZ, _P], ctypes.c_int),
    "coda_fold_gamma": ([_P, _P, _P, _I64, _I64, _P], ctypes.c_int),
    "coda_rms_rstd": ([_P, _I64, _I64, _I64, _F, _P, _P], ctypes.c_int),
    "coda_rmsnorm_scale": ([_P, _I64, _I64, _I64, _F, _P, _P, _P, _I64, _P], ctypes.c_int),
    "coda_rope_table": ([_F, _I32, _I32, _P, _P], ctypes.c_int),
    "coda_rmsnorm_linear_workspace_size": ([_I64, _I64, _I64], _SZ),
    "coda_rmsnorm_linear": ([_P, _P, _P, _P, _F, _P, _P, _I64, _I64, _I64, _P, _SZ, _P], ctypes.c_int),
    "coda_rmsnorm_linear_bwd_workspace_size": ([_I64, _I64, _I64], _SZ),
    "coda_rmsnorm_linear_bwd": ([_P] * 10 + [_I64, _I64, _I64, _P, _SZ, _P, _P], ctypes.c_int),
    "coda_linear_residual_workspace_size": ([_I64, _I64, _I64], _SZ),
    "coda_linear_residual": ([_P, _P, _P, _P, _F, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P], ctypes.c_int),
    "coda_linear_residual_bwd_workspace_size": ([_I64, _I64, _I64], _SZ),
    "coda_linear_residual_bwd": ([_P] * 5 + [_I64, _I64, _I64, _P, _SZ, _P], ctypes.c_int),
    "coda_linear_swiglu_workspace_size": ([_I64, _I64, _I64], _SZ),
    "coda_linear_swiglu": ([_P] * 7 + [_I64, _I64, _I64, _P, _SZ, _P], ctypes.c_int),
    "coda_linear_swiglu_bwd_workspace_size": ([_I64, _I64, _I64], _SZ),
    "coda_linear_swiglu_bwd": ([_P] * 16 + [_I64, _I64, _I64, _P, _SZ, _P, _P], ctypes.c_int),
    "coda_linear_qknorm_rope_workspace_size": ([_I64, _I64, _I32, _I32, _I32], _SZ),
    "coda_linear_qknorm_rope": ([_P] * 7 + [_I32, _F, _I32, _I32, _I32, _I32] + [_P] * 4 + [_I64, _I64, _P, _SZ, _P],
                                ctypes.c_int),
    "coda_linear_qknorm_rope_bwd_workspace_size": ([_I64, _I64, _I32, _I32, _I32], _SZ),
    "coda_linear_qknorm_rope_bwd": ([_P] * 9 + [_I32, _F, _I32, _I32, _I32, _I32] + [_P] * 10
                                    + [_I64, _I64, _P, _SZ, _P], ctypes.c_int),
    "coda_linear_cross_entropy_workspace_size": ([_I64, _I64, _I64], _SZ),
    "coda_linear_cross_entropy": ([_P, _P, _P, _I32, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P], ctypes.c_int),
    "coda_quantize_fp8_rows": ([_P, _I64, _I64, _I64, _P, _P, _P], ctypes.c_int),
    "coda_linear_fp8_workspace_size": ([_I64, _I64, _I64], _SZ),
    "coda_linear_fp8": ([_P] * 6 + [_I64, _I64, _I64, _P, _SZ, _P], ctypes.c_int),
    "coda_linear_swiglu_fp8_workspace_size": ([_I64, _I64, _I64], _SZ),
    "coda_linear_swiglu_fp8": ([_P] * 10 + [_I64, _I64, _I64, _P, _SZ, _P], ctypes.c_int),
    "coda_quantize_fp8_cols": ([_P, _I64, _I64, _P, _I64, _I64, _I64, _P, _I64, _P, _P], ctypes.c_int),
    "coda_linear_qknorm_rope_fp8_workspace_size": ([_I64, _I64, _I32, _I32, _I32], _SZ),
    "coda_linear_qknorm_rope_fp8": ([_P] * 9 + [_I32, _F, _I32, _I32, _I32, _I32] + [_P] * 4
                                    + [_I64, _I64, _P, _SZ, _P], ctypes.c_int),
    "coda_linear_cross_entropy_fp8_workspace_size": ([_I64, _I64, _I64], _SZ),
    "coda_linear_cross_entropy_fp8": ([_P] * 5 + [_I32, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P], ctypes.c_int),
    "coda_linear_cross_entropy_bwd_fp8_workspace_size": ([_I64, _I64, _I64], _SZ),
    "coda_linear_cross_entropy_bwd_fp8": ([_P] * 7 + [_I32, _P, _P, _F, _P, _P, _I64, _I64, _I64, _P, _SZ, _P],
                                          ctypes.c_int),
    "coda_linear_dswiglu_fp8_workspace_size": ([_I64, _I64, _I64], _SZ),
    "coda_linear_dswiglu_fp8": ([_P] * 10 + [_I64, _I64, _I64, _P, _SZ, _P], ctypes.c_int),
    "coda_rmsnorm_linear_dx_fp8_workspace_size": ([_I64, _I64, _I64], _SZ),
    "coda_rmsnorm_linear_dx_fp8": ([_P] * 10 + [_I64, _I64, _I64, _P, _SZ, _P], ctypes.c_int),
    "coda_linear_qknorm_rope_bwd_fp8_workspace_size": ([_I64, _I64, _I32, _I32, _I32], _SZ),
    "coda_linear_qknorm_rope_bwd_fp8": ([_P] * 9 + [_I32, _F, _I32, _I32, _I32, _I32] + [_P] * 13
                                        + [_I64, _I64, _P, _SZ, _P], ctypes.c_int),
    "coda_nvfp4_scale_bytes": ([_I64, _I64], _SZ),
    "coda_quantize_nvfp4_rows": ([_P, _I64, _I64, _I64, _P, _P, _P, _P], ctypes.c_int),
    "coda_rmsnorm_scale_nvfp4": ([_P, _I64, _I64, _I64, _F, _P, _P, _P, _P, _P, _P], ctypes.c_int),
    "coda_linear_nvfp4_workspace_size": ([_I64, _I64, _I64], _SZ),
    "coda_linear_nvfp4": ([_P] * 8 + [_I64, _I64, _I64, _P, _SZ, _P], ctypes.c_int),
    "coda_linear_swiglu_nvfp4_workspace_size": ([_I64, _I64, _I64], _SZ),
    "coda_linear_swiglu_nvfp4": ([_P] * 13 + [_I64, _I64, _I64, _P, _SZ, _P], ctypes.c_int),
    "coda_linear_sigmoid_workspace_size": ([_I64, _I64, _I64], _SZ),
    "coda_linear_sigmoid": ([_P, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P], ctypes.c_int),
    "coda_linear_sigmoid_bwd_workspace_size": ([_I64, _I64, _I64], _SZ),
    "coda_linear_sigmoid_bwd": ([_P] * 7 + [_I64, _I64, _I64, _P, _SZ, _P], ctypes.c_int),
    "coda_rmsnorm_linear_cross_entropy_workspace_size": ([_I64, _I64, _I64], _SZ),
    "coda_rmsnorm_linear_cross_entropy": ([_P, _P, _P, _P, _I32, _P, _P, _P, _I64, _I64, _I64, _P, _SZ, _P],
                                          ctypes.c_int),
    "coda_rmsnorm_linear_cross_entropy_bwd_workspace_size": ([_I64, _I64, _I64], _SZ),
    "coda_rmsnorm_linear_cross_entropy_bwd": ([_P, _P, _P, _P, _P, _P, _I32, _P, _P, _F, _P, _P, _P, _P,
                                               _I64, _I64, _I64, _P, _SZ, _P], ctypes.c_int),
    "coda_noalloc_scratch_bytes": ([], _SZ),
    "coda_linear_cross_entropy_noalloc": ([_P, _P, _P, _I32, _P, _P, _P, _P, _I64, _I64, _I64, _P], ctypes.c_int),
    "coda_linear_cross_entropy_bwd_workspace_size": ([_I64, _I64, _I64], _SZ),
    "coda_linear_cross_entropy_bwd": ([_P, _P, _P, _I32, _P, _P, _F, _P, _P, _I64, _I64, _I64, _P, _SZ, _P],
                                      ctypes.c_int),
}


class CodaError(RuntimeError):
    def __init__(self, fn, code):
        self.code = code
        super().__init__(f"{fn} failed: {status_string(code)} ({code})")


_lib = None


def lib_path():
    return _LIB_PATH


def load():
    """Load libcoda.so (raises if it was not built)."""
    global _lib
    if _lib is None:
        if not os.path.exists(_LIB_PATH):
            raise RuntimeError(f"{_LIB_PATH} is missing: build it with __graft_entry__.build() "
                               "(there is no fallback implementation)")
        lib = ctypes.CDLL(_LIB_PATH)
        for name, (args, res) in _SIGS.items():
            f = getattr(lib, name)
            f.argtypes = args
            f.restype = res
        _lib = lib
    return _lib


def status_string(code):
    return load().coda_status_string(int(code)).decode()


class EpilogueDesc(ctypes.Structure):
    _fields_ = [
        ("map", _I32), ("row_scale", _P), ("col_scale", _P),
        ("aux_in", _P * 2), ("ld_aux_in", _I64 * 2), ("row_coef", _P),
        ("aux_out", _P * 3), ("ld_aux_out", _I64 * 3), ("partials", _P), ("ld_partials", _I64),
        ("beta", _I32), ("B2", _P), ("ldb2", _I64), ("A2", _P), ("lda2", _I64), ("K2", _I64),
        ("labels", _P), ("ignore_index", _I32), ("lse", _P), ("n_valid", _P), ("dloss", _F),
        ("target_logit", _P), ("vocab_tiles_per_unit", _I32),
        ("positions", _P), ("cos_sin", _P), ("max_pos", _I32), ("n_q_heads", _I32),
        ("n_kv_heads", _I32), ("head_dim", _I32), ("eps", _F), ("gamma_q", _P), ("gamma_k", _P),
        ("Q", _P), ("K", _P), ("V", _P), ("rope_pairing", _I32),
        ("operand_type", _I32), ("acc_row_scale", _P), ("acc_col_scale", _P),
    ]


# ---------------------------------------------------------------------------
# marshalling helpers
# ---------------------------------------------------------------------------

def _ptr(t, dtype=None, name="tensor"):
    if t is None:
        return None
    if not isinstance(t, torch.Tensor):
        raise TypeError(f"{name}: expected a torch.Tensor")
    if not t.is_cuda:
        raise ValueError(f"{name}: must be a CUDA tensor (no CPU path)")
    if dtype is not None and t.dtype != dtype:
        raise TypeError(f"{name}: expected {dtype}, got {t.dtype}")
    if not t.is_contiguous():
        raise ValueError(f"{name}: must be contiguous")
    return t.data_ptr()


def _bf(t, name="tensor"):
    return _ptr(t, torch.bfloat16, name)


def _f32(t, name="tensor"):
    return _ptr(t, torch.float32, name)


def _i32(t, name="tensor"):
    return _ptr(t, torch.int32, name)


def _stream(stream=None):
    s = stream if stream is not None else torch.cuda.current_stream()
    return s.cuda_stream


def _check(fn, code):
    if code != 0:
        raise CodaError(fn, code)


def workspace(nbytes, device=None):
    """A zeroed byte workspace (status word cleared) of at least nbytes."""
    return torch.zeros(max(int(nbytes), 256), dtype=torch.uint8, device=device or "cuda")


def _ws(ws, need, device):
    if ws is None:
        return workspace(need, device)
    if ws.numel() < need:
        raise ValueError(f"workspace too small: {ws.numel()} < {need}")
    return ws


def _rows(t):
    """[..., F] -> ([M, F], leading shape) for the token-major operands of the
    forward calls; 2-D tensors and None pass through (leading shape None)."""
    if t is None or t.dim() == 2:
        return t, None
    if not t.is_contiguous():          # a copy would drop what the kernel writes
        raise ValueError("tensors with leading dimensions must be contiguous")
    return t.view(-1, t.shape[-1]), tuple(t.shape[:-1])


def _lead(t, lead):
    """Back to the caller's leading shape: [M, F] -> [*lead, F], [M] -> lead."""
    if t is None or lead is None:
        return t
    return t.view(*lead, t.shape[-1]) if t.dim() == 2 else t.view(lead)


def _vec(t, lead):
    """A per-token vector given in the caller's leading shape, as [M]."""
    return t if (t is None or lead is None) else t.view(-1)


ROPE_INTERLEAVED, ROPE_HALF = 0, 1


def _pairing(p):
    """RoPE pairing name -> coda_rope_pairing: "interleaved" pairs (2j, 2j+1),
    "half" pairs (j, j + head_dim/2)."""
    try:
        return {"interleaved": ROPE_INTERLEAVED, "half": ROPE_HALF}[p]
    except KeyError:
        raise ValueError(f"RoPE pairing must be 'interleaved' or 'half', not {p!r}") from None


def get_status(ws, stream=None):
    return load().coda_get_status(_ptr(ws), _stream(stream))


def reset_status(ws, stream=None):
    _check("coda_reset_status", load().coda_reset_status(_ptr(ws), _stream(stream)))


def launch_count():
    """Kernels this library has launched in this process (coda_launch_count)."""
    return int(load().coda_launch_count())


# ---------------------------------------------------------------------------
# operators
# ---------------------------------------------------------------------------

def fold_gamma(W, gamma, out=None, stream=None):
    N, K = W.shape
    out = torch.empty_like(W) if out is None else out
    _check("coda_fold_gamma", load().coda_fold_gamma(_bf(W, "W"), _f32(gamma, "gamma"), _bf(out, "Wf"), N, K,
                                                     _stream(stream)))
    return out


def rms_rstd(X, eps, out=None, stream=None):
    M, K = X.shape
    out = torch.empty(M, dtype=torch.float32, device=X.device) if out is None else out
    _check("coda_rms_rstd", load().coda_rms_rstd(_bf(X, "X"), K, M, K, float(eps), _f32(out, "rstd"),
                                                 _stream(stream)))
    return out


def rmsnorm_scale(X, gamma, eps, rstd=None, U=None, stream=None):
    """rstd = 1/rms(X) per row and U = X ⊙ gamma in one pass (coda_rmsnorm_scale).
    X may have leading dimensions ([..., K]); the outputs keep them."""
    X, lead = _rows(X)
    U, _ = _rows(U)
    rstd = _vec(rstd, lead)
    M, K = X.shape
    rstd = torch.empty(M, dtype=torch.float32, device=X.device) if rstd is None else rstd
    U = torch.empty_like(X) if U is None else U
    _check("coda_rmsnorm_scale", load().coda_rmsnorm_scale(_bf(X, "X"), K, M, K, float(eps), _f32(gamma, "gamma"),
                                                           _f32(rstd, "rstd"), _bf(U, "U"), K, _stream(stream)))
    return _lead(rstd, lead), _lead(U, lead)


def rope_table(theta, head_dim, max_pos, device="cuda", out=None, stream=None):
    out = torch.empty(max_pos, head_dim // 2, 2, dtype=torch.float32, device=device) if out is None else out
    _check("coda_rope_table", load().coda_rope_table(float(theta), int(head_dim), int(max_pos),
                                                     _f32(out, "cos_sin"), _stream(stream)))
    return out


def gemm_epilogue(desc, A, B, D, M, N, K, a_major=K_MAJOR, b_major=K_MAJOR, lda=None, ldb=None, ldd=None,
                  ws=None, stream=None):
    """Generic GEMM + epilogue (coda_gemm_epilogue).  `desc` is an
    EpilogueDesc whose pointer fields hold data_ptr() values."""
    lib = load()
    lda = lda if lda is not None else (K if a_major == K_MAJOR else M)
    ldb = ldb if ldb is not None else (K if b_major == K_MAJOR else N)
    ldd = ldd if ldd is not None else N
    dtype = F32 if (D is not None and D.dtype == torch.float32) else BF16
    ws = _ws(ws, lib.coda_gemm_epilogue_workspace_size(), A.device)
    _check("coda_gemm_epilogue", lib.coda_gemm_epilogue(
        ctypes.byref(desc), _bf(A, "A"), lda, a_major, _bf(B, "B"), ldb, b_major,
        _ptr(D, None, "D"), ldd, dtype, M, N, K, _ptr(ws), ws.numel(), _stream(stream)))
    return ws


def rmsnorm_linear(X, Wf, R=None, rstd_in=None, eps=1e-6, rstd_out=None, Y=None, ws=None, stream=None):
    lib = load()
    M, K = X.shape
    N = Wf.shape[0]
    Y = torch.empty(M, N, dtype=torch.bfloat16, device=X.device) if Y is None else Y
    if rstd_in is None and rstd_out is None:
        rstd_out = torch.empty(M, dtype=torch.float32, device=X.device)
    ws = _ws(ws, lib.coda_rmsnorm_linear_workspace_size(M, N, K), X.device)
    _check("coda_rmsnorm_linear", lib.coda_rmsnorm_linear(
        _bf(X, "X"), _f32(rstd_in, "rstd_in"), _bf(Wf, "Wf"), _bf(R, "R"), float(eps), _f32(rstd_out, "rstd_out"),
        _bf(Y, "Y"), M, N, K, _ptr(ws), ws.numel(), _stream(stream)))
    return Y, (rstd_in if rstd_in is not None else rstd_out)


def rmsnorm_linear_bwd(dY, X, W, gamma, rstd, Y, R=None, ws=None, out=None, stream=None, side_stream=None):
    """RMSNorm-reparameterised projection backward (coda_rmsnorm_linear_bwd);
    `side_stream`: optional second torch.cuda.Stream for the dW GEMM."""
    lib = load()
    M, K = X.shape
    N = W.shape[0]
    if out is None:
        out = {"dX": torch.empty_like(X), "dW": torch.empty_like(W),
               "dgamma": torch.empty(K, dtype=torch.float32, device=X.device)}
    ws = _ws(ws, lib.coda_rmsnorm_linear_bwd_workspace_size(M, N, K), X.device)
    _check("coda_rmsnorm_linear_bwd", lib.coda_rmsnorm_linear_bwd(
        _bf(dY, "dY"), _bf(X, "X"), _bf(W, "W"), _f32(gamma, "gamma"), _f32(rstd, "rstd"),
        _bf(Y, "Y"), _bf(R, "R"), _bf(out["dX"], "dX"), _bf(out["dW"], "dW"), _f32(out["dgamma"], "dgamma"),
        M, N, K, _ptr(ws), ws.numel(), _stream(stream),
        side_stream.cuda_stream if side_stream is not None else None))
    return out


def linear_residual(X, W, R=None, eps=1e-6, want_rstd=False, Y=None, rstd_out=None, gamma_next=None, U_out=None,
                    ws=None, stream=None):
    """Y = R + X W^T (coda_linear_residual); optionally the row factor of the
    next RMSNorm (rstd_out / want_rstd) and U_out = Y ⊙ gamma_next.  X, R, Y,
    U_out may have leading dimensions ([..., features]); outputs keep them."""
    lib = load()
    X, lead = _rows(X)
    R, _ = _rows(R)
    Y, _ = _rows(Y)
    U_out, _ = _rows(U_out)
    rstd_out = _vec(rstd_out, lead)
    M, K = X.shape
    N = W.shape[0]
    Y = torch.empty(M, N, dtype=torch.bfloat16, device=X.device) if Y is None else Y
    if want_rstd and rstd_out is None:
        rstd_out = torch.empty(M, dtype=torch.float32, device=X.device)
    ws = _ws(ws, lib.coda_linear_residual_workspace_size(M, N, K), X.device)
    _check("coda_linear_residual", lib.coda_linear_residual(
        _bf(X, "X"), _bf(W, "W"), _bf(R, "R"), _bf(Y, "Y"), float(eps), _f32(rstd_out, "rstd_out"),
        _f32(gamma_next, "gamma_next"), _bf(U_out, "U_out"), M, N, K, _ptr(ws), ws.numel(), _stream(stream)))
    Y, rstd_out = _lead(Y, lead), _lead(rstd_out, lead)
    return (Y, rstd_out) if want_rstd or rstd_out is not None else Y


def linear_residual_bwd(dY, X, W, ws=None, out=None, stream=None):
    lib = load()
    M, K = X.shape
    N = W.shape[0]
    if out is None:
        out = {"dX": torch.empty_like(X), "dW": torch.empty_like(W)}
    ws = _ws(ws, lib.coda_linear_residual_bwd_workspace_size(M, N, K), X.device)
    _check("coda_linear_residual_bwd", lib.coda_linear_residual_bwd(
        _bf(dY, "dY"), _bf(X, "X"), _bf(W, "W"), _bf(out["dX"], "dX"), _bf(out["dW"], "dW"),
        M, N, K, _ptr(ws), ws.numel(), _stream(stream)))
    return out


def linear_swiglu(X, Wg, Wu, rstd=None, save=True, H=None, g=None, u=None, ws=None, stream=None):
    """H = silu(r ⊙ X Wg^T) ⊙ (r ⊙ X Wu^T) (coda_linear_swiglu), and g, u when
    `save`.  X may have leading dimensions ([..., K]); the outputs keep them."""
    lib = load()
    X, lead = _rows(X)
    H, _ = _rows(H)
    g, _ = _rows(g)
    u, _ = _rows(u)
    rstd = _vec(rstd, lead)
    M, K = X.shape
    I = Wg.shape[0]
    dev = X.device
    H = torch.empty(M, I, dtype=torch.bfloat16, device=dev) if H is None else H
    if save:
        g = torch.empty(M, I, dtype=torch.bfloat16, device=dev) if g is None else g
        u = torch.empty(M, I, dtype=torch.bfloat16, device=dev) if u is None else u
    ws = _ws(ws, lib.coda_linear_swiglu_workspace_size(M, I, K), dev)
    _check("coda_linear_swiglu", lib.coda_linear_swiglu(
        _bf(X, "X"), _f32(rstd, "rstd"), _bf(Wg, "Wg"), _bf(Wu, "Wu"), _bf(H, "H"), _bf(g, "g"), _bf(u, "u"),
        M, I, K, _ptr(ws), ws.numel(), _stream(stream)))
    return _lead(H, lead), _lead(g, lead), _lead(u, lead)


def linear_swiglu_bwd(dY, X, Wg, Wu, Wd, g, u, H, rstd=None, gamma=None, dX_resid=None, ws=None, out=None,
                      stream=None, side_stream=None):
    """SwiGLU MLP backward (coda_linear_swiglu_bwd); Wg, Wu not folded.
    `side_stream`: optional second torch.cuda.Stream for the weight-gradient
    GEMMs."""
    lib = load()
    M, K = X.shape
    I = Wg.shape[0]
    dev = X.device
    if out is None:
        out = {"dX": torch.empty_like(X), "dWg": torch.empty_like(Wg), "dWu": torch.empty_like(Wu),
               "dWd": torch.empty_like(Wd),
               "dgamma": torch.empty(K, dtype=torch.float32, device=dev) if rstd is not None else None}
    ws = _ws(ws, lib.coda_linear_swiglu_bwd_workspace_size(M, I, K), dev)
    _check("coda_linear_swiglu_bwd", lib.coda_linear_swiglu_bwd(
        _bf(dY, "dY"), _bf(X, "X"), _f32(rstd, "rstd"), _f32(gamma, "gamma"), _bf(Wg, "Wg"), _bf(Wu, "Wu"),
        _bf(Wd, "Wd"), _bf(g, "g"), _bf(u, "u"), _bf(H, "H"), _bf(dX_resid, "dX_resid"), _bf(out["dX"], "dX"),
        _bf(out["dWg"], "dWg"), _bf(out["dWu"], "dWu"), _bf(out["dWd"], "dWd"), _f32(out.get("dgamma"), "dgamma"),
        M, I, K, _ptr(ws), ws.numel(), _stream(stream),
        side_stream.cuda_stream if side_stream is not None else None))
    return out


def linear_qknorm_rope(X, W, gamma_q, gamma_k, pos, cos_sin, n_q, n_kv, rstd=None, eps=1e-6,
                       head_dim=128, save=True, out=None, ws=None, stream=None, pairing="interleaved"):
    """QKV projection with per-head QK-RMSNorm and RoPE in the epilogue
    (coda_linear_qknorm_rope).  X may have leading dimensions ([..., Kdim],
    pos [...]); when it does and `out` is not given, Q, K, V, qk_save keep
    them."""
    lib = load()
    X, lead = _rows(X)
    pos = _vec(pos, lead)
    rstd = _vec(rstd, lead)
    M, Kd = X.shape
    dev = X.device
    shaped = out is None and lead is not None
    if out is None:
        out = {"Q": torch.empty(M, n_q * head_dim, dtype=torch.bfloat16, device=dev),
               "K": torch.empty(M, n_kv * head_dim, dtype=torch.bfloat16, device=dev),
               "V": torch.empty(M, n_kv * head_dim, dtype=torch.bfloat16, device=dev),
               "qk_save": torch.empty(M, (n_q + n_kv) * head_dim, dtype=torch.bfloat16, device=dev)
               if save else None}
    max_pos = cos_sin.shape[0]
    ws = _ws(ws, lib.coda_linear_qknorm_rope_workspace_size(M, Kd, n_q, n_kv, head_dim), dev)
    _check("coda_linear_qknorm_rope", lib.coda_linear_qknorm_rope(
        _bf(X, "X"), _f32(rstd, "rstd"), _bf(W, "W"), _f32(gamma_q, "gamma_q"),
        _f32(gamma_k, "gamma_k"), _i32(pos, "pos"), _f32(cos_sin, "cos_sin"), max_pos, float(eps),
        n_q, n_kv, head_dim, _pairing(pairing), _bf(out["Q"], "Q"), _bf(out["K"], "K"), _bf(out["V"], "V"),
        _bf(out.get("qk_save"), "qk_save"), M, Kd, _ptr(ws), ws.numel(), _stream(stream)))
    if shaped:
        out = {k: _lead(v, lead) for k, v in out.items()}
    return out


def linear_qknorm_rope_bwd(dQ, dK, dV, qk_save, V, gamma_q, gamma_k, pos, cos_sin, n_q, n_kv, X, W_qkv,
                           rstd=None, gamma_in=None, dX_resid=None, eps=1e-6, head_dim=128, ws=None, out=None,
                           stream=None, pairing="interleaved"):
    """QK-RMSNorm + RoPE projection backward (coda_linear_qknorm_rope_bwd);
    W_qkv not folded."""
    lib = load()
    M, Kd = X.shape
    dev = X.device
    if out is None:
        out = {"dX": torch.empty_like(X), "dW": torch.empty_like(W_qkv),
               "dgamma_in": torch.empty(Kd, dtype=torch.float32, device=dev) if rstd is not None else None,
               "dgamma_q": torch.empty(head_dim, dtype=torch.float32, device=dev),
               "dgamma_k": torch.empty(head_dim, dtype=torch.float32, device=dev)}
    max_pos = cos_sin.shape[0]
    ws = _ws(ws, lib.coda_linear_qknorm_rope_bwd_workspace_size(M, Kd, n_q, n_kv, head_dim), dev)
    _check("coda_linear_qknorm_rope_bwd", lib.coda_linear_qknorm_rope_bwd(
        _bf(dQ, "dQ"), _bf(dK, "dK"), _bf(dV, "dV"), _bf(qk_save, "qk_save"), _bf(V, "V"),
        _f32(gamma_q, "gamma_q"), _f32(gamma_k, "gamma_k"), _i32(pos, "pos"), _f32(cos_sin, "cos_sin"),
        max_pos, float(eps), n_q, n_kv, head_dim, _pairing(pairing), _bf(X, "X"), _f32(rstd, "rstd"),
        _f32(gamma_in, "gamma_in"),
        _bf(W_qkv, "W_qkv"), _bf(dX_resid, "dX_resid"), _bf(out["dX"], "dX"), _bf(out["dW"], "dW"),
        _f32(out.get("dgamma_in"), "dgamma_in"), _f32(out["dgamma_q"], "dgamma_q"), _f32(out["dgamma_k"], "dgamma_k"),
        M, Kd, _ptr(ws), ws.numel(), _stream(stream)))
    return out


def linear_cross_entropy(X, W, labels, ignore_index=-100, out=None, ws=None, stream=None):
    """Mean token cross-entropy of softmax(X W^T) against `labels` with an
    online log-sum-exp; logits never reach HBM (coda_linear_cross_entropy).
    X may have leading dimensions ([..., K], labels [...]); when it does and
    `out` is not given, lse keeps them."""
    lib = load()
    X, lead = _rows(X)
    labels = _vec(labels, lead)
    M, K = X.shape
    shaped = out is None and lead is not None
    V = W.shape[0]
    dev = X.device
    if out is None:
        out = {"loss": torch.empty(1, dtype=torch.float32, device=dev),
               "lse": torch.empty(M, dtype=torch.float32, device=dev),
               "n_valid": torch.empty(1, dtype=torch.int32, device=dev)}
    ws = _ws(ws, lib.coda_linear_cross_entropy_workspace_size(M, V, K), dev)
    _check("coda_linear_cross_entropy", lib.coda_linear_cross_entropy(
        _bf(X, "X"), _bf(W, "W"), _i32(labels, "labels"), int(ignore_index), _f32(out["loss"], "loss"),
        _f32(out["lse"], "lse"), _i32(out["n_valid"], "n_valid"), M, V, K, _ptr(ws), ws.numel(),
        _stream(stream)))
    out["ws"] = ws
    if shaped:
        out["lse"] = out["lse"].reshape(lead)
    return out


def _u8(t, name="tensor"):
    return _ptr(t, torch.uint8, name)


def quantize_fp8_rows(X, Xq=None, scale=None, stream=None):
    """Per-row e4m3 quantisation: returns (codes uint8 [M, K], scale fp32 [M])."""
    M, K = X.shape
    Xq = torch.empty(M, K, dtype=torch.uint8, device=X.device) if Xq is None else Xq
    scale = torch.empty(M, dtype=torch.float32, device=X.device) if scale is None else scale
    _check("coda_quantize_fp8_rows", load().coda_quantize_fp8_rows(_bf(X, "X"), K, M, K, _u8(Xq, "Xq"),
                                                                   _f32(scale, "scale"), _stream(stream)))
    return Xq, scale


def linear_fp8(Xq, sx, Wq, sw, R=None, Y=None, ws=None, stream=None):
    lib = load()
    M, K = Xq.shape
    N = Wq.shape[0]
    Y = torch.empty(M, N, dtype=torch.bfloat16, device=Xq.device) if Y is None else Y
    ws = _ws(ws, lib.coda_linear_fp8_workspace_size(M, N, K), Xq.device)
    _check("coda_linear_fp8", lib.coda_linear_fp8(_u8(Xq, "Xq"), _f32(sx, "sx"), _u8(Wq, "Wq"), _f32(sw, "sw"),
                                                  _bf(R, "R"), _bf(Y, "Y"), M, N, K, _ptr(ws), ws.numel(),
                                                  _stream(stream)))
    return Y


def linear_swiglu_fp8(Xq, sx, Wgq, sg, Wuq, su, rstd=None, save=True, H=None, g=None, u=None, ws=None,
                      stream=None):
    lib = load()
    M, K = Xq.shape
    I = Wgq.shape[0]
    dev = Xq.device
    H = torch.empty(M, I, dtype=torch.bfloat16, device=dev) if H is None else H
    if save:
        g = torch.empty(M, I, dtype=torch.bfloat16, device=dev) if g is None else g
        u = torch.empty(M, I, dtype=torch.bfloat16, device=dev) if u is None else u
    ws = _ws(ws, lib.coda_linear_swiglu_fp8_workspace_size(M, I, K), dev)
    _check("coda_linear_swiglu_fp8", lib.coda_linear_swiglu_fp8(
        _u8(Xq, "Xq"), _f32(sx, "sx"), _f32(rstd, "rstd"), _u8(Wgq, "Wgq"), _f32(sg, "sg"), _u8(Wuq, "Wuq"),
        _f32(su, "su"), _bf(H, "H"), _bf(g, "g"), _bf(u, "u"), M, I, K, _ptr(ws), ws.numel(), _stream(stream)))
    return H, g, u


def quantize_fp8_cols(X, X2=None, XTq=None, scale=None, stream=None):
    """Per-column e4m3 quantisation of X [R, C] (with X2 [R2, C] stacked
    below it): returns (codes uint8 [C, R + R2] of the transpose, scale fp32
    [C]) -- the K-major operand of a GEMM that contracts over X's rows."""
    R, C = X.shape
    R2 = 0 if X2 is None else X2.shape[0]
    XTq = torch.empty(C, R + R2, dtype=torch.uint8, device=X.device) if XTq is None else XTq
    scale = torch.empty(C, dtype=torch.float32, device=X.device) if scale is None else scale
    _check("coda_quantize_fp8_cols", load().coda_quantize_fp8_cols(
        _bf(X, "X"), X.stride(0), R, _bf(X2, "X2"), X2.stride(0) if X2 is not None else 0, R2, C,
        _u8(XTq, "XTq"), XTq.stride(0), _f32(scale, "scale"), _stream(stream)))
    return XTq, scale


def linear_qknorm_rope_fp8(Xq, sx, Wq, sw, gamma_q, gamma_k, pos, cos_sin, n_q, n_kv, rstd=None, eps=1e-6,
                           head_dim=128, save=True, out=None, ws=None, stream=None, pairing="interleaved"):
    """linear_qknorm_rope on e4m3 operands (coda_linear_qknorm_rope_fp8)."""
    lib = load()
    M, Kd = Xq.shape
    dev = Xq.device
    if out is None:
        out = {"Q": torch.empty(M, n_q * head_dim, dtype=torch.bfloat16, device=dev),
               "K": torch.empty(M, n_kv * head_dim, dtype=torch.bfloat16, device=dev),
               "V": torch.empty(M, n_kv * head_dim, dtype=torch.bfloat16, device=dev),
               "qk_save": torch.empty(M, (n_q + n_kv) * head_dim, dtype=torch.bfloat16, device=dev)
               if save else None}
    ws = _ws(ws, lib.coda_linear_qknorm_rope_fp8_workspace_size(M, Kd, n_q, n_kv, head_dim), dev)
    _check("coda_linear_qknorm_rope_fp8", lib.coda_linear_qknorm_rope_fp8(
        _u8(Xq, "Xq"), _f32(sx, "sx"), _f32(rstd, "rstd"), _u8(Wq, "Wq"), _f32(sw, "sw"),
        _f32(gamma_q, "gamma_q"), _f32(gamma_k, "gamma_k"), _i32(pos, "pos"), _f32(cos_sin, "cos_sin"),
        cos_sin.shape[0], float(eps), n_q, n_kv, head_dim, _pairing(pairing), _bf(out["Q"], "Q"),
        _bf(out["K"], "K"), _bf(out["V"], "V"), _bf(out.get("qk_save"), "qk_save"), M, Kd, _ptr(ws), ws.numel(),
        _stream(stream)))
    return out


def linear_cross_entropy_fp8(Xq, sx, Wq, sw, labels, ignore_index=-100, out=None, ws=None, stream=None):
    """linear_cross_entropy on e4m3 operands (coda_linear_cross_entropy_fp8)."""
    lib = load()
    M, K = Xq.shape
    V = Wq.shape[0]
    dev = Xq.device
    if out is None:
        out = {"loss": torch.empty(1, dtype=torch.float32, device=dev),
               "lse": torch.empty(M, dtype=torch.float32, device=dev),
               "n_valid": torch.empty(1, dtype=torch.int32, device=dev)}
    ws = _ws(ws, lib.coda_linear_cross_entropy_fp8_workspace_size(M, V, K), dev)
    _check("coda_linear_cross_entropy_fp8", lib.coda_linear_cross_entropy_fp8(
        _u8(Xq, "Xq"), _f32(sx, "sx"), _u8(Wq, "Wq"), _f32(sw, "sw"), _i32(labels, "labels"), int(ignore_index),
        _f32(out["loss"], "loss"), _f32(out["lse"], "lse"), _i32(out["n_valid"], "n_valid"), M, V, K, _ptr(ws),
        ws.numel(), _stream(stream)))
    out["ws"] = ws
    return out


def linear_cross_entropy_bwd_fp8(Xq, sx, Wq, sw, X, W, labels, lse, n_valid, dloss=1.0, ignore_index=-100,
                                 out=None, ws=None, stream=None):
    """Backward with the logits recomputed from the e4m3 operands and dX, dW
    from the bf16 X, W (coda_linear_cross_entropy_bwd_fp8)."""
    lib = load()
    M, K = X.shape
    V = W.shape[0]
    if out is None:
        out = {"dX": torch.empty_like(X), "dW": torch.empty_like(W)}
    ws = _ws(ws, lib.coda_linear_cross_entropy_bwd_fp8_workspace_size(M, V, K), X.device)
    _check("coda_linear_cross_entropy_bwd_fp8", lib.coda_linear_cross_entropy_bwd_fp8(
        _u8(Xq, "Xq"), _f32(sx, "sx"), _u8(Wq, "Wq"), _f32(sw, "sw"), _bf(X, "X"), _bf(W, "W"),
        _i32(labels, "labels"), int(ignore_index), _f32(lse, "lse"), _i32(n_valid, "n_valid"), float(dloss),
        _bf(out["dX"], "dX"), _bf(out["dW"], "dW"), M, V, K, _ptr(ws), ws.numel(), _stream(stream)))
    out["ws"] = ws
    return out


def linear_dswiglu_fp8(dYq, sdy, WdTq, swd, g, u, rstd=None, want_row=True, want_H=False, out=None, ws=None,
                       stream=None):
    """dH GEMM on e4m3 operands with the dSwiGLU epilogue
    (coda_linear_dswiglu_fp8): returns {"Gp": [M, 2I] = r [dG | dU],
    "row": [M] (with rstd the RMSNorm-backward coefficient c, else the row
    sum) or None, "H": [M, I] or None}."""
    lib = load()
    M, K = dYq.shape
    I = WdTq.shape[0]
    dev = dYq.device
    if out is None:
        out = {"Gp": torch.empty(M, 2 * I, dtype=torch.bfloat16, device=dev),
               "row": torch.empty(M, dtype=torch.float32, device=dev) if want_row else None,
               "H": torch.empty(M, I, dtype=torch.bfloat16, device=dev) if want_H else None}
    ws = _ws(ws, lib.coda_linear_dswiglu_fp8_workspace_size(M, I, K), dev)
    _check("coda_linear_dswiglu_fp8", lib.coda_linear_dswiglu_fp8(
        _u8(dYq, "dYq"), _f32(sdy, "sdy"), _u8(WdTq, "WdTq"), _f32(swd, "swd"), _bf(g, "g"), _bf(u, "u"),
        _f32(rstd, "rstd"), _bf(out["Gp"], "Gp"), _f32(out.get("row"), "row"), _bf(out.get("H"), "H"), M, I, K,
        _ptr(ws), ws.numel(), _stream(stream)))
    return out


def rmsnorm_linear_dx_fp8(Gq, sg, WTq, sw, X, gamma, coef, dX_resid=None, out=None, ws=None, stream=None):
    """Input gradient of an RMSNorm-reparameterised projection on e4m3
    operands (coda_rmsnorm_linear_dx_fp8): returns {"dX", "dgamma"}."""
    lib = load()
    M, N = Gq.shape
    K = WTq.shape[0]
    dev = Gq.device
    if out is None:
        out = {"dX": torch.empty(M, K, dtype=torch.bfloat16, device=dev),
               "dgamma": torch.empty(K, dtype=torch.float32, device=dev)}
    ws = _ws(ws, lib.coda_rmsnorm_linear_dx_fp8_workspace_size(M, N, K), dev)
    _check("coda_rmsnorm_linear_dx_fp8", lib.coda_rmsnorm_linear_dx_fp8(
        _u8(Gq, "Gq"), _f32(sg, "sg"), _u8(WTq, "WTq"), _f32(sw, "sw"), _bf(X, "X"), _f32(gamma, "gamma"),
        _f32(coef, "coef"), _bf(dX_resid, "dX_resid"), _bf(out["dX"], "dX"), _f32(out["dgamma"], "dgamma"), M, N,
        K, _ptr(ws), ws.numel(), _stream(stream)))
    return out


def linear_qknorm_rope_bwd_fp8(dQ, dK, dV, qk_save, V, gamma_q, gamma_k, pos, cos_sin, n_q, n_kv, WTq, sw, UTq,
                               su, X=None, rstd=None, gamma_in=None, dX_resid=None, eps=1e-6, head_dim=128, ws=None,
                               out=None, stream=None, pairing="interleaved"):
    """QK-RMSNorm + RoPE projection backward with both GEMMs on e4m3 operands
    (coda_linear_qknorm_rope_bwd_fp8): WTq, sw = quantize_fp8_cols(W_qkv),
    UTq, su = quantize_fp8_cols(U) of the forward GEMM's input U (x ⊙ gamma_in
    with the input RMSNorm, x without).  X (the un-normalised input) is
    needed with rstd only.  Returns {"dX", "dW", "dgamma_in", "dgamma_q",
    "dgamma_k"}."""
    lib = load()
    Kd, M = UTq.shape
    dev = UTq.device
    nqkv = (n_q + 2 * n_kv) * head_dim
    if out is None:
        out = {"dX": torch.empty(M, Kd, dtype=torch.bfloat16, device=dev),
               "dW": torch.empty(nqkv, Kd, dtype=torch.bfloat16, device=dev),
               "dgamma_in": torch.empty(Kd, dtype=torch.float32, device=dev) if rstd is not None else None,
               "dgamma_q": torch.empty(head_dim, dtype=torch.float32, device=dev),
               "dgamma_k": torch.empty(head_dim, dtype=torch.float32, device=dev)}
    max_pos = cos_sin.shape[0]
    ws = _ws(ws, lib.coda_linear_qknorm_rope_bwd_fp8_workspace_size(M, Kd, n_q, n_kv, head_dim), dev)
    _check("coda_linear_qknorm_rope_bwd_fp8", lib.coda_linear_qknorm_rope_bwd_fp8(
        _bf(dQ, "dQ"), _bf(dK, "dK"), _bf(dV, "dV"), _bf(qk_save, "qk_save"), _bf(V, "V"),
        _f32(gamma_q, "gamma_q"), _f32(gamma_k, "gamma_k"), _i32(pos, "pos"), _f32(cos_sin, "cos_sin"),
        max_pos, float(eps), n_q, n_kv, head_dim, _pairing(pairing), _bf(X, "X"), _f32(rstd, "rstd"),
        _f32(gamma_in, "gamma_in"), _u8(WTq, "WTq"), _f32(sw, "sw"), _u8(UTq, "UTq"), _f32(su, "su"),
        _bf(dX_resid, "dX_resid"), _bf(out["dX"], "dX"), _bf(out["dW"], "dW"),
        _f32(out.get("dgamma_in"), "dgamma_in"), _f32(out["dgamma_q"], "dgamma_q"), _f32(out["dgamma_k"], "dgamma_k"),
        M, Kd, _ptr(ws), ws.numel(), _stream(stream)))
    return out


def quantize_nvfp4_rows(X, stream=None):
    """Per-row NVFP4 quantisation (coda_quantize_nvfp4_rows): returns (codes
    uint8 [M, K/2], two e2m1 codes per byte; block scales uint8 in the
    tensor-core order of include/coda.h; row scales fp32 [M])."""
    lib = load()
    M, K = X.shape
    dev = X.device
    Xq = torch.empty(M, K // 2, dtype=torch.uint8, device=dev)
    sf = torch.empty(max(lib.coda_nvfp4_scale_bytes(M, K), 16), dtype=torch.uint8, device=dev)
    scale = torch.empty(M, dtype=torch.float32, device=dev)
    _check("coda_quantize_nvfp4_rows", lib.coda_quantize_nvfp4_rows(
        _bf(X, "X"), X.stride(0), M, K, _u8(Xq, "Xq"), _u8(sf, "sf"), _f32(scale, "scale"), _stream(stream)))
    return Xq, sf, scale


def rmsnorm_scale_nvfp4(X, gamma, eps, stream=None):
    """One pass over X (coda_rmsnorm_scale_nvfp4): the NVFP4 codes, block
    scales and row scales of u = X ⊙ gamma, and rstd = 1/rms(X).  Returns
    (codes, block scales, row scales, rstd)."""
    lib = load()
    M, K = X.shape
    dev = X.device
    Xq = torch.empty(M, K // 2, dtype=torch.uint8, device=dev)
    sf = torch.empty(max(lib.coda_nvfp4_scale_bytes(M, K), 16), dtype=torch.uint8, device=dev)
    scale = torch.empty(M, dtype=torch.float32, device=dev)
    rstd = torch.empty(M, dtype=torch.float32, device=dev)
    _check("coda_rmsnorm_scale_nvfp4", lib.coda_rmsnorm_scale_nvfp4(
        _bf(X, "X"), X.stride(0), M, K, float(eps), _f32(gamma, "gamma"), _f32(rstd, "rstd"), _u8(Xq, "Xq"),
        _u8(sf, "sf"), _f32(scale, "scale"), _stream(stream)))
    return Xq, sf, scale, rstd


def linear_nvfp4(Xq, sfx, sx, Wq, sfw, sw, R=None, Y=None, ws=None, stream=None):
    """Y = R + X̂ Ŵᵀ on NVFP4 operands (coda_linear_nvfp4)."""
    lib = load()
    M, K = Xq.shape[0], 2 * Xq.shape[1]
    N = Wq.shape[0]
    Y = torch.empty(M, N, dtype=torch.bfloat16, device=Xq.device) if Y is None else Y
    ws = _ws(ws, lib.coda_linear_nvfp4_workspace_size(M, N, K), Xq.device)
    _check("coda_linear_nvfp4", lib.coda_linear_nvfp4(
        _u8(Xq, "Xq"), _u8(sfx, "sfx"), _f32(sx, "sx"), _u8(Wq, "Wq"), _u8(sfw, "sfw"), _f32(sw, "sw"),
        _bf(R, "R"), _bf(Y, "Y"), M, N, K, _ptr(ws), ws.numel(), _stream(stream)))
    return Y


def linear_swiglu_nvfp4(Xq, sfx, sx, Wgq, sfg, sg, Wuq, sfu, su, rstd=None, save=True, H=None, g=None, u=None,
                        ws=None, stream=None):
    """SwiGLU gate/up projection on NVFP4 operands (coda_linear_swiglu_nvfp4)."""
    lib = load()
    M, K = Xq.shape[0], 2 * Xq.shape[1]
    I = Wgq.shape[0]
    dev = Xq.device
    H = torch.empty(M, I, dtype=torch.bfloat16, device=dev) if H is None else H
    if save:
        g = torch.empty(M, I, dtype=torch.bfloat16, device=dev) if g is None else g
        u = torch.empty(M, I, dtype=torch.bfloat16, device=dev) if u is None else u
    ws = _ws(ws, lib.coda_linear_swiglu_nvfp4_workspace_size(M, I, K), dev)
    _check("coda_linear_swiglu_nvfp4", lib.coda_linear_swiglu_nvfp4(
        _u8(Xq, "Xq"), _u8(sfx, "sfx"), _f32(sx, "sx"), _f32(rstd, "rstd"), _u8(Wgq, "Wgq"), _u8(sfg, "sfg"),
        _f32(sg, "sg"), _u8(Wuq, "Wuq"), _u8(sfu, "sfu"), _f32(su, "su"), _bf(H, "H"), _bf(g, "g"), _bf(u, "u"),
        M, I, K, _ptr(ws), ws.numel(), _stream(stream)))
    return H, g, u


def linear_sigmoid(X, W, Z=None, Y=None, ws=None, stream=None):
    """sigmoid(X W^T), gating Z when given.  X, Z, Y may have leading
    dimensions ([..., features]); Y keeps them."""
    lib = load()
    X, lead = _rows(X)
    Z, _ = _rows(Z)
    Y, _ = _rows(Y)
    M, K = X.shape
    N = W.shape[0]
    Y = torch.empty(M, N, dtype=torch.bfloat16, device=X.device) if Y is None else Y
    ws = _ws(ws, lib.coda_linear_sigmoid_workspace_size(M, N, K), X.device)
    _check("coda_linear_sigmoid", lib.coda_linear_sigmoid(_bf(X, "X"), _bf(W, "W"), _bf(Z, "Z"), _bf(Y, "Y"),
                                                          M, N, K, _ptr(ws), ws.numel(), _stream(stream)))
    return _lead(Y, lead)


def linear_sigmoid_bwd(dY, X, W, Z=None, out=None, ws=None, stream=None):
    lib = load()
    M, K = X.shape
    N = W.shape[0]
    if out is None:
        out = {"dX": torch.empty_like(X), "dW": torch.empty_like(W),
               "dZ": torch.empty_like(dY) if Z is not None else None}
    ws = _ws(ws, lib.coda_linear_sigmoid_bwd_workspace_size(M, N, K), X.device)
    _check("coda_linear_sigmoid_bwd", lib.coda_linear_sigmoid_bwd(
        _bf(dY, "dY"), _bf(X, "X"), _bf(W, "W"), _bf(Z, "Z"), _bf(out["dX"], "dX"), _bf(out["dW"], "dW"),
        _bf(out.get("dZ"), "dZ"), M, N, K, _ptr(ws), ws.numel(), _stream(stream)))
    return out


def rmsnorm_linear_cross_entropy(X, rstd, Wf, labels, ignore_index=-100, out=None, ws=None, stream=None):
    """Final RMSNorm folded into the LM head: CE of z = rstd ⊙ (X Wf^T)."""
    lib = load()
    M, K = X.shape
    V = Wf.shape[0]
    dev = X.device
    if out is None:
        out = {"loss": torch.empty(1, dtype=torch.float32, device=dev),
               "lse": torch.empty(M, dtype=torch.float32, device=dev),
               "n_valid": torch.empty(1, dtype=torch.int32, device=dev)}
    ws = _ws(ws, lib.coda_rmsnorm_linear_cross_entropy_workspace_size(M, V, K), dev)
    _check("coda_rmsnorm_linear_cross_entropy", lib.coda_rmsnorm_linear_cross_entropy(
        _bf(X, "X"), _f32(rstd, "rstd"), _bf(Wf, "Wf"), _i32(labels, "labels"), int(ignore_index),
        _f32(out["loss"], "loss"), _f32(out["lse"], "lse"), _i32(out["n_valid"], "n_valid"), M, V, K,
        _ptr(ws), ws.numel(), _stream(stream)))
    out["ws"] = ws
    return out


def rmsnorm_linear_cross_entropy_bwd(X, rstd, gamma, W, Wf, labels, lse, n_valid, dloss=1.0, ignore_index=-100,
                                     dX_resid=None, out=None, ws=None, stream=None):
    lib = load()
    M, K = X.shape
    V = W.shape[0]
    dev = X.device
    if out is None:
        out = {"dX": torch.empty_like(X), "dW": torch.empty_like(W),
               "dgamma": torch.empty(K, dtype=torch.float32, device=dev)}
    ws = _ws(ws, lib.coda_rmsnorm_linear_cross_entropy_bwd_workspace_size(M, V, K), dev)
    _check("coda_rmsnorm_linear_cross_entropy_bwd", lib.coda_rmsnorm_linear_cross_entropy_bwd(
        _bf(X, "X"), _f32(rstd, "rstd"), _f32(gamma, "gamma"), _bf(W, "W"), _bf(Wf, "Wf"),
        _i32(labels, "labels"), int(ignore_index), _f32(lse, "lse"), _i32(n_valid, "n_valid"), float(dloss),
        _bf(dX_resid, "dX_resid"), _bf(out["dX"], "dX"), _bf(out["dW"], "dW"), _f32(out["dgamma"], "dgamma"),
        M, V, K, _ptr(ws), ws.numel(), _stream(stream)))
    out["ws"] = ws
    return out


def linear_cross_entropy_noalloc(X, W, labels, ignore_index=-100, out=None, stream=None):
    """coda_linear_cross_entropy_noalloc: the forward with the library's fixed
    device scratch instead of a workspace, for callers that cannot allocate
    device memory (see include/coda.h).  Pass `out` (loss [1], lse [M],
    n_valid [1], status [1] int32) so that nothing is allocated here either."""
    lib = load()
    M, K = X.shape
    V = W.shape[0]
    dev = X.device
    if out is None:
        out = {"loss": torch.empty(1, dtype=torch.float32, device=dev),
               "lse": torch.empty(M, dtype=torch.float32, device=dev),
               "n_valid": torch.empty(1, dtype=torch.int32, device=dev),
               "status": torch.empty(1, dtype=torch.int32, device=dev)}
    _check("coda_linear_cross_entropy_noalloc", lib.coda_linear_cross_entropy_noalloc(
        _bf(X, "X"), _bf(W, "W"), _i32(labels, "labels"), int(ignore_index), _f32(out["loss"], "loss"),
        _f32(out["lse"], "lse"), _i32(out["n_valid"], "n_valid"), _i32(out.get("status"), "status"),
        M, V, K, _stream(stream)))
    return out


def linear_cross_entropy_bwd(X, W, labels, lse, n_valid, dloss=1.0, ignore_index=-100, out=None, ws=None,
                             stream=None):
    lib = load()
    M, K = X.shape
    V = W.shape[0]
    if out is None:
        out = {"dX": torch.empty_like(X), "dW": torch.empty_like(W)}
    ws = _ws(ws, lib.coda_linear_cross_entropy_bwd_workspace_size(M, V, K), X.device)
    _check("coda_linear_cross_entropy_bwd", lib.coda_linear_cross_entropy_bwd(
        _bf(X, "X"), _bf(W, "W"), _i32(labels, "labels"), int(ignore_index), _f32(lse, "lse"),
        _i32(n_valid, "n_valid"), float(dloss), _bf(out["dX"], "dX"), _bf(out["dW"], "dW"), M, V, K,
        _ptr(ws), ws.numel(), _stream(stream)))
    out["ws"] = ws
    return out
