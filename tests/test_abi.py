"""CPU tests of the C ABI: the library builds, loads without a GPU, exports
every function that include/coda.h declares, and rejects bad arguments on the
host before anything is enqueued (no CUDA call is reached in these cases)."""
import ctypes
import os
import re

import pytest

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))
HEADER = os.path.join(ROOT, "include", "coda.h")


@pytest.fixture(scope="module")
def lib():
    from gemm_epilogue_transformer_bf16_gb300 import _build
    import gemm_epilogue_transformer_bf16_gb300 as coda
    _build.build()
    return coda.load()


def declared_functions():
    src = open(HEADER).read()
    src = re.sub(r"/\*.*?\*/", "", src, flags=re.S)
    names = re.findall(r"\b(?:int|size_t|uint64_t|const char\s*\*)\s+(coda_\w+)\s*\(", src)
    return sorted(set(names))


def test_header_declares_the_operator_set():
    names = declared_functions()
    for required in ["coda_gemm_epilogue", "coda_rmsnorm_linear", "coda_linear_swiglu", "coda_linear_swiglu_bwd",
                     "coda_linear_residual", "coda_linear_qknorm_rope", "coda_linear_qknorm_rope_bwd",
                     "coda_linear_cross_entropy", "coda_linear_cross_entropy_bwd"]:
        assert required in names


def test_every_declared_symbol_is_exported(lib):
    missing = [n for n in declared_functions() if not hasattr(lib, n)]
    assert not missing, f"not exported: {missing}"


def test_binding_covers_every_symbol():
    import gemm_epilogue_transformer_bf16_gb300 as coda
    missing = [n for n in declared_functions() if n not in coda._SIGS]
    assert not missing, f"no ctypes signature for: {missing}"


def declared_parameters():
    """name -> list of parameter declarations, from include/coda.h."""
    src = re.sub(r"/\*.*?\*/", "", open(HEADER).read(), flags=re.S)
    out = {}
    for m in re.finditer(r"\b(?:int|size_t|uint64_t|const char\s*\*)\s+(coda_\w+)\s*\(([^)]*)\)", src):
        params = [p.strip() for p in m.group(2).split(",")]
        out[m.group(1)] = [] if params in ([""], ["void"]) else params
    return out


def _ctype_of(param):
    """The ctypes type a C parameter declaration is marshalled as."""
    if "*" in param or param.startswith("coda_stream"):
        return ctypes.c_void_p
    base = param.rsplit(" ", 1)[0].replace("const ", "").strip()
    return {"int64_t": ctypes.c_int64, "int32_t": ctypes.c_int32, "int": ctypes.c_int, "uint32_t": ctypes.c_uint32,
            "float": ctypes.c_float, "size_t": ctypes.c_size_t}[base]


def test_binding_signatures_match_header():
    """Every ctypes signature has the header's parameter count and, position
    by position, the type each parameter is passed as (a pointer or a
    stream handle as void*, each integer and float at its width)."""
    import gemm_epilogue_transformer_bf16_gb300 as coda
    bad = []
    for name, params in declared_parameters().items():
        want = [_ctype_of(p) for p in params]
        got = coda._SIGS[name][0]
        if len(got) != len(want) or any(ctypes.sizeof(a) != ctypes.sizeof(b) or
                                         (a is ctypes.c_void_p) != (b is ctypes.c_void_p) or
                                         (a is ctypes.c_float) != (b is ctypes.c_float)
                                         for a, b in zip(got, want)):
            bad.append((name, len(got), len(want)))
    assert not bad, f"ctypes signatures that differ from include/coda.h: {bad}"


def test_launch_count_without_launches(lib):
    """The launch counter is host state: readable without a GPU, and zero
    on a host without one (nothing can have been launched)."""
    import torch
    import gemm_epilogue_transformer_bf16_gb300 as coda
    assert "coda_launch_count" in declared_functions()
    n = coda.launch_count()
    assert n >= 0
    if not torch.cuda.is_available():
        assert n == 0


def test_version_and_status_strings(lib):
    assert b"sm_103a" in lib.coda_version()
    assert lib.coda_status_string(0) == b"CODA_OK"
    assert lib.coda_status_string(7) == b"CODA_ERR_LABEL_RANGE"


def test_epilogue_desc_layout_matches_header():
    """ctypes mirror of coda_epilogue_desc has the C layout (compiled probe)."""
    import subprocess
    import tempfile
    import gemm_epilogue_transformer_bf16_gb300 as coda
    src = r'''
#include <stdio.h>
#include <stddef.h>
#include "coda.h"
int main(void) {
  printf("%zu %zu %zu %zu %zu %zu %zu %zu %zu\n", sizeof(coda_epilogue_desc), offsetof(coda_epilogue_desc, partials),
         offsetof(coda_epilogue_desc, K2), offsetof(coda_epilogue_desc, dloss),
         offsetof(coda_epilogue_desc, eps), offsetof(coda_epilogue_desc, V),
         offsetof(coda_epilogue_desc, rope_pairing), offsetof(coda_epilogue_desc, operand_type),
         offsetof(coda_epilogue_desc, acc_col_scale));
  return 0;
}
'''
    with tempfile.TemporaryDirectory() as d:
        c = os.path.join(d, "p.c")
        exe = os.path.join(d, "p")
        open(c, "w").write(src)
        subprocess.check_call(["gcc", "-I", os.path.join(ROOT, "include"), c, "-o", exe])
        got = [int(x) for x in subprocess.check_output([exe]).split()]
    D = coda.EpilogueDesc
    want = [ctypes.sizeof(D), D.partials.offset, D.K2.offset, D.dloss.offset, D.eps.offset, D.V.offset,
            D.rope_pairing.offset, D.operand_type.offset, D.acc_col_scale.offset]
    assert got == want


# --------------------------------------------------------------------------- host validation
FAKE = 1 << 20          # a 16-byte aligned non-null address (never dereferenced)
FAKE_UNALIGNED = FAKE + 2


def test_rejects_bad_arguments_on_host(lib):
    ws = FAKE
    # null required pointer
    assert lib.coda_linear_swiglu(None, None, FAKE, FAKE, FAKE, None, None, 16, 64, 64, ws, 4096, None) == 1
    # misaligned pointer
    assert lib.coda_linear_swiglu(FAKE_UNALIGNED, None, FAKE, FAKE, FAKE, None, None, 16, 64, 64, ws, 4096,
                                  None) == 2
    # feature dims must be multiples of 8
    assert lib.coda_linear_swiglu(FAKE, None, FAKE, FAKE, FAKE, None, None, 16, 60, 64, ws, 4096, None) == 3
    # negative size
    assert lib.coda_linear_residual(FAKE, FAKE, None, FAKE, 1e-6, None, None, None, -1, 64, 64, ws, 4096, None) == 1
    # workspace too small
    need = lib.coda_rmsnorm_linear_bwd_workspace_size(128, 64, 64)
    assert lib.coda_rmsnorm_linear_bwd(*([FAKE] * 10), 128, 64, 64, ws, need - 1, None, None) == 4
    # null workspace
    assert lib.coda_linear_residual(FAKE, FAKE, None, FAKE, 1e-6, None, None, None, 16, 64, 64, None, 4096, None) == 4
    # head_dim other than 128 is unsupported
    assert lib.coda_linear_qknorm_rope(*([FAKE] * 7), 16, 1e-6, 2, 1, 64, 0, *([FAKE] * 4), 16, 64, ws, 4096,
                                       None) == 3
    # unknown RoPE pairing
    assert lib.coda_linear_qknorm_rope_bwd(*([FAKE] * 9), 16, 1e-6, 2, 1, 128, 7, *([FAKE] * 10), 16, 64, ws,
                                           1 << 30, None) == 1
    # K == 0 with work to do
    assert lib.coda_linear_residual_bwd(FAKE, FAKE, FAKE, FAKE, FAKE, 16, 64, 0, ws, 4096, None) == 3
    # gain output: gamma_next and U_out come together
    assert lib.coda_linear_residual(FAKE, FAKE, None, FAKE, 1e-6, None, FAKE, None, 16, 64, 64, ws, 4096,
                                    None) == 1
    # RMSNorm prepass: every pointer required and aligned, row strides >= K and multiples of 8
    assert lib.coda_rmsnorm_scale(FAKE, 64, 16, 64, 1e-6, None, FAKE, FAKE, 64, None) == 1
    assert lib.coda_rmsnorm_scale(FAKE, 64, 16, 64, 1e-6, FAKE, FAKE, FAKE_UNALIGNED, 64, None) == 2
    assert lib.coda_rmsnorm_scale(FAKE, 64, 16, 64, 1e-6, FAKE, FAKE, FAKE, 60, None) == 1
    assert lib.coda_rmsnorm_scale(FAKE, 64, 0, 64, 1e-6, FAKE, FAKE, FAKE, 64, None) == 0
    # NVFP4: K a multiple of 32; block scales required and aligned
    assert lib.coda_quantize_nvfp4_rows(FAKE, 48, 16, 48, FAKE, FAKE, FAKE, None) == 3
    assert lib.coda_quantize_nvfp4_rows(FAKE, 64, 16, 64, FAKE, None, FAKE, None) == 1
    assert lib.coda_quantize_nvfp4_rows(FAKE, 64, 16, 64, FAKE, FAKE_UNALIGNED, FAKE, None) == 2
    assert lib.coda_linear_nvfp4(*([FAKE] * 6), None, FAKE, 16, 64, 48, ws, 4096, None) == 3
    assert lib.coda_linear_nvfp4(FAKE, None, *([FAKE] * 4), None, FAKE, 16, 64, 64, ws, 4096, None) == 1
    assert lib.coda_linear_swiglu_nvfp4(*([FAKE] * 9), None, FAKE, None, None, 16, 64, 64, ws, 4096, None) == 1
    assert lib.coda_linear_swiglu_nvfp4(*([FAKE] * 10), FAKE, None, None, 0, 64, 64, ws, 4096, None) == 0
    assert lib.coda_rmsnorm_scale_nvfp4(FAKE, 64, 16, 64, 1e-6, None, None, FAKE, FAKE, FAKE, None) == 1
    assert lib.coda_rmsnorm_scale_nvfp4(FAKE, 48, 16, 48, 1e-6, FAKE, None, FAKE, FAKE, FAKE, None) == 3
    # FP8 QKV backward: the dW GEMM contracts over the tokens, M % 16 == 0
    assert lib.coda_linear_qknorm_rope_bwd_fp8(*([FAKE] * 9), 16, 1e-6, 2, 1, 128, 0, *([FAKE] * 13), 20, 64, ws,
                                               1 << 30, None) == 3
    assert lib.coda_linear_qknorm_rope_bwd_fp8(*([FAKE] * 9), 16, 1e-6, 2, 1, 128, 0, *([FAKE] * 13), 0, 64, ws,
                                               1 << 30, None) == 0
    assert lib.coda_nvfp4_scale_bytes(300, 224) == 4 * 1 * 2048
    assert lib.coda_nvfp4_scale_bytes(600, 512) == 8 * 2 * 2048


def test_empty_problem_is_a_noop(lib):
    ws = FAKE
    # M == 0: nothing to do, nothing enqueued, OK
    assert lib.coda_linear_swiglu(FAKE, None, FAKE, FAKE, FAKE, None, None, 0, 64, 64, ws, 4096, None) == 0
    assert lib.coda_linear_residual(FAKE, FAKE, None, FAKE, 1e-6, None, None, None, 0, 64, 64, ws, 4096, None) == 0


def test_generic_rejects_bad_descriptor(lib):
    import gemm_epilogue_transformer_bf16_gb300 as coda
    d = coda.EpilogueDesc()
    d.map = 99
    assert lib.coda_gemm_epilogue(ctypes.byref(d), FAKE, 64, 0, FAKE, 64, 0, FAKE, 64, 0, 16, 64, 64, FAKE, 4096,
                                  None) == 1
    d.map = coda.MAP_QKNORM_ROPE
    d.head_dim = 64
    assert lib.coda_gemm_epilogue(ctypes.byref(d), FAKE, 64, 0, FAKE, 64, 0, FAKE, 64, 0, 16, 64, 64, FAKE, 4096,
                                  None) == 3
    d = coda.EpilogueDesc()
    # fp32 output only with MAP_NONE
    d.map = coda.MAP_COLDOT
    d.aux_in[0] = FAKE
    d.ld_aux_in[0] = 64
    assert lib.coda_gemm_epilogue(ctypes.byref(d), FAKE, 64, 0, FAKE, 64, 0, FAKE, 64, 1, 16, 64, 64, FAKE, 4096,
                                  None) == 3
