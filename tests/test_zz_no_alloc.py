"""The allocation-free cross-entropy forward (coda_linear_cross_entropy_noalloc).

It exists for callers that cannot obtain device memory -- a plugin handed only
its input and output buffers by a host application that owns all device
memory, or a latency-critical loop that must not call cudaMalloc -- and runs
the regular kernels with the library's fixed device scratch.  This file is
named so that pytest collects it last.  The test calls the entry point through
the C ABI twice in a row (the scratch keeps the first call's contents) and
compares each result with the regular coda_linear_cross_entropy on the same
inputs, within the parity tolerances of the other tests."""
import pytest
import torch

import synth
from parity import assert_f32

pytestmark = pytest.mark.gpu
DEV = "cuda"


@pytest.fixture(scope="module")
def coda():
    import gemm_epilogue_transformer_bf16_gb300 as c
    from gemm_epilogue_transformer_bf16_gb300 import _build
    _build.build()
    c.load()
    return c


def _noalloc_via_abi(lib, X, W, labels, out, M, V, K):
    return lib.coda_linear_cross_entropy_noalloc(
        X.data_ptr(), W.data_ptr(), labels.data_ptr(), -100, out["loss"].data_ptr(), out["lse"].data_ptr(),
        out["n_valid"].data_ptr(), out["status"].data_ptr(), M, V, K,
        torch.cuda.current_stream().cuda_stream)


def _fresh_out(M):
    return {"loss": torch.full((1,), float("nan"), device=DEV),
            "lse": torch.full((M,), float("nan"), device=DEV),
            "n_valid": torch.full((1,), -1, dtype=torch.int32, device=DEV),
            "status": torch.full((1,), -1, dtype=torch.int32, device=DEV)}


def test_noalloc_matches_regular_twice(coda):
    lib = coda.load()
    shapes = [synth.CeShape(tokens=512, hidden=256, vocab=8200), synth.CeShape(tokens=300, hidden=136, vocab=4104)]
    for call, s in enumerate(shapes):      # two calls in a row, different problems
        t = synth.make_ce(s, seed=10 + call)
        X, W, lab = t["X"].to(DEV), t["W"].to(DEV), t["labels"].to(DEV)
        ref = coda.linear_cross_entropy(X, W, lab)
        out = _fresh_out(s.tokens)
        assert _noalloc_via_abi(lib, X, W, lab, out, s.tokens, s.vocab, s.hidden) == 0
        torch.cuda.synchronize()
        assert int(out["status"].item()) == 0
        assert int(out["n_valid"].item()) == int(ref["n_valid"].item())
        assert_f32(out["lse"], ref["lse"], f"lse call {call}")
        assert_f32(out["loss"], ref["loss"], f"loss call {call}")


def test_noalloc_reports_label_errors_and_rejects_oversize(coda):
    lib = coda.load()
    s = synth.CeShape(tokens=128, hidden=128, vocab=1024)
    t = synth.make_ce(s, seed=3)
    X, W, lab = t["X"].to(DEV), t["W"].to(DEV), t["labels"].to(DEV)
    lab[5] = s.vocab + 1
    out = _fresh_out(s.tokens)
    assert _noalloc_via_abi(lib, X, W, lab, out, s.tokens, s.vocab, s.hidden) == 0
    torch.cuda.synchronize()
    assert int(out["status"].item()) == 2          # label out of range, reported for this call
    lab[5] = 0
    assert _noalloc_via_abi(lib, X, W, lab, out, s.tokens, s.vocab, s.hidden) == 0
    torch.cuda.synchronize()
    assert int(out["status"].item()) == 0          # the shared status word starts clear on every call
    cap = lib.coda_noalloc_scratch_bytes()
    big_m = 2 * cap // 8                            # needs more scratch than the fixed array holds
    assert lib.coda_linear_cross_entropy_workspace_size(big_m, 128256, 2048) > cap
    assert lib.coda_linear_cross_entropy_noalloc(X.data_ptr(), W.data_ptr(), lab.data_ptr(), -100, None, None,
                                                 None, None, big_m, 128256, 2048, None) == 4
