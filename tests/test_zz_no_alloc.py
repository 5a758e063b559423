"""The allocation-free cross-entropy forward (coda_linear_cross_entropy_noalloc).

It exists for callers that cannot obtain device memory -- a plugin handed only
its input and output buffers by a host application that owns all device
memory, or a latency-critical loop that must not call cudaMalloc -- and runs
the regular kernels with the library's fixed device scratch.  This file is
named so that pytest collects it last.  The test calls the entry point through
the C ABI twice in a row (the scratch keeps the first call's contents) and
compares each result with the regular coda_linear_cross_entropy on the same
inputs and with the fp64 oracle, within the parity tolerances of the other
tests; a third call with every label ignored and a call with no rows check
that nothing the previous calls left in the shared scratch reaches the
result."""
import math

import pytest
import torch

import synth
from oracle import coda_oracle as O
from parity import assert_f32, to_np

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
        f = O.linear_cross_entropy_fwd(to_np(t["X"]), to_np(t["W"]), t["labels"].numpy())
        out = _fresh_out(s.tokens)
        assert _noalloc_via_abi(lib, X, W, lab, out, s.tokens, s.vocab, s.hidden) == 0
        torch.cuda.synchronize()
        assert int(out["status"].item()) == 0
        assert int(out["n_valid"].item()) == int(ref["n_valid"].item()) == f["n_valid"]
        assert_f32(out["lse"], ref["lse"], f"lse call {call} vs the regular entry point")
        assert_f32(out["loss"], ref["loss"], f"loss call {call} vs the regular entry point")
        assert_f32(out["lse"], f["lse"], f"lse call {call} vs the oracle")
        assert_f32(out["loss"], [f["loss"]], f"loss call {call} vs the oracle")
    # a third call with every row ignored: the combine must not read the
    # target logits the previous calls left in the shared scratch
    s = shapes[0]
    t = synth.make_ce(s, seed=10)
    X, W = t["X"].to(DEV), t["W"].to(DEV)
    lab = torch.full((s.tokens,), -100, dtype=torch.int32)
    ref = coda.linear_cross_entropy(X, W, lab.to(DEV))
    f = O.linear_cross_entropy_fwd(to_np(t["X"]), to_np(t["W"]), lab.numpy())
    out = _fresh_out(s.tokens)
    assert _noalloc_via_abi(lib, X, W, lab.to(DEV), out, s.tokens, s.vocab, s.hidden) == 0
    torch.cuda.synchronize()
    assert int(out["status"].item()) == 0
    assert int(out["n_valid"].item()) == int(ref["n_valid"].item()) == f["n_valid"] == 0
    assert math.isnan(out["loss"].item()) and math.isnan(ref["loss"].item()) and math.isnan(f["loss"])
    assert_f32(out["lse"], ref["lse"], "lse, all ignored, vs the regular entry point")
    assert_f32(out["lse"], f["lse"], "lse, all ignored, vs the oracle")
    # and a call with no rows: only the mean (NaN) and the count (0) are written
    out = _fresh_out(1)
    assert _noalloc_via_abi(lib, X, W, lab.to(DEV), out, 0, s.vocab, s.hidden) == 0
    torch.cuda.synchronize()
    assert int(out["status"].item()) == 0
    assert int(out["n_valid"].item()) == 0 and math.isnan(out["loss"].item())


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
