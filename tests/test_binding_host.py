"""CPU checks of the Python binding's marshalling: host tensors are refused
(there is no CPU path: every call runs the CUDA kernels or raises), dtypes
and contiguity are checked before any call, leading dimensions fold into
rows and back, and RoPE pairing names map to the C enum."""
import pytest
import torch

import gemm_epilogue_transformer_bf16_gb300 as coda


def test_host_tensors_are_refused():
    x = torch.zeros(4, 8, dtype=torch.bfloat16)
    with pytest.raises(ValueError, match="CUDA"):
        coda._ptr(x, torch.bfloat16, "X")
    with pytest.raises(TypeError):
        coda._ptr([1, 2, 3], None, "X")
    assert coda._ptr(None) is None


def test_public_calls_refuse_host_tensors():
    x = torch.zeros(128, 64, dtype=torch.bfloat16)
    w = torch.zeros(64, 64, dtype=torch.bfloat16)
    r = torch.zeros(128, 64, dtype=torch.bfloat16)
    # a host tensor never reaches a CPU computation: the call fails loudly
    with pytest.raises(ValueError, match="CUDA"):
        coda.linear_residual(x, w, r, ws=torch.zeros(1 << 20, dtype=torch.uint8))
    with pytest.raises(ValueError, match="workspace too small"):
        coda.linear_residual(x, w, r, ws=torch.zeros(256, dtype=torch.uint8))


def test_leading_dimensions_fold_and_unfold():
    t = torch.arange(2 * 3 * 5, dtype=torch.float32).view(2, 3, 5)
    rows, lead = coda._rows(t)
    assert rows.shape == (6, 5) and lead == (2, 3)
    assert rows.data_ptr() == t.data_ptr()           # a view, not a copy
    back = coda._lead(rows, lead)
    assert back.shape == (2, 3, 5) and torch.equal(back, t)
    v = torch.arange(6, dtype=torch.float32)
    assert coda._lead(v, lead).shape == (2, 3)
    assert coda._vec(torch.zeros(2, 3), lead).shape == (6,)
    two_d = torch.zeros(4, 5)
    assert coda._rows(two_d) == (two_d, None) and coda._lead(two_d, None) is two_d
    with pytest.raises(ValueError, match="contiguous"):
        coda._rows(torch.zeros(5, 3, 2).transpose(0, 1))


def test_rope_pairing_names():
    assert coda._pairing("interleaved") == coda.ROPE_INTERLEAVED == 0
    assert coda._pairing("half") == coda.ROPE_HALF == 1
    with pytest.raises(ValueError):
        coda._pairing("neox")
