"""Seeded synthetic inputs for the five CODA workloads.

This module is shared by the CUDA path's tests and benchmark and by the fp64
oracle's tests.  It draws random numbers and rounds them to the storage dtype;
it holds none of the operators' arithmetic.

Recipe (identical for every workload):
  * one ``torch.Generator('cpu')`` per tensor, ``manual_seed(base_seed + i)``
    where ``i`` is the tensor's position in the workload's fixed list below;
  * ``torch.randn`` in float32, drawn in *storage* order, times the std, then
    rounded to bfloat16 (round-to-nearest-even) for bf16 tensors;
  * weights are stored ``[out_features, in_features]`` (the nn.Linear layout
    the x-tip guide's functional-API example uses for ``w1``), with
    std = 1/sqrt(fan_in);
  * RMSNorm gains are ``1 + 0.1*N(0,1)`` in float32.

Shapes follow the hidden widths {2048, 4096, 8192} that the x-tip guide's
benchmark section names (about 1B / 7B / 70B models).
"""
from __future__ import annotations

import math
from dataclasses import dataclass, field

import torch


def randn_bf16(shape, std, seed):
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    x = torch.randn(*shape, generator=g, dtype=torch.float32)
    if std != 1.0:
        x.mul_(std)
    return x.to(torch.bfloat16)


def gain_f32(n, seed):
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    return 1.0 + 0.1 * torch.randn(n, generator=g, dtype=torch.float32)


def labels_i32(m, vocab, seed, ignore_frac=0.05, ignore_index=-100):
    """Uniform labels in [0, vocab); then floor(ignore_frac*m) rows, chosen by
    a seeded permutation (seed+1), are set to ignore_index."""
    g = torch.Generator(device="cpu")
    g.manual_seed(int(seed))
    lab = torch.randint(0, vocab, (m,), generator=g, dtype=torch.int64)
    n_ign = int(math.floor(ignore_frac * m))
    if n_ign > 0:
        g2 = torch.Generator(device="cpu")
        g2.manual_seed(int(seed) + 1)
        rows = torch.randperm(m, generator=g2)[:n_ign]
        lab[rows] = ignore_index
    return lab.to(torch.int32)


def positions_i32(tokens, seq_len):
    """Token t of a packed batch of sequences of length seq_len sits at
    position t mod seq_len (each sequence restarts at 0)."""
    return (torch.arange(tokens, dtype=torch.int64) % seq_len).to(torch.int32)


# --------------------------------------------------------------------------
# workload shapes
# --------------------------------------------------------------------------

@dataclass(frozen=True)
class SwigluShape:            # linear + SwiGLU forward, 256 x 512 -> 1024
    tokens: int = 256
    hidden: int = 512
    inter: int = 1024


@dataclass(frozen=True)
class RmsLinearShape:         # RMSNorm-reparameterised projection + residual, 4096 x 2048 -> 2048
    tokens: int = 4096
    hidden: int = 2048
    out: int = 2048
    eps: float = 1e-6


@dataclass(frozen=True)
class MlpShape:               # SwiGLU MLP fwd+bwd, 8192 x 4096, intermediate 11008
    tokens: int = 8192
    hidden: int = 4096
    inter: int = 11008


@dataclass(frozen=True)
class CeShape:                # linear + cross-entropy, 8192 x 2048, vocabulary 128256
    tokens: int = 8192
    hidden: int = 2048
    vocab: int = 128256
    ignore_index: int = -100
    ignore_frac: float = 0.05


@dataclass(frozen=True)
class BlockShape:             # non-attention block fwd+bwd, 8192 tokens, hidden 8192
    tokens: int = 8192
    hidden: int = 8192
    n_q: int = 64
    n_kv: int = 8
    head_dim: int = 128
    inter: int = 28672
    seq_len: int = 2048
    theta: float = 500000.0
    eps: float = 1e-6

    @property
    def qkv_out(self):
        return (self.n_q + 2 * self.n_kv) * self.head_dim


FULL = {
    "swiglu": SwigluShape(),
    "rmsnorm_linear": RmsLinearShape(),
    "mlp": MlpShape(),
    "linear_ce": CeShape(),
    "block": BlockShape(),
}


def make_swiglu(s: SwigluShape = SwigluShape(), seed=0):
    return {
        "X": randn_bf16((s.tokens, s.hidden), 1.0, seed + 0),
        "Wg": randn_bf16((s.inter, s.hidden), 1.0 / math.sqrt(s.hidden), seed + 1),
        "Wu": randn_bf16((s.inter, s.hidden), 1.0 / math.sqrt(s.hidden), seed + 2),
    }


def make_rms_linear(s: RmsLinearShape = RmsLinearShape(), seed=0):
    return {
        "X": randn_bf16((s.tokens, s.hidden), 1.0, seed + 0),
        "gamma": gain_f32(s.hidden, seed + 1),
        "W": randn_bf16((s.out, s.hidden), 1.0 / math.sqrt(s.hidden), seed + 2),
        "R": randn_bf16((s.tokens, s.out), 1.0, seed + 3),
        "G": randn_bf16((s.tokens, s.out), 1.0, seed + 4),
    }


def make_mlp(s: MlpShape = MlpShape(), seed=0):
    return {
        "X": randn_bf16((s.tokens, s.hidden), 1.0, seed + 0),
        "Wg": randn_bf16((s.inter, s.hidden), 1.0 / math.sqrt(s.hidden), seed + 1),
        "Wu": randn_bf16((s.inter, s.hidden), 1.0 / math.sqrt(s.hidden), seed + 2),
        "Wd": randn_bf16((s.hidden, s.inter), 1.0 / math.sqrt(s.inter), seed + 3),
        "R": randn_bf16((s.tokens, s.hidden), 1.0, seed + 4),
        "dY": randn_bf16((s.tokens, s.hidden), 1.0, seed + 5),
    }


def make_ce(s: CeShape = CeShape(), seed=0):
    return {
        "X": randn_bf16((s.tokens, s.hidden), 1.0, seed + 0),
        "W": randn_bf16((s.vocab, s.hidden), 1.0 / math.sqrt(s.hidden), seed + 1),
        "labels": labels_i32(s.tokens, s.vocab, seed + 2, s.ignore_frac, s.ignore_index),
    }


def make_block(s: BlockShape = BlockShape(), seed=0):
    h, d = s.hidden, s.head_dim
    return {
        "x0": randn_bf16((s.tokens, h), 1.0, seed + 0),
        "Wqkv": randn_bf16((s.qkv_out, h), 1.0 / math.sqrt(h), seed + 1),
        "Wo": randn_bf16((h, s.n_q * d), 1.0 / math.sqrt(s.n_q * d), seed + 2),
        "Wg": randn_bf16((s.inter, h), 1.0 / math.sqrt(h), seed + 3),
        "Wu": randn_bf16((s.inter, h), 1.0 / math.sqrt(h), seed + 4),
        "Wd": randn_bf16((h, s.inter), 1.0 / math.sqrt(s.inter), seed + 5),
        "gamma_attn": gain_f32(h, seed + 6),
        "gamma_mlp": gain_f32(h, seed + 7),
        "gamma_q": gain_f32(d, seed + 8),
        "gamma_k": gain_f32(d, seed + 9),
        "A": randn_bf16((s.tokens, s.n_q * d), 1.0, seed + 10),
        "dx2": randn_bf16((s.tokens, h), 1.0, seed + 11),
        "dQ": randn_bf16((s.tokens, s.n_q * d), 1.0, seed + 12),
        "dK": randn_bf16((s.tokens, s.n_kv * d), 1.0, seed + 13),
        "dV": randn_bf16((s.tokens, s.n_kv * d), 1.0, seed + 14),
        "pos": positions_i32(s.tokens, s.seq_len),
    }


def sample_rows(n_rows, n_sample, seed=1234):
    """Sorted, distinct row indices used to check large outputs row by row.
    Always includes the first and last rows (ragged tail)."""
    g = torch.Generator(device="cpu")
    g.manual_seed(seed)
    if n_sample >= n_rows:
        return torch.arange(n_rows)
    idx = torch.randperm(n_rows, generator=g)[: max(n_sample - 2, 0)]
    idx = torch.unique(torch.cat([idx, torch.tensor([0, n_rows - 1])]))
    return idx.sort().values


def to_f64(t):
    """Exact widening of a CPU tensor (bf16/fp32/int) to a float64 numpy array."""
    return t.detach().to("cpu").double().numpy()
