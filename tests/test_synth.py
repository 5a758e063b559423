"""CPU checks of the seeded input generators: the same seed gives the same
bits, each tensor of a workload has its own seed (base + position in the
workload's list), weights have std 1/sqrt(fan_in), gains 1 + 0.1 N(0, 1),
the cross-entropy workload ignores exactly floor(0.05 M) labels, positions
restart at every sequence, and the full-size shapes are the documented
ones."""
import math

import torch

import synth


def _std(t):
    return float(t.float().std())


def test_same_seed_same_bits_and_distinct_tensors():
    a, b = synth.make_swiglu(seed=0), synth.make_swiglu(seed=0)
    for k in a:
        assert torch.equal(a[k].view(torch.int16), b[k].view(torch.int16)), k
    c = synth.make_swiglu(seed=1)
    assert not torch.equal(a["X"], c["X"])
    # Wg and Wu have the same shape and std but different seeds
    assert not torch.equal(a["Wg"], a["Wu"])
    # tensor i of a workload is drawn with seed base + i
    s = synth.FULL["swiglu"]
    assert torch.equal(c["X"], synth.randn_bf16(a["X"].shape, 1.0, 1))
    assert torch.equal(a["Wg"], synth.randn_bf16(a["Wg"].shape, 1.0 / math.sqrt(s.hidden), 1))
    assert torch.equal(a["Wu"], synth.randn_bf16(a["Wu"].shape, 1.0 / math.sqrt(s.hidden), 2))


def test_storage_dtype_and_rounding():
    x = synth.randn_bf16((64, 33), 0.5, 7)
    assert x.dtype == torch.bfloat16
    g = torch.Generator(device="cpu")
    g.manual_seed(7)
    ref = (torch.randn(64, 33, generator=g, dtype=torch.float32) * 0.5).to(torch.bfloat16)
    assert torch.equal(x.view(torch.int16), ref.view(torch.int16))


def test_weight_and_gain_statistics():
    s = synth.FULL["swiglu"]
    d = synth.make_swiglu(s, seed=0)
    assert abs(_std(d["Wg"]) * math.sqrt(s.hidden) - 1.0) < 0.01
    assert abs(_std(d["X"]) - 1.0) < 0.01
    g = synth.gain_f32(8192, 3)
    assert g.dtype == torch.float32
    assert abs(float(g.mean()) - 1.0) < 0.005 and abs(_std(g) - 0.1) < 0.005


def test_cross_entropy_labels():
    s = synth.FULL["linear_ce"]
    lab = synth.labels_i32(s.tokens, s.vocab, 2, s.ignore_frac, s.ignore_index)
    assert lab.dtype == torch.int32 and lab.shape == (s.tokens,)
    ignored = lab == s.ignore_index
    assert int(ignored.sum()) == math.floor(0.05 * s.tokens) == 409
    valid = lab[~ignored]
    assert int(valid.min()) >= 0 and int(valid.max()) < s.vocab
    assert torch.equal(lab, synth.labels_i32(s.tokens, s.vocab, 2, s.ignore_frac, s.ignore_index))


def test_positions_restart_per_sequence():
    s = synth.FULL["block"]
    pos = synth.positions_i32(s.tokens, s.seq_len)
    assert pos.dtype == torch.int32
    assert int(pos[0]) == 0 and int(pos[s.seq_len - 1]) == s.seq_len - 1
    assert int(pos[s.seq_len]) == 0 and int(pos[-1]) == s.seq_len - 1
    assert s.tokens // s.seq_len == 4


def test_full_size_shapes():
    b = synth.FULL["block"]
    assert (b.tokens, b.hidden, b.inter, b.n_q, b.n_kv, b.head_dim) == (8192, 8192, 28672, 64, 8, 128)
    assert b.qkv_out == 10240 and b.theta == 500000.0 and b.eps == 1e-6
    assert synth.FULL["mlp"] == synth.MlpShape(8192, 4096, 11008)
    assert synth.FULL["linear_ce"].vocab == 128256 and synth.FULL["linear_ce"].hidden == 2048
    r = synth.FULL["rmsnorm_linear"]
    assert (r.tokens, r.hidden, r.out, r.eps) == (4096, 2048, 2048, 1e-6)
    w = synth.FULL["swiglu"]
    assert (w.tokens, w.hidden, w.inter) == (256, 512, 1024)
    # a scaled block draws the same kinds of tensors with the documented shapes
    small = synth.BlockShape(tokens=16, hidden=32, n_q=2, n_kv=1, head_dim=8, inter=48, seq_len=8)
    t = synth.make_block(small, seed=0)
    assert t["Wqkv"].shape == (small.qkv_out, 32) and t["Wd"].shape == (32, 48)
    assert t["dK"].shape == (16, 8) and t["pos"].tolist() == [i % 8 for i in range(16)]


def test_sample_rows_keep_both_ends():
    idx = synth.sample_rows(8192, 64)
    assert int(idx[0]) == 0 and int(idx[-1]) == 8191
    assert len(idx) <= 64 and bool((idx[1:] > idx[:-1]).all())
