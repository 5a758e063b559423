"""Pins of the fp64 oracle (CPU only).

``test_pin`` runs every check of ``pins.py`` on the oracle.  ``test_mutant``
plants a plausible mistake in a private copy of the oracle (on the CPU) and
asserts that at least one pin then fails, so the pins are shown to be able to
catch that class of error.
"""
import importlib.util
import os

import numpy as np
import pytest

import pins
from oracle import coda_oracle

ORACLE_SRC = os.path.join(os.path.dirname(coda_oracle.__file__), "coda_oracle.py")


@pytest.mark.parametrize("name", sorted(pins.ALL_CHECKS))
def test_pin(name):
    fn, tol = pins.ALL_CHECKS[name]
    err = fn(coda_oracle)
    assert err <= tol, f"{name}: {err:.3e} > {tol:.1e}"


def _fresh_copy(tag):
    spec = importlib.util.spec_from_file_location(f"oracle_mutant_{tag}", ORACLE_SRC)
    mod = importlib.util.module_from_spec(spec)
    spec.loader.exec_module(mod)
    return mod


def _mut_rms_eps_outside(m):
    m.rms_inv = lambda x, eps: 1.0 / (np.sqrt(np.mean(np.asarray(x) ** 2, axis=-1)) + eps)


def _mut_rmsnorm_bwd_drop_mean(m):
    def bad(x, gamma, eps, dy):
        r = m.rms_inv(x, eps)[..., None]
        dx = r * (dy * gamma)
        return dx, (dy * x * r).reshape(-1, x.shape[-1]).sum(axis=0)
    m.rmsnorm_bwd = bad


def _mut_rmsnorm_gamma_before(m):
    m.rmsnorm = lambda x, gamma, eps: (x * gamma) * m.rms_inv(x * gamma, eps)[..., None]


def _mut_silu_sign(m):
    m.silu = lambda a: np.asarray(a, dtype=np.float64) / (1.0 + np.exp(np.asarray(a, dtype=np.float64)))


def _mut_swiglu_swapped(m):
    def bad(X, Wg, Wu):
        g, u = X @ Wg.T, X @ Wu.T
        return m.silu(u) * g, g, u
    m.swiglu_fwd = bad


def _mut_rope_sign(m):
    orig = m.rope

    def bad(v, pos, theta):
        out = orig(v, pos, theta)
        out[..., 1::2] *= -1.0
        return out
    m.rope = bad


def _mut_rope_freq(m):
    def bad(pos, head_dim, theta):
        j = np.arange(head_dim // 2, dtype=np.float64)
        return np.asarray(pos, dtype=np.float64)[:, None] * (theta ** (-j / head_dim))[None, :]
    m.rope_angles = bad


def _mut_ce_mean_over_all(m):
    orig = m.linear_cross_entropy_fwd

    def bad(X, W, labels, ignore_index=-100):
        f = orig(X, W, labels, ignore_index)
        if f["n_valid"] > 0:
            f["loss"] = f["per_row"].sum() / len(labels)
        return f
    m.linear_cross_entropy_fwd = bad


def _mut_ce_grad_no_onehot(m):
    orig = m.linear_cross_entropy_bwd

    def bad(X, W, labels, ignore_index=-100, dloss=1.0):
        z = X @ W.T
        p = np.exp(z - m._lse(z)[:, None])
        valid = np.asarray(labels) != ignore_index
        dZ = np.where(valid[:, None], p, 0.0) / max(int(valid.sum()), 1)
        return {"dX": dZ @ W, "dW": dZ.T @ X, "dZ": dZ}
    m.linear_cross_entropy_bwd = bad


def _mut_block_mlp_on_x0(m):
    orig = m.block_fwd

    def bad(p, n_q, n_kv, head_dim, theta, eps):
        f = orig(p, n_q, n_kv, head_dim, theta, eps)
        mm = m.mlp_fwd(p["x0"], p["Wg"], p["Wu"], p["Wd"], p["x0"], p["gamma_mlp"], eps)
        f["x2"] = mm["y"]
        return f
    m.block_fwd = bad


def _mut_block_bwd_no_residual(m):
    orig = m.block_bwd

    def bad(p, n_q, n_kv, head_dim, theta, eps):
        b = orig(p, n_q, n_kv, head_dim, theta, eps)
        b["dx0"] = b["dx0"] - b["dx1"]
        return b
    m.block_bwd = bad


def _mut_mlp_bwd_transposed(m):
    orig = m.mlp_bwd

    def bad(*a, **k):
        b = orig(*a, **k)
        b["dWg"], b["dWu"] = b["dWu"], b["dWg"]
        return b
    m.mlp_bwd = bad


def _mut_gemm_transposed_scale(m):
    orig = m.gemm_epilogue_plain

    def bad(A, B, row_scale=None, col_scale=None, aux0=None, row_coef=None, aux1=None, D_old=None):
        return orig(A, B, row_scale, col_scale, aux0, None if row_coef is None else -np.asarray(row_coef),
                    aux1, D_old)
    m.gemm_epilogue_plain = bad


def _mut_rmsnorm_ce_skip_norm_bwd(m):
    def bad(X, gamma, W, labels, eps, ignore_index=-100, dloss=1.0):
        a = m.rmsnorm(X, gamma, eps)
        b = m.linear_cross_entropy_bwd(a, W, labels, ignore_index, dloss)
        return {"dX": b["dX"] * gamma, "dW": b["dW"], "dgamma": (b["dX"] * a).sum(axis=0)}
    m.rmsnorm_linear_cross_entropy_bwd = bad


def _mut_sigmoid_bwd_missing_factor(m):
    def bad(X, W, dY, Z=None):
        s = m.sigmoid(X @ W.T)
        g = dY if Z is None else dY * Z
        dz = g * s
        out = {"dX": dz @ W, "dW": dz.T @ X}
        if Z is not None:
            out["dZ"] = dY * s
        return out
    m.linear_sigmoid_bwd = bad


def _mut_fp8_truncate(m):
    import torch

    def bad(X):
        x32 = np.asarray(X, dtype=np.float32)
        amax = np.max(np.abs(x32), axis=1)
        scale = np.where(amax > 0, amax / np.float32(448.0), np.float32(1.0)).astype(np.float32)
        v = np.clip(x32 / scale[:, None], -448, 448)
        v = np.sign(v) * np.floor(np.abs(v) * 8) / 8       # truncation instead of rounding
        q = torch.from_numpy(v.astype(np.float32)).to(torch.float8_e4m3fn)
        return q.view(torch.uint8).numpy(), q.double().numpy(), scale
    m.quantize_fp8_rows = bad


def _source_mutant(old, new, *more):
    """A mutant that re-executes the oracle's source with one phrase replaced
    (or several: further (old, new) pairs)."""
    pairs = [(old, new)] + list(more)

    def apply(m):
        src = open(ORACLE_SRC).read()
        for a, b in pairs:
            assert src.count(a) == 1, a
            src = src.replace(a, b)
        exec(compile(src, ORACLE_SRC, "exec"), m.__dict__)
    return apply


MUTANTS = {
    "rope_half_swapped_halves": _source_mutant("a, b = v[..., : d // 2], v[..., d // 2:]",
                                               "a, b = v[..., d // 2:], v[..., : d // 2]"),
    "rmsnorm_nvfp4_rms_of_scaled_input": _source_mutant("(rms_inv(X, eps),)", "(rms_inv(u, eps),)"),
    "e2m1_ties_away_from_zero": _source_mutant("((d_hi == d_lo) & (hi % 2 == 0))", "(d_hi == d_lo)"),
    "nvfp4_block_scale_from_row_max": _source_mutant("ax.reshape(M, nb, NVFP4_BLOCK).max(axis=2)",
                                                     "np.repeat(amax[:, None], nb, axis=1)"),
    "nvfp4_codes_without_row_scale": _source_mutant("(sf_val * s[:, None]).astype(np.float32)",
                                                    "sf_val.astype(np.float32)"),
    "qknorm_bwd_forward_rotation": _source_mutant("dn = rope_inv(dout, pos, theta, pairing)",
                                                  "dn = rope(dout, pos, theta, pairing)"),
    "residual_rms_of_input": _source_mutant("return u, rms_inv(u, eps)", "return u, rms_inv(X, eps)"),
    "quantised_linear_drops_weight_scale": _source_mutant("B = Wv * np.asarray(sw, dtype=np.float64)[:, None]",
                                                          "B = Wv"),
    "lse_mean_instead_of_sum": _source_mutant("np.log(np.exp(z - m).sum(axis=-1, keepdims=True))",
                                              "np.log(np.exp(z - m).mean(axis=-1, keepdims=True))"),
    "swiglu_quantised_drops_row_factor": _source_mutant(
        "A = A * np.asarray(row_scale, dtype=np.float64)[:, None]", "A = A"),
    "e2m1_wrong_grid": _source_mutant("np.array([0.0, 0.5, 1.0, 1.5, 2.0, 3.0, 4.0, 6.0])",
                                      "np.array([0.0, 0.5, 1.0, 1.5, 2.0, 2.5, 4.0, 6.0])"),
    "sigmoid_gate_grad_without_s": _source_mutant('out["dZ"] = dY * s', 'out["dZ"] = dY'),
    "ce_grad_ignores_dloss": _source_mutant("dZ *= dloss / n_valid", "dZ *= 1.0 / n_valid"),
    "ce_dw_rows_without_onehot": _source_mutant("return {\"dW_rows\": dZ[:, np.asarray(vocab_rows)].T @ X}",
                                                "return {\"dW_rows\": (p * dloss / max(n_valid, 1))"
                                                "[:, np.asarray(vocab_rows)].T @ X}"),
    "fp8_cols_scale_from_whole_matrix": _source_mutant(
        "amax = np.max(np.abs(x32), axis=0) if x32.shape[0] else np.zeros(x32.shape[1], np.float32)",
        "amax = np.full(x32.shape[1], np.max(np.abs(x32)), np.float32)"),
    "dswiglu_fp8_gate_grad_is_silu": _source_mutant("dG = dH * u * silu_grad(g)", "dG = dH * u * silu(g)"),
    "rms_dx_fp8_drops_gamma": _source_mutant(
        "dX = D * np.asarray(gamma, dtype=np.float64)[None, :] - np.asarray(coef, dtype=np.float64)[:, None] * X",
        "dX = D - np.asarray(coef, dtype=np.float64)[:, None] * X"),
    "qkv_bwd_fp8_coef_single_r": _source_mutant("coef = r * r * (G * y).sum(axis=1) / Xf.shape[1]",
                                                "coef = r * (G * y).sum(axis=1) / Xf.shape[1]"),
    "qkv_bwd_fp8_dw_drops_u_scale": _source_mutant('"dW": _deq(gtv, sgt) @ _deq(UTv, su).T',
                                                   '"dW": _deq(gtv, sgt) @ np.asarray(UTv, dtype=np.float64).T'),
    "qkv_bwd_fp8_k_gain_q": _source_mutant("dk, dgk = qk_rmsnorm_rope_bwd(k, gamma_k, pos",
                                           "dk, dgk = qk_rmsnorm_rope_bwd(k, gamma_q, pos"),
    "qkv_bwd_fp8_g_unrounded": _source_mutant("Gp = _bf16(G * r[:, None])", "Gp = G * r[:, None]"),
    "qkv_bwd_fp8_d_from_column_codes": _source_mutant("D = _deq(gv, sg) @ _deq(WTv, sw).T",
                                                      "D = _deq(gtv, sgt).T @ _deq(WTv, sw).T"),
    # a negative label wraps around to column V + label (numpy indexing)
    "ce_negative_label_wraps": _source_mutant("in_range = (labels >= 0) & (labels < V)",
                                              "in_range = labels < V"),
    # the same wrong gain in the forward and the backward: the gradients stay
    # consistent, so only a forward pin can see it
    "block_k_uses_gamma_q": _source_mutant(
        'K = qk_rmsnorm_rope_fwd(k, p["gamma_k"], p["pos"], theta, eps)',
        'K = qk_rmsnorm_rope_fwd(k, p["gamma_q"], p["pos"], theta, eps)',
        ('dk, dgk = qk_rmsnorm_rope_bwd(k, p["gamma_k"]', 'dk, dgk = qk_rmsnorm_rope_bwd(k, p["gamma_q"]')),
    "fp8_truncates": _mut_fp8_truncate,
    "sigmoid_bwd_missing_derivative": _mut_sigmoid_bwd_missing_factor,
    "rmsnorm_ce_skips_norm_backward": _mut_rmsnorm_ce_skip_norm_bwd,
    "gemm_coef_sign": _mut_gemm_transposed_scale,
    "rms_eps_outside_root": _mut_rms_eps_outside,
    "rmsnorm_bwd_drop_mean": _mut_rmsnorm_bwd_drop_mean,
    "rmsnorm_gamma_before_norm": _mut_rmsnorm_gamma_before,
    "silu_sign": _mut_silu_sign,
    "swiglu_gate_on_up": _mut_swiglu_swapped,
    "rope_sign": _mut_rope_sign,
    "rope_frequency": _mut_rope_freq,
    "ce_mean_over_all_rows": _mut_ce_mean_over_all,
    "ce_grad_no_onehot": _mut_ce_grad_no_onehot,
    "block_mlp_residual_x0": _mut_block_mlp_on_x0,
    "block_bwd_no_residual": _mut_block_bwd_no_residual,
    "mlp_bwd_swapped_weights": _mut_mlp_bwd_transposed,
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant(name):
    m = _fresh_copy(name)
    MUTANTS[name](m)
    failed = []
    for cname, (fn, tol) in pins.ALL_CHECKS.items():
        try:
            err = fn(m)
        except Exception:
            err = float("inf")
        if not (err <= tol):
            failed.append(cname)
    assert failed, f"planted mistake {name!r} slipped past every pin"
