"""Planted mistakes in a copy of the oracle must each break at least one pin.

Every mutant is a one-line textual change to oracle/oracle.cpp (a dropped term, a wrong
sign or index, an off-by-one window, a transposed operand), compiled on the CPU into a
temporary library and run through the same pins as the real oracle. The real oracle is
never modified.
"""

import os

import pytest

from oracle import oracle as O
from tests import oracle_pins as P

MUTANTS = {
    "window_off_by_one": ("dist >= w", "dist > w"),
    "not_causal": ("dist < 0 || dist >= w", "dist >= w || -dist >= w"),
    "ln_unbiased_variance": ("var = sq / (double)H;", "var = sq / (double)(H - 1);"),
    "ln_no_eps": ("std::sqrt(var + eps)", "std::sqrt(var)"),
    "ln_no_beta": ("inv * gamma[c] + beta[c]", "inv * gamma[c]"),
    "ln_no_centering": ("o[c] = (xr[c] - mu) * inv", "o[c] = xr[c] * inv"),
    "attn_no_scale": ("scale = 1.0 / std::sqrt((double)dh);\n  const double neg_inf",
                      "scale = 1.0;\n  const double neg_inf"),
    "attn_no_max_shift_sign": ("std::exp(s[kk] - smax)", "std::exp(smax - s[kk])"),
    "attn_wrong_head_offset": ("k + kk * H + head * dh", "k + kk * H"),
    "gelu_no_half": ("out[i] = 0.5 * in[i]", "out[i] = in[i]"),
    "gelu_no_sqrt2": ("std::erf(in[i] * inv_sqrt2)", "std::erf(in[i])"),
    "linear_no_bias": ("bias ? bias[j] : 0.0", "0.0"),
    "linear_transposed": ("ci[j] += a * wk[j]", "ci[j] += a * W[(j % K) * ldw + (k % N)]"),
    "add3_drops_term": ("out[i] = a[i] + b[i] + c[i]", "out[i] = a[i] + b[i]"),
    "rms_no_eps": ("inv = 1.0 / std::sqrt(sq / (double)H + eps)", "inv = 1.0 / std::sqrt(sq / (double)H)"),
    "norm_bwd_no_eps": ("rs = 1.0 / std::sqrt(sq / (double)H + eps)", "rs = 1.0 / std::sqrt(sq / (double)H)"),
    "rms_mean_not_square": ("sq += xr[c] * xr[c]", "sq += xr[c] * std::fabs(xr[c])"),
    "rms_no_gamma": ("o[c] = xr[c] * inv * gamma[c]", "o[c] = xr[c] * inv"),
    "silu_sign": ("gate[i] / (1.0 + std::exp(-gate[i]))", "gate[i] / (1.0 + std::exp(gate[i]))"),
    "swiglu_bwd_sigmoid_sign": ("sg = 1.0 / (1.0 + std::exp(-gate[i]))",
                                "sg = 1.0 / (1.0 + std::exp(gate[i]))"),
    "swiglu_drops_up": ("std::exp(-gate[i])) * up[i]", "std::exp(-gate[i]))"),
    "e4m3_ties_away": ("q = std::nearbyint(a / step) * step;", "q = std::round(a / step) * step;"),
    "e4m3_subnormal_step": ("std::nearbyint(a * 512.0)", "std::nearbyint(a * 256.0)"),
    "e4m3_bias_8": ("code = uint8_t(((E + 7) << 3) | mant);", "code = uint8_t(((E + 8) << 3) | mant);"),
    "e4m3_two_mantissa_bits": ("std::ldexp(1.0, ex - 3)", "std::ldexp(1.0, ex - 2)"),
    "e4m3_scale_inverted": ("const float s = amax / 448.0f;", "const float s = 448.0f / amax;"),
    # backward
    "norm_bwd_no_mean_term": ("rs * (g[c] - mean_g - xhat[c] * mean_gx)",
                              "rs * (g[c] - xhat[c] * mean_gx)"),
    "norm_bwd_no_xhat_term": ("rs * (g[c] - mean_g - xhat[c] * mean_gx)", "rs * (g[c] - mean_g)"),
    "norm_bwd_dgamma_no_xhat": ("sg += d * (x[r * H + c] - mu[r]) * rstd[r];", "sg += d;"),
    "norm_bwd_no_gamma": ("g[c] = dout[r * H + c] * gamma[c];", "g[c] = dout[r * H + c];"),
    "gelu_bwd_no_z_phi": ("dz[i] = dout[i] * (Phi + z[i] * phi);", "dz[i] = dout[i] * Phi;"),
    "swiglu_bwd_no_chain": ("sg * (1.0 + gate[i] * (1.0 - sg))", "sg"),
    "swiglu_bwd_dup_sigma": ("dup[i] = dout[i] * gate[i] * sg;", "dup[i] = dout[i] * sg;"),
    "attn_bwd_no_delta": ("p[j] * (dp[j] - pdp)", "p[j] * dp[j]"),
    "attn_bwd_dk_no_scale": ("dk[j * H + off + d] += ds * qi[d] * scale;",
                             "dk[j * H + off + d] += ds * qi[d];"),
    "attn_bwd_dv_from_ds": ("dv[j * H + off + d] += p[j] * doi[d];",
                            "dv[j * H + off + d] += ds * doi[d];"),
    "attn_bwd_window_off_by_one": ("std::max<int64_t>(0, i - w + 1)", "std::max<int64_t>(0, i - w)"),
    "attn_bwd_dq_uses_v": ("dqi[d] += ds * k[j * H + off + d] * scale;",
                           "dqi[d] += ds * v[j * H + off + d] * scale;"),
}

# Planted mistakes in the Python composition of the backward (oracle.py), each a one-line
# change, run through the backward pins on a mutated copy of the module.
PY_MUTANTS = {
    "bwd_no_residual_grad": ('g["dx"] = (dY + dx_norm)', 'g["dx"] = (dx_norm)'),
    "bwd_drops_mlp_path_into_dxn": ("+ linear(dh, w1.T, None, threads, lib)", ""),
    "bwd_wo_grad_from_act": ('"wo": linear(attn.T, dY', '"wo": linear(act[:, :H].T, dY'),
    "bwd_act_grad_skips_activation": ("dh = gelu_backward(h, d_act, threads, lib)", "dh = d_act"),
    "bwd_dqkv_order": ("dqkv = np.concatenate([dq, dk, dv], axis=1)",
                       "dqkv = np.concatenate([dk, dq, dv], axis=1)"),
}


@pytest.mark.parametrize("name", sorted(MUTANTS))
def test_mutant_is_caught(name, tmp_path):
    old, new = MUTANTS[name]
    src = open(O._SRC).read()
    assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
    path = tmp_path / "oracle_mutant.cpp"
    path.write_text(src.replace(old, new))
    lib_path = O.build(force=True, src=str(path), out=str(tmp_path / "libmutant.so"))
    lib = O.load(lib_path)
    failed = []
    for pin in P.ALL_PINS:
        try:
            ok, _ = pin(lib)
        except Exception:  # a crash or shape error also exposes the mistake
            ok = False
        if not ok:
            failed.append(pin.__name__)
    assert failed, f"no pin catches mutant {name}"
    assert os.path.exists(lib_path)


@pytest.mark.parametrize("name", sorted(PY_MUTANTS))
def test_python_backward_mutant_is_caught(name):
    import types

    old, new = PY_MUTANTS[name]
    src = open(O.__file__).read()
    assert src.count(old) == 1, f"mutation anchor not unique: {old!r}"
    import sys

    mod = types.ModuleType("oracle_mutant")
    mod.__file__ = O.__file__
    sys.modules[mod.__name__] = mod  # dataclasses look their module up here
    try:
        exec(compile(src.replace(old, new), "oracle_mutant.py", "exec"), mod.__dict__)
    finally:
        del sys.modules[mod.__name__]
    lib = O.load()
    failed = []
    for pin in (P.pin_backward_finite_differences, P.pin_backward_autograd):
        try:
            ok, _ = pin(lib, mod=mod)
        except Exception:
            ok = False
        if not ok:
            failed.append(pin.__name__)
    assert failed, f"no pin catches mutant {name}"
