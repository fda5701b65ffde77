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
    "attn_no_scale": ("1.0 / std::sqrt((double)dh)", "1.0"),
    "attn_no_max_shift_sign": ("std::exp(s[kk] - smax)", "std::exp(smax - s[kk])"),
    "attn_wrong_head_offset": ("k + kk * H + head * dh", "k + kk * H"),
    "gelu_no_half": ("out[i] = 0.5 * in[i]", "out[i] = in[i]"),
    "gelu_no_sqrt2": ("std::erf(in[i] * inv_sqrt2)", "std::erf(in[i])"),
    "linear_no_bias": ("bias ? bias[j] : 0.0", "0.0"),
    "linear_transposed": ("ci[j] += a * wk[j]", "ci[j] += a * W[(j % K) * ldw + (k % N)]"),
    "add3_drops_term": ("out[i] = a[i] + b[i] + c[i]", "out[i] = a[i] + b[i]"),
    "rms_no_eps": ("std::sqrt(sq / (double)H + eps)", "std::sqrt(sq / (double)H)"),
    "rms_mean_not_square": ("sq += xr[c] * xr[c]", "sq += xr[c] * std::fabs(xr[c])"),
    "rms_no_gamma": ("o[c] = xr[c] * inv * gamma[c]", "o[c] = xr[c] * inv"),
    "silu_sign": ("(1.0 + std::exp(-gate[i]))", "(1.0 + std::exp(gate[i]))"),
    "swiglu_drops_up": ("std::exp(-gate[i])) * up[i]", "std::exp(-gate[i]))"),
    "e4m3_ties_away": ("q = std::nearbyint(a / step) * step;", "q = std::round(a / step) * step;"),
    "e4m3_subnormal_step": ("std::nearbyint(a * 512.0)", "std::nearbyint(a * 256.0)"),
    "e4m3_bias_8": ("code = uint8_t(((E + 7) << 3) | mant);", "code = uint8_t(((E + 8) << 3) | mant);"),
    "e4m3_two_mantissa_bits": ("std::ldexp(1.0, ex - 3)", "std::ldexp(1.0, ex - 2)"),
    "e4m3_scale_inverted": ("const float s = amax / 448.0f;", "const float s = 448.0f / amax;"),
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
