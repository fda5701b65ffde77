"""Constants the CUDA kernels take from published methods, checked against those methods'
stated accuracy (CPU only; the kernels' sources are read as text)."""

import math
import os
import re

import numpy as np

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def _gemm_source():
    return open(os.path.join(ROOT, "transformer_block_gb300", "csrc", "gemm.cu")).read()


def test_gelu_erf_constants_meet_the_published_bound():
    # The first GEMM's GeLU uses Abramowitz & Stegun 7.1.26: for x >= 0,
    # 1 - erf(x) = (a1 t + ... + a5 t^5) exp(-x^2), t = 1 / (1 + p x), |error| <= 1.5e-7.
    src = _gemm_source()
    names = ["kP", "kA1", "kA2", "kA3", "kA4", "kA5"]
    vals = {}
    for n in names:
        m = re.search(rf"\b{n}\s*=\s*(-?[0-9.]+)f", src)
        assert m, n
        vals[n] = float(m.group(1))
    x = np.linspace(0.0, 8.0, 80001)
    t = 1.0 / (1.0 + vals["kP"] * x)
    poly = t * (vals["kA1"] + t * (vals["kA2"] + t * (vals["kA3"] + t * (vals["kA4"] +
                                                                       t * vals["kA5"]))))
    approx = 1.0 - poly * np.exp(-x * x)
    exact = np.array([math.erf(v) for v in x])
    assert np.abs(approx - exact).max() <= 1.5e-7
    # a dropped or mistyped term would be far outside the bound
    bad = 1.0 - (poly - t * vals["kA1"]) * np.exp(-x * x)
    assert np.abs(bad - exact).max() > 1e-3
