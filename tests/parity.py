"""Shared helpers of the GPU parity tests: the acceptance metrics and oracle adapters.

Acceptance on the same seeded bf16 inputs (fp32-accumulate GPU path vs fp64 oracle):
    max|g - r| / (max|r| + 1e-6) <= 2e-2      and      mean|g - r| / mean|r| <= 3e-3
"""

from __future__ import annotations

import numpy as np
import torch

from oracle import oracle as O

MAX_REL_TOL = 2e-2
MEAN_REL_TOL = 3e-3


def metrics(g, r) -> tuple[float, float]:
    g = np.asarray(g, dtype=np.float64)
    r = np.asarray(r, dtype=np.float64)
    assert g.shape == r.shape, (g.shape, r.shape)
    err = np.abs(g - r)
    max_rel = float(err.max() / (np.abs(r).max() + 1e-6))
    mean_rel = float(err.mean() / max(np.abs(r).mean(), 1e-300))
    return max_rel, mean_rel


def assert_parity(g, r, what: str, max_tol=MAX_REL_TOL, mean_tol=MEAN_REL_TOL):
    g = np.asarray(g, dtype=np.float64)
    assert np.all(np.isfinite(g)), f"{what}: non-finite GPU output"
    mx, mn = metrics(g, r)
    print(f"{what}: max_rel={mx:.3e} mean_rel={mn:.3e}")
    assert mx <= max_tol and mn <= mean_tol, f"{what}: max_rel={mx:.3e} mean_rel={mn:.3e}"


def report(g, r, what: str):
    """Prints the metrics without asserting. Used for the branch sum y - x: its error is
    dominated by the bf16 rounding of y itself (|y| ~ 1 while |y - x| ~ 0.05), so it has
    no tolerance of its own; each branch is checked through the intermediates instead."""
    mx, mn = metrics(g, r)
    print(f"{what}: max_rel={mx:.3e} mean_rel={mn:.3e} (reported)")


def host(t: torch.Tensor) -> np.ndarray:
    """Exact float32 copy of a bf16 tensor (every bf16 value is a float32)."""
    return t.detach().float().cpu().numpy()


def host_params(params: dict) -> dict:
    return {k: host(v) for k, v in params.items()}


def oracle_dims(wl) -> O.Dims:
    return O.Dims(wl.batch, wl.seq, wl.hidden, wl.heads, wl.head_dim, wl.ffn, wl.window,
                  wl.ln_eps, getattr(wl, "variant", 0))
