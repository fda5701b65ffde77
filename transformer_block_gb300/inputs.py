"""Seeded synthetic inputs shared by the CUDA path's tests and the oracle.

This module holds none of the method's arithmetic: it only draws numbers. Every tensor
is drawn in float32 from ``torch.randn`` on a generator seeded with
``seed * 1000 + layer`` and rounded to bf16 (round to nearest even), so both sides
consume identical bf16 values. Draw order per layer stream: ``x`` (layer 0 only), then
``ln_gamma = 1 + 0.1 N``, ``ln_beta = 0.1 N``, ``Wq, Wk, Wv, W1, Wo, W2 = std * N``
(``[in, out]`` layout; for the RMSNorm + SwiGLU variant W1 is ``[H, 2F]`` = gate | up and
``ln_beta`` is drawn but unused), then, if requested, the biases ``b_qkv, b1, b_o, b2 = 0.02 N``,
then, if requested, a second LayerNorm ``ln2_gamma = 1 + 0.1 N``, ``ln2_beta = 0.1 N`` (the
serial block's). ``x ~ N(0, 1)``.
"""

from __future__ import annotations

import torch

from .configs import Workload


def _gen(device, seed: int, layer: int) -> torch.Generator:
    g = torch.Generator(device=device)
    g.manual_seed(seed * 1000 + layer)
    return g


def _draw(g, shape, device, scale=1.0, shift=0.0) -> torch.Tensor:
    t = torch.randn(shape, generator=g, device=device, dtype=torch.float32)
    if scale != 1.0:
        t.mul_(scale)
    if shift != 0.0:
        t.add_(shift)
    return t.to(torch.bfloat16)


def make_layer(wl: Workload, layer: int = 0, seed: int = 0, device="cpu", biases: bool = False,
               ln2: bool = False):
    """Returns ``(x or None, params)``; ``x`` is ``[B*S, H]`` bf16 and only drawn for layer 0."""
    H, F = wl.hidden, wl.ffn
    g = _gen(device, seed, layer)
    x = _draw(g, (wl.tokens, H), device) if layer == 0 else None
    p = {
        "ln_gamma": _draw(g, (H,), device, 0.1, 1.0),
        "ln_beta": _draw(g, (H,), device, 0.1),
    }
    wq = _draw(g, (H, H), device, wl.weight_std)
    wk = _draw(g, (H, H), device, wl.weight_std)
    wv = _draw(g, (H, H), device, wl.weight_std)
    p["wqkv"] = torch.cat([wq, wk, wv], dim=1).contiguous()
    del wq, wk, wv
    glu = getattr(wl, "variant", 0) == 1  # SwiGLU: w1 = [W_gate | W_up]
    p["w1"] = _draw(g, (H, 2 * F if glu else F), device, wl.weight_std)
    p["wo"] = _draw(g, (H, H), device, wl.weight_std)
    p["w2"] = _draw(g, (F, H), device, wl.weight_std)
    if biases:
        p["b_qkv"] = _draw(g, (3 * H,), device, 0.02)
        p["b1"] = _draw(g, (2 * F if glu else F,), device, 0.02)
        p["b_o"] = _draw(g, (H,), device, 0.02)
        p["b2"] = _draw(g, (H,), device, 0.02)
    if ln2:
        p["ln2_gamma"] = _draw(g, (H,), device, 0.1, 1.0)
        p["ln2_beta"] = _draw(g, (H,), device, 0.1)
    return x, p


def make_stack(wl: Workload, seed: int = 0, device="cpu", biases: bool = False):
    """``x`` and one parameter dict per layer (independent streams per layer)."""
    x, p0 = make_layer(wl, 0, seed, device, biases)
    layers = [p0] + [make_layer(wl, l, seed, device, biases)[1] for l in range(1, wl.layers)]
    return x, layers
