"""Model FLOPs of the parallel block forward pass.

The count follows the MFU convention of the Megatron-LM performance notes ("MFU" section):
model FLOPs are 2 per weight per token in the forward pass plus the attention term, and
work a method adds (recomputation) or skips is not counted. For sliding-window causal
attention the attention term counts the (query, key) pairs the window actually admits:
QK^T and PV each take 2*dh multiply-adds per pair and head, i.e. 4*H FLOPs per pair.
LayerNorm, bias, GeLU and softmax arithmetic are not counted.
"""

from __future__ import annotations

from .configs import Workload


def windowed_pairs(seq: int, window: int) -> int:
    """sum_{i<seq} min(i+1, window): visible (query, key) pairs in one sequence."""
    if window >= seq:
        return seq * (seq + 1) // 2
    return window * (window + 1) // 2 + (seq - window) * window


def gemm_flops(wl: Workload) -> int:
    """Per layer: 2 * tokens * (Wq, Wk, Wv, Wo: 4 H^2  +  W1, W2: 2 H F); the SwiGLU
    variant has W_gate, W_up, W2: 3 H F."""
    H, F = wl.hidden, wl.ffn
    mlp = 3 if getattr(wl, "variant", 0) == 1 else 2
    return 2 * wl.tokens * (4 * H * H + mlp * H * F)


def attention_flops(wl: Workload) -> int:
    """Per layer: 4 * H * batch * windowed pairs."""
    return 4 * wl.hidden * wl.batch * windowed_pairs(wl.seq, wl.window)


def model_flops(wl: Workload) -> int:
    return wl.layers * (gemm_flops(wl) + attention_flops(wl))
