"""The five workloads of the parallel transformer block forward pass.

Shapes and value distributions follow the workloads the pages' method is run on:
a tiny block, a hidden-2048 block, one layer shaped like GPT-3 175B (hidden 12288,
96 heads, Megatron-LM notes section 5.6 shape table), a 32k-token sliding-window
stress case (window 4096, the window MegaScale trains with, reading notes section 1.1)
and an 8-layer stack of residual blocks.
"""

from __future__ import annotations

from dataclasses import dataclass


@dataclass(frozen=True)
class Workload:
    name: str
    batch: int
    seq: int
    hidden: int
    heads: int
    head_dim: int
    ffn: int
    window: int
    layers: int
    weight_std: float
    ln_eps: float = 1e-5
    # 0: LayerNorm + GeLU MLP; 1: RMSNorm + SwiGLU MLP (w1 = [W_gate | W_up], [H, 2F])
    variant: int = 0

    @property
    def tokens(self) -> int:
        return self.batch * self.seq

    def with_(self, **kw) -> "Workload":
        d = dict(self.__dict__)
        d.update(kw)
        return Workload(**d)


WORKLOADS = {
    "tiny": Workload("tiny", 1, 128, 256, 4, 64, 1024, 32, 1, 0.02),
    "block-h2048": Workload("block-h2048", 4, 2048, 2048, 16, 128, 8192, 512, 1, 0.02),
    "gpt3-175b-layer": Workload("gpt3-175b-layer", 1, 2048, 12288, 96, 128, 49152, 2048, 1,
                                0.006),
    "long-swa-32k": Workload("long-swa-32k", 1, 32768, 4096, 32, 128, 16384, 4096, 1, 0.02),
    "stack8-h5120": Workload("stack8-h5120", 2, 4096, 5120, 40, 128, 20480, 1024, 8, 0.01),
    # RMSNorm + SwiGLU variants; F = 8H/3 keeps the MLP's weights and FLOPs equal to the
    # GeLU block's with F = 4H
    "tiny-swiglu": Workload("tiny-swiglu", 1, 128, 256, 4, 64, 704, 32, 1, 0.02, variant=1),
    "gpt3-175b-layer-swiglu": Workload("gpt3-175b-layer-swiglu", 1, 2048, 12288, 96, 128, 32768,
                                       2048, 1, 0.006, variant=1),
}

# The single-GPU workload the throughput figure is quoted on.
BENCH_WORKLOAD = "gpt3-175b-layer"
