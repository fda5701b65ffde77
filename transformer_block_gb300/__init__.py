"""GB300-native forward pass of the parallel transformer block
``y = x + Attn_SWA(LN(x)) + MLP_GeLU(LN(x))``.

The compute path is the C-ABI library ``libpb.so`` (hand-written sm_103a kernels); the
Python side only marshals arguments (``transformer_block_gb300.pb``). Importing this
package does not load the library; the first call into ``pb`` does, and fails loudly
when it has not been built.
"""

from .configs import BENCH_WORKLOAD, WORKLOADS, Workload  # noqa: F401
