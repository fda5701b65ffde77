"""pb_gemm_bf16_static: the stream-K GEMM for callers that cannot allocate device memory
(plugins whose device memory all belongs to a host engine's allocator, paths where a
cudaMalloc could block), with its scratch in the library's own fixed device array.

It runs the same stream-K schedule as pb_gemm_bf16 with caller scratch, so on two calls in
a row (the second with new inputs, which stale partial tiles or flags left by the first
would corrupt) its output must equal that entry point's bit for bit, and so also meet the
oracle bar. The shapes leave a partial last wave, so tiles really are split along K: the
result differs in rounding from the whole-tile GEMM (no scratch). Collected last, so that
a failure here stops nothing else.
"""

import numpy as np
import pytest
import torch

from oracle import oracle as O
from tests.parity import assert_parity, host
from transformer_block_gb300 import pb

pytestmark = pytest.mark.gpu


# (4096, 5120, 16384): a long K, where the GEMM works in units of two 256-row M tiles and
# splits the leftover units into their tiles for stream-K.
@pytest.mark.parametrize("M,N,K", [(2048, 12288, 1024), (4160, 2080, 512), (4096, 5120, 16384)])
def test_static_scratch_gemm_matches_caller_scratch_gemm(M, N, K):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    g = torch.Generator(device="cuda").manual_seed(7 * M + N + K)
    a1 = torch.randn(M, K, generator=g, device="cuda").to(torch.bfloat16)
    a2 = torch.randn(M, K, generator=g, device="cuda").to(torch.bfloat16)
    b = torch.randn(N, K, generator=g, device="cuda").to(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    scratch = torch.zeros(pb.gemm_scratch_bytes(), dtype=torch.uint8, device="cuda")
    ref1 = pb.gemm(a1, b, scratch=scratch, status=status)
    ref2 = pb.gemm(a2, b, scratch=scratch, status=status)
    whole1 = pb.gemm(a1, b, status=status)
    first = pb.gemm_static(a1, b, status=status)
    second = pb.gemm_static(a2, b, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert torch.equal(first, ref1), "static-scratch gemm, first call"
    assert torch.equal(second, ref2), "static-scratch gemm, second call (new inputs)"
    # the K split changes the fp32 summation order of the split tiles: stream-K ran
    assert not torch.equal(first, whole1)
    rows = torch.randperm(M, generator=torch.Generator().manual_seed(3))[:256].sort().values
    r = rows.numpy()
    for out, a, what in ((first, a1, "first"), (second, a2, "second")):
        ref = O.linear(host(a)[r], host(b).T)
        assert_parity(host(out)[r], ref, f"static-scratch gemm {M}x{N}x{K}, {what} call")
