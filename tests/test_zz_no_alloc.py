"""pb_gemm_bf16_static: the stream-K GEMM for callers that cannot allocate device memory
(graph capture, engine-owned memory, allocation-free paths), with its scratch in the
library's own fixed device array. Its output must match the caller-scratch entry point,
pb_gemm_bf16, on two calls in a row. Collected last, so a failure here stops nothing else.
"""

import pytest
import torch

from tests.parity import assert_parity, host
from transformer_block_gb300 import pb

pytestmark = pytest.mark.gpu


@pytest.mark.parametrize("M,N,K", [(2048, 12288, 1024), (4160, 2080, 512)])
def test_static_scratch_gemm_matches_caller_scratch_gemm(M, N, K):
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    g = torch.Generator(device="cuda").manual_seed(7 * M + N + K)
    a = torch.randn(M, K, generator=g, device="cuda").to(torch.bfloat16)
    b = torch.randn(N, K, generator=g, device="cuda").to(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    scratch = torch.empty(pb.gemm_scratch_bytes(), dtype=torch.uint8, device="cuda")
    ref = pb.gemm(a, b, scratch=scratch, status=status)
    first = pb.gemm_static(a, b, status=status)
    second = pb.gemm_static(a, b, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert_parity(host(first), host(ref), f"static-scratch gemm {M}x{N}x{K}, first call")
    assert_parity(host(second), host(ref), f"static-scratch gemm {M}x{N}x{K}, second call")
