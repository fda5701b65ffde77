"""GPU parity of the backward pass's pieces and of the whole block backward against the fp64
oracle (``oracle.block_backward``): the GEMM with MN-major operands (the weight gradients
contract over tokens, so token-major activations are MN-major operands there), then the
block's gradients."""

import numpy as np
import pytest
import torch

from oracle import oracle as O
from tests.parity import assert_parity, host
from transformer_block_gb300 import pb

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    pb.lib()


# --------------------------------------------------------------------------- GEMM layouts

@pytest.mark.parametrize("a_mn,b_mn", [(True, False), (False, True), (True, True)])
@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 512, 192), (200, 288, 128),
                                   (512, 768, 200), (1000, 1024, 1000), (264, 96, 8)])
def test_gemm_layouts_match_oracle(M, N, K, a_mn, b_mn):
    if not (a_mn and b_mn) and K % 8:
        pytest.skip("a K-major operand needs K % 8 == 0")
    g = torch.Generator(device="cuda").manual_seed(M * 5 + N * 3 + K + 7 * a_mn + 11 * b_mn)
    a = torch.randn(M, K, generator=g, device="cuda").to(torch.bfloat16)
    b = torch.randn(N, K, generator=g, device="cuda").to(torch.bfloat16)
    a_st = a.t().contiguous() if a_mn else a
    b_st = b.t().contiguous() if b_mn else b
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    scratch = torch.empty(pb.gemm_scratch_bytes(), dtype=torch.uint8, device="cuda")
    c = pb.gemm_layout(a_st, b_st, a_mn, b_mn, scratch=scratch, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = O.linear(host(a), host(b).T)
    assert_parity(host(c), ref, f"gemm {M}x{N}x{K} a_mn={a_mn} b_mn={b_mn}")


def test_gemm_layout_stream_k_ragged_tokens():
    # a weight-gradient shape: M = H + F rows, N = H, K = tokens not a multiple of 64,
    # enough tiles for a partial last wave (stream-K)
    M, N, K = 2560 + 256, 2048, 1000
    g = torch.Generator(device="cuda").manual_seed(3)
    a_st = torch.randn(K, M, generator=g, device="cuda").to(torch.bfloat16)
    b_st = torch.randn(K, N, generator=g, device="cuda").to(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    scratch = torch.empty(pb.gemm_scratch_bytes(), dtype=torch.uint8, device="cuda")
    c = pb.gemm_layout(a_st, b_st, True, True, scratch=scratch, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rows = np.sort(np.random.default_rng(4).choice(M, 128, replace=False))
    ref = O.linear(host(a_st).T[rows], host(b_st))
    assert_parity(host(c)[rows], ref, f"gemm {M}x{N}x{K} MN-major both")
