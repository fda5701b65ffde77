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


# --------------------------------------------------------------------------- block backward

from tests.parity import host_params, metrics, oracle_dims, report  # noqa: E402
from transformer_block_gb300 import inputs  # noqa: E402
from transformer_block_gb300.configs import Workload  # noqa: E402


# Bars of the backward (mean relative error; the max bar stays 2e-2). A product of bf16
# operands accumulated in fp32 meets 3e-3; one that compounds the rounding of two bf16
# intermediates (dv = P^T dO with P and dO rounded, dW from rounded activations and
# gradients) gets 4e-3, the bar already used for compounded roundings. dq and dk read
# dS = P (dP - D), which subtracts two nearly equal numbers (D is the P-weighted mean of
# dP per row), so the rounding of dO, V and O reaches dS enlarged; measured, dq and dk sit
# at 1.5 - 1.6 times dv's error on every case here, hence 1.5 x 4e-3 for them and for
# what is computed from them (dLN(x), dWqkv, db_qkv, dgamma, dbeta).
COMPOUND_MEAN_TOL = 4e-3
DS_MEAN_TOL = 6e-3


def wl_b(name, B, S, H, nh, dh, F, w, variant=0):
    return Workload(name, B, S, H, nh, dh, F, w, 1, 0.02, variant=variant)


BWD = [
    wl_b("bwd-b1-s128-h256-w32", 1, 128, 256, 2, 128, 512, 32),
    wl_b("bwd-b2-s130-h256-w64", 2, 130, 256, 2, 128, 512, 64),
    wl_b("bwd-b2-s257-h384-w129", 2, 257, 384, 3, 128, 768, 129),
    wl_b("bwd-b1-s300-w300", 1, 300, 256, 2, 128, 512, 300),
    wl_b("bwd-b1-s1", 1, 1, 256, 2, 128, 512, 4),
    wl_b("bwd-glu-b2-s130-w64", 2, 130, 256, 2, 128, 512, 64, variant=1),
    wl_b("bwd-glu-b1-s200-w200", 1, 200, 256, 2, 128, 768, 200, variant=1),
    # head size 64: the tiny workload's shape, ragged tiles, and the SwiGLU variant
    wl_b("bwd-dh64-b1-s128-h256-w32", 1, 128, 256, 4, 64, 1024, 32),
    wl_b("bwd-dh64-b2-s130-h256-w64", 2, 130, 256, 4, 64, 512, 64),
    wl_b("bwd-dh64-b1-s257-h192-w129", 1, 257, 192, 3, 64, 384, 129),
    wl_b("bwd-glu-dh64-b3-s33-h128-w5", 3, 33, 128, 2, 64, 256, 5, variant=1),
    # rows wider than 4096: the normalisation backward's four-warps-per-row kernel, with
    # a ragged last vector per thread (528 vectors of 8 over 128 threads); weights at the
    # scale of the wide workloads (std 0.006), so each branch stays below x as there
    Workload("bwd-b1-s64-h4224", 1, 64, 4224, 33, 128, 256, 64, 1, 0.006),
    Workload("bwd-glu-b1-s64-h4224", 1, 64, 4224, 33, 128, 256, 64, 1, 0.006, variant=1),
]


def deinterleave(F):
    """Column order of [gate | up] from W1cat's interleave of the SwiGLU h columns."""
    idx = np.empty(2 * F, dtype=np.int64)
    for c in range(2 * F):
        t, i = divmod(c, 32)
        idx[16 * t + i if i < 16 else F + 16 * t + i - 16] = c
    return idx


def run_backward(wl, biases=False, seed=0):
    x, params = inputs.make_layer(wl, 0, seed=seed, device="cuda", biases=biases)
    dims = pb.make_dims(wl)
    block = pb.ParallelBlock(dims, params)
    scratch = pb.new_train_scratch(dims)
    y = block.forward_train(x, scratch)
    g = torch.Generator(device="cuda").manual_seed(1000 + seed)
    dy = torch.randn(x.shape, generator=g, device="cuda").to(torch.bfloat16)
    grads = block.backward(x, dy, scratch, biases=biases)
    torch.cuda.synchronize()
    assert block.status() == pb.PB_OK
    return x, params, dims, block, scratch, y, dy, grads


def check_backward(wl, biases=False, branch_tol=None):
    x, params, dims, block, scratch, y, dy, grads = run_backward(wl, biases)
    B, S, H, F = wl.batch, wl.seq, wl.hidden, wl.ffn
    T = B * S
    ref = O.block_backward(oracle_dims(wl), host(x).reshape(B, S, H), host_params(params),
                           host(dy).reshape(B, S, H), keep_stages=True)
    st = ref["stages"]
    # the training forward's output is the forward's
    yref = O.block_forward(oracle_dims(wl), host(x).reshape(B, S, H), host_params(params))
    assert_parity(host(y), yref.reshape(T, H), f"{wl.name} forward y")
    # intermediates of the backward
    assert_parity(host(pb.scratch_view(scratch, dims, "d_attn")), st["d_attn"],
                  f"{wl.name} d_attn")
    dz = host(pb.scratch_view(scratch, dims, "dz"))
    dh = dz[:, 3 * H:]
    if wl.variant == 1:
        dh = dh[:, deinterleave(F)]
    assert_parity(dh, st["dh"], f"{wl.name} dh")
    assert_parity(dz[:, 2 * H:3 * H], st["dv"], f"{wl.name} dv", mean_tol=COMPOUND_MEAN_TOL)
    if S == 1 or wl.window == 1:
        # one visible key: softmax has no freedom, dq = dk = 0 exactly; the kernel's dP - D
        # is a difference of two fp32 sums of the same products
        scale = float(np.abs(st["dv"]).max())
        assert np.abs(dz[:, :2 * H]).max() <= 1e-3 * scale
    else:
        assert_parity(dz[:, H:2 * H], st["dk"], f"{wl.name} dk", mean_tol=DS_MEAN_TOL)
        assert_parity(dz[:, :H], st["dq"], f"{wl.name} dq", mean_tol=DS_MEAN_TOL)
    assert_parity(pb.scratch_view(scratch, dims, "dxn").cpu().numpy(), st["dxn"],
                  f"{wl.name} dLN(x)", mean_tol=DS_MEAN_TOL)
    # the gradients
    dx = host(grads["dx"])
    assert_parity(dx, ref["dx"].reshape(T, H), f"{wl.name} dx")
    if branch_tol is None:  # dy dominates dx: its bf16 rounding hides the branches
        report(dx - host(dy), ref["dx"].reshape(T, H) - host(dy), f"{wl.name} dx - dy")
    else:
        assert_parity(dx - host(dy), ref["dx"].reshape(T, H) - host(dy), f"{wl.name} dx - dy",
                      mean_tol=branch_tol)
    names = ["ln_gamma", "wqkv", "w1", "wo", "w2"] + ([] if wl.variant == 1 else ["ln_beta"])
    if biases:
        names += ["b_qkv", "b1", "b_o", "b2"]
    key = {"ln_gamma": "dgamma", "ln_beta": "dbeta", "wqkv": "dwqkv", "w1": "dw1", "wo": "dwo",
           "w2": "dw2", "b_qkv": "db_qkv", "b1": "db1", "b_o": "db_o", "b2": "db2"}
    for n in names:
        tol = DS_MEAN_TOL if n in ("ln_gamma", "ln_beta", "wqkv", "b_qkv") else COMPOUND_MEAN_TOL
        assert_parity(grads[key[n]].cpu().numpy(), ref[n], f"{wl.name} d{n}", mean_tol=tol)
    return x, params, dims, block, scratch, dy, grads


@pytest.mark.parametrize("wl", BWD, ids=lambda w: w.name)
def test_backward_matches_oracle(wl):
    check_backward(wl)


@pytest.mark.parametrize("variant", [0, 1])
def test_backward_strong_branches(variant):
    # weights of std 1 / sqrt(H) (3x the default): the branches' gradient is then about 9x
    # larger, enough that dx - dy (the normalisation backward) shows through dx's rounding
    # (larger logits make the recomputed P's error larger too: the other gradients are
    # reported here, checked at the default init above)
    wl = Workload(f"bwd-strong-v{variant}", 2, 140, 256, 2, 128, 512, 48, 1, 0.0625,
                  variant=variant)
    x, params, dims, block, scratch, y, dy, grads = run_backward(wl)
    B, S, H = wl.batch, wl.seq, wl.hidden
    ref = O.block_backward(oracle_dims(wl), host(x).reshape(B, S, H), host_params(params),
                           host(dy).reshape(B, S, H))
    dyh = host(dy)
    dxr = ref["dx"].reshape(B * S, H)
    mx, mn = metrics(dyh, dxr)
    print(f"{wl.name}: |dx - dy| / |dx| = {np.abs(dxr - dyh).mean() / np.abs(dxr).mean():.3f}")
    assert_parity(host(grads["dx"]) - dyh, dxr - dyh, f"{wl.name} dx - dy",
                  mean_tol=DS_MEAN_TOL)
    for n, k in (("ln_gamma", "dgamma"), ("wqkv", "dwqkv"), ("w1", "dw1"), ("wo", "dwo"),
                 ("w2", "dw2")):
        report(grads[k].cpu().numpy(), ref[n], f"{wl.name} d{n}")


@pytest.mark.parametrize("variant", [0, 1])
def test_backward_with_biases(variant):
    check_backward(wl_b(f"bwd-bias-v{variant}", 2, 150, 256, 2, 128, 512, 40, variant),
                   biases=True)


# dq is summed over key tiles with floating-point atomics, so what depends on it (dx,
# dgamma, dbeta, dWqkv, db_qkv) may differ in the last bits from run to run; the rest is
# computed in a fixed order.
DQ_FREE = ("dwo", "dw2", "dw1", "db_o", "db2", "db1")


def test_backward_accumulates_and_is_deterministic():
    wl = BWD[1]
    x, params, dims, block, scratch, y, dy, g1 = run_backward(wl, biases=True)
    g2 = block.backward(x, dy, scratch, biases=True)
    g3 = block.backward(x, dy, scratch, grads={k: v.clone() for k, v in g2.items()},
                        accumulate=True)
    torch.cuda.synchronize()
    for k in g1:
        if k in DQ_FREE:
            assert torch.equal(g1[k], g2[k]), k
            assert torch.allclose(g3[k], 2 * g2[k], rtol=1e-6, atol=1e-7), k
        else:
            a, b = g1[k].float(), g2[k].float()
            assert torch.allclose(a, b, rtol=1e-2, atol=1e-3 * float(b.abs().max())), k
            if k != "dx":
                assert torch.allclose(g3[k], 2 * g2[k], rtol=1e-2,
                                      atol=1e-3 * float(g2[k].abs().max())), k


def test_backward_rejects_unsupported_handles():
    wl = BWD[0]
    x, params = inputs.make_layer(wl, 0, device="cuda")
    dims = pb.make_dims(wl)
    scratch = pb.new_train_scratch(dims)
    with pytest.raises(pb.PbError):
        pb.ParallelBlock(dims, params, operand_precision=pb.PB_OPERANDS_FP16).forward_train(
            x, scratch)
    with pytest.raises(pb.PbError):  # y must not overwrite x
        pb.ParallelBlock(dims, params).forward_train(x, scratch, y=x)


def test_two_layer_training_through_per_layer_calls():
    # A stack trains through per-layer calls, each layer with its own training scratch:
    # forward layer by layer, then backward in reverse, layer l's dx the dy of layer l - 1.
    wl = Workload("bwd-stack2", 2, 130, 256, 2, 128, 512, 48, 2, 0.02)
    x, layers = inputs.make_stack(wl, device="cuda")
    dims = pb.make_dims(wl)
    blocks = [pb.ParallelBlock(dims, p) for p in layers]
    scr = [pb.new_train_scratch(dims) for _ in blocks]
    acts = [x]
    for b, s in zip(blocks, scr):
        acts.append(b.forward_train(acts[-1], s))
    g = torch.Generator(device="cuda").manual_seed(5)
    dy = torch.randn(x.shape, generator=g, device="cuda").to(torch.bfloat16)
    grads = [None, None]
    d = dy
    for i in (1, 0):
        grads[i] = blocks[i].backward(acts[i], d, scr[i], biases=False)
        d = grads[i]["dx"]
    torch.cuda.synchronize()
    for b in blocks:
        assert b.status() == pb.PB_OK
    # the oracle, on its own fp64 activations
    B, S, H = wl.batch, wl.seq, wl.hidden
    od = oracle_dims(wl)
    hp = [host_params(p) for p in layers]
    xs = [host(x).reshape(B, S, H)]
    xs.append(O.block_forward(od, xs[0], hp[0]))
    ref1 = O.block_backward(od, xs[1], hp[1], host(dy).reshape(B, S, H))
    ref0 = O.block_backward(od, xs[0], hp[0], ref1["dx"])
    assert_parity(host(grads[0]["dx"]), ref0["dx"].reshape(-1, H), "stack2 dx")
    for i, ref in ((0, ref0), (1, ref1)):
        for n, k in (("wqkv", "dwqkv"), ("w1", "dw1"), ("wo", "dwo"), ("w2", "dw2"),
                     ("ln_gamma", "dgamma")):
            tol = DS_MEAN_TOL if n in ("wqkv", "ln_gamma") else COMPOUND_MEAN_TOL
            assert_parity(grads[i][k].cpu().numpy(), ref[n], f"stack2 layer {i} d{n}",
                          mean_tol=tol)


def test_backward_full_width_matches_oracle():
    # The width of gpt3-175b-layer (H 12288, 96 heads of 128), full causal attention over
    # 640 tokens (five key tiles, a ragged last query tile) with F cut to 4096 so the fp64
    # oracle stays near 4 TFLOP. Every backward GEMM runs several waves of tiles and splits
    # its last waves along K (stream-K): d act (640 x 16384, K 12288), dLN(x) (640 x 12288,
    # K 40960), [dWo ; dW2] (16384 x 12288, K 640) and [dWqkv | dW1] (12288 x 40960, K 640).
    wl = Workload("bwd-h12288-s640", 1, 640, 12288, 96, 128, 4096, 640, 1, 0.006)
    check_backward(wl)
