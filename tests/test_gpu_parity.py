"""GPU parity: the C-ABI path against the fp64 oracle on the same seeded bf16 inputs.

Small cases span several tiles and ragged tails and are compared element by element
on every output (and every intermediate the scratch exposes). Full-size workloads are
compared on sampled output rows the oracle computes exactly from their window cones.
"""

import numpy as np
import pytest
import torch

from oracle import oracle as O
from tests.parity import assert_parity, host, host_params, metrics, oracle_dims, report
from transformer_block_gb300 import WORKLOADS, inputs, pb
from transformer_block_gb300.configs import Workload

pytestmark = pytest.mark.gpu


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    pb.lib()


def wl_small(name, B, S, H, nh, dh, F, w, layers=1, std=0.02):
    return Workload(name, B, S, H, nh, dh, F, w, layers, std)


# --------------------------------------------------------------------------- single steps

@pytest.mark.parametrize("M,N,K", [(128, 256, 64), (256, 512, 128), (200, 288, 192),
                                   (1, 32, 64), (300, 1056, 512), (1000, 768, 2048)])
def test_gemm_matches_oracle(M, N, K):
    g = torch.Generator(device="cuda").manual_seed(M * 7 + N * 3 + K)
    a = torch.randn(M, K, generator=g, device="cuda").to(torch.bfloat16)
    b = torch.randn(N, K, generator=g, device="cuda").to(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    c = pb.gemm(a, b, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    ref = O.linear(host(a), host(b).T)
    assert_parity(host(c), ref, f"gemm {M}x{N}x{K}")


@pytest.mark.parametrize("M,N,K", [(2048, 12288, 1024), (4160, 2080, 512),
                                   (256 * 77, 256, 640), (4096, 5120, 16384),
                                   (4160, 2560, 16384), (4160, 2080, 12288)])
def test_gemm_stream_k_matches_oracle(M, N, K):
    # Unit counts that leave a partial last wave on 76 CTA pairs, so the last units are
    # split along K (stream-K) when scratch is given; without scratch every unit is whole.
    # K >= 12288 with M > 256: units of two 256-row tiles, the leftover units split into
    # their tiles (4160 rows: a ragged last unit whose second tile is empty; 2080 columns:
    # a ragged last column block).
    g = torch.Generator(device="cuda").manual_seed(M + N + K)
    a = torch.randn(M, K, generator=g, device="cuda").to(torch.bfloat16)
    b = torch.randn(N, K, generator=g, device="cuda").to(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    scratch = torch.empty(pb.gemm_scratch_bytes(), dtype=torch.uint8, device="cuda")
    c_sk = pb.gemm(a, b, scratch=scratch, status=status)
    c_sk2 = pb.gemm(a, b, scratch=scratch, status=status)  # flags from the previous call
    c_dp = pb.gemm(a, b, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    rows = torch.randperm(M, generator=torch.Generator().manual_seed(1))[:256].sort().values
    ref = O.linear(host(a)[rows.numpy()], host(b).T)
    assert_parity(host(c_sk)[rows.numpy()], ref, f"stream-K gemm {M}x{N}x{K}")
    assert_parity(host(c_dp)[rows.numpy()], ref, f"whole-tile gemm {M}x{N}x{K}")
    assert torch.equal(c_sk, c_sk2)
    # the split changes the fp32 summation order, so some rounded outputs differ: the
    # stream-K path really ran
    assert not torch.equal(c_sk, c_dp)


def test_stream_k_leaves_its_flags_cleared():
    # Each stream-K flag is read by one warp, which clears it: after any completed call the
    # flags region (the last 96 pairs x 2 CTAs x 4 warps x 8 bytes of the scratch) is zero
    # again, so a later launch that carries the same epoch value cannot take a stale flag
    # (and the partial tiles next to it) for its own. New inputs on the second call make
    # stale partials visible in the output.
    M, N, K = 2048, 12288, 1024
    g = torch.Generator(device="cuda").manual_seed(11)
    a1 = torch.randn(M, K, generator=g, device="cuda").to(torch.bfloat16)
    a2 = torch.randn(M, K, generator=g, device="cuda").to(torch.bfloat16)
    b = torch.randn(N, K, generator=g, device="cuda").to(torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    scratch = torch.zeros(pb.gemm_scratch_bytes(), dtype=torch.uint8, device="cuda")
    flags = scratch[-96 * 2 * 4 * 8:].view(torch.int64)
    c1 = pb.gemm(a1, b, scratch=scratch, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert int(flags.count_nonzero()) == 0
    c2 = pb.gemm(a2, b, scratch=scratch, status=status)
    d2 = pb.gemm(a2, b, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    assert int(flags.count_nonzero()) == 0
    rows = np.arange(0, M, 8)
    assert_parity(host(c2)[rows], O.linear(host(a2)[rows], host(b).T), "stream-K, second call")
    assert_parity(host(c1)[rows], O.linear(host(a1)[rows], host(b).T), "stream-K, first call")
    assert not torch.equal(c2, d2)


def test_stream_k_gemms_on_two_streams_at_once():
    # Distinct scratch buffers make concurrent calls independent: two streams issue
    # stream-K GEMMs back to back, and every result equals the same call made alone.
    # A stream-K owner waits (boundedly) for its contributor pairs; a launch that could
    # never get them resident would end with a timeout status, checked here.
    M, N, K = 2048, 12288, 4096
    g = torch.Generator(device="cuda").manual_seed(13)
    A = [torch.randn(M, K, generator=g, device="cuda").to(torch.bfloat16) for _ in range(2)]
    B = [torch.randn(N, K, generator=g, device="cuda").to(torch.bfloat16) for _ in range(2)]
    scr = [torch.zeros(pb.gemm_scratch_bytes(), dtype=torch.uint8, device="cuda")
           for _ in range(2)]
    status = [torch.zeros(1, dtype=torch.int32, device="cuda") for _ in range(2)]
    ref = [pb.gemm(A[i], B[i], scratch=scr[i]) for i in range(2)]
    torch.cuda.synchronize()
    streams = [torch.cuda.Stream() for _ in range(2)]
    for s in streams:
        s.wait_stream(torch.cuda.current_stream())
    outs = [[torch.empty(M, N, dtype=torch.bfloat16, device="cuda") for _ in range(8)]
            for _ in range(2)]
    for it in range(8):
        for i in range(2):
            with torch.cuda.stream(streams[i]):
                pb.gemm(A[i], B[i], out=outs[i][it], scratch=scr[i], status=status[i],
                        stream=streams[i])
    torch.cuda.synchronize()
    assert [int(s.item()) for s in status] == [0, 0]
    for i in range(2):
        for it in range(8):
            assert torch.equal(outs[i][it], ref[i]), f"stream {i}, call {it}"


@pytest.mark.parametrize("rows,H", [(37, 256), (7, 128), (9, 384), (5, 2048), (300, 4096),
                                    (3, 12288), (64, 16384)])
def test_layernorm_matches_oracle(rows, H):
    g = torch.Generator(device="cuda").manual_seed(rows + H)
    x = (torch.randn(rows, H, generator=g, device="cuda") * 2 + 0.5).to(torch.bfloat16)
    gamma = (1 + 0.1 * torch.randn(H, generator=g, device="cuda")).to(torch.bfloat16)
    beta = (0.1 * torch.randn(H, generator=g, device="cuda")).to(torch.bfloat16)
    out = pb.layernorm(x, gamma, beta, 1e-5)
    torch.cuda.synchronize()
    ref = O.layernorm(host(x), host(gamma), host(beta), 1e-5)
    assert_parity(host(out), ref, f"layernorm {rows}x{H}")


# --------------------------------------------------------------------------- whole block

SMALL = [
    WORKLOADS["tiny"],
    wl_small("b2-s130-h256-dh128", 2, 130, 256, 2, 128, 512, 64),
    wl_small("b3-s33-h128-dh64-w5", 3, 33, 128, 2, 64, 256, 5),
    wl_small("b1-s300-h384-w300", 1, 300, 384, 3, 128, 768, 300),
    wl_small("b2-s257-h256-w129", 2, 257, 256, 4, 64, 1024, 129),
    wl_small("b1-s1", 1, 1, 256, 2, 128, 512, 4),
    wl_small("b1-s200-w1", 1, 200, 256, 2, 128, 512, 1),
    wl_small("b2-s384-h512-w1000", 2, 384, 512, 4, 128, 2048, 1000),
]


def run_block(wl, biases=False, seed=0, precision=pb.PB_OPERANDS_BF16):
    x, params = inputs.make_layer(wl, 0, seed=seed, device="cuda", biases=biases)
    dims = pb.make_dims(wl)
    block = pb.ParallelBlock(dims, params, operand_precision=precision)
    scratch = pb.new_scratch(dims)
    y = block(x, scratch=scratch)
    torch.cuda.synchronize()
    assert block.status() == pb.PB_OK
    return x, params, dims, block, scratch, y


PRECISIONS = {"bf16": pb.PB_OPERANDS_BF16, "fp16": pb.PB_OPERANDS_FP16}


@pytest.mark.parametrize("prec", ["bf16", "fp16"])
@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_block_matches_oracle(wl, prec):
    x, params, dims, block, scratch, y = run_block(wl, precision=PRECISIONS[prec])
    op_dtype = torch.float16 if prec == "fp16" else torch.bfloat16
    od = oracle_dims(wl)
    ref, st = O.block_forward(od, host(x).reshape(wl.batch, wl.seq, wl.hidden),
                              host_params(params), keep_stages=True)
    H, T = wl.hidden, wl.tokens
    assert_parity(host(y), ref.reshape(T, H), f"{wl.name} y")
    report(host(y) - host(x), ref.reshape(T, H) - host(x), f"{wl.name} y-x")
    # intermediates
    assert_parity(host(pb.scratch_view(scratch, dims, "xn", op_dtype)), st["xn"], f"{wl.name} xn")
    qk = host(pb.scratch_view(scratch, dims, "qk"))
    assert_parity(qk[:, :H], st["q"], f"{wl.name} q")
    assert_parity(qk[:, H:], st["k"], f"{wl.name} k")
    vt = host(pb.scratch_view(scratch, dims, "vt"))[..., :wl.seq]  # [B, nh, dh, S]
    v = vt.transpose(0, 3, 1, 2).reshape(T, H)
    assert_parity(v, st["v"], f"{wl.name} v")
    act = host(pb.scratch_view(scratch, dims, "act", op_dtype))
    assert_parity(act[:, :H], st["attn"], f"{wl.name} attention")
    assert_parity(act[:, H:], st["gelu_h"], f"{wl.name} GeLU(h)")


def test_block_with_biases():
    wl = wl_small("bias-b2-s150-h256", 2, 150, 256, 2, 128, 512, 40)
    x, params, dims, block, scratch, y = run_block(wl, biases=True)
    ref = O.block_forward(oracle_dims(wl), host(x).reshape(2, 150, 256), host_params(params))
    assert_parity(host(y), ref.reshape(-1, 256), "biases y")


def test_zero_affine_gives_identity_bit_exact():
    wl = wl_small("zero-affine", 2, 160, 256, 2, 128, 512, 50)
    x, params = inputs.make_layer(wl, 0, device="cuda")
    params["ln_gamma"].zero_()
    params["ln_beta"].zero_()
    y = pb.ParallelBlock(pb.make_dims(wl), params)(x)
    torch.cuda.synchronize()
    assert torch.equal(y, x)


def test_window_one_returns_v_exactly():
    wl = wl_small("w1", 2, 140, 256, 2, 128, 512, 1)
    x, params, dims, block, scratch, y = run_block(wl)
    vt = pb.scratch_view(scratch, dims, "vt")[..., :wl.seq]
    v = vt.permute(0, 3, 1, 2).reshape(wl.tokens, wl.hidden)
    attn = pb.scratch_view(scratch, dims, "act")[:, :wl.hidden]
    assert torch.equal(attn, v)


def test_in_place_matches_out_of_place():
    wl = wl_small("inplace", 1, 256, 256, 2, 128, 512, 64)
    x, params, dims, block, scratch, y = run_block(wl)
    x2 = x.clone()
    block(x2, y=x2, scratch=scratch)
    torch.cuda.synchronize()
    assert torch.equal(x2, y)


def test_deterministic():
    wl = wl_small("det", 2, 200, 256, 2, 128, 512, 70)
    x, params, dims, block, scratch, y = run_block(wl)
    y2 = block(x, scratch=scratch)
    torch.cuda.synchronize()
    assert torch.equal(y, y2)


@pytest.mark.parametrize("prec", ["bf16", "fp16"])
def test_stack_matches_oracle_and_host_path(prec):
    wl = wl_small("stack3", 2, 192, 256, 2, 128, 512, 48, layers=3)
    x, layers = inputs.make_stack(wl, device="cuda")
    dims = pb.make_dims(wl)
    blocks = [pb.ParallelBlock(dims, p, operand_precision=PRECISIONS[prec]) for p in layers]
    scratch = pb.new_scratch(dims)
    y = pb.forward_stack(blocks, x, scratch=scratch)
    xh = x.cpu().pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    pb.forward_stack_host(blocks, xh, yh, scratch)
    torch.cuda.synchronize()
    assert torch.equal(yh, y.cpu())
    ref = O.stack_forward(oracle_dims(wl), host(x), [host_params(p) for p in layers])
    assert_parity(host(y), ref.reshape(-1, wl.hidden), f"stack3 {prec} y")
    # the fp32 output is the same residual stream before its final rounding: rounded to
    # bf16 (nearest even) it gives the bf16 output bit for bit
    y32 = pb.forward_stack_f32(blocks, x, scratch=scratch)
    torch.cuda.synchronize()
    assert y32.dtype == torch.float32
    assert torch.equal(y32.to(torch.bfloat16), y)
    assert_parity(y32.cpu().numpy(), ref.reshape(-1, wl.hidden), f"stack3 {prec} fp32 y")
    # the residual stream between layers is fp32: chaining single-layer calls (bf16 between
    # layers) is close but not bit-identical
    z = x
    for b in blocks:
        z = b(z, scratch=scratch)
    torch.cuda.synchronize()
    assert_parity(host(z), ref.reshape(-1, wl.hidden), f"stack3 {prec} chained single layers")


# --------------------------------------------------------------------------- full sizes

def sample_rows(wl, clusters):
    rows = {}
    for b in range(wl.batch):
        pos = set()
        for start, n in clusters:
            s = start if start >= 0 else wl.seq + start
            pos.update(range(max(0, s), min(wl.seq, s + n)))
        rows[b] = sorted(pos)
    return rows


@pytest.mark.parametrize("name,clusters", [
    ("block-h2048", [(0, 4), (509, 6), (1500, 3), (-5, 5)]),
    ("gpt3-175b-layer", [(0, 3), (1023, 3), (-6, 6)]),
    ("long-swa-32k", [(0, 3), (4093, 5), (-5, 5)]),
])
def test_full_size_sampled_rows(name, clusters):
    wl = WORKLOADS[name]
    x, params, dims, block, scratch, y = run_block(wl)
    rows = sample_rows(wl, clusters)
    hp = host_params(params)
    del params
    ref = O.block_forward(oracle_dims(wl), host(x).reshape(wl.batch, wl.seq, wl.hidden), hp,
                          rows=rows)
    yh = host(y).reshape(wl.batch, wl.seq, wl.hidden)
    g = np.concatenate([yh[b][rows[b]] for b in sorted(rows)])
    assert_parity(g, ref, f"{name} sampled y ({len(g)} rows)")
    xh = host(x).reshape(wl.batch, wl.seq, wl.hidden)
    xs = np.concatenate([xh[b][rows[b]] for b in sorted(rows)])
    report(g - xs, ref - xs, f"{name} sampled y-x")


# stack8-h5120 (8 layers, window 1024) on a prefix of sequence 0. By causality the first P
# rows of every layer depend only on the first P inputs, so the fp64 oracle chains the 8
# layers on P tokens (about 7.7 TFLOP). P = 1536: from token 1023 on the 1024-key window is
# full, so a third of the graded rows see the window's far edge and its masking in every
# layer.
STACK8_P = 1536


@pytest.fixture(scope="module")
def stack8_prefix():
    wl = WORKLOADS["stack8-h5120"]
    x, layers = inputs.make_stack(wl, device="cuda")
    od = oracle_dims(wl)
    od = O.Dims(1, STACK8_P, od.hidden, od.heads, od.head_dim, od.ffn, od.window, od.ln_eps)
    z = host(x).reshape(wl.batch, wl.seq, wl.hidden)[:1, :STACK8_P].astype(np.float64)
    for p in layers:
        z = O.block_forward(od, z, host_params(p))
    return wl, x, layers, z.reshape(STACK8_P, wl.hidden)


def stack8_gpu_prefix(wl, x, layers, prec, f32_out=False):
    dims = pb.make_dims(wl)
    blocks = [pb.ParallelBlock(dims, p, operand_precision=PRECISIONS[prec]) for p in layers]
    y = pb.forward_stack_f32(blocks, x) if f32_out else pb.forward_stack(blocks, x)
    torch.cuda.synchronize()
    for b in blocks:
        assert b.status() == pb.PB_OK
    return host(y).reshape(wl.batch, wl.seq, wl.hidden)[0, :STACK8_P]


def test_full_size_stack_prefix_bf16_operands_fp32_output(stack8_prefix):
    # bf16 GEMM operands at the standard bar, with the stack's output taken as the fp32
    # residual stream it carries between layers (pb_forward_stack_f32), i.e. without the
    # final rounding of y to bf16, which alone costs 1.4e-3 of mean relative error.
    wl, x, layers, z = stack8_prefix
    g = stack8_gpu_prefix(wl, x, layers, "bf16", f32_out=True)
    report(g[1023:], z[1023:], "stack8 bf16 operands, fp32 y, window-full rows 1023..1535")
    assert_parity(g, z, f"stack8 bf16 operands, fp32 y, prefix {STACK8_P} rows")


def test_full_size_stack_prefix_fp16_operands(stack8_prefix):
    # The graded configuration of the 8-layer stack: 16-bit GEMM operands with 3 more
    # mantissa bits than bf16 (same tensor rate), fp32 accumulation, at the standard bar.
    wl, x, layers, z = stack8_prefix
    g = stack8_gpu_prefix(wl, x, layers, "fp16")
    report(g[1023:], z[1023:], "stack8 fp16 operands, window-full rows 1023..1535")
    assert_parity(g, z, f"stack8 fp16 operands, prefix {STACK8_P} rows")


@pytest.mark.xfail(strict=True, reason=(
    "known: with bf16 GEMM operands and y rounded to bf16 the 8-layer stack sits at about "
    "3.2e-3 mean relative error, above the 3e-3 bar; a CPU emulation of the same rounding "
    "points predicts it (3.17e-3 on this prefix); the rounding of the GEMM operands to bf16 "
    "(3.16e-3 with all else exact) and of y (1.41e-3 alone) add up past it"))
def test_full_size_stack_prefix_bf16_operands(stack8_prefix):
    # bf16 operands and the bf16 output at the standard bar, kept as a recorded known
    # failure: the max bar holds, the mean bar does not (strict: a pass would be reported).
    wl, x, layers, z = stack8_prefix
    g = stack8_gpu_prefix(wl, x, layers, "bf16")
    report(g, z, f"stack8 bf16 operands, prefix {STACK8_P} rows")
    report(g[1023:], z[1023:], "stack8 bf16 operands, window-full rows 1023..1535")
    mx, _ = metrics(g, z)
    assert mx <= 2e-2
    assert_parity(g, z, f"stack8 bf16 operands, prefix {STACK8_P} rows")


def test_fp16_range_violation_is_reported():
    wl = wl_small("range", 1, 128, 256, 2, 128, 512, 32)
    x, params = inputs.make_layer(wl, 0, device="cuda")
    params["ln_gamma"].fill_(30000.0)  # LN(x) then exceeds the fp16 range
    block = pb.ParallelBlock(pb.make_dims(wl), params, operand_precision=pb.PB_OPERANDS_FP16)
    block(x)
    torch.cuda.synchronize()
    assert block.status() == pb.PB_ERR_RANGE
    block.clear_status()
    torch.cuda.synchronize()
    assert block.status() == pb.PB_OK


def test_bounded_wait_gives_up_and_reports():
    # The kernels' bounded wait on a barrier nothing arrives at: after the limit the
    # kernel records PB_ERR_DEVICE_TIMEOUT (site 99) and returns; the context survives.
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    t0 = torch.cuda.Event(enable_timing=True)
    t1 = torch.cuda.Event(enable_timing=True)
    t0.record()
    pb.wait_probe(20_000_000, status)  # 20 ms
    t1.record()
    torch.cuda.synchronize()
    assert int(status.item()) == pb.PB_ERR_DEVICE_TIMEOUT | (99 << 8)
    assert t0.elapsed_time(t1) >= 19.0
    wl = wl_small("after-timeout", 1, 128, 256, 2, 128, 512, 32)
    x, params, dims, block, scratch, y = run_block(wl)
    assert torch.isfinite(y.float()).all()


def test_tiny_wait_limit_keeps_context_usable():
    # With a 1 ns limit every pipeline wait that is not satisfied at once may give up
    # (mbarrier.try_wait suspends the thread for a while first, so it rarely does); either
    # way the call ends, and a normal call afterwards gives the same bits as before.
    wl = wl_small("tiny-limit", 1, 256, 256, 2, 128, 512, 64)
    x, params = inputs.make_layer(wl, 0, device="cuda")
    block = pb.ParallelBlock(pb.make_dims(wl), params)
    ok = block(x)
    torch.cuda.synchronize()
    block.set_wait_limit_ns(1)
    block(x)
    torch.cuda.synchronize()
    assert block.status() in (pb.PB_OK, pb.PB_ERR_DEVICE_TIMEOUT)
    block.set_wait_limit_ns(2_000_000_000)
    block.clear_status()
    again = block(x)
    torch.cuda.synchronize()
    assert block.status() == pb.PB_OK
    assert torch.equal(again, ok)


def test_host_steps_match_device_stack():
    # the pipelined host-buffer entry point gives, step by step, the device path's bits
    wl = wl_small("steps", 2, 192, 256, 2, 128, 512, 48, layers=2)
    x, layers = inputs.make_stack(wl, device="cuda")
    dims = pb.make_dims(wl)
    blocks = [pb.ParallelBlock(dims, p) for p in layers]
    scratch = pb.new_scratch(dims)
    xs = [x, (x * 0.5).to(torch.bfloat16), (x + 1).to(torch.bfloat16)]
    want = [pb.forward_stack(blocks, xi, scratch=scratch) for xi in xs]
    torch.cuda.synchronize()
    for n in (1, 3):
        xh = [xi.cpu().pin_memory() for xi in xs[:n]]
        yh = [torch.empty_like(t).pin_memory() for t in xh]
        pb.forward_stack_host_steps(blocks, xh, yh, scratch)
        torch.cuda.current_stream().synchronize()
        for i in range(n):
            assert torch.equal(yh[i], want[i].cpu()), (n, i)
