"""GPU parity of the FP8 operand mode (``PB_OPERANDS_FP8``) against the oracle's FP8 block.

The oracle quantizes the same operands with the same current scaling (E4M3 for the forward
GEMMs, one scale per row of LN(x) and of [attention | GeLU(h)], one per output channel of the
packed weights; performance notes, "BF16 / FP16 / FP8"), so what is compared is the kernels,
not the FP8 rounding:

* the row quantizer on its own: bit-exact codes and scales on seeded bf16 rows (its fp32
  steps are fixed, so a correct implementation reproduces the bytes);
* the block: the output y, and the two branches att + mlp read in fp32 (the first layer of
  a two-layer stack keeps its output in the fp32 residual buffer; y's own bf16 rounding
  would hide a branch error), plus the intermediates before each quantization.

Tolerance of the branches (derived, written here): the GPU quantizes its own bf16 act, the
oracle the bf16 rounding of its fp64 act. Where the two bf16 values differ by one bf16 unit
(2^-8 relative), the E4M3 code (3 mantissa bits, 2^-4 relative spacing) differs with
probability about 2^-8 / 2^-4 = 1/16, and by one E4M3 unit when it does. The squared error
per element is then about 16 times that of the bf16 path, so the branches get 4 times the
bf16 path's bar on the quantized intermediate in the mean: 1.2e-2 (GeLU: act is checked
against 3e-3 in bf16), 1.6e-2 (SwiGLU: silu(gate) * up compounds three 16-bit roundings
and is checked against 4e-3), and 2.5 times the bf16 bar in the max (5e-2). Everything
upstream of the second quantization (q, k, v, attention, the MLP activation) keeps the
bf16 bar; the LN(x) codes are checked code by code.
"""

import numpy as np
import pytest
import torch

from oracle import oracle as O
from tests.parity import assert_parity, host, host_params, metrics, oracle_dims, report
from transformer_block_gb300 import WORKLOADS, inputs, pb
from transformer_block_gb300.configs import Workload

pytestmark = pytest.mark.gpu

BRANCH_MAX_TOL = 5e-2
BRANCH_MEAN_TOL = {0: 1.2e-2, 1: 1.6e-2}  # by block variant: LN + GeLU, RMSNorm + SwiGLU


@pytest.fixture(scope="module", autouse=True)
def _cuda():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    pb.lib()


def e4m3_values(codes: np.ndarray) -> np.ndarray:
    """Values of E4M3 codes from the format definition: sign bit, 4 exponent bits with bias
    7, 3 mantissa bits; exponent field 0 is subnormal (m * 2^-9). (0x7F / 0xFF, NaN, never
    comes out of a saturating quantizer of finite inputs.)"""
    c = codes.astype(np.int64)
    sign = np.where(c & 0x80, -1.0, 1.0)
    e, m = (c >> 3) & 0xF, c & 0x7
    normal = (1.0 + m / 8.0) * np.exp2(e - 7.0)
    sub = m * 2.0 ** -9
    return sign * np.where(e == 0, sub, normal)


# --------------------------------------------------------------------------- quantizer

def seeded_rows(rows, cols, seed):
    """bf16 rows of N(0, 1) values, row r scaled by 2^((r % 41) - 20) (so codes run into
    the subnormals and up to the saturation point), with row 0 all zero and row 1 a single
    non-zero value when there are enough rows."""
    g = torch.Generator().manual_seed(seed)
    x = torch.randn(rows, cols, generator=g, dtype=torch.float32)
    x *= torch.exp2(torch.arange(rows, dtype=torch.float32) % 41 - 20)[:, None]
    if rows > 2:
        x[0] = 0
        x[1] = 0
        x[1, cols // 2] = -3.0
    return x.to(torch.bfloat16)


@pytest.mark.parametrize("rows,cols", [(1, 8), (37, 264), (130, 4096), (5, 61440)])
def test_quantize_rows_bit_exact(rows, cols):
    x = seeded_rows(rows, cols, seed=rows * 7919 + cols)
    codes, scales = pb.quantize_rows_e4m3(x.cuda())
    torch.cuda.synchronize()
    want_codes, want_scales, _ = O.quantize_e4m3_rows(x.float().numpy())
    got_codes, got_scales = codes.cpu().numpy(), scales.cpu().numpy()
    assert np.array_equal(got_scales.view(np.uint32), want_scales.view(np.uint32))
    bad = np.argwhere(got_codes != want_codes)
    assert bad.size == 0, (f"{len(bad)} codes differ, first at {bad[0].tolist()}: "
                           f"{got_codes[tuple(bad[0])]:#x} vs {want_codes[tuple(bad[0])]:#x}")


def test_quantize_rows_rejects_ragged_columns():
    x = torch.zeros(4, 12, dtype=torch.bfloat16, device="cuda")
    with pytest.raises(pb.PbError):
        pb.quantize_rows_e4m3(x)


# --------------------------------------------------------------------------- block

def wl_fp8(name, B, S, H, nh, dh, F, w, variant=0):
    return Workload(name, B, S, H, nh, dh, F, w, 1, 0.02, variant=variant)


SMALL = [
    wl_fp8("fp8-b2-s130-h256", 2, 130, 256, 2, 128, 768, 64),
    wl_fp8("fp8-b3-s33-h128-dh64-w5", 3, 33, 128, 2, 64, 384, 5),
    wl_fp8("fp8-b2-s257-h256-w129", 2, 257, 256, 4, 64, 1024, 129),
    wl_fp8("fp8-b1-s1", 1, 1, 256, 2, 128, 768, 4),
    wl_fp8("fp8-glu-b2-s130-h256", 2, 130, 256, 2, 128, 768, 64, variant=1),
    wl_fp8("fp8-glu-b3-s33-h128-dh64", 3, 33, 128, 2, 64, 384, 5, variant=1),
]


def run_fp8(wl, biases=False):
    """The block in FP8 as the first layer of a two-layer stack of the same weights: the
    scratch then holds layer 1's intermediates and its output in fp32 (res0)."""
    x, params = inputs.make_layer(wl, 0, device="cuda", biases=biases)
    dims = pb.make_dims(wl)
    block = pb.ParallelBlock(dims, params, operand_precision=pb.PB_OPERANDS_FP8)
    scratch = pb.new_scratch(dims)
    y = block(x, scratch=scratch)
    torch.cuda.synchronize()
    assert block.status() == pb.PB_OK
    views = {n: pb.scratch_view(scratch, dims, n).clone()
             for n in ("qk", "vt", "act", "q8", "qscale")}
    views["xn"] = pb.scratch_view(scratch, dims, "xn", torch.uint8).clone()
    pb.forward_stack([block, block], x, scratch=scratch)
    torch.cuda.synchronize()
    assert block.status() == pb.PB_OK
    y32 = pb.scratch_view(scratch, dims, "res0").clone()
    return x, params, dims, y, y32, views


def check_block(wl, biases=False):
    x, params, dims, y, y32, v = run_fp8(wl, biases)
    B, S, H, T = wl.batch, wl.seq, wl.hidden, wl.tokens
    xh, hp = host(x).reshape(B, S, H), host_params(params)
    ref, st = O.block_forward(oracle_dims(wl), xh, hp, keep_stages=True, fp8=True)
    ref = ref.reshape(T, H)
    assert_parity(host(y), ref, f"{wl.name} y")
    x2 = xh.reshape(T, H)
    assert_parity(y32.cpu().numpy() - x2, ref - x2, f"{wl.name} att + mlp (fp32)",
                  BRANCH_MAX_TOL, BRANCH_MEAN_TOL[wl.variant])
    # LN(x) codes and scales, dequantized, against the oracle's quantized LN(x). The GPU
    # normalises in fp32, the oracle in fp64, so a value within ~1e-7 of an E4M3 rounding
    # boundary may take the neighbouring code: such flips must be rare and one step wide.
    qs = v["qscale"].cpu().numpy().astype(np.float64)
    xn = e4m3_values(v["xn"].cpu().numpy()) * qs[:T, None]
    r = st["xn"]
    diff = np.abs(xn - r)
    step = np.maximum(np.abs(r) * 2.0 ** -3, 2.0 ** -9 * qs[:T, None])  # >= one E4M3 unit
    flips = diff > 1e-6 * np.abs(r) + 1e-30
    print(f"{wl.name} E4M3 LN(x): {int(flips.sum())} of {flips.size} codes differ by one "
          f"step; max_rel={metrics(xn, r)[0]:.3e}")
    assert np.all(diff <= step * (1 + 1e-6))
    assert flips.mean() <= 1e-3
    qk = host(v["qk"])
    assert_parity(qk[:, :H], st["q"], f"{wl.name} q")
    assert_parity(qk[:, H:], st["k"], f"{wl.name} k")
    vt = host(v["vt"])[..., :S]
    assert_parity(vt.transpose(0, 3, 1, 2).reshape(T, H), st["v"], f"{wl.name} v")
    act = host(v["act"])
    assert_parity(act[:, :H], st["attn"], f"{wl.name} attention")
    assert_parity(act[:, H:], st["mlp_act"], f"{wl.name} MLP activation")
    # the second quantization, from the GPU's act against the oracle's: reported (its
    # effect on the result is what the branch check above bounds)
    q8 = e4m3_values(v["q8"].cpu().numpy()) * qs[T:, None]
    want = O.quantize_e4m3_rows(O.round_bf16(np.concatenate([st["attn"], st["mlp_act"]], 1)))[2]
    report(q8, want, f"{wl.name} E4M3 act")
    # properties of the fused quantizer's output against the GPU's own bf16 act: each row's
    # scale is its amax / 448, the largest code of a non-zero row is +-448, and every code
    # is within half an E4M3 step of act / scale (2^-4 relative for normal values, 2^-10
    # absolute in the subnormal range)
    sa = qs[T:]
    amax = np.abs(act).max(axis=1)
    assert np.allclose(sa, amax / 448.0, rtol=2e-7, atol=0)
    vals = e4m3_values(v["q8"].cpu().numpy())
    nz = amax > 0
    assert np.all(np.abs(vals[nz]).max(axis=1) == 448.0)
    scaled = np.divide(act, sa[:, None], out=np.zeros_like(act, dtype=np.float64),
                       where=sa[:, None] > 0)
    assert np.all(np.abs(vals - scaled) <= np.maximum(np.abs(scaled) * 2.0 ** -4, 2.0 ** -10)
                  * (1 + 1e-6))


@pytest.mark.parametrize("wl", SMALL, ids=lambda w: w.name)
def test_fp8_block_matches_oracle(wl):
    check_block(wl)


@pytest.mark.parametrize("variant", [0, 1])
def test_fp8_block_with_biases(variant):
    check_block(wl_fp8(f"fp8-bias-v{variant}", 2, 150, 256, 2, 128, 768, 40, variant), biases=True)


def test_fp8_against_bf16_oracle_reported():
    """How far FP8 operands move the block from the unquantized fp64 result (reported: the
    pages give FP8 as a speed option, with no accuracy figure for this block)."""
    wl = SMALL[0]
    x, params, dims, y, y32, v = run_fp8(wl)
    T, H = wl.tokens, wl.hidden
    x2 = host(x)
    ref = O.block_forward(oracle_dims(wl), x2.reshape(wl.batch, wl.seq, H),
                          host_params(params)).reshape(T, H)
    mx, mn = metrics(y32.cpu().numpy() - x2, ref - x2)
    print(f"FP8 vs unquantized, att + mlp: max_rel={mx:.3e} mean_rel={mn:.3e} (reported)")
    assert mn < 0.1  # gross-failure guard only


def test_fp8_rejects_unaligned_dims_and_serial():
    wl = wl_fp8("fp8-bad", 1, 64, 256, 2, 128, 704, 32)  # H + F = 960, not a multiple of 128
    x, params = inputs.make_layer(wl, 0, device="cuda")
    with pytest.raises(pb.PbError):
        pb.ParallelBlock(pb.make_dims(wl), params, operand_precision=pb.PB_OPERANDS_FP8)
    wl = SMALL[0]
    x, params = inputs.make_layer(wl, 0, device="cuda")
    block = pb.ParallelBlock(pb.make_dims(wl), params, operand_precision=pb.PB_OPERANDS_FP8)
    with pytest.raises(pb.PbError):
        block.forward_serial(x)


@pytest.mark.parametrize("name,clusters", [
    ("block-h2048", [(0, 3), (2047, 1), (1000, 3)]),
    ("gpt3-175b-layer", [(0, 2), (1023, 2), (-3, 3)]),
])
def test_fp8_full_size_sampled_rows(name, clusters):
    wl = WORKLOADS[name]
    x, params = inputs.make_layer(wl, 0, device="cuda")
    dims = pb.make_dims(wl)
    block = pb.ParallelBlock(dims, params, operand_precision=pb.PB_OPERANDS_FP8)
    y = block(x)
    torch.cuda.synchronize()
    assert block.status() == pb.PB_OK
    rows = {b: sorted({p for s, n in clusters
                       for p in range(max(0, s if s >= 0 else wl.seq + s),
                                      min(wl.seq, (s if s >= 0 else wl.seq + s) + n))})
            for b in range(wl.batch)}
    hp = host_params(params)
    del params, block
    xh = host(x).reshape(wl.batch, wl.seq, wl.hidden)
    ref = O.block_forward(oracle_dims(wl), xh, hp, rows=rows, fp8=True)
    yh = host(y).reshape(wl.batch, wl.seq, wl.hidden)
    g = np.concatenate([yh[b][rows[b]] for b in sorted(rows)])
    assert_parity(g, ref, f"{name} FP8 sampled y ({len(g)} rows)")
