"""Guard regions: no kernel writes outside the buffer regions it was given.

With ``pb_set_guard_bytes(G)`` every workspace and scratch layout leaves G unused bytes
after each region. Each test fills the weight workspace, the scratch, the outputs and the
gradient buffers with a canary byte (plus G canary bytes before and after every buffer),
runs calls on ragged shapes (sequence lengths 1, 33, 130 and 257; partial tiles of every
kernel), and checks byte for byte that every guard gap still holds the canary: an epilogue,
a TMA store or a reduction that ran past the end of a region, or wrote a neighbour's
gap, fails here even when the neighbour is rewritten later and every parity test passes.

A region's gap is found without its size: the next region starts at
align_up(end + G, 1024), so the G bytes just before each region's start (and before the
layout's end) always lie in the gap of the region before it.
"""

import pytest
import torch

from transformer_block_gb300 import inputs, pb
from transformer_block_gb300.configs import Workload

pytestmark = pytest.mark.gpu

G = 4096
CANARY = 0xA5

SCRATCH_REGIONS = ["xn", "qk", "vt", "act", "io", "io2", "res0", "res1", "sk", "q8", "qscale"]
TRAIN_REGIONS = ["hpre", "lse", "d_attn", "delta", "dq_acc", "dz", "dxn", "stats", "partials"]


@pytest.fixture(autouse=True)
def _guarded():
    if not torch.cuda.is_available():
        pytest.skip("no CUDA device")
    torch.cuda.set_device(0)
    pb.set_guard_bytes(G)
    yield
    pb.set_guard_bytes(0)


class Guarded:
    """n bytes of CUDA memory with G canary bytes before and after, all canary-filled."""

    def __init__(self, n: int):
        self.n = n
        self.buf = torch.full((n + 2 * G,), CANARY, dtype=torch.uint8, device="cuda")
        self.t = self.buf[G:G + n]  # 4096-byte offset: keeps the base 256-byte aligned

    def view(self, dtype, *shape):
        return self.t.view(dtype).view(*shape)

    def check_edges(self, what: str):
        bad = []
        for name, seg in (("before", self.buf[:G]), ("after", self.buf[G + self.n:])):
            n = int((seg != CANARY).sum())
            if n:
                bad.append(f"{what}: {n} canary bytes changed {name} the buffer")
        return bad


def guarded_tensor(shape, dtype) -> tuple[Guarded, torch.Tensor]:
    n = 1
    for s in shape:
        n *= s
    g = Guarded(n * torch.empty((), dtype=dtype).element_size())
    return g, g.view(dtype, *shape)


def layout_gaps(dims, train: bool):
    L = pb.scratch_layout(dims)
    names = SCRATCH_REGIONS + (TRAIN_REGIONS if train else [])
    starts = [getattr(L, n) for n in names]
    ends = starts[1:] + [L.train_total if train else L.total]
    return [(n, e - G, e) for n, e in zip(names, ends)]


def check_scratch(g: Guarded, dims, train: bool, what: str):
    bad = g.check_edges(what + " scratch")
    for name, lo, hi in layout_gaps(dims, train):
        n = int((g.t[lo:hi] != CANARY).sum())
        if n:
            bad.append(f"{what}: {n} canary bytes changed in the gap after scratch region {name}")
    return bad


def new_block(dims, params, precision=pb.PB_OPERANDS_BF16):
    ws = Guarded(pb.weight_workspace_bytes(dims))
    return ws, pb.ParallelBlock(dims, params, operand_precision=precision, workspace=ws.t)


def finish(what, blocks, guards):
    torch.cuda.synchronize()
    for b in blocks:
        assert b.status() == pb.PB_OK, what
    bad = []
    for gw, kind in guards:
        bad += gw() if callable(gw) else gw.check_edges(f"{what} {kind}")
    assert not bad, "\n".join(bad)


def wl(name, B, S, H, nh, dh, F, w, layers=1, variant=0):
    return Workload(name, B, S, H, nh, dh, F, w, layers, 0.02, variant=variant)


RAGGED = [
    wl("s1", 1, 1, 256, 2, 128, 512, 4),
    wl("s33-dh64", 3, 33, 128, 2, 64, 256, 5),
    wl("s130", 2, 130, 256, 2, 128, 512, 64),
    wl("s257-dh64", 2, 257, 256, 4, 64, 1024, 129),
]
RAGGED_DH128 = [
    wl("s1", 1, 1, 256, 2, 128, 512, 4),
    wl("s33", 3, 33, 256, 2, 128, 512, 5),
    wl("s130", 2, 130, 256, 2, 128, 512, 64),
    wl("s257", 2, 257, 384, 3, 128, 768, 129),
]
PRECISIONS = {"bf16": pb.PB_OPERANDS_BF16, "fp16": pb.PB_OPERANDS_FP16,
              "fp8": pb.PB_OPERANDS_FP8}


def test_checker_sees_a_planted_write():
    # the checker itself: a byte changed (by torch, not a kernel of this library) in one gap
    wl0 = RAGGED[2]
    dims = pb.make_dims(wl0)
    sg = Guarded(pb.scratch_bytes(dims))
    assert not check_scratch(sg, dims, False, "clean")
    name, lo, hi = layout_gaps(dims, False)[3]
    sg.t[hi - 1] = 0
    bad = check_scratch(sg, dims, False, "planted")
    assert len(bad) == 1 and f"region {name}" in bad[0]
    sg.buf[-1] = 0
    assert len(sg.check_edges("planted")) == 1


@pytest.mark.parametrize("prec", ["bf16", "fp16", "fp8"])
@pytest.mark.parametrize("w", RAGGED, ids=lambda w: w.name)
def test_forward_writes_stay_inside_their_regions(w, prec):
    dims = pb.make_dims(w)
    x, params = inputs.make_layer(w, 0, device="cuda")
    ws, block = new_block(dims, params, PRECISIONS[prec])
    sg = Guarded(pb.scratch_bytes(dims))
    yg, y = guarded_tensor((w.tokens, w.hidden), torch.bfloat16)
    block(x, y=y, scratch=sg.t)
    what = f"{w.name} {prec} forward"
    finish(what, [block], [(ws, "workspace"), (yg, "y"),
                           (lambda: check_scratch(sg, dims, False, what), "")])
    assert torch.isfinite(y.float()).all()


@pytest.mark.parametrize("w", RAGGED, ids=lambda w: w.name)
def test_swiglu_and_serial_writes_stay_inside_their_regions(w):
    wg = w.with_(variant=1)
    dims = pb.make_dims(wg)
    x, params = inputs.make_layer(wg, 0, device="cuda", ln2=True)
    ws, block = new_block(dims, params)
    sg = Guarded(pb.scratch_bytes(dims))
    yg, y = guarded_tensor((w.tokens, w.hidden), torch.bfloat16)
    block(x, y=y, scratch=sg.t)
    zg, z = guarded_tensor((w.tokens, w.hidden), torch.bfloat16)
    block.forward_serial(x, y=z, ln2_gamma=params["ln2_gamma"], ln2_beta=params["ln2_beta"],
                         scratch=sg.t)
    what = f"{w.name} swiglu forward + serial"
    finish(what, [block], [(ws, "workspace"), (yg, "y"), (zg, "serial y"),
                           (lambda: check_scratch(sg, dims, False, what), "")])


@pytest.mark.parametrize("w", RAGGED, ids=lambda w: w.name)
def test_stack_and_host_paths_stay_inside_their_regions(w):
    w2 = w.with_(layers=2)
    dims = pb.make_dims(w2)
    x, layers = inputs.make_stack(w2, device="cuda")
    made = [new_block(dims, p) for p in layers]
    blocks = [b for _, b in made]
    sg = Guarded(pb.scratch_bytes(dims))
    yg, y = guarded_tensor((w.tokens, w.hidden), torch.bfloat16)
    pb.forward_stack(blocks, x, y=y, scratch=sg.t)
    xh = x.cpu().pin_memory()
    yh = torch.empty_like(xh).pin_memory()
    pb.forward_stack_host(blocks, xh, yh, sg.t)
    xs = [xh, (x * 0.5).to(torch.bfloat16).cpu().pin_memory()]
    ys = [torch.empty_like(t).pin_memory() for t in xs]
    pb.forward_stack_host_steps(blocks, xs, ys, sg.t)
    y32g, y32 = guarded_tensor((w.tokens, w.hidden), torch.float32)
    pb.forward_stack_f32(blocks, x, y=y32, scratch=sg.t)
    what = f"{w.name} stack of 2"
    finish(what, blocks, [(ws, "workspace") for ws, _ in made] +
           [(yg, "y"), (y32g, "fp32 y"), (lambda: check_scratch(sg, dims, False, what), "")])
    assert torch.equal(yh, y.cpu())


@pytest.mark.parametrize("w", RAGGED + [RAGGED_DH128[1], RAGGED_DH128[3]], ids=lambda w: w.name)
def test_backward_writes_stay_inside_their_regions(w):
    dims = pb.make_dims(w)
    x, params = inputs.make_layer(w, 0, device="cuda", biases=True)
    ws, block = new_block(dims, params)
    sg = Guarded(pb.train_scratch_bytes(dims))
    yg, y = guarded_tensor((w.tokens, w.hidden), torch.bfloat16)
    block.forward_train(x, sg.t, y=y)
    dy = (torch.randn(w.tokens, w.hidden, device="cuda") * 0.1).to(torch.bfloat16)
    H, F, T = w.hidden, w.ffn, w.tokens
    shapes = {"dx": (T, H), "dgamma": (H,), "dbeta": (H,), "dwqkv": (H, 3 * H), "dw1": (H, F),
              "dwo": (H, H), "dw2": (F, H), "db_qkv": (3 * H,), "db1": (F,), "db_o": (H,),
              "db2": (H,)}
    guards, grads = [], {}
    for n, shp in shapes.items():
        g, t = guarded_tensor(shp, torch.bfloat16 if n == "dx" else torch.float32)
        t.zero_()
        guards.append((g, n))
        grads[n] = t
    block.backward(x, dy, sg.t, grads=grads)
    what = f"{w.name} forward_train + backward"
    finish(what, [block], [(ws, "workspace"), (yg, "y")] + guards +
           [(lambda: check_scratch(sg, dims, True, what), "")])
    assert torch.isfinite(grads["dx"].float()).all()


# 2048 x 12288 x 1024: 384 tiles on 76 pairs, the last waves split along K; 4160 x 2080 x
# 12288: units of two M tiles (long K), a ragged last unit and column block, the leftover
# units split into their tiles
@pytest.mark.parametrize("M,N,K", [(2048, 12288, 1024), (4160, 2080, 12288)])
def test_stream_k_gemm_stays_inside_its_scratch(M, N, K):
    g = torch.Generator(device="cuda").manual_seed(5)
    a = torch.randn(M, K, generator=g, device="cuda").to(torch.bfloat16)
    b = torch.randn(N, K, generator=g, device="cuda").to(torch.bfloat16)
    sg = Guarded(pb.gemm_scratch_bytes())
    sg.t.zero_()
    cg, c = guarded_tensor((M, N), torch.bfloat16)
    status = torch.zeros(1, dtype=torch.int32, device="cuda")
    pb.gemm(a, b, out=c, scratch=sg.t, status=status)
    torch.cuda.synchronize()
    assert int(status.item()) == 0
    bad = sg.check_edges("stream-K scratch") + cg.check_edges("gemm output")
    assert not bad, "\n".join(bad)
