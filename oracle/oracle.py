"""fp64 CPU oracle for the parallel transformer block, forward and backward.

TEST INFRASTRUCTURE ONLY: imported by tests/, ``__graft_entry__.smoke()`` and the CPU
baseline leg of ``bench.py``; never by the product package. It shares no code with the
CUDA path (it does not import ``transformer_block_gb300``).

What it computes (MegaScale reading notes, section 1.1, eq. (4)):

    y = x + MLP(LN(x)) + Attention(LN(x))

step by step, in the pages' order, with the ORIGINAL separate weights:

1. ``xn = LN(x)`` -- LayerNorm with gamma/beta, one LN shared by both branches (eq. (4)).
2. ``q = xn Wq``, ``k = xn Wk``, ``v = xn Wv`` (columns [Q | K | V] of Wqkv, the
   ``[b, s, 3h]`` projection of the Megatron-LM notes, section 2.2) and ``h = xn W1``
   (section 2.1, ``Y = GeLU(XA)B``), four separate matmuls, optional biases.
3. Per sequence, head and query: explicit masked softmax over the most recent ``w``
   tokens, self included (section 1.1, eqs. (5)-(6)), scale ``1/sqrt(dh)``.
4. ``attn = concat_heads(o) Wo``, ``mlp = GeLU(h) W2``.
5. ``y = x + mlp + attn``.

Two further block forms, on the same primitives:
* ``Dims(variant=1)``: RMSNorm and a SwiGLU MLP (the fused "RMSNorm" and "SiLU +
  elementwise multiply" kernels of section 1.3, which the pages name without defining;
  the standard forms are taken: ``x / sqrt(mean x^2 + eps) * gamma`` and
  ``silu(x W_gate) * (x W_up)``, ``w1 = [W_gate | W_up]``).
* ``serial_block_forward``: the standard block of eq. (3), for comparison.
* ``block_backward``: the gradients of eq. (4) for an upstream ``dy`` (training; the
  performance notes count the backward as 4 of the 6 FLOPs per weight and token), by the
  chain rule through the steps above in reverse, with the attention probabilities
  recomputed from q and k (the pages' selective recomputation). Its primitives
  (``oracle_norm_backward``, ``oracle_gelu_backward``, ``oracle_swiglu_backward``,
  ``oracle_swa_attention_backward``) are the derivatives of the forward ones.
* ``block_forward(fp8=True)``: both GEMMs on FP8 E4M3 operands with per-row current
  scaling (the performance notes' FP8 recipe), the quantizer's fp32 steps in
  ``oracle_quantize_e4m3_rows`` (E4M3 rounding written from the format definition).

All arithmetic is float64 in oracle.cpp (built here with g++); inputs are the exact
bf16 values the GPU receives, passed as float32/float64 arrays.

Row sampling (``rows=``): output row ``i`` of sequence ``b`` depends only on rows
``max(0, i-w+1) .. i`` of the same sequence (the window), so the oracle can compute a
chosen set of output rows exactly from that cone. ``stack_forward(prefix=P)`` uses
causality the same way: the first ``P`` rows of every layer depend only on the first
``P`` input rows.
"""

from __future__ import annotations

import ctypes
import os
import subprocess
from dataclasses import dataclass

import numpy as np

_HERE = os.path.dirname(os.path.abspath(__file__))
_SRC = os.path.join(_HERE, "oracle.cpp")
_BUILD = os.path.join(_HERE, "_build")
_LIB_PATH = os.path.join(_BUILD, "liboracle.so")

_lib = None


def build(force: bool = False, src: str = _SRC, out: str = _LIB_PATH) -> str:
    """Compile oracle.cpp into a shared library with g++ (no GPU, no CUDA)."""
    if not force and os.path.exists(out) and os.path.getmtime(out) >= os.path.getmtime(src):
        return out
    os.makedirs(os.path.dirname(out), exist_ok=True)
    tmp = out + f".tmp{os.getpid()}"
    cmd = ["g++", "-O2", "-std=c++17", "-shared", "-fPIC", "-pthread", src, "-o", tmp]
    subprocess.run(cmd, check=True)
    os.replace(tmp, out)
    return out


def _bind(lib):
    d, i64, i32 = ctypes.c_void_p, ctypes.c_int64, ctypes.c_int
    lib.oracle_threads.argtypes = [i32]
    lib.oracle_threads.restype = i32
    lib.oracle_layernorm.argtypes = [i64, i64, d, d, d, ctypes.c_double, d, i32]
    lib.oracle_linear.argtypes = [i64, i64, i64, d, i64, d, i64, d, d, i64, i32]
    lib.oracle_gelu.argtypes = [i64, d, d, i32]
    lib.oracle_swa_attention.argtypes = [i64, d, d, i64, d, d, d, i64, i64, i64, d, i32]
    lib.oracle_add3.argtypes = [i64, d, d, d, d]
    lib.oracle_rmsnorm.argtypes = [i64, i64, d, d, ctypes.c_double, d, i32]
    lib.oracle_swiglu.argtypes = [i64, d, d, d, i32]
    lib.oracle_quantize_e4m3_rows.argtypes = [i64, i64, d, d, d, d, i32]
    lib.oracle_norm_backward.argtypes = [i64, i64, d, d, d, ctypes.c_double, i32, d, d, d, i32]
    lib.oracle_gelu_backward.argtypes = [i64, d, d, d, i32]
    lib.oracle_swiglu_backward.argtypes = [i64, d, d, d, d, d, i32]
    lib.oracle_swa_attention_backward.argtypes = [i64, d, d, d, d, i64, i64, i64, d, d, d, i32]
    for f in ("oracle_layernorm", "oracle_linear", "oracle_gelu", "oracle_swa_attention",
              "oracle_add3", "oracle_rmsnorm", "oracle_swiglu", "oracle_quantize_e4m3_rows",
              "oracle_norm_backward", "oracle_gelu_backward", "oracle_swiglu_backward",
              "oracle_swa_attention_backward"):
        getattr(lib, f).restype = None
    return lib


def load(path: str | None = None):
    """Load (building first if needed) the oracle library; ``path`` loads another build."""
    global _lib
    if path is not None:
        return _bind(ctypes.CDLL(path))
    if _lib is None:
        _lib = _bind(ctypes.CDLL(build()))
    return _lib


def _f64(a) -> np.ndarray:
    return np.ascontiguousarray(a, dtype=np.float64)


def _ptr(a: np.ndarray):
    return ctypes.c_void_p(a.ctypes.data)


@dataclass(frozen=True)
class Dims:
    batch: int
    seq: int
    hidden: int
    heads: int
    head_dim: int
    ffn: int
    window: int
    ln_eps: float = 1e-5
    # 0: LayerNorm + GeLU MLP (eq. (4) as written); 1: RMSNorm + SwiGLU MLP (the fused
    # kernels of section 1.3), w1 = [W_gate | W_up] of [H, 2F].
    variant: int = 0


# ----------------------------------------------------------------------------- primitives


def threads_used(threads: int = 0, lib=None) -> int:
    return (lib or load()).oracle_threads(threads)


def layernorm(x, gamma, beta, eps, threads=0, lib=None) -> np.ndarray:
    lib = lib or load()
    x, g, b = _f64(x), _f64(gamma), _f64(beta)
    rows, H = x.shape
    out = np.empty_like(x)
    lib.oracle_layernorm(rows, H, _ptr(x), _ptr(g), _ptr(b), float(eps), _ptr(out), threads)
    return out


def rmsnorm(x, gamma, eps, threads=0, lib=None) -> np.ndarray:
    lib = lib or load()
    x, g = _f64(x), _f64(gamma)
    rows, H = x.shape
    out = np.empty_like(x)
    lib.oracle_rmsnorm(rows, H, _ptr(x), _ptr(g), float(eps), _ptr(out), threads)
    return out


def swiglu(gate, up, threads=0, lib=None) -> np.ndarray:
    lib = lib or load()
    gate, up = _f64(gate), _f64(up)
    assert gate.shape == up.shape
    out = np.empty_like(gate)
    lib.oracle_swiglu(gate.size, _ptr(gate), _ptr(up), _ptr(out), threads)
    return out


def quantize_e4m3_rows(x, threads=0, lib=None):
    """Per-row current scaling to FP8 E4M3 with the quantizer's fp32 steps (oracle.cpp):
    returns ``(codes uint8 [rows, cols], scales float32 [rows], dequantized float64)``."""
    lib = lib or load()
    x = _f64(x)
    rows, cols = x.shape
    codes = np.empty((rows, cols), dtype=np.uint8)
    scales = np.empty(rows, dtype=np.float32)
    deq = np.empty_like(x)
    lib.oracle_quantize_e4m3_rows(rows, cols, _ptr(x), codes.ctypes.data_as(ctypes.c_void_p),
                                  scales.ctypes.data_as(ctypes.c_void_p), _ptr(deq), threads)
    return codes, scales, deq


def round_bf16(x) -> np.ndarray:
    """Round to bf16 (nearest even) and back: the storage of a 16-bit intermediate."""
    import torch
    return torch.from_numpy(_f64(x)).to(torch.bfloat16).to(torch.float64).numpy()


def _norm(dims, x, gamma, beta, threads, lib):
    """The block's normalisation: LayerNorm (variant 0) or RMSNorm (variant 1, no beta)."""
    if dims.variant == 1:
        return rmsnorm(x, gamma, dims.ln_eps, threads, lib)
    return layernorm(x, gamma, beta, dims.ln_eps, threads, lib)


def _mlp_act(dims, h, threads, lib):
    """GeLU(h) (variant 0), or SwiGLU over h = [gate | up] (variant 1)."""
    if dims.variant == 1:
        F = dims.ffn
        return swiglu(h[:, :F], h[:, F:], threads, lib)
    return gelu(h, threads, lib)


def linear(a, w, bias=None, threads=0, lib=None) -> np.ndarray:
    """``a [M, K] @ w [K, N] (+ bias [N])`` in float64."""
    lib = lib or load()
    a, w = _f64(a), _f64(w)
    M, K = a.shape
    K2, N = w.shape
    assert K == K2, (a.shape, w.shape)
    b = None if bias is None else _f64(bias)
    out = np.empty((M, N), dtype=np.float64)
    lib.oracle_linear(M, K, N, _ptr(a), K, _ptr(w), N, None if b is None else _ptr(b),
                      _ptr(out), N, threads)
    return out


def gelu(z, threads=0, lib=None) -> np.ndarray:
    lib = lib or load()
    z = _f64(z)
    out = np.empty_like(z)
    lib.oracle_gelu(z.size, _ptr(z), _ptr(out), threads)
    return out


def swa_attention(q, q_pos, k, v, k_pos, heads, head_dim, window, threads=0, lib=None):
    """Sliding-window causal attention of one sequence; positions index the sequence."""
    lib = lib or load()
    q, k, v = _f64(q), _f64(k), _f64(v)
    qp = np.ascontiguousarray(q_pos, dtype=np.int64)
    kp = np.ascontiguousarray(k_pos, dtype=np.int64)
    out = np.empty_like(q)
    lib.oracle_swa_attention(q.shape[0], _ptr(qp), _ptr(q), k.shape[0], _ptr(kp), _ptr(k),
                             _ptr(v), heads, head_dim, window, _ptr(out), threads)
    return out


def norm_backward(x, gamma, dout, eps, rms=False, threads=0, lib=None):
    """LayerNorm (or RMSNorm) backward: returns ``(dx, dgamma, dbeta)`` (dbeta None for
    RMSNorm)."""
    lib = lib or load()
    x, g, do = _f64(x), _f64(gamma), _f64(dout)
    rows, H = x.shape
    dx, dg = np.empty_like(x), np.empty(H)
    db = None if rms else np.empty(H)
    lib.oracle_norm_backward(rows, H, _ptr(x), _ptr(g), _ptr(do), float(eps), int(rms),
                             _ptr(dx), _ptr(dg), None if db is None else _ptr(db), threads)
    return dx, dg, db


def gelu_backward(z, dout, threads=0, lib=None) -> np.ndarray:
    lib = lib or load()
    z, do = _f64(z), _f64(dout)
    out = np.empty_like(z)
    lib.oracle_gelu_backward(z.size, _ptr(z), _ptr(do), _ptr(out), threads)
    return out


def swiglu_backward(gate, up, dout, threads=0, lib=None):
    """Returns ``(dgate, dup)`` for ``out = silu(gate) * up``."""
    lib = lib or load()
    gate, up, do = _f64(gate), _f64(up), _f64(dout)
    dg, du = np.empty_like(gate), np.empty_like(up)
    lib.oracle_swiglu_backward(gate.size, _ptr(gate), _ptr(up), _ptr(do), _ptr(dg), _ptr(du),
                               threads)
    return dg, du


def swa_attention_backward(q, k, v, dout, heads, head_dim, window, threads=0, lib=None):
    """Backward of the sliding-window attention of one whole sequence: ``(dq, dk, dv)``."""
    lib = lib or load()
    q, k, v, do = _f64(q), _f64(k), _f64(v), _f64(dout)
    dq, dk, dv = np.empty_like(q), np.empty_like(k), np.empty_like(v)
    lib.oracle_swa_attention_backward(q.shape[0], _ptr(q), _ptr(k), _ptr(v), _ptr(do), heads,
                                      head_dim, window, _ptr(dq), _ptr(dk), _ptr(dv), threads)
    return dq, dk, dv


# ----------------------------------------------------------------------------- the block


def _param(params, name):
    t = params.get(name)
    return None if t is None else _f64(t)


def block_forward(dims: Dims, x, params: dict, rows: dict | None = None, threads: int = 0,
                  keep_stages: bool = False, lib=None, fp8: bool = False):
    """One parallel transformer block (eq. (4)) in float64.

    ``x``: ``[B, S, H]``; ``params``: ``ln_gamma, ln_beta [H]``, ``wqkv [H, 3H]``,
    ``w1 [H, F]``, ``wo [H, H]``, ``w2 [F, H]`` (all ``Y = X W``, ``[in, out]``) and
    optional ``b_qkv [3H]``, ``b1 [F]``, ``b_o [H]``, ``b2 [H]``. With ``dims.variant == 1``
    the normalisation is RMSNorm (``ln_beta`` unused) and the MLP is SwiGLU:
    ``w1 = [W_gate | W_up]`` is ``[H, 2F]``, ``b1`` is ``[2F]``, and the MLP's activation is
    ``silu(gate) * up`` (the fused kernels of section 1.3).

    ``rows=None`` returns ``y [B, S, H]``. ``rows={b: positions}`` returns only those
    output rows, ``[sum_b len(positions), H]``, ordered by ``b`` then position.
    ``keep_stages=True`` also returns the intermediates of step 1-4 for the same rows.

    ``fp8=True``: both GEMMs take FP8 E4M3 operands with per-row current scaling (the
    performance notes' FP8 recipe, "BF16 / FP16 / FP8": E4M3 for the forward pass, only the
    GEMMs in FP8). The operands are quantized where the fused path quantizes them and from
    the precision it holds them in: LN(x) rows (the quantizer casts to fp32), the output
    channels of [Wqkv | W1] and of [Wo ; W2] (bf16 weights), and the rows of
    [attn | GeLU(h)] after rounding to bf16 (how that intermediate is stored). Everything
    else stays float64.
    """
    lib = lib or load()
    B, S, H = dims.batch, dims.seq, dims.hidden
    nh, dh, F, w = dims.heads, dims.head_dim, dims.ffn, dims.window
    assert nh * dh == H
    x = np.asarray(x).reshape(B, S, H)

    # Which query rows are wanted, and which rows their windows reach (the cone).
    want, cone = {}, {}
    for b in range(B):
        if rows is None:
            pos = np.arange(S, dtype=np.int64)
            need = pos
        else:
            pos = np.unique(np.asarray(rows.get(b, []), dtype=np.int64))
            if pos.size == 0:
                continue
            assert pos.min() >= 0 and pos.max() < S
            mask = np.zeros(S, dtype=bool)
            for i in pos:
                mask[max(0, i - w + 1): i + 1] = True
            need = np.nonzero(mask)[0].astype(np.int64)
        want[b], cone[b] = pos, need

    gamma, beta = _param(params, "ln_gamma"), _param(params, "ln_beta")
    wqkv = params["wqkv"]
    bqkv = _param(params, "b_qkv")
    bq, bk, bv = (None, None, None) if bqkv is None else (bqkv[:H], bqkv[H:2 * H], bqkv[2 * H:])

    cone_x = np.concatenate([x[b][cone[b]] for b in want]) if want else np.zeros((0, H))
    # 1. one LayerNorm, shared by both branches
    xn_cone = _norm(dims, cone_x, gamma, beta, threads, lib)
    # rows of the cone that are wanted queries
    sel, off = [], 0
    for b in want:
        sel.append(off + np.searchsorted(cone[b], want[b]))
        off += cone[b].size
    sel = np.concatenate(sel) if sel else np.zeros(0, dtype=np.int64)
    xn_q = xn_cone[sel]

    w1 = params["w1"]
    if fp8:
        # one scale per output channel of [Wqkv | W1] and per row of LN(x)
        w1cat = np.concatenate([_f64(wqkv), _f64(w1)], axis=1)
        w1cat = quantize_e4m3_rows(w1cat.T, threads, lib)[2].T
        wqkv, w1 = w1cat[:, :3 * H], w1cat[:, 3 * H:]
        xn_cone = quantize_e4m3_rows(xn_cone, threads, lib)[2]
        xn_q = xn_cone[sel]

    # 2. four separate projections
    q = linear(xn_q, wqkv[:, 0:H], bq, threads, lib)
    k = linear(xn_cone, wqkv[:, H:2 * H], bk, threads, lib)
    v = linear(xn_cone, wqkv[:, 2 * H:3 * H], bv, threads, lib)
    h = linear(xn_q, w1, _param(params, "b1"), threads, lib)

    # 3. sliding-window attention, per sequence
    attn = np.empty_like(q)
    qoff, koff = 0, 0
    for b in want:
        nq, nk = want[b].size, cone[b].size
        attn[qoff:qoff + nq] = swa_attention(q[qoff:qoff + nq], want[b], k[koff:koff + nk],
                                             v[koff:koff + nk], cone[b], nh, dh, w, threads, lib)
        qoff += nq
        koff += nk

    # 4. the two output projections
    g = _mlp_act(dims, h, threads, lib)
    wo, w2 = params["wo"], params["w2"]
    if fp8:
        # one scale per row of [attn | act(h)] (stored as bf16) and per output channel of
        # [Wo ; W2]
        act = quantize_e4m3_rows(round_bf16(np.concatenate([attn, g], axis=1)), threads, lib)[2]
        attn_in, g_in = act[:, :H], act[:, H:]
        w2cat = quantize_e4m3_rows(np.concatenate([_f64(wo), _f64(w2)], axis=0).T, threads,
                                   lib)[2].T
        wo, w2 = w2cat[:H], w2cat[H:]
    else:
        attn_in, g_in = attn, g
    mlp = linear(g_in, w2, _param(params, "b2"), threads, lib)
    att = linear(attn_in, wo, _param(params, "b_o"), threads, lib)

    # 5. residual sum of the three terms of eq. (4)
    xq = _f64(np.concatenate([x[b][want[b]] for b in want]) if want else np.zeros((0, H)))
    y = np.empty_like(xq)
    lib.oracle_add3(y.size, _ptr(xq), _ptr(mlp), _ptr(att), _ptr(y))
    if rows is None:
        y = y.reshape(B, S, H)
    if not keep_stages:
        return y
    stages = {"xn": xn_q, "q": q, "k": k[sel], "v": v[sel], "h": h, "gelu_h": g, "mlp_act": g,
              "attn": attn, "mlp": mlp, "att_proj": att}
    return y, stages


def serial_block_forward(dims: Dims, x, params: dict, rows: dict | None = None,
                         threads: int = 0, lib=None):
    """The standard (serial) transformer block of eq. (3), in float64, on the same weights:

        h = x + Attn(LN(x)),   y = h + MLP(LN'(h))

    (MegaScale reading notes, section 1.1, "Parallel Transformer Block", eq. (3)). The
    printed eq. (3) leaves the attention term out of the outer sum; the derivation under it
    (the parallel block replaces the MLP input LN(x + h2) by LN(x), h2 = Attention(LN(x)))
    only holds with the attention output in the residual stream, as in eq. (4), so it is
    kept here. LN' uses ``ln2_gamma``/``ln2_beta`` when given, else the block's one
    LayerNorm (eq. (3) writes the same LN twice). ``Attn(LN(x)) = softmax(..) V Wo + b_o``
    is the attention term of eq. (4), taken from ``block_forward``; the MLP is
    ``GeLU(LN'(h) W1 + b1) W2 + b2``. ``rows`` as in ``block_forward``.
    """
    lib = lib or load()
    B, S, H = dims.batch, dims.seq, dims.hidden
    x = np.asarray(x).reshape(B, S, H)
    _, st = block_forward(dims, x, params, rows=rows, threads=threads, keep_stages=True,
                          lib=lib)
    if rows is None:
        xq = _f64(x.reshape(B * S, H))
    else:
        parts = []
        for b in range(B):
            pos = np.unique(np.asarray(rows.get(b, []), dtype=np.int64))
            if pos.size:
                parts.append(x[b][pos])
        xq = _f64(np.concatenate(parts)) if parts else np.zeros((0, H))
    h = xq + st["att_proj"]
    g2 = _param(params, "ln2_gamma")
    b2n = _param(params, "ln2_beta")
    if g2 is None:
        g2, b2n = _param(params, "ln_gamma"), _param(params, "ln_beta")
    hn = _norm(dims, h, g2, b2n, threads, lib)
    m = linear(_mlp_act(dims, linear(hn, params["w1"], _param(params, "b1"), threads, lib),
                        threads, lib),
               params["w2"], _param(params, "b2"), threads, lib)
    y = h + m
    return y.reshape(B, S, H) if rows is None else y


def stack_forward(dims: Dims, x, layers: list, prefix: int | None = None, threads: int = 0,
                  lib=None):
    """``len(layers)`` blocks applied in turn, ``x_{l+1} = block_l(x_l)`` (float64 between
    layers). ``prefix=P`` computes only the first ``P`` rows of every sequence, which by
    causality equal the first ``P`` rows of the full computation."""
    lib = lib or load()
    x = _f64(np.asarray(x).reshape(dims.batch, dims.seq, dims.hidden))
    if prefix is not None:
        x = np.ascontiguousarray(x[:, :prefix])
        dims = Dims(dims.batch, prefix, dims.hidden, dims.heads, dims.head_dim, dims.ffn,
                    dims.window, dims.ln_eps)
    for p in layers:
        x = block_forward(dims, x, p, threads=threads, lib=lib)
    return x


# ----------------------------------------------------------------------------- backward


def block_backward(dims: Dims, x, params: dict, dy, threads: int = 0, lib=None,
                   keep_stages: bool = False):
    """Gradients of the parallel block (eq. (4)) for an upstream gradient ``dy [B, S, H]``,
    in float64, by the chain rule through the forward's steps in reverse:

    1. ``y = x + attn Wo + b_o + act(h) W2 + b2``: ``d_attn = dy Wo^T``, ``d_act = dy W2^T``,
       ``dWo = attn^T dy``, ``dW2 = act^T dy``, ``db_o = db2 = sum_t dy``.
    2. the MLP activation: ``dh = d_act * gelu'(h)`` (SwiGLU: the gate and up parts).
    3. the attention, per sequence: ``(dq, dk, dv)`` from its definition (the probabilities
       are recomputed from q and k, as the pages' selective recomputation does).
    4. ``[q | k | v | h] = xn [Wqkv | W1] + b``: ``dxn = dq Wq^T + dk Wk^T + dv Wv^T + dh W1^T``,
       ``dWqkv = xn^T [dq | dk | dv]``, ``dW1 = xn^T dh``, biases the column sums.
    5. the shared normalisation: ``dx = dy + LN'(x)^T dxn`` (both branches and the residual
       meet here), ``dgamma``, ``dbeta``.

    Returns a dict with ``dx [B, S, H]`` and one entry per parameter of ``params`` (the
    same names and shapes; ``ln_beta`` is None for RMSNorm). ``keep_stages=True`` also
    returns ``d_attn, d_act, dh, dq, dk, dv, dxn`` ([T, .] each).
    """
    lib = lib or load()
    B, S, H = dims.batch, dims.seq, dims.hidden
    nh, dh_, F, w = dims.heads, dims.head_dim, dims.ffn, dims.window
    T = B * S
    X = _f64(np.asarray(x).reshape(T, H))
    dY = _f64(np.asarray(dy).reshape(T, H))
    gamma, beta = _param(params, "ln_gamma"), _param(params, "ln_beta")
    wqkv, w1 = _f64(params["wqkv"]), _f64(params["w1"])
    wo, w2 = _f64(params["wo"]), _f64(params["w2"])
    bqkv, b1 = _param(params, "b_qkv"), _param(params, "b1")
    glu = dims.variant == 1

    # forward, keeping what the backward reads
    xn = _norm(dims, X, gamma, beta, threads, lib)
    qkv = linear(xn, wqkv, bqkv, threads, lib)
    q, k, v = qkv[:, :H], qkv[:, H:2 * H], qkv[:, 2 * H:]
    h = linear(xn, w1, b1, threads, lib)
    pos = np.arange(S, dtype=np.int64)
    attn = np.concatenate([swa_attention(q[b * S:(b + 1) * S], pos, k[b * S:(b + 1) * S],
                                         v[b * S:(b + 1) * S], pos, nh, dh_, w, threads, lib)
                           for b in range(B)])
    act = _mlp_act(dims, h, threads, lib)

    # 1. the two output projections and the residual
    d_attn = linear(dY, wo.T, None, threads, lib)
    d_act = linear(dY, w2.T, None, threads, lib)
    g = {"wo": linear(attn.T, dY, None, threads, lib), "w2": linear(act.T, dY, None, threads, lib)}
    if params.get("b_o") is not None:
        g["b_o"] = dY.sum(axis=0)
    if params.get("b2") is not None:
        g["b2"] = dY.sum(axis=0)
    # 2. the MLP activation
    if glu:
        dgate, dup = swiglu_backward(h[:, :F], h[:, F:], d_act, threads, lib)
        dh = np.concatenate([dgate, dup], axis=1)
    else:
        dh = gelu_backward(h, d_act, threads, lib)
    # 3. the attention, per sequence
    dq, dk, dv = (np.empty((T, H)) for _ in range(3))
    for b in range(B):
        r = slice(b * S, (b + 1) * S)
        dq[r], dk[r], dv[r] = swa_attention_backward(q[r], k[r], v[r], d_attn[r], nh, dh_, w,
                                                     threads, lib)
    dqkv = np.concatenate([dq, dk, dv], axis=1)
    # 4. the input projections
    g["wqkv"] = linear(xn.T, dqkv, None, threads, lib)
    g["w1"] = linear(xn.T, dh, None, threads, lib)
    if bqkv is not None:
        g["b_qkv"] = dqkv.sum(axis=0)
    if b1 is not None:
        g["b1"] = dh.sum(axis=0)
    dxn = linear(dqkv, wqkv.T, None, threads, lib) + linear(dh, w1.T, None, threads, lib)
    # 5. the shared normalisation and the residual
    dx_norm, g["ln_gamma"], dbeta = norm_backward(X, gamma, dxn, dims.ln_eps, glu, threads, lib)
    g["ln_beta"] = None if glu else dbeta
    g["dx"] = (dY + dx_norm).reshape(B, S, H)
    if keep_stages:
        g["stages"] = {"d_attn": d_attn, "d_act": d_act, "dh": dh, "dq": dq, "dk": dk, "dv": dv,
                       "dxn": dxn}
    return g
