"""Pins of the fp64 oracle against facts that do not come from the oracle itself.

Each ``pin_*`` takes a loaded oracle library and returns ``(ok, detail)``; the test
suite asserts every pin holds for the real oracle and that each planted mistake (a
mutated copy of oracle.cpp, see test_oracle_mutants.py) breaks at least one pin.

What pins what:
* closed forms: GeLU at standard-normal-table points, LayerNorm of a 2-vector,
  two-key softmax (window 2) as a logistic weight, window 1 returning V exactly;
* library routines in float64: ``numpy`` matmul, ``torch.nn.functional.layer_norm``,
  ``F.gelu``, ``F.scaled_dot_product_attention`` (causal, and with an explicit band
  mask), and a full block restated with them;
* identities of the method: window >= seq is full causal attention; the concatenated
  weight form ``x + [attn | GeLU(h)] [Wo ; W2]`` equals the two-branch sum;
* invariants: LayerNorm statistics, value rows all equal give that value, head
  permutation, translation of a window, per-row shift of x, batch independence;
* RMSNorm + SwiGLU (the fused kernels of section 1.3): closed forms (constant rows,
  sigmoid(ln 3) = 3/4), torch ``rms_norm`` / ``silu``, RMSNorm's scale invariance, and
  the variant block restated with torch routines;
* FP8 E4M3 with per-row current scaling: the code table of the format definition, a
  round trip of every code through an independent decoder, ties to even, torch's
  ``float8_e4m3fn`` casts, the per-row scale invariants, and the FP8 block restated with
  torch;
* the serial block of eq. (3): restated with torch routines, equal to the parallel
  block when either branch's output weight is zero, and first-order in the attention
  term when compared with the parallel block;
* the backward pass: central finite differences of the pinned forward at random entries
  of x and of every parameter (both block variants), torch autograd through the torch
  restatements, closed forms of gelu' and silu' (normal table, sigmoid(ln 3) = 3/4), the
  normalisation's invariants (dx orthogonal to ones and to xhat) and softmax's (each
  head's key gradients sum to zero; window 1 passes dout to dv and nothing to q, k).
"""

from __future__ import annotations

import math

import numpy as np
import torch
import torch.nn.functional as F

from oracle import oracle as O

# Standard normal CDF at a few points, from any printed normal table (textbook values).
NORMAL_TABLE = {0.0: 0.5, 0.5: 0.6914624612740131, 1.0: 0.8413447460685429,
                1.96: 0.9750021048517795, 2.0: 0.9772498680518208,
                -1.0: 0.15865525393145707, -2.0: 0.022750131948179195}


def _rng(seed):
    return np.random.default_rng(seed)


def _close(a, b, tol):
    a, b = np.asarray(a, dtype=np.float64), np.asarray(b, dtype=np.float64)
    err = float(np.max(np.abs(a - b))) if a.size else 0.0
    return err <= tol, f"max|diff|={err:.3e} (tol {tol:g})"


# ----------------------------------------------------------------------------- GeLU


def pin_gelu_table(lib):
    z = np.array(list(NORMAL_TABLE.keys()))
    want = z * np.array(list(NORMAL_TABLE.values()))
    return _close(O.gelu(z, lib=lib), want, 1e-15)


def pin_gelu_library(lib):
    z = _rng(1).normal(0, 3, 1000)
    want = F.gelu(torch.from_numpy(z), approximate="none").numpy()
    return _close(O.gelu(z, lib=lib), want, 1e-14)


# ----------------------------------------------------------------------------- LayerNorm


def pin_layernorm_two_vector(lib):
    # x = [1, 3]: mean 2, variance 1 -> normalised [-1, 1] / sqrt(1 + eps)
    eps = 1e-5
    x = np.array([[1.0, 3.0]])
    g, b = np.array([2.0, 3.0]), np.array([0.5, -0.5])
    s = 1.0 / math.sqrt(1.0 + eps)
    want = np.array([[-2.0 * s + 0.5, 3.0 * s - 0.5]])
    return _close(O.layernorm(x, g, b, eps, lib=lib), want, 1e-15)


def pin_layernorm_library(lib):
    r = _rng(2)
    x = r.normal(0.3, 2.0, (37, 96))
    g, b = r.normal(1, 0.1, 96), r.normal(0, 0.1, 96)
    want = F.layer_norm(torch.from_numpy(x), (96,), torch.from_numpy(g), torch.from_numpy(b),
                        1e-5).numpy()
    return _close(O.layernorm(x, g, b, 1e-5, lib=lib), want, 1e-12)


def pin_layernorm_stats(lib):
    # Before the affine map each row has mean 0 and variance var / (var + eps).
    r = _rng(3)
    x = r.normal(1.0, 0.01, (5, 64))  # small variance so eps matters
    eps = 1e-5
    out = O.layernorm(x, np.ones(64), np.zeros(64), eps, lib=lib)
    var = x.var(axis=1)
    ok1, d1 = _close(out.mean(axis=1), 0.0, 1e-12)
    ok2, d2 = _close(out.var(axis=1), var / (var + eps), 1e-12)
    return ok1 and ok2, d1 + "; " + d2


# ----------------------------------------------------------------------------- linear


def pin_linear_library(lib):
    r = _rng(4)
    a, w, b = r.normal(size=(37, 19)), r.normal(size=(19, 1030)), r.normal(size=1030)
    return _close(O.linear(a, w, b, lib=lib), a @ w + b, 1e-12)


# ----------------------------------------------------------------------------- attention


def _qkv(seed, S, nh, dh):
    r = _rng(seed)
    return (r.normal(size=(S, nh * dh)), r.normal(size=(S, nh * dh)), r.normal(size=(S, nh * dh)))


def _attn(q, k, v, nh, dh, w, lib):
    pos = np.arange(q.shape[0])
    return O.swa_attention(q, pos, k, v, pos, nh, dh, w, lib=lib)


def _sdpa(q, k, v, nh, dh, mask=None, causal=False):
    S = q.shape[0]
    t = lambda a: torch.from_numpy(a).reshape(S, nh, dh).transpose(0, 1)
    o = F.scaled_dot_product_attention(t(q), t(k), t(v), attn_mask=mask, is_causal=causal)
    return o.transpose(0, 1).reshape(S, nh * dh).numpy()


def band_mask(S, w):
    i = torch.arange(S).unsqueeze(1)
    k = torch.arange(S).unsqueeze(0)
    return (k <= i) & (i - k < w)


def pin_attention_window1_is_v(lib):
    q, k, v = _qkv(5, 9, 2, 4)
    out = _attn(q, k, v, 2, 4, 1, lib)
    return bool(np.array_equal(out, v)), "window 1 must return v exactly"


def pin_attention_window2_closed_form(lib):
    # Two visible keys (i-1, i): o_i = v_{i-1} + sigmoid(s_i - s_{i-1}) (v_i - v_{i-1}).
    S, nh, dh = 7, 2, 4
    q, k, v = _qkv(6, S, nh, dh)
    out = _attn(q, k, v, nh, dh, 2, lib)
    want = np.empty_like(v)
    for h in range(nh):
        c = slice(h * dh, (h + 1) * dh)
        want[0, c] = v[0, c]
        for i in range(1, S):
            s_prev = q[i, c] @ k[i - 1, c] / math.sqrt(dh)
            s_self = q[i, c] @ k[i, c] / math.sqrt(dh)
            lam = 1.0 / (1.0 + math.exp(-(s_self - s_prev)))
            want[i, c] = v[i - 1, c] + lam * (v[i, c] - v[i - 1, c])
    return _close(out, want, 1e-13)


def pin_attention_full_causal(lib):
    # Identity: window >= seq is full causal attention.
    S, nh, dh = 11, 3, 8
    q, k, v = _qkv(7, S, nh, dh)
    want = _sdpa(q, k, v, nh, dh, causal=True)
    ok = True
    detail = []
    for w in (S, S + 17):
        o, d = _close(_attn(q, k, v, nh, dh, w, lib), want, 1e-13)
        ok &= o
        detail.append(f"w={w}: {d}")
    return ok, "; ".join(detail)


def pin_attention_band_library(lib):
    S, nh, dh = 23, 2, 8
    q, k, v = _qkv(8, S, nh, dh)
    ok, detail = True, []
    for w in (1, 2, 3, 5, 22):
        o, d = _close(_attn(q, k, v, nh, dh, w, lib), _sdpa(q, k, v, nh, dh, band_mask(S, w)),
                      1e-13)
        ok &= o
        detail.append(f"w={w}: {d}")
    return ok, "; ".join(detail)


def pin_attention_rows_sum_to_one(lib):
    # Softmax weights sum to 1: with every value row equal to c the output is c.
    S, nh, dh = 13, 2, 4
    q, k, _ = _qkv(9, S, nh, dh)
    c = np.linspace(-1, 2, nh * dh)
    v = np.tile(c, (S, 1))
    return _close(_attn(q, k, v, nh, dh, 4, lib), v, 1e-14)


def pin_attention_translation(lib):
    # A row i >= w-1 depends only on rows i-w+1..i: recomputing on that slice alone,
    # with shifted positions, gives the same row.
    S, nh, dh, w = 20, 2, 4, 5
    q, k, v = _qkv(10, S, nh, dh)
    full = _attn(q, k, v, nh, dh, w, lib)
    i = 15
    part = _attn(q[i - w + 1:i + 1], k[i - w + 1:i + 1], v[i - w + 1:i + 1], nh, dh, w, lib)
    return _close(part[-1], full[i], 1e-14)


# ----------------------------------------------------------------------------- the block


def tiny_params(H, nh, F_, seed, biases=True, std=0.3):
    r = _rng(seed)
    p = {"ln_gamma": 1 + 0.1 * r.normal(size=H), "ln_beta": 0.1 * r.normal(size=H),
         "wqkv": std * r.normal(size=(H, 3 * H)), "w1": std * r.normal(size=(H, F_)),
         "wo": std * r.normal(size=(H, H)), "w2": std * r.normal(size=(F_, H))}
    if biases:
        p.update(b_qkv=0.1 * r.normal(size=3 * H), b1=0.1 * r.normal(size=F_),
                 b_o=0.1 * r.normal(size=H), b2=0.1 * r.normal(size=H))
    return p


def torch_block(dims, x, p):
    """The block restated with torch float64 library routines (layer_norm, gelu, sdpa)."""
    B, S, H, nh, dh = dims.batch, dims.seq, dims.hidden, dims.heads, dims.head_dim
    T = lambda a: None if a is None else torch.from_numpy(np.asarray(a, dtype=np.float64))
    X = T(x).reshape(B, S, H)
    xn = F.layer_norm(X, (H,), T(p["ln_gamma"]), T(p["ln_beta"]), dims.ln_eps)
    qkv = xn @ T(p["wqkv"])
    if p.get("b_qkv") is not None:
        qkv = qkv + T(p["b_qkv"])
    q, k, v = (qkv[..., i * H:(i + 1) * H].reshape(B, S, nh, dh).transpose(1, 2) for i in range(3))
    a = F.scaled_dot_product_attention(q, k, v, attn_mask=band_mask(S, dims.window))
    a = a.transpose(1, 2).reshape(B, S, H) @ T(p["wo"])
    h = xn @ T(p["w1"])
    if p.get("b1") is not None:
        h = h + T(p["b1"])
    m = F.gelu(h, approximate="none") @ T(p["w2"])
    if p.get("b_o") is not None:
        a = a + T(p["b_o"])
    if p.get("b2") is not None:
        m = m + T(p["b2"])
    return (X + m + a).numpy()


def pin_block_library(lib):
    ok, detail = True, []
    for w in (1, 2, 3, 8, 13):
        dims = O.Dims(2, 8, 8, 2, 4, 16, w)
        p = tiny_params(8, 2, 16, seed=20 + w)
        x = _rng(30 + w).normal(size=(2, 8, 8))
        o, d = _close(O.block_forward(dims, x, p, lib=lib), torch_block(dims, x, p), 1e-12)
        ok &= o
        detail.append(f"w={w}: {d}")
    return ok, "; ".join(detail)


def pin_block_concat_identity(lib):
    # y = x + [attn | GeLU(h)] [Wo ; W2] with [q|k|v|h] = xn [Wqkv | W1] (one GEMM each).
    dims = O.Dims(2, 9, 16, 4, 4, 32, 3)
    H = 16
    p = tiny_params(H, 4, 32, seed=40)
    x = _rng(41).normal(size=(2, 9, H))
    y = O.block_forward(dims, x, p, lib=lib)
    w1cat = np.concatenate([p["wqkv"], p["w1"]], axis=1)
    w2cat = np.concatenate([p["wo"], p["w2"]], axis=0)
    b1cat = np.concatenate([p["b_qkv"], p["b1"]])
    X = x.reshape(-1, H)
    mu = X.mean(1, keepdims=True)
    xn = (X - mu) / np.sqrt(X.var(1, keepdims=True) + dims.ln_eps) * p["ln_gamma"] + p["ln_beta"]
    z = xn @ w1cat + b1cat
    attn = np.concatenate([_sdpa(z[b * 9:(b + 1) * 9, 0:H], z[b * 9:(b + 1) * 9, H:2 * H],
                                 z[b * 9:(b + 1) * 9, 2 * H:3 * H], 4, 4, band_mask(9, 3))
                           for b in range(2)])
    act = np.concatenate([attn, F.gelu(torch.from_numpy(z[:, 3 * H:])).numpy()], axis=1)
    y2 = X + act @ w2cat + (p["b_o"] + p["b2"])
    return _close(y.reshape(-1, H), y2, 1e-10 * np.abs(y2).max())


def pin_block_zero_affine(lib):
    # gamma = beta = 0 and no biases: LN(x) = 0 -> every branch is 0 -> y = x exactly.
    dims = O.Dims(2, 6, 8, 2, 4, 16, 3)
    p = tiny_params(8, 2, 16, seed=50, biases=False)
    p["ln_gamma"] = np.zeros(8)
    p["ln_beta"] = np.zeros(8)
    x = _rng(51).normal(size=(2, 6, 8))
    return bool(np.array_equal(O.block_forward(dims, x, p, lib=lib), x)), "y must equal x"


def pin_block_zero_output_weights(lib):
    dims = O.Dims(1, 6, 8, 2, 4, 16, 4)
    p = tiny_params(8, 2, 16, seed=52, biases=False)
    p["wo"] = np.zeros((8, 8))
    p["w2"] = np.zeros((16, 8))
    x = _rng(53).normal(size=(1, 6, 8))
    return bool(np.array_equal(O.block_forward(dims, x, p, lib=lib), x)), "y must equal x"


def pin_block_invariants(lib):
    dims = O.Dims(3, 10, 16, 4, 4, 32, 4)
    p = tiny_params(16, 4, 32, seed=60)
    x = _rng(61).normal(size=(3, 10, 16))
    y = O.block_forward(dims, x, p, lib=lib)
    out = []
    # batch independence
    one = O.Dims(1, 10, 16, 4, 4, 32, 4)
    yb = np.stack([O.block_forward(one, x[b:b + 1], p, lib=lib)[0] for b in range(3)])
    out.append(("batch", _close(yb, y, 1e-13)))
    # per-row shift of x leaves y - x unchanged (LN removes the row mean)
    c = _rng(62).normal(size=(3, 10, 1)) * 5
    ys = O.block_forward(dims, x + c, p, lib=lib)
    out.append(("shift", _close(ys - (x + c), y - x, 1e-10)))
    # permuting heads consistently in Wq, Wk, Wv (columns) and Wo (rows)
    perm = [2, 0, 3, 1]
    idx = np.concatenate([np.arange(h * 4, h * 4 + 4) for h in perm])
    pp = dict(p)
    pp["wqkv"] = np.concatenate([p["wqkv"][:, i * 16:(i + 1) * 16][:, idx] for i in range(3)], 1)
    pp["b_qkv"] = np.concatenate([p["b_qkv"][i * 16:(i + 1) * 16][idx] for i in range(3)])
    pp["wo"] = p["wo"][idx, :]
    out.append(("heads", _close(O.block_forward(dims, x, pp, lib=lib), y, 1e-12)))
    ok = all(o for _, (o, _) in out)
    return ok, "; ".join(f"{n}: {d}" for n, (_, d) in out)


def pin_block_rows_mode(lib):
    dims = O.Dims(2, 40, 16, 4, 4, 32, 7)
    p = tiny_params(16, 4, 32, seed=70)
    x = _rng(71).normal(size=(2, 40, 16))
    full = O.block_forward(dims, x, p, lib=lib)
    rows = {0: [0, 5, 39], 1: [6, 7, 20, 33]}
    part = O.block_forward(dims, x, p, rows=rows, lib=lib)
    want = np.concatenate([full[b][rows[b]] for b in (0, 1)])
    return _close(part, want, 1e-13)


# ----------------------------------------------------------------------------- serial block


def torch_serial_block(dims, x, p):
    """The serial block (h = x + Attn(LN(x)), y = h + MLP(LN'(h))) with torch float64
    library routines."""
    B, S, H, nh, dh = dims.batch, dims.seq, dims.hidden, dims.heads, dims.head_dim
    T = lambda a: None if a is None else torch.from_numpy(np.asarray(a, dtype=np.float64))
    X = T(x).reshape(B, S, H)
    xn = F.layer_norm(X, (H,), T(p["ln_gamma"]), T(p["ln_beta"]), dims.ln_eps)
    qkv = xn @ T(p["wqkv"])
    if p.get("b_qkv") is not None:
        qkv = qkv + T(p["b_qkv"])
    q, k, v = (qkv[..., i * H:(i + 1) * H].reshape(B, S, nh, dh).transpose(1, 2) for i in range(3))
    a = F.scaled_dot_product_attention(q, k, v, attn_mask=band_mask(S, dims.window))
    a = a.transpose(1, 2).reshape(B, S, H) @ T(p["wo"])
    if p.get("b_o") is not None:
        a = a + T(p["b_o"])
    h = X + a
    g2 = T(p.get("ln2_gamma", p["ln_gamma"]))
    b2 = T(p.get("ln2_beta", p["ln_beta"]))
    hn = F.layer_norm(h, (H,), g2, b2, dims.ln_eps)
    z = hn @ T(p["w1"])
    if p.get("b1") is not None:
        z = z + T(p["b1"])
    m = F.gelu(z, approximate="none") @ T(p["w2"])
    if p.get("b2") is not None:
        m = m + T(p["b2"])
    return (h + m).numpy()


def pin_serial_library(lib):
    ok, detail = True, []
    for w, second_ln in ((1, False), (3, True), (8, False), (13, True)):
        dims = O.Dims(2, 8, 8, 2, 4, 16, w)
        p = tiny_params(8, 2, 16, seed=120 + w)
        if second_ln:
            r = _rng(130 + w)
            p["ln2_gamma"] = 1 + 0.1 * r.normal(size=8)
            p["ln2_beta"] = 0.1 * r.normal(size=8)
        x = _rng(140 + w).normal(size=(2, 8, 8))
        o, d = _close(O.serial_block_forward(dims, x, p, lib=lib), torch_serial_block(dims, x, p),
                      1e-12)
        ok &= o
        detail.append(f"w={w}: {d}")
    return ok, "; ".join(detail)


def pin_serial_reduces_to_parallel(lib):
    # Without the attention output (Wo = 0, b_o absent) or without the MLP output
    # (W2 = 0, b2 absent), eq. (3) and eq. (4) are the same function.
    dims = O.Dims(2, 10, 16, 4, 4, 32, 4)
    x = _rng(151).normal(size=(2, 10, 16))
    out = []
    for name, zero in (("no attention", {"wo": np.zeros((16, 16)), "b_o": None}),
                       ("no MLP", {"w2": np.zeros((32, 16)), "b2": None})):
        p = tiny_params(16, 4, 32, seed=150)
        p.update(zero)
        out.append((name, _close(O.serial_block_forward(dims, x, p, lib=lib),
                                 O.block_forward(dims, x, p, lib=lib), 1e-12)))
    return all(o for _, (o, _) in out), "; ".join(f"{n}: {d}" for n, (_, d) in out)


def pin_serial_first_order(lib):
    # With the attention term scaled by eps, serial - parallel = J_MLP(LN) . h2 + O(eps^2):
    # nonzero, and halving eps halves it (the MLP really reads LN(x + h2)).
    dims = O.Dims(1, 12, 16, 4, 4, 32, 5)
    x = _rng(161).normal(size=(1, 12, 16))
    diffs = []
    for eps in (1e-3, 5e-4):
        p = tiny_params(16, 4, 32, seed=160, biases=False)
        p["wo"] = eps * p["wo"]
        diffs.append(np.max(np.abs(O.serial_block_forward(dims, x, p, lib=lib)
                                   - O.block_forward(dims, x, p, lib=lib))))
    ratio = diffs[0] / diffs[1] if diffs[1] > 0 else float("inf")
    return bool(diffs[1] > 0 and abs(ratio - 2.0) < 0.05), f"diffs={diffs}, ratio={ratio:.4f}"


def pin_serial_rows_mode(lib):
    dims = O.Dims(2, 30, 16, 4, 4, 32, 6)
    p = tiny_params(16, 4, 32, seed=170)
    x = _rng(171).normal(size=(2, 30, 16))
    full = O.serial_block_forward(dims, x, p, lib=lib)
    rows = {0: [0, 29], 1: [4, 5, 17]}
    part = O.serial_block_forward(dims, x, p, rows=rows, lib=lib)
    return _close(part, np.concatenate([full[b][rows[b]] for b in (0, 1)]), 1e-13)


# ----------------------------------------------------------------------------- RMSNorm + SwiGLU


def pin_rmsnorm_closed_form(lib):
    # a constant row c: rms = |c|; a 2-vector (a, b): rms = sqrt((a^2 + b^2) / 2)
    eps = 1e-5
    x = np.array([[3.0, 3.0, 3.0, 3.0], [-2.0, -2.0, -2.0, -2.0]])
    g = np.array([1.0, 2.0, -1.0, 0.5])
    want = np.sign(x) * np.abs(x) / np.sqrt(x ** 2 + eps) * g
    ok1, d1 = _close(O.rmsnorm(x, g, eps, lib=lib), want, 1e-15)
    x2 = np.array([[3.0, 4.0]])
    want2 = x2 / math.sqrt(12.5 + eps)
    ok2, d2 = _close(O.rmsnorm(x2, np.ones(2), eps, lib=lib), want2, 1e-15)
    return ok1 and ok2, f"{d1}; {d2}"


def pin_rmsnorm_library(lib):
    x = _rng(180).normal(0, 2, size=(7, 48))
    g = 1 + 0.1 * _rng(181).normal(size=48)
    want = F.rms_norm(torch.from_numpy(x), (48,), torch.from_numpy(g), 1e-5).numpy()
    return _close(O.rmsnorm(x, g, 1e-5, lib=lib), want, 1e-14)


def pin_rmsnorm_scale_invariance(lib):
    # RMSNorm(a x) = RMSNorm(x) for a > 0 (eps -> 0), and it does not remove the row mean
    x = _rng(182).normal(0.5, 1, size=(5, 32))
    g = _rng(183).normal(size=32)
    a = O.rmsnorm(x, g, 1e-30, lib=lib)
    b = O.rmsnorm(7.5 * x, g, 1e-30, lib=lib)
    ok, d = _close(a, b, 1e-13)
    shifted = O.rmsnorm(x + 3.0, g, 1e-30, lib=lib)
    return ok and float(np.max(np.abs(shifted - a))) > 1e-3, d


def pin_swiglu_closed_form(lib):
    # sigmoid(ln 3) = 3/4 and sigmoid(-ln 3) = 1/4; silu(0) = 0
    l3 = math.log(3.0)
    gate = np.array([l3, -l3, 0.0, l3])
    up = np.array([1.0, 1.0, 5.0, -2.0])
    want = np.array([0.75 * l3, -0.25 * l3, 0.0, -1.5 * l3])
    return _close(O.swiglu(gate, up, lib=lib), want, 1e-15)


def pin_swiglu_library(lib):
    gate = _rng(184).normal(0, 4, 500)
    up = _rng(185).normal(0, 1, 500)
    want = (F.silu(torch.from_numpy(gate)) * torch.from_numpy(up)).numpy()
    return _close(O.swiglu(gate, up, lib=lib), want, 1e-14)


def swiglu_params(H, nh, F_, seed, biases=True, std=0.3):
    p = tiny_params(H, nh, F_, seed, biases, std)
    r = _rng(seed + 1000)
    p["w1"] = std * r.normal(size=(H, 2 * F_))
    if biases:
        p["b1"] = 0.1 * r.normal(size=2 * F_)
    return p


def torch_block_swiglu(dims, x, p):
    """The RMSNorm + SwiGLU parallel block restated with torch float64 routines."""
    B, S, H, nh, dh, F_ = dims.batch, dims.seq, dims.hidden, dims.heads, dims.head_dim, dims.ffn
    T = lambda a: None if a is None else torch.from_numpy(np.asarray(a, dtype=np.float64))
    X = T(x).reshape(B, S, H)
    xn = F.rms_norm(X, (H,), T(p["ln_gamma"]), dims.ln_eps)
    qkv = xn @ T(p["wqkv"])
    if p.get("b_qkv") is not None:
        qkv = qkv + T(p["b_qkv"])
    q, k, v = (qkv[..., i * H:(i + 1) * H].reshape(B, S, nh, dh).transpose(1, 2) for i in range(3))
    a = F.scaled_dot_product_attention(q, k, v, attn_mask=band_mask(S, dims.window))
    a = a.transpose(1, 2).reshape(B, S, H) @ T(p["wo"])
    if p.get("b_o") is not None:
        a = a + T(p["b_o"])
    z = xn @ T(p["w1"])
    if p.get("b1") is not None:
        z = z + T(p["b1"])
    m = (F.silu(z[..., :F_]) * z[..., F_:]) @ T(p["w2"])
    if p.get("b2") is not None:
        m = m + T(p["b2"])
    return (X + m + a).numpy()


def pin_block_swiglu_library(lib):
    ok, detail = True, []
    for w in (1, 3, 13):
        dims = O.Dims(2, 8, 8, 2, 4, 16, w, variant=1)
        p = swiglu_params(8, 2, 16, seed=190 + w)
        x = _rng(200 + w).normal(size=(2, 8, 8))
        o, d = _close(O.block_forward(dims, x, p, lib=lib), torch_block_swiglu(dims, x, p), 1e-12)
        ok &= o
        detail.append(f"w={w}: {d}")
    return ok, "; ".join(detail)


def pin_block_swiglu_rows_mode(lib):
    dims = O.Dims(2, 30, 16, 4, 4, 32, 6, variant=1)
    p = swiglu_params(16, 4, 32, seed=210)
    x = _rng(211).normal(size=(2, 30, 16))
    full = O.block_forward(dims, x, p, lib=lib)
    rows = {0: [0, 29], 1: [4, 5, 17]}
    part = O.block_forward(dims, x, p, rows=rows, lib=lib)
    return _close(part, np.concatenate([full[b][rows[b]] for b in (0, 1)]), 1e-13)


# ----------------------------------------------------------------------------- FP8 E4M3


def e4m3_decode(code: int) -> float:
    """Value of an E4M3 code from the format definition (sign, 4 exponent bits with bias 7,
    3 mantissa bits; exponent field 0 is subnormal: m * 2^-9)."""
    sign = -1.0 if code & 0x80 else 1.0
    e, m = (code >> 3) & 0xF, code & 0x7
    if e == 0:
        return sign * m * 2.0 ** -9
    return sign * (1.0 + m / 8.0) * 2.0 ** (e - 7)


def _q1(values, lib):
    """Quantize values with a unit scale: each row gets 448 as its amax."""
    v = np.asarray(values, dtype=np.float64)
    x = np.stack([v, np.full_like(v, 448.0)], axis=1)
    codes, scales, deq = O.quantize_e4m3_rows(x, lib=lib)
    assert np.all(scales == 1.0)
    return codes[:, 0], deq[:, 0]


def pin_e4m3_table(lib):
    table = {448.0: 0x7E, 1.0: 0x38, 0.5: 0x30, 2.0 ** -6: 0x08, 2.0 ** -9: 0x01,
             7 * 2.0 ** -9: 0x07, 240.0: 0x77, 1.125: 0x39, -1.0: 0xB8, 0.0: 0x00, -2.0: 0xC0}
    codes, _ = _q1(list(table), lib)
    want = np.array(list(table.values()), dtype=np.uint8)
    return bool(np.array_equal(codes, want)), f"codes {codes.tolist()} want {want.tolist()}"


def pin_e4m3_roundtrip_all_codes(lib):
    codes = [c for c in range(256) if c not in (0x7F, 0xFF)]
    vals = [e4m3_decode(c) for c in codes]
    got, deq = _q1(vals, lib)
    # -0 (0x80) decodes to -0.0 and keeps its sign
    want = np.array(codes, dtype=np.uint8)
    ok = bool(np.array_equal(got, want)) and bool(np.array_equal(deq, np.array(vals)))
    return ok, f"{int(np.sum(got != want))} codes differ"


def pin_e4m3_ties_to_even(lib):
    # halfway cases: 1.0625 between 1.0 (m 0) and 1.125 (m 1) -> 1.0; 1.1875 -> 1.25 (m 2);
    # 3 * 2^-10 between 2^-9 (m 1) and 2^-8 (m 2) -> 2^-8; 27 * 2^-5 -> 0.875 (m 6)
    vals = [1.0625, 1.1875, 3 * 2.0 ** -10, 29 * 2.0 ** -5, -1.0625]
    want = [1.0, 1.25, 2.0 ** -8, 0.875, -1.0]
    _, deq = _q1(vals, lib)
    return bool(np.array_equal(deq, np.array(want))), f"{deq.tolist()} want {want}"


def pin_e4m3_library(lib):
    v = _rng(220).normal(0, 60, 4000).clip(-448, 448)
    v = np.concatenate([v, _rng(221).normal(0, 0.01, 1000)])
    codes, _ = _q1(v, lib)
    want = torch.from_numpy(v).to(torch.float32).to(torch.float8_e4m3fn).view(torch.uint8)
    want = want.numpy()
    # torch keeps the sign of a negative value that rounds to zero (0x80); so does the oracle
    return bool(np.array_equal(codes, want)), f"{int(np.sum(codes != want))} differ"


def pin_e4m3_row_scaling(lib):
    # each row's largest magnitude maps to +-448 exactly (scale amax / 448 in fp32), the
    # dequantized value is within half an E4M3 step of the input, and all-zero rows stay 0
    x = _rng(222).normal(0, 3, size=(6, 40))
    x[3] = 0.0
    codes, scales, deq = O.quantize_e4m3_rows(x, lib=lib)
    amax = np.abs(x.astype(np.float32)).max(axis=1)
    ok = bool(np.array_equal(scales, (amax / np.float32(448.0)).astype(np.float32)))
    big = np.abs(np.array([[e4m3_decode(int(c)) for c in r] for r in codes])).max(axis=1)
    ok &= bool(np.all(big[[0, 1, 2, 4, 5]] == 448.0)) and bool(np.all(codes[3] == 0))
    rel = np.abs(deq - x) / np.maximum(np.maximum(np.abs(x), 2.0 ** -6 * scales[:, None]),
                                       1e-300)
    ok &= bool(np.all(rel <= 2.0 ** -4 + 1e-6))
    return ok, f"max relative error {rel.max():.3e}"


def torch_block_fp8(dims, x, p):
    """The FP8 block restated with torch: float8_e4m3fn casts with per-row fp32 scales."""
    B, S, H, nh, dh = dims.batch, dims.seq, dims.hidden, dims.heads, dims.head_dim
    T64 = lambda a: torch.from_numpy(np.asarray(a, dtype=np.float64))

    def q(a):  # rows of a (float64 tensor) -> dequantized float64
        a32 = a.to(torch.float32)
        amax = a32.abs().amax(dim=1, keepdim=True)
        inv = torch.where(amax > 0, torch.tensor(448.0, dtype=torch.float32) / amax,
                          torch.zeros_like(amax))
        codes = (a32 * inv).to(torch.float8_e4m3fn)
        return codes.to(torch.float64) * (amax / 448.0).to(torch.float64)

    X = T64(x).reshape(B * S, H)
    xn = q(F.layer_norm(X, (H,), T64(p["ln_gamma"]), T64(p["ln_beta"]), dims.ln_eps))
    w1cat = q(torch.cat([T64(p["wqkv"]), T64(p["w1"])], dim=1).T).T
    z = xn @ w1cat
    qkv, h = z[:, :3 * H], z[:, 3 * H:]
    q4, k4, v4 = (qkv[:, i * H:(i + 1) * H].reshape(B, S, nh, dh).transpose(1, 2) for i in range(3))
    a = F.scaled_dot_product_attention(q4, k4, v4, attn_mask=band_mask(S, dims.window))
    a = a.transpose(1, 2).reshape(B * S, H)
    act = torch.cat([a, F.gelu(h, approximate="none")], dim=1)
    act = q(act.to(torch.bfloat16).to(torch.float64))
    w2cat = q(torch.cat([T64(p["wo"]), T64(p["w2"])], dim=0).T).T
    return (X + act @ w2cat).reshape(B, S, H).numpy()


def pin_block_fp8_library(lib):
    ok, detail = True, []
    for w in (2, 9):
        dims = O.Dims(2, 12, 16, 4, 4, 32, w)
        p = tiny_params(16, 4, 32, seed=230 + w, biases=False)
        x = _rng(240 + w).normal(size=(2, 12, 16))
        o, d = _close(O.block_forward(dims, x, p, lib=lib, fp8=True), torch_block_fp8(dims, x, p),
                      1e-9)
        ok &= o
        detail.append(f"w={w}: {d}")
    return ok, "; ".join(detail)


def pin_block_fp8_rows_mode(lib):
    dims = O.Dims(2, 30, 16, 4, 4, 32, 6)
    p = tiny_params(16, 4, 32, seed=250)
    x = _rng(251).normal(size=(2, 30, 16))
    full = O.block_forward(dims, x, p, lib=lib, fp8=True)
    rows = {0: [0, 29], 1: [4, 5, 17]}
    part = O.block_forward(dims, x, p, rows=rows, lib=lib, fp8=True)
    return _close(part, np.concatenate([full[b][rows[b]] for b in (0, 1)]), 1e-13)


# ----------------------------------------------------------------------------- backward
# The block's backward pass (training; performance notes "MFU": the backward is 4 of the 6
# FLOPs per weight and token). Pinned by central finite differences of the pinned forward,
# by torch autograd through the torch restatements above, by closed forms of the
# activation derivatives and by invariants of the normalisation and of softmax.

PHI_1 = 0.24197072451914337  # standard normal density at 1, from a printed normal table


def pin_gelu_backward_closed_form(lib):
    z = np.array([0.0, 1.0, -1.0])
    want = np.array([0.5, NORMAL_TABLE[1.0] + PHI_1, NORMAL_TABLE[-1.0] - PHI_1])
    return _close(O.gelu_backward(z, np.ones(3), lib=lib), want, 1e-14)


def pin_swiglu_backward_closed_form(lib):
    # sigmoid(ln 3) = 3/4: silu(ln 3) = 3 ln3 / 4, silu'(ln 3) = 3/4 (1 + ln3 / 4)
    g, u, d = np.array([math.log(3.0)]), np.array([2.0]), np.array([-1.5])
    dg, du = O.swiglu_backward(g, u, d, lib=lib)
    want_du = -1.5 * 0.75 * math.log(3.0)
    want_dg = -1.5 * 2.0 * 0.75 * (1.0 + math.log(3.0) / 4.0)
    return _close([dg[0], du[0]], [want_dg, want_du], 1e-14)


def pin_norm_backward_invariants(lib):
    # LayerNorm's output ignores a shift and a scale of its input row, so dx is orthogonal
    # to the all-ones row and to xhat; RMSNorm's only to xhat (a scale). Also against torch.
    x = _rng(300).normal(1.0, 2.0, size=(5, 24))
    gam, do = 1 + 0.2 * _rng(301).normal(size=24), _rng(302).normal(size=(5, 24))
    # (exact only without eps, which breaks the scale invariance by eps / var)
    ok, det = True, []
    for rms in (False, True):
        dx = O.norm_backward(x, gam, do, 0.0, rms, lib=lib)[0]
        mu = 0.0 if rms else x.mean(axis=1, keepdims=True)
        xhat = (x - mu) / np.sqrt(((x - mu) ** 2).mean(axis=1, keepdims=True))
        ok &= bool(np.all(np.abs((dx * xhat).sum(axis=1)) < 1e-12))
        if not rms:
            ok &= bool(np.all(np.abs(dx.sum(axis=1)) < 1e-12))
        dx, dg, db = O.norm_backward(x, gam, do, 1e-5, rms, lib=lib)
        X = torch.tensor(x, requires_grad=True)
        G = torch.tensor(gam, requires_grad=True)
        out = F.rms_norm(X, (24,), G, 1e-5) if rms else F.layer_norm(X, (24,), G, None, 1e-5)
        tx, tg = torch.autograd.grad((out * torch.tensor(do)).sum(), (X, G))
        o1, d1 = _close(dx, tx.numpy(), 1e-12)
        o2, d2 = _close(dg, tg.numpy(), 1e-12)
        ok &= o1 and o2
        if not rms:
            ok &= _close(db, do.sum(axis=0), 1e-12)[0]
        det.append(f"rms={rms}: {d1}, {d2}")
    return ok, "; ".join(det)


def pin_attention_backward_invariants(lib):
    # softmax ignores a shift of its scores, so per query sum_j ds_j = 0 and the keys'
    # gradients of one head sum to zero; window 1 attends to itself only: dq = dk = 0 and
    # dv = dout; and against torch autograd through sdpa with the band mask.
    S, nh, dh = 11, 2, 4
    q, k, v = _qkv(310, S, nh, dh)
    do = _rng(311).normal(size=(S, nh * dh))
    ok, det = True, []
    dq, dk, dv = O.swa_attention_backward(q, k, v, do, nh, dh, 1, lib=lib)
    ok &= bool(np.all(dq == 0) and np.all(dk == 0)) and _close(dv, do, 0.0)[0]
    for w in (2, 4, 11):
        dq, dk, dv = O.swa_attention_backward(q, k, v, do, nh, dh, w, lib=lib)
        ok &= bool(np.all(np.abs(dk.sum(axis=0)) < 1e-12))
        Q, K, V = (torch.tensor(a.reshape(S, nh, dh).transpose(1, 0, 2), requires_grad=True)
                   for a in (q, k, v))
        o = F.scaled_dot_product_attention(Q, K, V, attn_mask=band_mask(S, w))
        D = torch.tensor(do.reshape(S, nh, dh).transpose(1, 0, 2))
        tq, tk, tv = (t.transpose(0, 1).reshape(S, nh * dh).numpy()
                      for t in torch.autograd.grad((o * D).sum(), (Q, K, V)))
        for a, b in ((dq, tq), (dk, tk), (dv, tv)):
            o1, d1 = _close(a, b, 1e-12)
            ok &= o1
        det.append(f"w={w}: {d1}")
    return ok, "; ".join(det)


GRAD_NAMES = ["ln_gamma", "ln_beta", "wqkv", "w1", "wo", "w2", "b_qkv", "b1", "b_o", "b2"]


def _grad_names(dims, p):
    """Parameters with a gradient: RMSNorm has no beta."""
    return [n for n in GRAD_NAMES
            if p.get(n) is not None and not (dims.variant == 1 and n == "ln_beta")]


def _bwd_case(variant, seed):
    dims = O.Dims(2, 9, 8, 2, 4, 16, 4, variant=variant)
    p = (swiglu_params if variant else tiny_params)(8, 2, 16, seed=seed)
    x = _rng(seed + 1).normal(size=(2, 9, 8))
    dy = _rng(seed + 2).normal(size=(2, 9, 8))
    return dims, p, x, dy


def pin_backward_finite_differences(lib, mod=O):
    # central differences of L = sum(y * dy) through the pinned forward, at random entries
    # of x and of every parameter
    ok, det = True, []
    for variant in (0, 1):
        dims, p, x, dy = _bwd_case(variant, 320 + variant)
        g = mod.block_backward(dims, x, p, dy, lib=lib)
        L = lambda: float((O.block_forward(dims, x, p, lib=lib) * dy).sum())
        r, eps, worst = _rng(330 + variant), 1e-6, 0.0
        for name in ["x"] + _grad_names(dims, p):
            a = x if name == "x" else p[name]
            want = g["dx"] if name == "x" else g[name]
            for _ in range(3):
                idx = tuple(int(r.integers(0, n)) for n in a.shape)
                old = a[idx]
                a[idx] = old + eps
                lp = L()
                a[idx] = old - eps
                lm = L()
                a[idx] = old
                err = abs((lp - lm) / (2 * eps) - want[idx]) / max(1.0, abs(want[idx]))
                worst = max(worst, err)
        ok &= worst < 1e-6
        det.append(f"variant {variant}: worst relative {worst:.2e}")
    return ok, "; ".join(det)


def pin_backward_autograd(lib, mod=O):
    # every gradient against torch autograd through torch_block / torch_block_swiglu
    ok, det = True, []
    for variant in (0, 1):
        dims, p, x, dy = _bwd_case(variant, 340 + variant)
        g = mod.block_backward(dims, x, p, dy, lib=lib)
        names = _grad_names(dims, p)
        leaves = {n: torch.tensor(np.asarray(p[n], dtype=np.float64), requires_grad=True)
                  for n in names}
        X = torch.tensor(x, requires_grad=True)
        y = _torch_block_autograd(dims, X, leaves)
        grads = torch.autograd.grad((y * torch.tensor(dy)).sum(), [X] + [leaves[n] for n in names])
        worst = 0.0
        for n, t in zip(["dx"] + names, grads):
            a = g[n] if n != "dx" else g["dx"]
            worst = max(worst, float(np.max(np.abs(np.asarray(a) - t.numpy()))))
        ok &= worst < 1e-10
        det.append(f"variant {variant}: max|diff| {worst:.2e}")
    return ok, "; ".join(det)


def _torch_block_autograd(dims, X, p):
    """The block of torch_block / torch_block_swiglu on torch leaves (for autograd)."""
    B, S, H, nh, dh, F_ = dims.batch, dims.seq, dims.hidden, dims.heads, dims.head_dim, dims.ffn
    if dims.variant == 1:
        xn = F.rms_norm(X, (H,), p["ln_gamma"], dims.ln_eps)
    else:
        xn = F.layer_norm(X, (H,), p["ln_gamma"], p["ln_beta"], dims.ln_eps)
    qkv = xn @ p["wqkv"] + p["b_qkv"]
    q, k, v = (qkv[..., i * H:(i + 1) * H].reshape(B, S, nh, dh).transpose(1, 2) for i in range(3))
    a = F.scaled_dot_product_attention(q, k, v, attn_mask=band_mask(S, dims.window))
    a = a.transpose(1, 2).reshape(B, S, H) @ p["wo"] + p["b_o"]
    z = xn @ p["w1"] + p["b1"]
    act = F.silu(z[..., :F_]) * z[..., F_:] if dims.variant == 1 else F.gelu(z, approximate="none")
    return X + act @ p["w2"] + p["b2"] + a


BACKWARD_PINS = [pin_gelu_backward_closed_form, pin_swiglu_backward_closed_form,
                 pin_norm_backward_invariants, pin_attention_backward_invariants,
                 pin_backward_finite_differences, pin_backward_autograd]


ALL_PINS = [pin_gelu_table, pin_gelu_library, pin_layernorm_two_vector, pin_layernorm_library,
            pin_layernorm_stats, pin_linear_library, pin_attention_window1_is_v,
            pin_attention_window2_closed_form, pin_attention_full_causal,
            pin_attention_band_library, pin_attention_rows_sum_to_one,
            pin_attention_translation, pin_block_library, pin_block_concat_identity,
            pin_block_zero_affine, pin_block_zero_output_weights, pin_block_invariants,
            pin_block_rows_mode, pin_serial_library, pin_serial_reduces_to_parallel,
            pin_serial_first_order, pin_serial_rows_mode, pin_rmsnorm_closed_form,
            pin_rmsnorm_library, pin_rmsnorm_scale_invariance, pin_swiglu_closed_form,
            pin_swiglu_library, pin_block_swiglu_library, pin_block_swiglu_rows_mode,
            pin_e4m3_table, pin_e4m3_roundtrip_all_codes, pin_e4m3_ties_to_even,
            pin_e4m3_library, pin_e4m3_row_scaling, pin_block_fp8_library,
            pin_block_fp8_rows_mode,
            *BACKWARD_PINS]
