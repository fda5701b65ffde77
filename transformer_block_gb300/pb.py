"""Python binding of the C ABI in ``include/pb.h`` (argument marshalling only).

Every step of the forward pass runs in ``libpb.so``'s kernels; PyTorch only supplies
device memory and the current CUDA stream. There is no fallback: if the library has not
been built, or a call fails, an exception is raised.
"""

from __future__ import annotations

import ctypes
import os

import torch

from . import build as _build
from .configs import Workload

PB_OK = 0
PB_ERR_DEVICE_TIMEOUT = 5
PB_ERR_RANGE = 7
STATUS_NAMES = {0: "PB_OK", 1: "PB_ERR_INVALID_ARG", 2: "PB_ERR_UNSUPPORTED",
                3: "PB_ERR_WORKSPACE", 4: "PB_ERR_CUDA", 5: "PB_ERR_DEVICE_TIMEOUT",
                6: "PB_ERR_BAD_HANDLE", 7: "PB_ERR_RANGE"}
PB_OPERANDS_BF16, PB_OPERANDS_FP16, PB_OPERANDS_FP8 = 0, 1, 2


class PbError(RuntimeError):
    def __init__(self, func: str, status: int, message: str):
        super().__init__(f"{func}: {STATUS_NAMES.get(status, status)}: {message}")
        self.status = status


class pb_dims(ctypes.Structure):
    _fields_ = [("batch", ctypes.c_int32), ("seq", ctypes.c_int32), ("hidden", ctypes.c_int32),
                ("heads", ctypes.c_int32), ("head_dim", ctypes.c_int32), ("ffn", ctypes.c_int32),
                ("window", ctypes.c_int32), ("ln_eps", ctypes.c_float),
                ("variant", ctypes.c_int32)]


WEIGHT_FIELDS = ["ln_gamma", "ln_beta", "wqkv", "w1", "wo", "w2", "b_qkv", "b1", "b_o", "b2"]


class pb_weights(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in WEIGHT_FIELDS]


class pb_scratch_layout(ctypes.Structure):
    _fields_ = [(n, ctypes.c_size_t) for n in
                ("xn", "qk", "vt", "act", "io", "io2", "res0", "res1", "sk", "q8", "qscale", "seq_pad",
                 "total", "hpre", "lse", "d_attn", "delta", "dq_acc", "dz", "dxn", "stats",
                 "partials", "train_total")]


GRAD_FIELDS = ("dx", "dgamma", "dbeta", "dwqkv", "dw1", "dwo", "dw2", "db_qkv", "db1", "db_o",
               "db2")


class pb_grads(ctypes.Structure):
    _fields_ = [(n, ctypes.c_void_p) for n in GRAD_FIELDS]


class pb_options(ctypes.Structure):
    _fields_ = [("operand_precision", ctypes.c_int32), ("wait_limit_ns", ctypes.c_uint64)]


# name -> (restype, argtypes); every function of include/pb.h
_P, _S, _I32, _I64, _U64 = ctypes.c_void_p, ctypes.c_size_t, ctypes.c_int32, ctypes.c_int64, \
    ctypes.c_uint64
_DP = ctypes.POINTER(pb_dims)
SIGNATURES = {
    "pb_weight_workspace_bytes": (ctypes.c_int, [_DP, ctypes.POINTER(_S)]),
    "pb_scratch_bytes": (ctypes.c_int, [_DP, ctypes.POINTER(_S)]),
    "pb_get_scratch_layout": (ctypes.c_int, [_DP, ctypes.POINTER(pb_scratch_layout)]),
    "pb_create": (ctypes.c_int, [_DP, ctypes.POINTER(pb_weights), _P, _S, _P,
                                 ctypes.POINTER(_P)]),
    "pb_create_ex": (ctypes.c_int, [_DP, ctypes.POINTER(pb_weights),
                                    ctypes.POINTER(pb_options), _P, _S, _P, ctypes.POINTER(_P)]),
    "pb_forward": (ctypes.c_int, [_P, _P, _P, _P, _S, _P]),
    "pb_forward_serial": (ctypes.c_int, [_P, _P, _P, _P, _P, _P, _S, _P]),
    "pb_forward_stack": (ctypes.c_int, [ctypes.POINTER(_P), _I32, _P, _P, _P, _S, _P]),
    "pb_forward_stack_host": (ctypes.c_int, [ctypes.POINTER(_P), _I32, _P, _P, _P, _S, _P]),
    "pb_forward_stack_f32": (ctypes.c_int, [ctypes.POINTER(_P), _I32, _P, _P, _P, _S, _P]),
    "pb_get_status": (ctypes.c_int, [_P]),
    "pb_clear_status": (ctypes.c_int, [_P, _P]),
    "pb_set_wait_limit_ns": (ctypes.c_int, [_P, _U64]),
    "pb_trace_enable": (ctypes.c_int, [_P, _I32]),
    "pb_trace_read": (ctypes.c_int, [_P, ctypes.POINTER(ctypes.c_float), ctypes.POINTER(_I32)]),
    "pb_destroy": (ctypes.c_int, [_P]),
    "pb_status_string": (ctypes.c_char_p, [ctypes.c_int]),
    "pb_last_error_message": (ctypes.c_char_p, []),
    "pb_layernorm": (ctypes.c_int, [_I64, _I32, _P, _P, _P, ctypes.c_float, _P, _P]),
    "pb_quantize_rows_e4m3": (ctypes.c_int, [_I64, _I32, _P, _P, _P, _P]),
    "pb_train_scratch_bytes": (ctypes.c_int, [_P, _P]),
    "pb_forward_train": (ctypes.c_int, [_P, _P, _P, _P, _S, _P]),
    "pb_forward_stack_host_steps": (ctypes.c_int, [_P, _I32, _I32, _P, _P, _P, _S, _P]),
    "pb_backward": (ctypes.c_int, [_P, _P, _P, _P, _I32, _P, _S, _P]),
    "pb_gemm_scratch_bytes": (ctypes.c_int, [ctypes.POINTER(_S)]),
    "pb_gemm_bf16": (ctypes.c_int, [_I32, _I32, _I32, _P, _P, _P, _P, _S, _P, _P]),
    "pb_gemm_bf16_layout": (ctypes.c_int, [_I32, _I32, _I32, _P, _I32, _P, _I32, _P, _P, _S, _P,
                                           _P]),
    "pb_swa_attention": (ctypes.c_int, [_DP, _P, _P, _P, _I64, _P, _P]),
    "pb_wait_probe": (ctypes.c_int, [_U64, _P, _P]),
    "pb_gemm_bf16_static": (ctypes.c_int, [_I32, _I32, _I32, _P, _P, _P, _P, _P]),
    "pb_set_guard_bytes": (ctypes.c_int, [_S]),
    "pb_get_guard_bytes": (ctypes.c_int, [ctypes.POINTER(_S)]),
}

_lib = None


def library_path() -> str:
    return _build.LIB


def lib():
    """The loaded ``libpb.so`` (raises if it has not been built)."""
    global _lib
    if _lib is None:
        path = library_path()
        if not os.path.exists(path):
            raise RuntimeError(f"{path} is missing: build it with transformer_block_gb300.build."
                               "build(); the forward pass has no other implementation")
        L = ctypes.CDLL(path)
        for name, (res, args) in SIGNATURES.items():
            f = getattr(L, name)
            f.restype = res
            f.argtypes = args
        _lib = L
    return _lib


def _check(func: str, status: int):
    if status != PB_OK:
        msg = lib().pb_last_error_message()
        raise PbError(func, status, msg.decode() if msg else "")


def _ptr(t: torch.Tensor | None):
    return None if t is None else ctypes.c_void_p(t.data_ptr())


def _stream(stream) -> ctypes.c_void_p:
    if stream is None:
        stream = torch.cuda.current_stream()
    return ctypes.c_void_p(stream.cuda_stream if hasattr(stream, "cuda_stream") else int(stream))


def make_dims(wl: Workload | None = None, **kw) -> pb_dims:
    src = dict(wl.__dict__) if wl is not None else {}
    src.update(kw)
    return pb_dims(src["batch"], src["seq"], src["hidden"], src["heads"], src["head_dim"],
                   src["ffn"], src["window"], float(src.get("ln_eps", 1e-5)),
                   int(src.get("variant", 0)))


def weight_workspace_bytes(dims: pb_dims) -> int:
    n = ctypes.c_size_t()
    _check("pb_weight_workspace_bytes", lib().pb_weight_workspace_bytes(ctypes.byref(dims),
                                                                        ctypes.byref(n)))
    return n.value


def scratch_bytes(dims: pb_dims) -> int:
    n = ctypes.c_size_t()
    _check("pb_scratch_bytes", lib().pb_scratch_bytes(ctypes.byref(dims), ctypes.byref(n)))
    return n.value


def train_scratch_bytes(dims: pb_dims) -> int:
    n = ctypes.c_size_t()
    _check("pb_train_scratch_bytes", lib().pb_train_scratch_bytes(ctypes.byref(dims),
                                                                  ctypes.byref(n)))
    return n.value


def new_train_scratch(dims: pb_dims, device="cuda") -> torch.Tensor:
    return torch.empty(train_scratch_bytes(dims), dtype=torch.uint8, device=device)


def scratch_layout(dims: pb_dims) -> pb_scratch_layout:
    L = pb_scratch_layout()
    _check("pb_get_scratch_layout", lib().pb_get_scratch_layout(ctypes.byref(dims),
                                                                ctypes.byref(L)))
    return L


def new_scratch(dims: pb_dims, device="cuda") -> torch.Tensor:
    return torch.empty(scratch_bytes(dims), dtype=torch.uint8, device=device)


def scratch_view(scratch: torch.Tensor, dims: pb_dims, name: str,
                 dtype=torch.bfloat16) -> torch.Tensor:
    """A view of one intermediate in the scratch (``xn, qk, vt, act, io, res0, res1, q8,
    qscale``); ``dtype`` is the element type it holds (fp16 for ``xn``/``act`` with fp16
    operands, uint8 E4M3 codes for ``xn`` with FP8 operands; ``res0``/``res1``/``qscale``
    are always fp32 and ``q8`` uint8)."""
    L = scratch_layout(dims)
    T, H, F = dims.batch * dims.seq, dims.hidden, dims.ffn
    shapes = {"xn": (T, H), "qk": (T, 2 * H), "act": (T, H + F), "io": (T, H),
              "res0": (T, H), "res1": (T, H),
              "vt": (dims.batch, dims.heads, dims.head_dim, L.seq_pad),
              "q8": (T, H + F), "qscale": (2 * T,)}
    Fp = 2 * F if dims.variant == 1 else F
    nrow = dims.batch * dims.heads * ((dims.seq + 63) // 64 * 64)
    shapes.update({"hpre": (T, Fp), "lse": (nrow,), "d_attn": (T, H), "delta": (nrow,),
                   "dq_acc": (T, H), "dz": (T, 3 * H + Fp), "dxn": (T, H)})
    if name in ("res0", "res1", "qscale", "lse", "delta", "dq_acc", "dxn"):
        dtype = torch.float32
    elif name == "q8":
        dtype = torch.uint8
    shape = shapes[name]
    n = 1
    for s in shape:
        n *= s
    off = getattr(L, name)
    nbytes = n * torch.empty((), dtype=dtype).element_size()
    return scratch[off:off + nbytes].view(dtype).view(*shape)


class ParallelBlock:
    """One parallel transformer block: a ``pb_handle`` plus the workspace it owns."""

    def __init__(self, dims: pb_dims, params: dict, stream=None,
                 operand_precision: int = PB_OPERANDS_BF16, wait_limit_ns: int = 0,
                 workspace: torch.Tensor | None = None):
        """``workspace``: a caller-provided uint8 CUDA tensor of at least
        ``weight_workspace_bytes(dims)`` (256-byte aligned), else one is allocated."""
        self.dims = dims
        self.operand_precision = operand_precision
        self._lib = lib()
        dev = params["wqkv"].device
        if workspace is None:
            workspace = torch.empty(weight_workspace_bytes(dims), dtype=torch.uint8, device=dev)
        self.workspace = workspace
        w = pb_weights(*[_ptr(params.get(n)) for n in WEIGHT_FIELDS])
        opt = pb_options(operand_precision, wait_limit_ns)
        h = ctypes.c_void_p()
        _check("pb_create_ex", self._lib.pb_create_ex(ctypes.byref(dims), ctypes.byref(w),
                                                      ctypes.byref(opt), _ptr(self.workspace),
                                                      self.workspace.numel(), _stream(stream),
                                                      ctypes.byref(h)))
        self.handle = h

    def forward(self, x: torch.Tensor, y: torch.Tensor | None = None,
                scratch: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        if y is None:
            y = torch.empty_like(x)
        if scratch is None:
            scratch = new_scratch(self.dims, x.device)
        _check("pb_forward", self._lib.pb_forward(self.handle, _ptr(x), _ptr(y), _ptr(scratch),
                                                  scratch.numel(), _stream(stream)))
        return y

    __call__ = forward

    def forward_serial(self, x: torch.Tensor, y: torch.Tensor | None = None,
                       ln2_gamma: torch.Tensor | None = None, ln2_beta: torch.Tensor | None = None,
                       scratch: torch.Tensor | None = None, stream=None) -> torch.Tensor:
        """The serial block of eq. (3) on the same weights (``pb_forward_serial``)."""
        if y is None:
            y = torch.empty_like(x)
        if scratch is None:
            scratch = new_scratch(self.dims, x.device)
        _check("pb_forward_serial",
               self._lib.pb_forward_serial(self.handle, _ptr(x), _ptr(y), _ptr(ln2_gamma),
                                           _ptr(ln2_beta), _ptr(scratch), scratch.numel(),
                                           _stream(stream)))
        return y

    def forward_train(self, x: torch.Tensor, scratch: torch.Tensor, y: torch.Tensor | None = None,
                      stream=None) -> torch.Tensor:
        """``pb_forward_train``: the forward pass, keeping in ``scratch`` (a training
        scratch, ``new_train_scratch``) what ``backward`` reads."""
        if y is None:
            y = torch.empty_like(x)
        _check("pb_forward_train",
               self._lib.pb_forward_train(self.handle, _ptr(x), _ptr(y), _ptr(scratch),
                                          scratch.numel(), _stream(stream)))
        return y

    def backward(self, x: torch.Tensor, dy: torch.Tensor, scratch: torch.Tensor,
                 grads: dict | None = None, accumulate: bool = False, biases: bool = True,
                 stream=None) -> dict:
        """``pb_backward`` after ``forward_train(x, scratch)``: returns the gradients (``dx``
        bf16, the parameter gradients fp32 in their ``pb_weights`` layout, keyed like
        ``GRAD_FIELDS``). ``grads`` may hold preallocated buffers (needed for
        ``accumulate``)."""
        d = self.dims
        H, F, T = d.hidden, d.ffn, d.batch * d.seq
        Fp = 2 * F if d.variant == 1 else F
        shapes = {"dx": (T, H), "dgamma": (H,), "dbeta": (H,), "dwqkv": (H, 3 * H),
                  "dw1": (H, Fp), "dwo": (H, H), "dw2": (F, H), "db_qkv": (3 * H,),
                  "db1": (Fp,), "db_o": (H,), "db2": (H,)}
        g = dict(grads or {})
        for n, shp in shapes.items():
            if n in g:
                continue
            if n in ("db_qkv", "db1", "db_o", "db2") and not biases:
                continue
            if n == "dbeta" and d.variant == 1:
                continue
            dt = torch.bfloat16 if n == "dx" else torch.float32
            g[n] = torch.zeros(shp, dtype=dt, device=x.device)
        gs = pb_grads(*[_ptr(g.get(n)) for n in GRAD_FIELDS])
        _check("pb_backward",
               self._lib.pb_backward(self.handle, _ptr(x), _ptr(dy), ctypes.byref(gs),
                                     int(accumulate), _ptr(scratch), scratch.numel(),
                                     _stream(stream)))
        return g

    def status(self) -> int:
        return self._lib.pb_get_status(self.handle)

    def clear_status(self, stream=None):
        _check("pb_clear_status", self._lib.pb_clear_status(self.handle, _stream(stream)))

    def set_wait_limit_ns(self, ns: int):
        _check("pb_set_wait_limit_ns", self._lib.pb_set_wait_limit_ns(self.handle, int(ns)))

    def trace_enable(self, n_calls: int):
        _check("pb_trace_enable", self._lib.pb_trace_enable(self.handle, int(n_calls)))

    def trace_read(self):
        """Summed ms of [LayerNorm, first GEMM, attention, second GEMM] and the call count."""
        ms = (ctypes.c_float * 4)()
        n = ctypes.c_int32()
        _check("pb_trace_read", self._lib.pb_trace_read(self.handle, ms, ctypes.byref(n)))
        return list(ms), n.value

    def close(self):
        if getattr(self, "handle", None) is not None and self.handle.value:
            _check("pb_destroy", self._lib.pb_destroy(self.handle))
            self.handle = None

    def __del__(self):
        try:
            self.close()
        except Exception:
            pass


def _handles(blocks):
    arr = (ctypes.c_void_p * len(blocks))(*[b.handle.value for b in blocks])
    return arr


def forward_stack(blocks, x, y=None, scratch=None, stream=None):
    if y is None:
        y = torch.empty_like(x)
    if scratch is None:
        scratch = new_scratch(blocks[0].dims, x.device)
    _check("pb_forward_stack", lib().pb_forward_stack(_handles(blocks), len(blocks), _ptr(x),
                                                      _ptr(y), _ptr(scratch), scratch.numel(),
                                                      _stream(stream)))
    return y


def forward_stack_f32(blocks, x, y=None, scratch=None, stream=None):
    """``forward_stack`` returning the fp32 residual stream (float32 [T, H]) instead of its
    bf16 rounding (``pb_forward_stack_f32``)."""
    if y is None:
        y = torch.empty(x.shape, dtype=torch.float32, device=x.device)
    if scratch is None:
        scratch = new_scratch(blocks[0].dims, x.device)
    _check("pb_forward_stack_f32", lib().pb_forward_stack_f32(_handles(blocks), len(blocks),
                                                              _ptr(x), _ptr(y), _ptr(scratch),
                                                              scratch.numel(), _stream(stream)))
    return y


def forward_stack_host(blocks, x_host, y_host, scratch, stream=None):
    """Host (pinned) x -> device -> stack -> host y, enqueued on ``stream``."""
    _check("pb_forward_stack_host",
           lib().pb_forward_stack_host(_handles(blocks), len(blocks), _ptr(x_host), _ptr(y_host),
                                       _ptr(scratch), scratch.numel(), _stream(stream)))
    return y_host


def forward_stack_host_steps(blocks, x_hosts, y_hosts, scratch, stream=None):
    """Host (pinned) x_hosts[s] -> stack -> y_hosts[s] for every step s, the copies of
    neighbouring steps overlapping each step's compute (``pb_forward_stack_host_steps``)."""
    n = len(x_hosts)
    assert len(y_hosts) == n
    xs = (ctypes.c_void_p * n)(*[t.data_ptr() for t in x_hosts])
    ys = (ctypes.c_void_p * n)(*[t.data_ptr() for t in y_hosts])
    _check("pb_forward_stack_host_steps",
           lib().pb_forward_stack_host_steps(_handles(blocks), len(blocks), n, xs, ys,
                                             _ptr(scratch), scratch.numel(), _stream(stream)))
    return y_hosts


def layernorm(x, gamma, beta, eps=1e-5, out=None, stream=None):
    if out is None:
        out = torch.empty_like(x)
    _check("pb_layernorm", lib().pb_layernorm(x.shape[0], x.shape[1], _ptr(x), _ptr(gamma),
                                              _ptr(beta), float(eps), _ptr(out),
                                              _stream(stream)))
    return out


def set_guard_bytes(n: int):
    """Unused bytes after every workspace and scratch region of the layouts computed from
    now on (``pb_set_guard_bytes``; process-wide, a debugging aid)."""
    _check("pb_set_guard_bytes", lib().pb_set_guard_bytes(int(n)))


def guard_bytes() -> int:
    n = ctypes.c_size_t()
    _check("pb_get_guard_bytes", lib().pb_get_guard_bytes(ctypes.byref(n)))
    return n.value


def gemm_scratch_bytes() -> int:
    n = ctypes.c_size_t()
    _check("pb_gemm_scratch_bytes", lib().pb_gemm_scratch_bytes(ctypes.byref(n)))
    return n.value


def gemm(a, b, out=None, scratch=None, status=None, stream=None):
    """``a [M, K] @ b[N, K]^T`` -> bf16 ``[M, N]`` on the tensor cores; ``scratch`` (a uint8
    CUDA tensor of ``gemm_scratch_bytes()``) enables stream-K for the last waves."""
    M, K = a.shape
    N = b.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    nbytes = 0 if scratch is None else scratch.numel()
    _check("pb_gemm_bf16", lib().pb_gemm_bf16(M, N, K, _ptr(a), _ptr(b), _ptr(out), _ptr(scratch),
                                              nbytes, _ptr(status), _stream(stream)))
    return out


def gemm_layout(a, b, a_mn=False, b_mn=False, out=None, scratch=None, status=None,
                stream=None):
    """``C[m, n] = sum_k A(m, k) B(n, k)`` -> bf16 ``[M, N]`` with ``a`` stored ``[M, K]``
    (or ``[K, M]`` when ``a_mn``) and ``b`` stored ``[N, K]`` (or ``[K, N]`` when ``b_mn``)."""
    M, K = (a.shape[1], a.shape[0]) if a_mn else a.shape
    N = b.shape[1] if b_mn else b.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    nbytes = 0 if scratch is None else scratch.numel()
    _check("pb_gemm_bf16_layout",
           lib().pb_gemm_bf16_layout(M, N, K, _ptr(a), int(a_mn), _ptr(b), int(b_mn), _ptr(out),
                                     _ptr(scratch), nbytes, _ptr(status), _stream(stream)))
    return out


def gemm_static(a, b, out=None, status=None, stream=None):
    """``gemm`` without caller scratch: the stream-K partial tiles live in the library's
    own fixed device array (for callers that cannot allocate; calls must not overlap)."""
    M, K = a.shape
    N = b.shape[0]
    if out is None:
        out = torch.empty((M, N), dtype=torch.bfloat16, device=a.device)
    _check("pb_gemm_bf16_static", lib().pb_gemm_bf16_static(M, N, K, _ptr(a), _ptr(b), _ptr(out),
                                                            _ptr(status), _stream(stream)))
    return out


def quantize_rows_e4m3(x: torch.Tensor, stream=None):
    """Per-row current scaling of a bf16 [rows, cols] CUDA tensor to FP8 E4M3 codes
    (``pb_quantize_rows_e4m3``): returns ``(codes uint8 [rows, cols], scales fp32 [rows])``."""
    rows, cols = x.shape
    codes = torch.empty((rows, cols), dtype=torch.uint8, device=x.device)
    scales = torch.empty(rows, dtype=torch.float32, device=x.device)
    _check("pb_quantize_rows_e4m3", lib().pb_quantize_rows_e4m3(rows, cols, _ptr(x), _ptr(codes),
                                                                _ptr(scales), _stream(stream)))
    return codes, scales


def swa_attention(dims: pb_dims, qk, vt, act, status=None, stream=None):
    _check("pb_swa_attention", lib().pb_swa_attention(ctypes.byref(dims), _ptr(qk), _ptr(vt),
                                                      _ptr(act), act.shape[1], _ptr(status),
                                                      _stream(stream)))
    return act


def wait_probe(limit_ns: int, status: torch.Tensor, stream=None):
    """Runs the bounded-wait self-test kernel; ``status`` is a 1-element int32 CUDA tensor."""
    _check("pb_wait_probe", lib().pb_wait_probe(int(limit_ns), _ptr(status), _stream(stream)))
