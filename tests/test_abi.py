"""The C-ABI library loads, exports every function include/pb.h declares, and rejects bad
arguments on the host before touching a GPU (CPU only)."""

import ctypes
import os
import re

import pytest

from transformer_block_gb300 import build, pb

ROOT = os.path.dirname(os.path.dirname(os.path.abspath(__file__)))


def declared_functions():
    text = open(os.path.join(ROOT, "include", "pb.h")).read()
    return sorted(set(re.findall(r"^\s*(?:pb_status|const char\s*\*)\s*(pb_\w+)\s*\(", text, re.M)))


@pytest.fixture(scope="module")
def lib():
    build.build()
    return pb.lib()


def test_header_declares_the_api():
    names = declared_functions()
    for required in ("pb_create", "pb_forward", "pb_destroy", "pb_forward_stack_host"):
        assert required in names


def test_header_is_plain_c_and_links(lib, tmp_path):
    # A C program (not C++) that includes the header and calls into the library: the
    # declarations are C, and the exported names link without C++ mangling.
    import shutil
    import subprocess
    cc = shutil.which("gcc") or shutil.which("cc")
    if cc is None:
        pytest.skip("no C compiler")
    src = tmp_path / "use_pb.c"
    src.write_text(
        '#include <stdio.h>\n#include "pb.h"\n'
        "int main(void) {\n"
        "  pb_dims d = {1, 128, 256, 4, 64, 1024, 32, 1e-5f, PB_BLOCK_LN_GELU};\n"
        "  size_t ws = 0, scr = 0;\n"
        "  if (pb_weight_workspace_bytes(&d, &ws) != PB_OK) return 1;\n"
        "  if (pb_scratch_bytes(&d, &scr) != PB_OK) return 2;\n"
        "  d.head_dim = 96;\n  d.hidden = 384;\n"
        "  if (pb_scratch_bytes(&d, &scr) != PB_ERR_UNSUPPORTED) return 3;\n"
        '  printf("%zu %zu %s\\n", ws, scr, pb_status_string(PB_ERR_UNSUPPORTED));\n'
        "  return 0;\n}\n")
    exe = tmp_path / "use_pb"
    libdir = os.path.dirname(pb.library_path())
    subprocess.run([cc, "-std=c99", "-Wall", "-Werror", "-I", os.path.join(ROOT, "include"),
                    str(src), "-o", str(exe), "-L", libdir, "-lpb", "-Wl,-rpath," + libdir],
                   check=True)
    out = subprocess.run([str(exe)], check=True, capture_output=True, text=True).stdout.split()
    assert int(out[0]) == pb.weight_workspace_bytes(pb.make_dims(
        batch=1, seq=128, hidden=256, heads=4, head_dim=64, ffn=1024, window=32))
    assert out[2] == "PB_ERR_UNSUPPORTED"


def test_every_declared_symbol_is_exported(lib):
    for name in declared_functions():
        assert hasattr(lib, name), name
    # and the binding wraps exactly the declared functions
    assert set(pb.SIGNATURES) == set(declared_functions())


def test_status_strings(lib):
    for code, name in pb.STATUS_NAMES.items():
        assert lib.pb_status_string(code).decode() == name


def dims(**kw):
    base = dict(batch=1, seq=128, hidden=256, heads=4, head_dim=64, ffn=1024, window=32)
    base.update(kw)
    return pb.make_dims(**base)


@pytest.mark.parametrize("bad,code", [
    (dict(hidden=250), pb.STATUS_NAMES and 1),          # heads * head_dim != hidden
    (dict(head_dim=32, heads=8), 2),                     # unsupported head_dim
    (dict(ffn=1000), 2),                                 # ffn % 64
    (dict(window=0), 1),
    (dict(seq=0), 1),
    (dict(ln_eps=0.0), 1),
    (dict(batch=65536, seq=65536), 2),                   # 2^32 tokens
])
def test_bad_dims_rejected(lib, bad, code):
    n = ctypes.c_size_t()
    d = dims(**bad)
    assert lib.pb_weight_workspace_bytes(ctypes.byref(d), ctypes.byref(n)) == code
    assert lib.pb_last_error_message().decode()


def test_workspace_and_scratch_sizes(lib):
    d = dims()
    H, F, T = 256, 1024, 128
    ws = pb.weight_workspace_bytes(d)
    assert ws >= 2 * ((3 * H + F) * H + H * (H + F))
    L = pb.scratch_layout(d)
    assert L.seq_pad == 128
    assert L.total == pb.scratch_bytes(d)
    order = ["xn", "qk", "vt", "act", "io", "res0", "res1", "sk"]
    for a, b in zip(order, order[1:]):
        assert getattr(L, a) < getattr(L, b) and getattr(L, b) % 1024 == 0
    assert L.act - L.vt >= 2 * 1 * H * 128
    assert L.res0 - L.io >= 2 * T * H
    assert L.res1 - L.res0 >= 4 * T * H          # fp32 residual stream
    assert L.sk - L.res1 >= 4 * T * H
    assert L.total - L.sk >= pb.gemm_scratch_bytes()
    # ragged sequences pad the transposed V to a multiple of 8 tokens
    assert pb.scratch_layout(dims(seq=130)).seq_pad == 136


def test_create_rejects_missing_weights_before_cuda(lib):
    d = dims()
    w = pb.pb_weights()
    h = ctypes.c_void_p()
    assert lib.pb_create(ctypes.byref(d), ctypes.byref(w), ctypes.c_void_p(1 << 20), 1 << 30,
                         None, ctypes.byref(h)) == 1
    assert "NULL" in lib.pb_last_error_message().decode()
    assert not h.value


def test_create_rejects_small_workspace(lib):
    d = dims()
    ptrs = [ctypes.c_void_p(0x100000 + 0x10000 * i) for i in range(6)] + [None] * 4
    w = pb.pb_weights(*ptrs)
    h = ctypes.c_void_p()
    assert lib.pb_create(ctypes.byref(d), ctypes.byref(w), ctypes.c_void_p(0x4000000), 16, None,
                         ctypes.byref(h)) == 3
    assert lib.pb_create(ctypes.byref(d), ctypes.byref(w), ctypes.c_void_p(0x4000001), 1 << 40,
                         None, ctypes.byref(h)) == 1  # misaligned workspace


def test_create_rejects_bad_options(lib):
    d = dims()
    ptrs = [ctypes.c_void_p(0x100000 + 0x10000 * i) for i in range(6)] + [None] * 4
    w = pb.pb_weights(*ptrs)
    h = ctypes.c_void_p()
    opt = pb.pb_options(5, 0)
    assert lib.pb_create_ex(ctypes.byref(d), ctypes.byref(w), ctypes.byref(opt),
                            ctypes.c_void_p(0x4000000), 1 << 40, None, ctypes.byref(h)) == 1
    assert "operand_precision" in lib.pb_last_error_message().decode()


def test_null_handles(lib):
    assert lib.pb_forward(None, None, None, None, 0, None) == 6
    assert lib.pb_forward_serial(None, None, None, None, None, None, 0, None) == 6
    assert lib.pb_destroy(None) == 6
    assert lib.pb_get_status(None) == 6
    arr = (ctypes.c_void_p * 1)(None)
    assert lib.pb_forward_stack(arr, 1, None, None, None, 0, None) == 6
    assert lib.pb_forward_stack(arr, 0, None, None, None, 0, None) == 1


def test_step_entry_points_validate(lib):
    assert lib.pb_gemm_bf16(128, 100, 64, None, None, None, None, 0, None, None) == 2  # N % 32
    assert lib.pb_gemm_bf16(128, 128, 64, None, None, None, None, 0, None, None) == 1  # NULL
    n = ctypes.c_size_t()
    assert lib.pb_gemm_scratch_bytes(ctypes.byref(n)) == 0 and n.value > 0
    assert lib.pb_layernorm(4, 12, None, None, None, 1e-5, None, None) == 2   # H % 8
    assert lib.pb_layernorm(4, 16, None, None, None, 1e-5, None, None) == 1   # NULL


def test_guard_gaps_in_every_layout(lib):
    # pb_set_guard_bytes leaves the requested gap after every region (CPU only: layouts are
    # host arithmetic), keeps 1024-byte alignment, and rejects more than 1 MiB.
    d = dims(batch=2, seq=130, head_dim=128, heads=2)
    assert pb.guard_bytes() == 0
    plain = pb.scratch_layout(d)
    ws0 = pb.weight_workspace_bytes(d)
    try:
        pb.set_guard_bytes(4096)
        assert pb.guard_bytes() == 4096
        g = pb.scratch_layout(d)
        names = ["xn", "qk", "vt", "act", "io", "io2", "res0", "res1", "sk", "q8", "qscale",
                 "hpre", "lse", "d_attn", "delta", "dq_acc", "dz", "dxn", "stats", "partials"]
        offs = [getattr(g, n) for n in names] + [g.train_total]
        plain_offs = [getattr(plain, n) for n in names] + [plain.train_total]
        for k in range(len(names)):
            assert offs[k] % 1024 == 0
            # the region keeps its size and is followed by at least 4096 unused bytes
            size = plain_offs[k + 1] - plain_offs[k]  # an upper bound of the region's size
            assert offs[k + 1] - offs[k] >= 4096
            assert offs[k + 1] - offs[k] <= size + 4096 + 1024
        assert g.total == g.hpre and g.total > plain.total
        assert pb.scratch_bytes(d) == g.total
        assert pb.train_scratch_bytes(d) == g.train_total
        assert pb.weight_workspace_bytes(d) >= ws0 + 13 * 4096
        with pytest.raises(pb.PbError):
            pb.set_guard_bytes((1 << 20) + 1)
        assert pb.guard_bytes() == 4096
    finally:
        pb.set_guard_bytes(0)
    assert pb.scratch_bytes(d) == plain.total
